"""Seeded synthetic inputs for the MoE feed-forward layer.

This module only draws random numbers and lays them out in the byte formats the
layer consumes. It computes nothing of the layer itself (no decode, no routing,
no FFN arithmetic), so that both the CPU oracle and the CUDA path can take their
inputs from it without sharing any of the method's arithmetic.

Workloads (shapes and distributions follow the layer described in "Cascadia:
Resident 975B MoE Inference on Eleven AI PCs" §3.1/§3.4 and the MXFP4 expert
format of "DeepSeek-V4-Flash on a four-GPU Ampere workstation", section "MXFP4
is not NVFP4, and the difference matters on Ampere"):

* ``tiny``     T=16, H=256, I=128, E=8, top-2, no shared expert, seed 0
* ``decode``   T=1, H=7168, I=2048, E=256 + 1 shared, top-8, seed 1
* ``sweep``    same layer, T in {1, 15, 88, 176}, logits N(0,1) + b_e with a
               per-expert bias b_e ~ N(0, 0.5), seed 2
* ``prefill``  same layer, T=8192, Zipf(1.1) expert popularity, seed 3
  (decode, sweep and prefill share the expert weights, seeded by 1)
* ``dense``    dense SwiGLU FFN H=7168, I=18432 as 9 slices of 2048, T in
               {1, 88, 4096}; BF16 weights N(0, 0.02) and an MXFP4 variant, seed 4

Byte formats:

* ``x`` is BF16 stored as ``uint16`` bit patterns, shape [T, H].
* logits are ``float32`` [T, E].
* an MXFP4 matrix [rows, cols] is ``codes`` uint8 [rows, cols/2] (element 2j in
  the low nibble of byte j, 2j+1 in the high nibble) plus ``scales`` uint8
  [rows, cols/32] (one E8M0 exponent per 32 consecutive elements of a row).
* gate|up of one expert is one MXFP4 matrix [2I, H] (gate rows first, then up
  rows); down is [H, I].
* BF16 weights are ``uint16`` bit patterns.

Every tensor is drawn from its own ``numpy.random.SeedSequence`` keyed by
(seed, tag, index), so any single expert can be regenerated on its own.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np

# SeedSequence tags, one per tensor kind.
_TAG_X = 1
_TAG_LOGITS = 2
_TAG_BIAS = 3
_TAG_ZIPF_PERM = 4
_TAG_GUMBEL = 5
_TAG_GATE_UP = 10
_TAG_DOWN = 11
_TAG_DENSE_G = 20
_TAG_DENSE_U = 21
_TAG_DENSE_D = 22


@dataclasses.dataclass(frozen=True)
class LayerConfig:
    """Shape and input recipe of one synthetic MoE (or dense) layer."""

    name: str
    T: int
    hidden: int
    inter: int
    n_experts: int
    n_shared: int
    k: int
    seed: int                       # seeds x and the router logits
    logits: str = "normal"          # "normal" | "biased" | "zipf"
    weight_seed: int = -1           # seeds the expert weights (-1: same as seed)
    e8m0_lo: int = 120              # E8M0 exponents are uniform in [lo, hi]
    e8m0_hi: int = 130
    # dense layer only
    dense: bool = False
    n_slices: int = 0
    weight_format: str = "mxfp4"    # "mxfp4" | "bf16" | "int4g32"

    @property
    def n_groups(self) -> int:
        return self.n_experts + self.n_shared

    @property
    def wseed(self) -> int:
        return self.seed if self.weight_seed < 0 else self.weight_seed


def tiny() -> LayerConfig:
    return LayerConfig("tiny", T=16, hidden=256, inter=128, n_experts=8, n_shared=0, k=2, seed=0)


# The decode, sweep and prefill workloads run on one and the same layer (expert
# weights seeded by 1); each workload seeds its own tokens and logits.
LAYER_WEIGHT_SEED = 1


def decode(T: int = 1) -> LayerConfig:
    return LayerConfig(f"decode_T{T}", T=T, hidden=7168, inter=2048, n_experts=256, n_shared=1, k=8, seed=1,
                       weight_seed=LAYER_WEIGHT_SEED)


def sweep(T: int) -> LayerConfig:
    assert T in (1, 15, 88, 176)
    return LayerConfig(f"sweep_T{T}", T=T, hidden=7168, inter=2048, n_experts=256, n_shared=1, k=8, seed=2,
                       logits="biased", weight_seed=LAYER_WEIGHT_SEED)


def prefill(T: int = 8192) -> LayerConfig:
    return LayerConfig(f"prefill_T{T}", T=T, hidden=7168, inter=2048, n_experts=256, n_shared=1, k=8, seed=3,
                       logits="zipf", weight_seed=LAYER_WEIGHT_SEED)


def dense(T: int, weight_format: str = "bf16") -> LayerConfig:
    # Dense FFN I_total = 18432 = 9 slices of 2048.  The MXFP4 variant draws
    # codes uniformly and E8M0 exponents in [117, 121]: decoded weights then have
    # an rms of about 0.024, the scale of the BF16 variant's N(0, 0.02).
    return LayerConfig(f"dense_{weight_format}_T{T}", T=T, hidden=7168, inter=18432, n_experts=9, n_shared=0,
                       k=9, seed=4, dense=True, n_slices=9, weight_format=weight_format,
                       e8m0_lo=117, e8m0_hi=121)


def custom(name: str, T: int, hidden: int, inter: int, n_experts: int, n_shared: int, k: int, seed: int,
           logits: str = "normal", e8m0_lo: int = 120, e8m0_hi: int = 130) -> LayerConfig:
    """Any other shape with the same distributions (used for ragged/edge tests)."""
    return LayerConfig(name, T=T, hidden=hidden, inter=inter, n_experts=n_experts, n_shared=n_shared, k=k,
                       seed=seed, logits=logits, e8m0_lo=e8m0_lo, e8m0_hi=e8m0_hi)


def _rng(seed: int, tag: int, index: int = 0) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, tag, index])))


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 to BF16 (round to nearest even) and return the uint16 bits."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounding = ((u >> 16) & 1) + 0x7FFF
    return ((u + rounding) >> 16).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen BF16 bit patterns to float32 (exact)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def tokens(cfg: LayerConfig, T: Optional[int] = None) -> np.ndarray:
    """x as BF16 bits [T, H], drawn as float32 N(0, 1) then rounded."""
    T = cfg.T if T is None else T
    x = _rng(cfg.seed, _TAG_X).standard_normal((T, cfg.hidden), dtype=np.float32)
    return f32_to_bf16_bits(x)


def router_logits(cfg: LayerConfig) -> np.ndarray:
    """float32 [T, E] router logits following the config's recipe.

    * normal: iid N(0, 1)
    * biased: N(0, 1) + b_e with b_e ~ N(0, 0.5) drawn once per layer
    * zipf:   log p_{pi(e)} + Gumbel(0, 1) iid, p_r proportional to r^-1.1 over
              ranks r = 1..E mapped to experts by a seeded permutation pi.  The
              top-k of Gumbel-perturbed log-probabilities is a draw without
              replacement proportional to p, so expert popularity is Zipf(1.1).
    """
    T, E = cfg.T, cfg.n_experts
    if cfg.logits == "normal":
        return _rng(cfg.seed, _TAG_LOGITS).standard_normal((T, E), dtype=np.float32)
    if cfg.logits == "biased":
        b = _rng(cfg.seed, _TAG_BIAS).normal(0.0, 0.5, size=E)
        l = _rng(cfg.seed, _TAG_LOGITS).standard_normal((T, E))
        return (l + b[None, :]).astype(np.float32)
    if cfg.logits == "zipf":
        r = np.arange(1, E + 1, dtype=np.float64)
        p = r ** -1.1
        p /= p.sum()
        perm = _rng(cfg.seed, _TAG_ZIPF_PERM).permutation(E)
        lp = np.log(p)[perm]
        g = _rng(cfg.seed, _TAG_GUMBEL).gumbel(size=(T, E))
        return (lp[None, :] + g).astype(np.float32)
    raise ValueError(cfg.logits)


def mx_matrix(rng: np.random.Generator, rows: int, cols: int, e_lo: int, e_hi: int):
    """Random MXFP4 matrix [rows, cols]: uniform 4-bit codes, uniform E8M0 in [e_lo, e_hi]."""
    assert cols % 32 == 0
    codes = np.frombuffer(rng.bytes(rows * cols // 2), dtype=np.uint8).reshape(rows, cols // 2).copy()
    scales = rng.integers(e_lo, e_hi + 1, size=(rows, cols // 32), dtype=np.uint8)
    return codes, scales


def i4_matrix(rng: np.random.Generator, rows: int, cols: int, scale_lo: float, scale_hi: float, zero_lo: int = 8,
              zero_hi: int = 8, signed_scales: bool = False):
    """Random group-32 INT4 matrix [rows, cols]: uniform 4-bit codes, FP16 group
    scales with magnitude log-uniform in [scale_lo, scale_hi] (each with a random
    sign when signed_scales), and zero points uniform in [zero_lo, zero_hi].

    Returns (codes uint8 [rows, cols/2], scales uint16 FP16 bits [rows, cols/32],
    zeros uint8 [rows, cols/32]).
    """
    assert cols % 32 == 0 and 0 <= zero_lo <= zero_hi <= 15
    codes = np.frombuffer(rng.bytes(rows * cols // 2), dtype=np.uint8).reshape(rows, cols // 2).copy()
    mag = np.exp(rng.uniform(np.log(scale_lo), np.log(scale_hi), size=(rows, cols // 32)))
    sign = np.where(rng.integers(0, 2, size=mag.shape) == 1, -1.0, 1.0) if signed_scales else 1.0
    scales = (sign * mag).astype(np.float16).view(np.uint16)
    zeros = rng.integers(zero_lo, zero_hi + 1, size=(rows, cols // 32), dtype=np.uint8)
    return codes, scales, zeros


def _i4_scale_range(cfg: LayerConfig):
    # group-32 INT4 scales log-uniform over the same powers of two as the MXFP4
    # block scales, halved (|q - z| reaches 15 where |v(c)| reaches 6); zero
    # points uniform in [6, 10]
    return 2.0 ** (cfg.e8m0_lo - 128), 2.0 ** (cfg.e8m0_hi - 128), 6, 10


def expert_weights(cfg: LayerConfig, e: int):
    """Weights of expert e (0..E-1 routed, E..E+S-1 shared).

    MXFP4: (gate_up_codes [2I, H/2], gate_up_scales [2I, H/32],
            down_codes [H, I/2], down_scales [H, I/32]), all uint8.
    INT4G32: (gate_up_codes, gate_up_scales, down_codes, down_scales,
              gate_up_zeros, down_zeros): scales are FP16 bits (uint16), the
              rest uint8, shapes as for MXFP4.
    """
    H, I = cfg.hidden, cfg.inter
    if cfg.weight_format == "int4g32":
        lo, hi, zlo, zhi = _i4_scale_range(cfg)
        gc, gs, gz = i4_matrix(_rng(cfg.wseed, _TAG_GATE_UP, e), 2 * I, H, lo, hi, zlo, zhi)
        dc, ds, dz = i4_matrix(_rng(cfg.wseed, _TAG_DOWN, e), H, I, lo, hi, zlo, zhi)
        return gc, gs, dc, ds, gz, dz
    gc, gs = mx_matrix(_rng(cfg.wseed, _TAG_GATE_UP, e), 2 * I, H, cfg.e8m0_lo, cfg.e8m0_hi)
    dc, ds = mx_matrix(_rng(cfg.wseed, _TAG_DOWN, e), H, I, cfg.e8m0_lo, cfg.e8m0_hi)
    return gc, gs, dc, ds


def dense_weights(cfg: LayerConfig):
    """Unsliced dense FFN weights.

    BF16: (W_g [I, H], W_u [I, H], W_d [H, I]) as uint16 bits, N(0, 0.02).
    MXFP4: ((g_codes, g_scales), (u_codes, u_scales), (d_codes, d_scales)).
    INT4G32: ((g_codes, g_scales, g_zeros), (u_...), (d_...)).
    """
    H, I = cfg.hidden, cfg.inter
    if cfg.weight_format == "bf16":
        out = []
        for tag, shape in ((_TAG_DENSE_G, (I, H)), (_TAG_DENSE_U, (I, H)), (_TAG_DENSE_D, (H, I))):
            w = _rng(cfg.wseed, tag).standard_normal(shape, dtype=np.float32) * np.float32(0.02)
            out.append(f32_to_bf16_bits(w))
        return tuple(out)
    if cfg.weight_format == "int4g32":
        lo, hi, zlo, zhi = _i4_scale_range(cfg)
        return tuple(i4_matrix(_rng(cfg.wseed, tag), r, c, lo, hi, zlo, zhi)
                     for tag, r, c in ((_TAG_DENSE_G, I, H), (_TAG_DENSE_U, I, H), (_TAG_DENSE_D, H, I)))
    g = mx_matrix(_rng(cfg.wseed, _TAG_DENSE_G), I, H, cfg.e8m0_lo, cfg.e8m0_hi)
    u = mx_matrix(_rng(cfg.wseed, _TAG_DENSE_U), I, H, cfg.e8m0_lo, cfg.e8m0_hi)
    d = mx_matrix(_rng(cfg.wseed, _TAG_DENSE_D), H, I, cfg.e8m0_lo, cfg.e8m0_hi)
    return g, u, d


def sample_tokens(T: int, n: int, seed: int = 1234) -> np.ndarray:
    """A seeded sorted subset of n token indices out of T (always includes 0 and T-1)."""
    if n >= T:
        return np.arange(T, dtype=np.int64)
    rng = np.random.default_rng(seed)
    idx = set(rng.choice(T, size=n - 2, replace=False).tolist()) | {0, T - 1}
    return np.array(sorted(idx), dtype=np.int64)
