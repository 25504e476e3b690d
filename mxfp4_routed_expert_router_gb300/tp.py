"""Tensor parallelism of the MoE layer over its intermediate dimension.

The dense FFN of "Cascadia: Resident 975B MoE Inference on Eleven AI PCs"
§3.4 (Eq. 2) is a sum of slices of the intermediate dimension, each an
independent SwiGLU block: h_n depends only on row n of W_g and W_u, and
y = sum_n h_n W_d[:, n].  The same identity splits every expert of a routed
layer: rank r owns intermediate features [f0_r, f1_r) of every expert (the
gate rows, the up rows and the down columns of that range, with their block
scales), runs the layer on its slice with the same routing, and the ranks'
FP32 partial outputs add up to the layer's output -- one all-reduce of
[T, H] per layer, the rank-local partials plus in-place all-reduce of
"DeepSeek-V4-Flash on a four-GPU Ampere workstation" (section "The
architecture, in one diagram").

Slices start and end on multiples of 32 so that no MXFP4 block (one E8M0
exponent per 32 values along the intermediate dimension of the down matrix)
is cut; the loader's rule for dense slices is the same.

This module is host logic only: it computes the ranges, cuts the caller's
weight arrays, and wraps one rank's library handle; every step of the layer
runs in libmoe_gb300.so, and the sum across ranks is torch.distributed's
all-reduce (NCCL between GPUs).  The tests run the ranks one after another on
a single device and the all-reduce over gloo on the CPU.
"""
from __future__ import annotations

import dataclasses
from typing import List, Sequence, Tuple

import numpy as np

from . import workloads as wl

MX_BLOCK = 32


def shard_ranges(inter: int, world: int) -> List[Tuple[int, int]]:
    """[f0, f1) of every rank: contiguous, covering [0, inter), each a multiple
    of 32 wide, as equal as the 32-value blocks allow (earlier ranks take the
    extra blocks)."""
    if inter % MX_BLOCK:
        raise ValueError(f"inter = {inter} is not a multiple of {MX_BLOCK}")
    blocks = inter // MX_BLOCK
    if world < 1 or world > blocks:
        raise ValueError(f"cannot cut {blocks} blocks of {MX_BLOCK} over {world} ranks")
    base, extra = divmod(blocks, world)
    out, b0 = [], 0
    for r in range(world):
        nb = base + (1 if r < extra else 0)
        out.append((b0 * MX_BLOCK, (b0 + nb) * MX_BLOCK))
        b0 += nb
    return out


def shard_mx_expert(gu_codes: np.ndarray, gu_scales: np.ndarray, dn_codes: np.ndarray, dn_scales: np.ndarray,
                    inter: int, f0: int, f1: int):
    """One expert's MXFP4 weights restricted to intermediate features [f0, f1).

    gu_codes [2I, H/2] / gu_scales [2I, H/32]: gate rows 0..I-1, up rows I..2I-1
    -> rows [f0, f1) and [I + f0, I + f1), still gate rows first.
    dn_codes [H, I/2] / dn_scales [H, I/32] -> columns [f0, f1) (code bytes
    [f0/2, f1/2), scale bytes [f0/32, f1/32)).  Copies, contiguous."""
    if f0 % MX_BLOCK or f1 % MX_BLOCK or not 0 <= f0 < f1 <= inter:
        raise ValueError(f"feature range [{f0}, {f1}) is not a block-aligned part of [0, {inter})")
    rows = np.r_[f0:f1, inter + f0:inter + f1]
    g_c = np.ascontiguousarray(gu_codes[rows])
    g_s = np.ascontiguousarray(gu_scales[rows])
    d_c = np.ascontiguousarray(dn_codes[:, f0 // 2:f1 // 2])
    d_s = np.ascontiguousarray(dn_scales[:, f0 // MX_BLOCK:f1 // MX_BLOCK])
    return g_c, g_s, d_c, d_s


def shard_config(cfg: wl.LayerConfig, f0: int, f1: int) -> wl.LayerConfig:
    """The rank's layer: same experts, routing inputs and tokens, intermediate width f1 - f0."""
    return dataclasses.replace(cfg, name=f"{cfg.name}_tp{f0}_{f1}", inter=f1 - f0)


def shard_weights(cfg: wl.LayerConfig, f0: int, f1: int) -> Sequence[tuple]:
    """Every expert group's MXFP4 weights of the seeded layer cfg, cut to [f0, f1)."""
    if cfg.weight_format != "mxfp4" or cfg.dense:
        raise ValueError("tensor-parallel shards are cut from routed MXFP4 layers")
    return [shard_mx_expert(*wl.expert_weights(cfg, e), cfg.inter, f0, f1) for e in range(cfg.n_groups)]


class TensorParallelMoe:
    """One rank of a routed MXFP4 layer split over the intermediate dimension.

    forward() runs the rank's slice of every expert through the library and,
    when a process group is given, sums the partial outputs across ranks in
    place (torch.distributed all-reduce); without one it returns the rank's
    partial output."""

    def __init__(self, cfg: wl.LayerConfig, rank: int, world: int, device: str = "cuda", k_max=None):
        import torch

        from . import binding as B
        from .layer import u8_tensor

        self.cfg, self.rank, self.world = cfg, rank, world
        self.f0, self.f1 = shard_ranges(cfg.inter, world)[rank]
        self.device = torch.device(device)
        shards = shard_weights(cfg, self.f0, self.f1)
        gate_up = [(u8_tensor(g, device), u8_tensor(s, device)) for g, s, _, _ in shards]
        down = [(u8_tensor(c, device), u8_tensor(s, device)) for _, _, c, s in shards]
        c = B.MoeConfig(hidden=cfg.hidden, inter=self.f1 - self.f0, n_experts=cfg.n_experts, n_shared=cfg.n_shared,
                        k_max=k_max or cfg.k, n_slices=0, fmt=B.MOE_W_MXFP4)
        self.B = B
        self.handle = B.moe_load_weights(c, gate_up, down)
        self._ws = None

    def forward(self, x, logits, k=None, group=None, stream=None):
        import torch

        B = self.B
        T, k = x.shape[0], k or self.cfg.k
        n = B.moe_workspace_bytes(self.handle, T, k)
        if self._ws is None or self._ws.numel() < n:
            self._ws = torch.empty(max(n, 256), dtype=torch.uint8, device=self.device)
        out = torch.empty((T, self.cfg.hidden), dtype=torch.float32, device=self.device)
        B.moe_forward(self.handle, x, logits, T, k, out, False, self._ws, n, None, stream)
        if group is not None:
            import torch.distributed as dist
            dist.all_reduce(out, op=dist.ReduceOp.SUM, group=group)
        return out

    def free(self):
        if self.handle:
            self.B.moe_free(self.handle)
            self.handle = None
