"""GPU parity of group-32 INT4 weights ("Cascadia: Resident 975B MoE Inference
on Eleven AI PCs" §3.1: packed 4-bit codes with one FP16 scale per 32-value
group; §3.5: zero points; w = s * (q - z)) on both compute paths, against
the oracle's INT4 layer on the same seeded inputs:

* routing ids bit-exact, weights within 1e-6; outputs within the layer's bound
  (max|gpu - oracle| / rms(oracle) <= 1e-2) for every token-tile class of the
  kernel, ragged K tails, full hidden and intermediate sizes, and a dense layer
* weights that decode to the same values as INT4 and as MXFP4 give the same
  outputs to within 1e-6: the FP16 MMAs then see operands that differ only by
  exact powers of two
* stored zero points that are all 8 give the outputs of no zero points
* a non-finite scale or a zero point above 15 is rejected at load
* batches beyond the single kernel run the tensor-core GEMMs (each weight an FP16
  hi + lo pair, two MMAs per K step): the same bound against the oracle, on
  ragged shapes, on full H and I with a group over several token tiles (every
  element), on a dense layer of 4096 tokens (sampled tokens), and with large
  spreads of group scales inside a row
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from parity_util import TOL, TOL_W, oracle_dense, oracle_moe, rel_err

from mxfp4_routed_expert_router_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _mods():
    from mxfp4_routed_expert_router_gb300 import binding, layer
    return binding, layer


def i4(cfg):
    return dataclasses.replace(cfg, weight_format="int4g32")


CASES = [
    i4(wl.custom("i4_T1_H7168_I2048_E16_S1_k8", 1, 7168, 2048, 16, 1, 8, seed=61)),  # two-token kernel, full H, I
    i4(wl.custom("i4_T2_H416_I224_E8_S1_k3", 2, 416, 224, 8, 1, 3, seed=62)),         # ragged K tails
    i4(wl.custom("i4_T6_H320_I192_E16_S1_k4", 6, 320, 192, 16, 1, 4, seed=63)),       # 8-token kernel, local routing
    i4(wl.custom("i4_T13_H288_I160_E32_S1_k4", 13, 288, 160, 32, 1, 4, seed=64)),     # 16-token kernel
    i4(wl.custom("i4_T30_H256_I128_E24_S1_k4", 30, 256, 128, 24, 1, 4, seed=65)),     # 32-token kernel
    i4(wl.custom("i4_T60_H256_I128_E64_S1_k4", 60, 256, 128, 64, 1, 4, seed=66)),     # 64-token kernel
]


def _forward(L, cfg, x_bits, logits):
    B, layer = _mods()
    ids = torch.empty((cfg.T, cfg.k), dtype=torch.int32, device="cuda")
    w = torch.empty((cfg.T, cfg.k), dtype=torch.float32, device="cuda")
    out = L.forward(layer.bf16_tensor(x_bits), torch.from_numpy(logits).cuda(), cfg.k,
                    routing=B.routing_out(topk_ids=ids, topk_w=w))
    L.sync()
    return out.cpu().numpy(), ids.cpu().numpy(), w.cpu().numpy()


@pytest.mark.parametrize("cfg", CASES, ids=lambda c: c.name)
def test_int4_layer_parity(cfg):
    _, layer = _mods()
    L = layer.MoeLayer(cfg)
    x, lg = wl.tokens(cfg), wl.router_logits(cfg)
    out, ids, w = _forward(L, cfg, x, lg)
    rid, rw = oracle.route(lg, cfg.k)
    np.testing.assert_array_equal(ids, rid)
    assert np.max(np.abs(w - rw)) <= TOL_W
    ref = oracle_moe(cfg, x, lg, np.arange(cfg.T))
    assert rel_err(out, ref) <= TOL
    assert np.all(np.isfinite(out))
    L.free()


def test_int4_dense_slices():
    _, layer = _mods()
    cfg = dataclasses.replace(wl.dense(1, "int4g32"), name="i4_dense_small", T=37, hidden=256, inter=4 * 96,
                              n_experts=4, n_slices=4, k=4, seed=67)
    L = layer.MoeLayer(cfg)
    x = wl.tokens(cfg)
    out = L.forward(layer.bf16_tensor(x), None).cpu().numpy()
    L.sync()
    assert rel_err(out, oracle_dense(cfg, x, np.arange(cfg.T))) <= TOL
    L.free()


def test_int4_dense_full_size():
    # H = 7168, I = 18432 in 9 slices of 2048, at one and at 64 tokens
    _, layer = _mods()
    cfg = wl.dense(64, "int4g32")
    L = layer.MoeLayer(cfg)
    weights = wl.dense_weights(cfg)
    x = wl.tokens(cfg)
    for T, n_sample in ((1, 1), (64, 2)):
        out = L.forward(layer.bf16_tensor(x[:T]), None).cpu().numpy()
        L.sync()
        tok = wl.sample_tokens(T, n_sample)
        assert rel_err(out[tok], oracle_dense(cfg, x[:T], tok, weights)) <= TOL, T
    L.free()


# E2M1 codes with magnitude index m <= 5 have |v| = 0, .5, 1, 1.5, 2, 3, so
# 2|v| = 0, 1, 2, 3, 4, 6: with E8M0 126 (scale 1/2) the weight is v / 2, and
# as INT4 with scale 1/4 it is (q - z) / 4 for q - z = 2v.
_TWICE_V = np.array([0, 1, 2, 3, 4, 6])


def _small_mx(rng, rows, cols):
    m = rng.integers(0, 6, (rows, cols))
    sign = rng.integers(0, 2, (rows, cols))
    codes = (m | (sign << 3)).astype(np.uint8)
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    twice_v = np.where(sign == 1, -_TWICE_V[m], _TWICE_V[m])
    zeros = rng.integers(6, 10, (rows, cols // 32)).astype(np.uint8)
    q = twice_v + np.repeat(zeros.astype(np.int64), 32, axis=1)
    assert q.min() >= 0 and q.max() <= 15
    q_packed = (q[:, 0::2] | (q[:, 1::2] << 4)).astype(np.uint8)
    mx = (packed, np.full((rows, cols // 32), 126, np.uint8))
    i4w = (q_packed, np.full((rows, cols // 32), 0x3400, np.uint16), zeros)  # FP16 0x3400 = 1/4
    return mx, i4w


def _load(fmt, H, I, E, S, k, gu, dn):
    B, layer = _mods()
    c = B.MoeConfig(hidden=H, inter=I, n_experts=E, n_shared=S, k_max=k, n_slices=0, fmt=fmt)

    def dev(m):
        return tuple(None if a is None else (layer.u16_tensor(a) if a.dtype == np.uint16 else layer.u8_tensor(a))
                     for a in m)

    return B.moe_load_weights(c, [dev(m) for m in gu], [dev(m) for m in dn])


def _run(h, x, lg, T, k, H):
    B, layer = _mods()
    out = torch.empty((T, H), dtype=torch.float32, device="cuda")
    n = B.moe_workspace_bytes(h, T, k)
    ws = torch.empty(max(n, 256), dtype=torch.uint8, device="cuda")
    B.moe_forward(h, x, lg, T, k, out, False, ws, n)
    B.moe_sync_status(h)
    return out.cpu().numpy()


@pytest.mark.parametrize("T", [1, 5, 24])
def test_int4_equals_mxfp4_on_equal_weights(T):
    B, layer = _mods()
    H, I, E, S, k = 320, 192, 8, 1, 3
    rng = np.random.default_rng(68 + T)
    gu, dn = [_small_mx(rng, 2 * I, H) for _ in range(E + S)], [_small_mx(rng, H, I) for _ in range(E + S)]
    hm = _load(B.MOE_W_MXFP4, H, I, E, S, k, [g[0] for g in gu], [d[0] for d in dn])
    hi = _load(B.MOE_W_INT4G32, H, I, E, S, k, [g[1] for g in gu], [d[1] for d in dn])
    cfg = wl.custom("i4_eq", T, H, I, E, S, k, seed=69)
    x = layer.bf16_tensor(wl.tokens(cfg))
    lg = torch.from_numpy(wl.router_logits(cfg)).cuda()
    a, b = _run(hm, x, lg, T, k, H), _run(hi, x, lg, T, k, H)
    assert rel_err(b, a) <= 1e-6
    B.moe_free(hm)
    B.moe_free(hi)


def test_int4_zero_points_all_8_equal_none():
    B, layer = _mods()
    cfg = i4(wl.custom("i4_z8", 4, 256, 128, 8, 1, 2, seed=70))
    rng = np.random.default_rng(70)
    ws = [(wl.i4_matrix(rng, 256, 256, 2.0 ** -8, 2.0 ** -4), wl.i4_matrix(rng, 256, 128, 2.0 ** -8, 2.0 ** -4))
          for _ in range(9)]
    with_z = _load(B.MOE_W_INT4G32, 256, 128, 8, 1, 2, [g for g, _ in ws], [d for _, d in ws])
    no_z = _load(B.MOE_W_INT4G32, 256, 128, 8, 1, 2, [(g[0], g[1], None) for g, _ in ws],
                 [(d[0], d[1], None) for _, d in ws])
    x = layer.bf16_tensor(wl.tokens(cfg))
    lg = torch.from_numpy(wl.router_logits(cfg)).cuda()
    assert np.array_equal(_run(with_z, x, lg, 4, 2, 256), _run(no_z, x, lg, 4, 2, 256))
    B.moe_free(with_z)
    B.moe_free(no_z)


@pytest.mark.parametrize("bad", ["inf_scale", "nan_scale", "zero_16"])
def test_int4_bad_scale_or_zero_rejected_at_load(bad):
    B, _ = _mods()
    cfg = i4(wl.custom("i4_bad", 1, 256, 128, 4, 0, 2, seed=71))
    ex = [wl.expert_weights(cfg, e) for e in range(cfg.n_groups)]
    gc, gs, dc, ds, gz, dz = ex[2]
    if bad == "inf_scale":
        ds[7, 3] = 0x7C00
    elif bad == "nan_scale":
        gs[100, 5] = 0xFE00
    else:
        dz[0, 0] = 16
    with pytest.raises(B.MoeError) as e:
        _load(B.MOE_W_INT4G32, 256, 128, 4, 0, 2, [(a[0], a[1], a[4]) for a in ex], [(a[2], a[3], a[5]) for a in ex])
    assert e.value.status == B.MOE_ESCALE


TC_CASES = [
    # 80 routed slots for 4 experts: past the single kernel (16 per expert)
    i4(wl.custom("i4_tc_T40_H256_I128_E4_S0_k2", 40, 256, 128, 4, 0, 2, seed=72)),
    # ragged row tiles of both GEMMs (H and I not multiples of 128), a shared group
    i4(wl.custom("i4_tc_T300_H416_I288_E16_S1_k4", 300, 416, 288, 16, 1, 4, seed=73)),
]


@pytest.mark.parametrize("cfg", TC_CASES, ids=lambda c: c.name)
def test_int4_tensor_core_parity(cfg):
    _, layer = _mods()
    L = layer.MoeLayer(cfg)
    x, lg = wl.tokens(cfg), wl.router_logits(cfg)
    out, ids, w = _forward(L, cfg, x, lg)
    rid, rw = oracle.route(lg, cfg.k)
    np.testing.assert_array_equal(ids, rid)
    assert np.max(np.abs(w - rw)) <= TOL_W
    ref = oracle_moe(cfg, x, lg, np.arange(cfg.T))
    assert np.all(np.isfinite(out))
    assert rel_err(out, ref) <= TOL
    L.free()


def test_int4_tensor_core_full_hidden_multi_tile_every_element():
    # full H and I; one routed group of ~950 tokens spans several token tiles of
    # both GEMMs with a ragged last tile; every output element against the oracle
    from parity_util import skewed_logits
    _, layer = _mods()
    cfg = i4(wl.custom("i4_tc_T1000_H7168_I2048_E6_S1_k2", 1000, 7168, 2048, 6, 1, 2, seed=74))
    L = layer.MoeLayer(cfg)
    x, lg = wl.tokens(cfg), skewed_logits(cfg, 0, 950)
    out, ids, w = _forward(L, cfg, x, lg)
    rid, _ = oracle.route(lg, cfg.k)
    np.testing.assert_array_equal(ids, rid)
    assert int(np.sum(ids == 0)) >= 950
    ref = oracle_moe(cfg, x, lg, np.arange(cfg.T))
    assert np.all(np.isfinite(out))
    assert rel_err(out, ref) <= TOL
    L.free()


def test_int4_tensor_core_dense_4096():
    # the dense FFN (H = 7168, I = 18432 in 9 slices) at 4096 tokens, sampled tokens
    _, layer = _mods()
    cfg = wl.dense(4096, "int4g32")
    L = layer.MoeLayer(cfg)
    weights = wl.dense_weights(cfg)
    x = wl.tokens(cfg)
    out = L.forward(layer.bf16_tensor(x), None).cpu().numpy()
    L.sync()
    tok = wl.sample_tokens(cfg.T, 3)
    assert np.all(np.isfinite(out[tok]))
    assert rel_err(out[tok], oracle_dense(cfg, x, tok, weights)) <= TOL
    L.free()


def test_int4_tensor_core_wide_scale_spread():
    # group scales spread over 2^-24 .. 2^1 inside every row (FP16 subnormal
    # scales included): the decode against the row's power of two stays exact,
    # and the powers of two of h and y, fixed from norm bounds, still keep the
    # bound (a numpy model of the pipeline gives 4.9e-3 on these inputs; a
    # spread of 2^-30 gives 1.01e-2, on the model and on the GPU alike)
    B, layer = _mods()
    rng = np.random.default_rng(75)
    H, I, E, k, T = 256, 128, 4, 2, 48
    ex = []
    for e in range(E):
        mats = []
        for rows, cols in ((2 * I, H), (H, I)):
            q = rng.integers(0, 16, (rows, cols)).astype(np.uint8)
            packed = (q[:, 0::2] | (q[:, 1::2] << 4)).astype(np.uint8)
            expo = rng.integers(-24, 1, (rows, cols // 32)).astype(np.float64)
            sc = (np.exp2(expo) * rng.uniform(1.0, 2.0, expo.shape)).astype(np.float16).view(np.uint16)
            zp = rng.integers(6, 10, (rows, cols // 32)).astype(np.uint8)
            mats.append((packed, sc, zp))
        ex.append(mats)
    h = _load(B.MOE_W_INT4G32, H, I, E, 0, k, [m[0] for m in ex], [m[1] for m in ex])
    cfg = i4(wl.custom("i4_spread", T, H, I, E, 0, k, seed=76))
    x_bits, lg = wl.tokens(cfg), wl.router_logits(cfg)
    out = _run(h, layer.bf16_tensor(x_bits), torch.from_numpy(lg).cuda(), T, k, H)
    B.moe_free(h)
    W = oracle.OracleWeights(H, I, E, 0, "int4g32")
    for e in range(E):
        (g, gs, gz), (d, ds, dz) = ex[e]
        W.set_expert(e, g, gs, d, ds, gz, dz)
    ref, _, _ = oracle.moe_layer(W, x_bits, lg, k)
    assert np.all(np.isfinite(out))
    assert rel_err(out, ref) <= TOL
