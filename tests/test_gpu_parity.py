"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle on the
same seeded inputs.

* routing ids, expert offsets and the permutation: bit-exact
* routing weights: within 1e-6 absolute
* FP32 outputs: max|gpu - oracle| / rms(oracle) <= 1e-2

Small layers are compared on every output; full-size layers on every output
of a seeded token sample (the oracle computes a token from its own x and
logits rows alone), with routing and permutation always checked for all
tokens.
"""
import numpy as np
import pytest
import torch

import oracle
from parity_util import TOL, TOL_W, oracle_dense, oracle_moe, rel_err, skewed_logits

from mxfp4_routed_expert_router_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _binding():
    from mxfp4_routed_expert_router_gb300 import binding, layer
    return binding, layer


def run_routed(L, cfg, x_bits, logits, k=None):
    B, layer = _binding()
    k = k or cfg.k
    T = x_bits.shape[0]
    x = layer.bf16_tensor(x_bits)
    lg = torch.from_numpy(logits).cuda()
    ids = torch.empty((T, k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, k), dtype=torch.float32, device="cuda")
    off = torch.empty(cfg.n_experts + 1, dtype=torch.int32, device="cuda")
    ss = torch.empty(T * k, dtype=torch.int32, device="cuda")
    sp = torch.empty(T * k, dtype=torch.int32, device="cuda")
    r = B.routing_out(ids, w, off, ss, sp)
    out = L.forward(x, lg, k, routing=r)
    L.sync()
    return out.cpu().numpy(), ids.cpu().numpy(), w.cpu().numpy(), off.cpu().numpy(), ss.cpu().numpy(), sp.cpu().numpy()


def check_routing(cfg, logits, ids, w, off, ss, sp, k=None):
    k = k or cfg.k
    rid, rw = oracle.route(logits, k)
    np.testing.assert_array_equal(ids, rid)
    assert np.max(np.abs(w - rw)) <= TOL_W
    roff, rss, rsp = oracle.permute(rid, cfg.n_experts)
    np.testing.assert_array_equal(off, roff)
    np.testing.assert_array_equal(ss, rss)
    np.testing.assert_array_equal(sp, rsp)


# ------------------------------------------------------------------ small layers, every output

SMALL = [
    wl.tiny(),
    wl.custom("ragged_T100_H288_I160_E16_S1_k4", 100, 288, 160, 16, 1, 4, seed=21),
    wl.custom("k_eq_E_T33_H64_I96_E8", 33, 64, 96, 8, 0, 8, seed=22),
    wl.custom("single_expert_T7_H96_I64", 7, 96, 64, 1, 0, 1, seed=23),
    wl.custom("wide_T300_H512_I256_E32_S2_k6", 300, 512, 256, 32, 2, 6, seed=24),
    wl.custom("T1_H7168_I2048_E4_S1_k2", 1, 7168, 2048, 4, 1, 2, seed=25),
    # decode-sized batch (register-streaming path) with K not a multiple of 64
    wl.custom("stream_ragged_T3_H288_I160_E16_S1_k4", 3, 288, 160, 16, 1, 4, seed=31),
    # streaming path, largest token tile (64 tokens per group tile)
    wl.custom("stream_T60_H256_I128_E64_S1_k4", 60, 256, 128, 64, 1, 4, seed=32),
    # streaming path, batch of two tokens (two reserved token rows per stage), ragged K
    wl.custom("stream_T2_H416_I224_E8_S1_k3", 2, 416, 224, 8, 1, 3, seed=36),
    # streaming path, items of every tile class: groups of 9-16 and 17-32 tokens
    wl.custom("stream_classes_T40_H256_I192_E16_S1_k4", 40, 256, 192, 16, 1, 4, seed=33),
    wl.custom("stream_classes_T21_H320_I128_E4_S1_k3", 21, 320, 128, 4, 1, 3, seed=35),
    # 32-token kernel: down items of 1-4 tokens (packed) and of 5-8 and 11 tokens (class 2)
    wl.custom("stream_T30_H256_I128_E24_S1_k4", 30, 256, 128, 24, 1, 4, seed=39),
    # tensor-core path, FP16 operands at the widest exponent span they take (23 within a row):
    # weights down to 0.5 * 2^-23 relative to the row's largest scale are FP16 subnormals
    wl.custom("tc_span23_T100_H288_I160_E16_S1_k4", 100, 288, 160, 16, 1, 4, seed=64, e8m0_lo=107, e8m0_hi=130),
    # tensor-core path, exponents spanning more than 23 within rows: BF16 operands
    wl.custom("tc_span34_T100_H288_I160_E16_S1_k4", 100, 288, 160, 16, 1, 4, seed=65, e8m0_lo=96, e8m0_hi=130),
]


@pytest.mark.parametrize("cfg", SMALL, ids=lambda c: c.name)
def test_small_layer_parity(cfg):
    _, layer = _binding()
    L = layer.MoeLayer(cfg)
    x, lg = wl.tokens(cfg), wl.router_logits(cfg)
    out, ids, w, off, ss, sp = run_routed(L, cfg, x, lg)
    check_routing(cfg, lg, ids, w, off, ss, sp)
    ref = oracle_moe(cfg, x, lg, np.arange(cfg.T))
    assert rel_err(out, ref) <= TOL
    L.free()


def test_accumulate_adds_into_residual():
    _, layer = _binding()
    cfg = wl.tiny()
    L = layer.MoeLayer(cfg)
    x, lg = wl.tokens(cfg), wl.router_logits(cfg)
    resid = np.random.default_rng(3).standard_normal((cfg.T, cfg.hidden)).astype(np.float32) * 100
    out = torch.from_numpy(resid.copy()).cuda()
    L.forward(layer.bf16_tensor(x), torch.from_numpy(lg).cuda(), out=out, accumulate=True)
    L.sync()
    ref = oracle_moe(cfg, x, lg, np.arange(cfg.T))
    got = out.cpu().numpy().astype(np.float64) - resid
    assert np.max(np.abs(got - ref)) / np.sqrt(np.mean(ref ** 2)) <= TOL + 1e-4
    L.free()


def test_deterministic_and_token_order_equivariant():
    _, layer = _binding()
    cfg = wl.custom("det", 64, 256, 128, 8, 1, 2, seed=26)
    L = layer.MoeLayer(cfg)
    x, lg = wl.tokens(cfg), wl.router_logits(cfg)
    xt, lt = layer.bf16_tensor(x), torch.from_numpy(lg).cuda()
    a = L.forward(xt, lt).cpu().numpy()
    b = L.forward(xt, lt).cpu().numpy()
    np.testing.assert_array_equal(a, b)
    perm = np.random.default_rng(4).permutation(cfg.T)
    c = L.forward(layer.bf16_tensor(x[perm]), torch.from_numpy(lg[perm]).cuda()).cpu().numpy()
    assert rel_err(c, a[perm]) <= 1e-5
    L.free()


def test_down_exponent_plus_one_doubles_output():
    """Powers of two change exponents exactly ("Cascadia" §3.3): +1 on every
    down-projection E8M0 exponent doubles the output bit for bit."""
    B, layer = _binding()
    cfg = wl.custom("dbl", 24, 128, 64, 4, 1, 2, seed=27)
    ex = [wl.expert_weights(cfg, e) for e in range(cfg.n_groups)]
    handles = []
    for bump in (0, 1):
        gu = [(layer.u8_tensor(gc), layer.u8_tensor(gs)) for gc, gs, _, _ in ex]
        dn = [(layer.u8_tensor(dc), layer.u8_tensor(ds + bump)) for _, _, dc, ds in ex]
        c = B.MoeConfig(hidden=128, inter=64, n_experts=4, n_shared=1, k_max=2, n_slices=0, fmt=B.MOE_W_MXFP4)
        handles.append(B.moe_load_weights(c, gu, dn))
    x, lg = layer.bf16_tensor(wl.tokens(cfg)), torch.from_numpy(wl.router_logits(cfg)).cuda()
    outs = []
    for h in handles:
        n = B.moe_workspace_bytes(h, cfg.T, 2)
        ws = torch.empty(n, dtype=torch.uint8, device="cuda")
        o = torch.empty((cfg.T, 128), dtype=torch.float32, device="cuda")
        B.moe_forward(h, x, lg, cfg.T, 2, o, False, ws, n)
        B.moe_sync_status(h)
        outs.append(o.cpu().numpy())
        B.moe_free(h)
    np.testing.assert_array_equal(outs[1], 2 * outs[0])


def test_T0_is_a_noop():
    B, layer = _binding()
    cfg = wl.tiny()
    L = layer.MoeLayer(cfg)
    out = torch.full((1, cfg.hidden), 7.0, device="cuda")
    B.moe_forward(L.handle, out, out, 0, 2, out, False, out, 0)
    L.sync()
    assert torch.all(out == 7.0)
    L.free()


def test_routing_ties_signed_zero_nan_on_device():
    """Tie-laden logits: selection must match the oracle bit for bit."""
    _, layer = _binding()
    cfg = wl.custom("ties", 200, 64, 64, 40, 0, 6, seed=28)
    L = layer.MoeLayer(cfg)
    rng = np.random.default_rng(29)
    vals = np.array([0.0, -0.0, 1.0, -1.0, 0.5, 2.0, np.nan, -np.inf, np.inf], np.float32)
    lg = rng.choice(vals, size=(cfg.T, cfg.n_experts)).astype(np.float32)
    lg[:, 0] = 3.0  # keep every row's softmax finite: the largest logit is finite
    lg[:5, 1] = np.inf
    x = wl.tokens(cfg)
    _, ids, w, off, ss, sp = run_routed(L, cfg, x, lg)
    rid, _ = oracle.route(lg, cfg.k)
    np.testing.assert_array_equal(ids, rid)
    roff, rss, rsp = oracle.permute(rid, cfg.n_experts)
    np.testing.assert_array_equal(off, roff)
    np.testing.assert_array_equal(ss, rss)
    np.testing.assert_array_equal(sp, rsp)
    L.free()


# ------------------------------------------------------------------ error paths on the device

def test_scale_255_rejected_at_load():
    B, layer = _binding()
    cfg = wl.tiny()
    ex = [wl.expert_weights(cfg, e) for e in range(cfg.n_groups)]
    ex[3][3][5, 1] = 255
    gu = [(layer.u8_tensor(a), layer.u8_tensor(b)) for a, b, _, _ in ex]
    dn = [(layer.u8_tensor(c), layer.u8_tensor(d)) for _, _, c, d in ex]
    c = B.MoeConfig(hidden=256, inter=128, n_experts=8, n_shared=0, k_max=2, n_slices=0, fmt=B.MOE_W_MXFP4)
    with pytest.raises(B.MoeError) as e:
        B.moe_load_weights(c, gu, dn)
    assert e.value.status == B.MOE_ESCALE


def test_bad_forward_arguments():
    B, layer = _binding()
    cfg = wl.tiny()
    L = layer.MoeLayer(cfg)
    x = layer.bf16_tensor(wl.tokens(cfg))
    lg = torch.from_numpy(wl.router_logits(cfg)).cuda()
    out = torch.empty((cfg.T, cfg.hidden), device="cuda")
    n = B.moe_workspace_bytes(L.handle, cfg.T, 2)
    ws = torch.empty(n + 512, dtype=torch.uint8, device="cuda")
    cases = [
        (dict(k=3), B.MOE_EINVAL),                       # k > k_max
        (dict(k=0), B.MOE_EINVAL),
        (dict(ws_bytes=n - 1), B.MOE_EWORKSPACE),
        (dict(ws=ws.data_ptr() + 16), B.MOE_EWORKSPACE),  # misaligned workspace
        (dict(x=x.data_ptr() + 2), B.MOE_EINVAL),         # misaligned x
        (dict(T=-1), B.MOE_EINVAL),
    ]
    for over, status in cases:
        a = dict(x=x, k=2, ws=ws, ws_bytes=n, T=cfg.T)
        a.update(over)
        with pytest.raises(B.MoeError) as e:
            B.moe_forward(L.handle, a["x"], lg, a["T"], a["k"], out, False, a["ws"], a["ws_bytes"])
        assert e.value.status == status, over
    with pytest.raises(B.MoeError) as e:
        B.moe_dense_sliced_forward(L.handle, x, cfg.T, out, False, ws, n)
    assert e.value.status == B.MOE_EINVAL
    L.free()


def test_wait_expiry_reports_device_error_and_a_fresh_handle_works():
    """A bounded wait that runs out: the single kernel's grid-wide completion wait
    is armed with a target no launch reaches and a 1 ms limit.  The kernel must
    leave cleanly, the handle must report MOE_EDEVICE (a timeout), the context
    must stay usable, and a fresh handle must still match the oracle."""
    B, layer = _binding()
    cfg = wl.custom("expire_T4_H256_I128_E16_S1_k4", 4, 256, 128, 16, 1, 4, seed=63)
    x, lg = wl.tokens(cfg), wl.router_logits(cfg)
    L = layer.MoeLayer(cfg)
    with pytest.raises(B.MoeError) as e:
        B.moe_debug_expire_next_wait(L.handle, 0)
    assert e.value.status == B.MOE_EINVAL
    B.moe_debug_expire_next_wait(L.handle, 1000)
    L.forward(layer.bf16_tensor(x), torch.from_numpy(lg).cuda())
    with pytest.raises(B.MoeError) as e:
        L.sync()
    assert e.value.status == B.MOE_EDEVICE and "device error 3" in str(e.value)
    # the error is sticky on this handle: the next call is refused before any launch
    with pytest.raises(B.MoeError) as e:
        L.forward(layer.bf16_tensor(x), torch.from_numpy(lg).cuda())
    assert e.value.status == B.MOE_EDEVICE
    L.free()
    torch.cuda.synchronize()
    L2 = layer.MoeLayer(cfg)
    out, ids, w, off, ss, sp = run_routed(L2, cfg, x, lg)
    check_routing(cfg, lg, ids, w, off, ss, sp)
    assert rel_err(out, oracle_moe(cfg, x, lg, np.arange(cfg.T))) <= TOL
    L2.free()


# ------------------------------------------------------------------ the full-size layer (bench shapes)

@pytest.fixture(scope="module")
def big_layer():
    _, layer = _binding()
    L = layer.MoeLayer(wl.decode(1))
    yield L
    L.free()


@pytest.mark.parametrize("cfg,n_sample", [
    (wl.decode(1), 1),
    (wl.sweep(15), 15),
    (wl.sweep(88), 10),
    (wl.sweep(176), 10),
    (wl.prefill(8192), 6),
], ids=lambda v: v.name if hasattr(v, "name") else str(v))
def test_full_size_layer(big_layer, cfg, n_sample):
    x, lg = wl.tokens(cfg), wl.router_logits(cfg)
    out, ids, w, off, ss, sp = run_routed(big_layer, cfg, x, lg)
    check_routing(cfg, lg, ids, w, off, ss, sp)
    tok = wl.sample_tokens(cfg.T, n_sample)
    ref = oracle_moe(cfg, x, lg, tok)
    assert rel_err(out[tok], ref) <= TOL
    assert np.all(np.isfinite(out))


@pytest.mark.parametrize("cfg,hot_tokens", [
    # one routed group of ~950 tokens: 4 gate|up token tiles of up to 256 and 8 down
    # tiles of up to 128, both with a ragged last tile; the shared group spans all
    # 1000 tokens; the other routed groups are small (one partial tile each)
    (wl.custom("multi_tile_T1000_H7168_I2048_E6_S1_k2", 1000, 7168, 2048, 6, 1, 2, seed=61), 950),
    # a group just past one tile boundary next to near-empty groups
    (wl.custom("multi_tile_T300_H7168_I2048_E5_S1_k1", 300, 7168, 2048, 5, 1, 1, seed=62), 257),
], ids=lambda v: v.name if hasattr(v, "name") else str(v))
def test_full_hidden_multi_tile_every_element(cfg, hot_tokens):
    """Full H and I on the tensor-core path, with groups that span several token
    tiles of both GEMMs: every output element against the oracle."""
    _, layer = _binding()
    L = layer.MoeLayer(cfg)
    x, lg = wl.tokens(cfg), skewed_logits(cfg, 0, hot_tokens)
    out, ids, w, off, ss, sp = run_routed(L, cfg, x, lg)
    L.free()
    check_routing(cfg, lg, ids, w, off, ss, sp)
    counts = np.diff(off)
    assert counts[0] >= hot_tokens
    ref = oracle_moe(cfg, x, lg, np.arange(cfg.T))
    assert np.all(np.isfinite(out))
    assert rel_err(out, ref) <= TOL


# ------------------------------------------------------------------ dense FFN as all-active slices

@pytest.mark.parametrize("fmt", ["bf16", "mxfp4"])
def test_dense_small_sliced_vs_unsliced(fmt):
    """Eq. 2: the sliced GPU result matches the oracle's unsliced FFN."""
    _, layer = _binding()
    base = wl.dense(1, fmt)
    import dataclasses
    cfg = dataclasses.replace(base, name=f"dense_small_{fmt}", T=37, hidden=256, inter=4 * 96, n_experts=4,
                              n_slices=4, k=4, seed=30)
    L = layer.MoeLayer(cfg)
    x = wl.tokens(cfg)
    out = L.forward(layer.bf16_tensor(x), None).cpu().numpy()
    ref = oracle_dense(cfg, x, np.arange(cfg.T))
    assert rel_err(out, ref) <= TOL
    L.free()


@pytest.mark.parametrize("fmt", ["bf16", "mxfp4"])
def test_dense_full_size(fmt):
    _, layer = _binding()
    cfg = wl.dense(4096, fmt)
    L = layer.MoeLayer(cfg)
    weights = wl.dense_weights(cfg)
    x = wl.tokens(cfg)
    for T, n_sample in ((1, 1), (88, 4), (4096, 4)):
        xs = x[:T]
        out = L.forward(layer.bf16_tensor(xs), None).cpu().numpy()
        L.sync()
        tok = wl.sample_tokens(T, n_sample)
        ref = oracle_dense(cfg, xs, tok, weights)
        assert rel_err(out[tok], ref) <= TOL, (fmt, T)
    L.free()
