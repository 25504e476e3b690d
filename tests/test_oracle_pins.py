"""Pins of the CPU oracle against facts that do not come from the oracle itself.

Each test checks the oracle against one of: the tables and identities the pages
print (golden files under tests/golden/, each citing its passage), exact closed
forms evaluated with rational arithmetic, mathematical invariants, brute force
on tiny inputs written independently in numpy / plain Python, or special cases
that reduce to a textbook SwiGLU FFN.  They are chosen so that a plausible slip
in the oracle (nibble order, sign bit, magnitude order, exponent bias, block
index, tie-break, renormalisation, permutation stability, gate/up swap, a
dropped shared expert, a dropped slice; for group-32 INT4 the zero point's
sign or default, the group index and the FP16 scale decode) fails at least one
of them.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from mxfp4_routed_expert_router_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def load_e2m1_table():
    table = {}
    with open(os.path.join(GOLDEN, "e2m1_table.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            c, v = line.split()
            table[int(c)] = float(v)
    assert sorted(table) == list(range(16))
    return table


E2M1 = load_e2m1_table()


def exact_decode(code, e):
    """v(c) * 2^(e-127) from the golden table with exact rational arithmetic."""
    v = Fraction(E2M1[code])
    val = float(v * Fraction(2) ** (e - 127))
    return math.copysign(val, E2M1[code]) if val == 0 else val


def np_decode_golden(codes, scales):
    """Independent numpy decode of an MXFP4 matrix via the golden table."""
    tab = np.array([E2M1[c] for c in range(16)], np.float64)
    lo = codes & 0xF
    hi = codes >> 4
    c = np.stack([lo, hi], axis=-1).reshape(codes.shape[0], -1)
    v = tab[c]
    s = np.repeat(scales.astype(np.int64), 32, axis=1)
    return np.ldexp(v, s - 127)


# ------------------------------------------------------------------ decode pins

@pytest.mark.parametrize("e", [0, 1, 2, 120, 126, 127, 128, 130, 200, 252])
def test_e2m1_table_all_codes(e):
    for code in range(16):
        got = oracle.mx_value(code, e)
        want = exact_decode(code, e)
        assert got == want and math.copysign(1, got) == math.copysign(1, want), (code, e, got, want)


def test_e2m1_value_table():
    for code in range(16):
        got = oracle.e2m1_value(code)
        assert got == E2M1[code] and math.copysign(1, got) == math.copysign(1, E2M1[code])


def test_e8m0_zero_is_subnormal_not_zero():
    # 0.5 * 2^-127 = 2^-128 is a float32 subnormal; it must not flush to zero.
    assert oracle.mx_value(1, 0) == 2.0 ** -128
    assert oracle.mx_value(7, 0) == 6 * 2.0 ** -127


def test_nibble_order_low_is_even():
    codes = np.zeros((1, 16), np.uint8)
    codes[0, 0] = 0x21          # element 0 = code 1 (0.5), element 1 = code 2 (1.0)
    codes[0, 5] = 0xF0          # element 10 = code 0, element 11 = code 15 (-6)
    out = oracle.mx_decode(codes, np.full((1, 1), 127, np.uint8))
    assert out[0, 0] == 0.5 and out[0, 1] == 1.0
    assert out[0, 10] == 0.0 and out[0, 11] == -6.0
    assert np.count_nonzero(out) == 3


def test_block_index_is_floor_k_over_32():
    codes = np.full((1, 48), 0x22, np.uint8)  # every element code 2 = 1.0
    scales = np.array([[127, 128, 125]], np.uint8)
    out = oracle.mx_decode(codes, scales)
    assert np.all(out[0, :32] == 1.0)
    assert np.all(out[0, 32:64] == 2.0)
    assert np.all(out[0, 64:] == 0.25)


def test_decode_matches_independent_numpy_random():
    rng = np.random.default_rng(5)
    codes = rng.integers(0, 256, (7, 64), dtype=np.uint8)
    scales = rng.integers(0, 255, (7, 4), dtype=np.uint8)
    got = oracle.mx_decode(codes, scales).astype(np.float64)
    want = np_decode_golden(codes, scales).astype(np.float32).astype(np.float64)
    np.testing.assert_array_equal(got, want)


def test_scale_255_rejected():
    with pytest.raises(ValueError):
        oracle.mx_decode(np.zeros((1, 16), np.uint8), np.array([[255]], np.uint8))


def test_size_identity_4_25_bits():
    with open(os.path.join(GOLDEN, "mxfp4_sizes.txt")) as f:
        rows = [l.split() for l in f if l.strip() and not l.startswith("#")]
    for r, c, b in rows:
        r, c, b = int(r), int(c), int(b)
        assert oracle.mx_bytes(r, c) == b
        assert Fraction(8 * b, r * c) == Fraction(17, 4)
    # one expert at H=7168, I=2048 and the decode working set of 9 experts
    per_expert = oracle.mx_bytes(4096, 7168) + oracle.mx_bytes(7168, 2048)
    assert per_expert == 23_396_352
    assert 9 * per_expert == 210_567_168


# ------------------------------------------------------------------ routing pins

def brute_route(l, k):
    """Plain-Python selection: larger first, equal (incl. +-0) by lower index, NaN last."""
    E = len(l)
    order = sorted(range(E), key=lambda e: (math.isnan(l[e]), 0.0 if math.isnan(l[e]) else -l[e], e))
    return order[:k]


def test_route_ties_and_signed_zero_brute_force():
    rng = np.random.default_rng(11)
    vals = np.array([0.0, -0.0, 1.0, -1.0, 0.5, 2.0, 2.0, -3.0], np.float32)
    for trial in range(200):
        E = int(rng.integers(1, 40))
        k = int(rng.integers(1, E + 1))
        l = rng.choice(vals, size=(1, E)).astype(np.float32)
        ids, w = oracle.route(l, k)
        assert ids[0].tolist() == brute_route(l[0].tolist(), k)


def test_route_nan_ranks_last():
    l = np.array([[np.nan, -np.inf, 0.0, np.nan, 1.0, -5.0]], np.float32)
    ids, _ = oracle.route(l, 6)
    assert ids[0].tolist() == [4, 2, 5, 1, 0, 3]


def test_route_weights_invariants():
    rng = np.random.default_rng(12)
    l = rng.standard_normal((64, 256)).astype(np.float32)
    ids, w = oracle.route(l, 8)
    assert np.all(np.abs(w.sum(1) - 1.0) <= 1e-12)
    assert np.all(np.diff(w, axis=1) <= 0)
    # the ratio of two kept weights is exp of their logit difference
    for t in range(64):
        lt = l[t, ids[t]].astype(np.float64)
        for j in range(1, 8):
            assert math.isclose(w[t, 0] / w[t, j], math.exp(lt[0] - lt[j]), rel_tol=1e-12)
    # k = 1 gives weight exactly 1
    _, w1 = oracle.route(l, 1)
    assert np.all(w1 == 1.0)


def test_route_metamorphic_unselected_logits_do_not_matter():
    rng = np.random.default_rng(13)
    l = rng.standard_normal((32, 64)).astype(np.float32)
    ids, w = oracle.route(l, 6)
    l2 = l.copy()
    for t in range(32):
        kth = l[t, ids[t, -1]]
        mask = np.ones(64, bool)
        mask[ids[t]] = False
        l2[t, mask] = np.minimum(l[t, mask], kth) - rng.uniform(0.01, 5.0, mask.sum()).astype(np.float32)
    ids2, w2 = oracle.route(l2, 6)
    np.testing.assert_array_equal(ids, ids2)
    np.testing.assert_array_equal(w, w2)


# ------------------------------------------------------------------ permutation pins

def test_permute_against_python_stable_sort():
    rng = np.random.default_rng(14)
    for trial in range(20):
        T, E = int(rng.integers(0, 50)), int(rng.integers(1, 20))
        k = int(rng.integers(1, E + 1))
        ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32).reshape(T, k)
        off, ss, sp = oracle.permute(ids, E)
        flat = ids.ravel().tolist()
        want_ss = sorted(range(T * k), key=lambda s: flat[s])  # Python sort is stable
        assert ss.tolist() == want_ss
        counts = np.bincount(ids.ravel(), minlength=E)
        assert off.tolist() == [0] + np.cumsum(counts).tolist()
        assert np.all(sp[ss] == np.arange(T * k))


def test_permute_empty_slots_take_no_position():
    # id -1 marks an empty slot: the placed slots sort exactly as if the empty
    # ones were not there, the empty ones get slot_pos -1 and the positions past
    # the placed ones hold -1
    rng = np.random.default_rng(15)
    for trial in range(20):
        T, E = int(rng.integers(1, 40)), int(rng.integers(1, 12))
        k = int(rng.integers(1, 6))
        ids = rng.integers(-1, E, (T, k)).astype(np.int32)
        off, ss, sp = oracle.permute(ids, E)
        flat = ids.ravel().tolist()
        placed = [s for s in range(T * k) if flat[s] != -1]
        want_ss = sorted(placed, key=lambda s: flat[s])
        assert ss[:len(placed)].tolist() == want_ss
        assert np.all(ss[len(placed):] == -1)
        assert off[E] == len(placed)
        counts = np.bincount(ids.ravel()[ids.ravel() >= 0], minlength=E)
        assert off.tolist() == [0] + np.cumsum(counts).tolist()
        assert [sp[s] for s in range(T * k) if flat[s] == -1] == [-1] * (T * k - len(placed))
        assert np.all(sp[np.array(want_ss, np.int64)] == np.arange(len(placed)))


# ------------------------------------------------------------------ expert / layer pins

def silu(z):
    return z / (1.0 + math.exp(-z))


def onehot_mx(rows, cols, positions, code, e=127):
    """MXFP4 matrix with a single nonzero code per row at positions[r]."""
    codes = np.zeros((rows, cols // 2), np.uint8)
    for r, c in enumerate(positions):
        codes[r, c // 2] |= (code << 4) if c % 2 else code
    return codes, np.full((rows, cols // 32), e, np.uint8)


def test_onehot_expert_closed_form():
    H, I = 64, 32
    rng = np.random.default_rng(15)
    a = rng.integers(0, H, I)
    b = rng.integers(0, H, I)
    dn = rng.integers(0, I, H)
    gc, gs = onehot_mx(I, H, a, 2)          # gate row n = e_{a_n} (1.0)
    uc, us = onehot_mx(I, H, b, 5, 128)     # up row n = 3 * 2 * e_{b_n}
    gu_c = np.concatenate([gc, uc])
    gu_s = np.concatenate([gs, us])
    dc, ds = onehot_mx(H, I, dn, 12, 126)   # down row m = -2 * 0.5 * e_{dn_m}
    W = oracle.OracleWeights(H, I, 1, 0)
    W.set_expert(0, gu_c, gu_s, dc, ds)
    x = wl.f32_to_bf16_bits(rng.standard_normal((3, H)).astype(np.float32))
    xf = wl.bf16_bits_to_f32(x).astype(np.float64)
    out, ids, w = oracle.moe_layer(W, x, np.zeros((3, 1), np.float32), 1)
    assert np.all(ids == 0) and np.all(w == 1.0)
    for t in range(3):
        h = [silu(xf[t, a[n]]) * 6.0 * xf[t, b[n]] for n in range(I)]
        want = [-1.0 * h[dn[m]] for m in range(H)]
        np.testing.assert_allclose(out[t], want, rtol=1e-15, atol=0)


def test_silu_known_values():
    # x = e_0 with value 1 through a one-hot gate/up/down: out = silu(1) * 1
    H, I = 32, 32
    gc, gs = onehot_mx(I, H, [0] * I, 2)
    dc, ds = onehot_mx(H, I, [0] * H, 2)
    W = oracle.OracleWeights(H, I, 1, 0)
    W.set_expert(0, np.concatenate([gc, gc]), np.concatenate([gs, gs]), dc, ds)
    for xv, want in ((1.0, 0.7310585786300049), (0.0, 0.0), (-1.0, 0.2689414213699951)):
        x = np.zeros((1, H), np.float32)
        x[0, 0] = xv
        out, _, _ = oracle.moe_layer(W, wl.f32_to_bf16_bits(x), np.zeros((1, 1), np.float32), 1)
        # h = silu(x0) * x0; for x0 = -1 this is -silu(-1) = 0.2689...
        assert math.isclose(out[0, 0], want, rel_tol=1e-15, abs_tol=1e-300)


def numpy_layer(cfg, x_bits, logits, experts):
    """Independent brute force: every expert on every token (numpy FP64), then select."""
    H, I, E, S, k = cfg.hidden, cfg.inter, cfg.n_experts, cfg.n_shared, cfg.k
    x = wl.bf16_bits_to_f32(x_bits).astype(np.float64)
    Y = []
    for e in range(E + S):
        gc, gs, dc, ds = experts[e]
        Wgu = np_decode_golden(gc, gs)
        Wd = np_decode_golden(dc, ds)
        g = x @ Wgu[:I].T
        u = x @ Wgu[I:].T
        h = g / (1.0 + np.exp(-g)) * u
        Y.append(h @ Wd.T)
    out = np.zeros((x.shape[0], H))
    for t in range(x.shape[0]):
        sel = brute_route(logits[t].tolist(), k)
        lv = np.array([float(logits[t, e]) for e in sel])
        p = np.exp(lv - lv.max())
        p /= p.sum()
        for j, e in enumerate(sel):
            out[t] += p[j] * Y[e][t]
        for s in range(S):
            out[t] += Y[E + s][t]
    return out


@pytest.mark.parametrize("cfg", [wl.tiny(), wl.custom("tiny_shared", 12, 96, 64, 5, 1, 3, seed=7)],
                         ids=lambda c: c.name)
def test_layer_brute_force_tiny(cfg):
    x = wl.tokens(cfg)
    l = wl.router_logits(cfg)
    experts = [wl.expert_weights(cfg, e) for e in range(cfg.n_groups)]
    W = oracle.OracleWeights(cfg.hidden, cfg.inter, cfg.n_experts, cfg.n_shared)
    for e, ws in enumerate(experts):
        W.set_expert(e, *ws)
    out, ids, w = oracle.moe_layer(W, x, l, cfg.k, nthreads=2)
    want = numpy_layer(cfg, x, l, experts)
    scale = np.sqrt(np.mean(want ** 2))
    assert np.max(np.abs(out - want)) / scale <= 1e-12


def test_layer_single_expert_is_textbook_swiglu():
    cfg = wl.custom("e1", 5, 128, 96, 1, 0, 1, seed=8)
    x = wl.tokens(cfg)
    gc, gs, dc, ds = wl.expert_weights(cfg, 0)
    W = oracle.OracleWeights(cfg.hidden, cfg.inter, 1, 0)
    W.set_expert(0, gc, gs, dc, ds)
    out, _, _ = oracle.moe_layer(W, x, wl.router_logits(cfg), 1)
    Wgu = np_decode_golden(gc, gs)
    Wd = np_decode_golden(dc, ds)
    xf = wl.bf16_bits_to_f32(x).astype(np.float64)
    g, u = xf @ Wgu[:96].T, xf @ Wgu[96:].T
    want = (g / (1 + np.exp(-g)) * u) @ Wd.T
    assert np.max(np.abs(out - want)) / np.sqrt(np.mean(want ** 2)) <= 1e-12
    # the dense path on the same weights gives the same result
    dense = oracle.dense_ffn(((gc[:96], gs[:96]), (gc[96:], gs[96:]), (dc, ds)), x, 0)
    assert np.max(np.abs(dense - want)) / np.sqrt(np.mean(want ** 2)) <= 1e-12


def test_layer_down_exponent_plus_one_doubles_exactly():
    # Powers of two change exponents exactly ("Cascadia" §3.3): +1 on every
    # down-projection E8M0 exponent doubles the output bit for bit.
    cfg = wl.custom("dbl", 6, 64, 64, 4, 1, 2, seed=9)
    x, l = wl.tokens(cfg), wl.router_logits(cfg)
    W1 = oracle.OracleWeights(64, 64, 4, 1)
    W2 = oracle.OracleWeights(64, 64, 4, 1)
    for e in range(5):
        gc, gs, dc, ds = wl.expert_weights(cfg, e)
        W1.set_expert(e, gc, gs, dc, ds)
        W2.set_expert(e, gc, gs, dc, ds + 1)
    o1, _, _ = oracle.moe_layer(W1, x, l, 2)
    o2, _, _ = oracle.moe_layer(W2, x, l, 2)
    np.testing.assert_array_equal(o2, 2 * o1)


def test_layer_shared_expert_is_added_with_unit_weight():
    cfg = wl.custom("sh", 4, 64, 32, 3, 1, 1, seed=10)
    x, l = wl.tokens(cfg), wl.router_logits(cfg)
    ws = [wl.expert_weights(cfg, e) for e in range(4)]
    with_s = oracle.OracleWeights(64, 32, 3, 1)
    without = oracle.OracleWeights(64, 32, 3, 0)
    only_s = oracle.OracleWeights(64, 32, 1, 0)
    for e in range(3):
        with_s.set_expert(e, *ws[e])
        without.set_expert(e, *ws[e])
    with_s.set_expert(3, *ws[3])
    only_s.set_expert(0, *ws[3])
    a, _, _ = oracle.moe_layer(with_s, x, l, 1)
    b, _, _ = oracle.moe_layer(without, x, l, 1)
    c, _, _ = oracle.moe_layer(only_s, x, np.zeros((4, 1), np.float32), 1)
    np.testing.assert_allclose(a, b + c, rtol=1e-14, atol=1e-14 * np.abs(a).max())


@pytest.mark.parametrize("fmt", ["mxfp4", "bf16"])
def test_dense_slices_equal_unsliced(fmt):
    # Eq. (2) of "Cascadia" §3.4 with 4 slices of 32 over I = 128.
    H, I = 64, 128
    rng = np.random.default_rng(16)
    if fmt == "bf16":
        w = tuple(wl.f32_to_bf16_bits(rng.standard_normal(s).astype(np.float32) * 0.1)
                  for s in ((I, H), (I, H), (H, I)))
    else:
        w = (wl.mx_matrix(rng, I, H, 120, 130), wl.mx_matrix(rng, I, H, 120, 130), wl.mx_matrix(rng, H, I, 120, 130))
    x = wl.f32_to_bf16_bits(rng.standard_normal((3, H)).astype(np.float32))
    full = oracle.dense_ffn(w, x, 0, fmt)
    sliced = oracle.dense_ffn(w, x, 4, fmt)
    assert np.max(np.abs(full - sliced)) / np.sqrt(np.mean(full ** 2)) <= 1e-12
    # and against the textbook FFN in numpy
    if fmt == "bf16":
        Wg, Wu, Wd = (wl.bf16_bits_to_f32(a).astype(np.float64) for a in w)
    else:
        Wg, Wu, Wd = (np_decode_golden(c, s) for c, s in w)
    xf = wl.bf16_bits_to_f32(x).astype(np.float64)
    g, u = xf @ Wg.T, xf @ Wu.T
    want = (g / (1 + np.exp(-g)) * u) @ Wd.T
    assert np.max(np.abs(full - want)) / np.sqrt(np.mean(want ** 2)) <= 1e-12


def test_dense_rejects_slice_cutting_a_block():
    # A slice width that is not a multiple of 32 would cut an MX block.
    H, I = 64, 96
    rng = np.random.default_rng(17)
    w = (wl.mx_matrix(rng, I, H, 127, 127), wl.mx_matrix(rng, I, H, 127, 127), wl.mx_matrix(rng, H, I, 127, 127))
    x = wl.f32_to_bf16_bits(np.ones((1, H), np.float32))
    with pytest.raises(ValueError):
        oracle.dense_ffn(w, x, 2)   # 48-wide slices


# ------------------------------------------------------------------ sigmoid + bias routing pins
# "Cascadia: Resident 975B MoE Inference on Eleven AI PCs" §3.1: sigmoid scores,
# bias-adjusted top-k selection, weights normalised over the selected experts.

def brute_route_sigmoid(l, b, k, scale):
    """Plain-Python: key = sigmoid(l) + b (double), larger first, equal by lower
    index, NaN last; weights = scale * sigmoid(l_j) / sum of the kept sigmoids."""
    E = len(l)
    s = [1.0 / (1.0 + math.exp(-float(v))) if not math.isnan(v) else float("nan") for v in l]
    key = [s[e] + float(b[e]) for e in range(E)]
    order = sorted(range(E), key=lambda e: (math.isnan(key[e]), 0.0 if math.isnan(key[e]) else -key[e], e))
    sel = order[:k]
    tot = sum(s[e] for e in sel)
    return sel, [scale * s[e] / tot for e in sel]


def test_route_sigmoid_brute_force():
    rng = np.random.default_rng(31)
    for trial in range(100):
        E = int(rng.integers(1, 48))
        k = int(rng.integers(1, min(E, 8) + 1))
        l = (rng.standard_normal((3, E)) * 2).astype(np.float32)
        b = (rng.standard_normal(E) * 0.3).astype(np.float32)
        scale = float(rng.uniform(0.5, 3.0))
        ids, w = oracle.route_sigmoid(l, b, k, scale)
        for t in range(3):
            sel, ww = brute_route_sigmoid(l[t].tolist(), b.tolist(), k, scale)
            assert ids[t].tolist() == sel
            np.testing.assert_allclose(w[t], ww, rtol=1e-14, atol=0)


def test_route_sigmoid_zero_bias_selects_like_softmax():
    # sigmoid is increasing, so without a bias the selection is the softmax router's
    rng = np.random.default_rng(32)
    l = rng.standard_normal((64, 128)).astype(np.float32)
    ids_s, w_s = oracle.route_sigmoid(l, None, 6)
    ids_m, _ = oracle.route(l, 6)
    np.testing.assert_array_equal(ids_s, ids_m)
    assert np.all(np.abs(w_s.sum(1) - 1.0) <= 1e-12)
    sig = 1.0 / (1.0 + np.exp(-l.astype(np.float64)))
    for t in range(64):
        ratio = sig[t, ids_s[t]] / sig[t, ids_s[t]].sum()
        np.testing.assert_allclose(w_s[t], ratio, rtol=1e-13)


def test_route_sigmoid_bias_decides_selection_not_weights():
    rng = np.random.default_rng(33)
    l = rng.standard_normal((16, 32)).astype(np.float32)
    b = np.zeros(32, np.float32)
    b[5] = 10.0    # always selected ...
    b[9] = -10.0   # ... never selected
    ids, w = oracle.route_sigmoid(l, b, 4, 2.0)
    assert np.all(ids[:, 0] == 5) and not np.any(ids == 9)
    sig = 1.0 / (1.0 + np.exp(-l.astype(np.float64)))
    for t in range(16):
        np.testing.assert_allclose(w[t], 2.0 * sig[t, ids[t]] / sig[t, ids[t]].sum(), rtol=1e-13)
    assert np.all(np.abs(w.sum(1) - 2.0) <= 1e-12)


def test_route_sigmoid_ties_and_nan():
    l = np.array([[0.5, 0.5, np.nan, -1.0, 0.5]], np.float32)
    ids, _ = oracle.route_sigmoid(l, np.zeros(5, np.float32), 5)
    assert ids[0].tolist() == [0, 1, 4, 3, 2]
    # equal keys from different logits and biases tie exactly only if equal; lower index first
    ids2, _ = oracle.route_sigmoid(np.zeros((1, 4), np.float32), np.array([0.0, 0.25, 0.25, 0.0], np.float32), 2)
    assert ids2[0].tolist() == [1, 2]


# ------------------------------------------------------------------ layer for given routing

def test_layer_routed_equals_layer_on_its_own_routing():
    cfg = wl.custom("rt", 7, 64, 64, 6, 1, 2, seed=34)
    x, l = wl.tokens(cfg), wl.router_logits(cfg)
    W = oracle.OracleWeights(64, 64, 6, 1)
    for e in range(7):
        W.set_expert(e, *wl.expert_weights(cfg, e))
    out, ids, w = oracle.moe_layer(W, x, l, 2)
    np.testing.assert_array_equal(oracle.moe_layer_routed(W, x, ids, w), out)


def test_layer_routed_single_selection_closed_form():
    # one selected expert with weight alpha and no shared expert: alpha times the
    # textbook SwiGLU FFN of that expert, whatever the other experts hold
    cfg = wl.custom("rt1", 5, 96, 64, 3, 0, 1, seed=35)
    x = wl.tokens(cfg)
    ws = [wl.expert_weights(cfg, e) for e in range(3)]
    W = oracle.OracleWeights(96, 64, 3, 0)
    for e in range(3):
        W.set_expert(e, *ws[e])
    ids = np.array([[2], [0], [2], [1], [2]], np.int32)
    alpha = np.array([[0.5], [1.75], [-2.0], [3.0], [0.0]])
    out = oracle.moe_layer_routed(W, x, ids, alpha)
    xf = wl.bf16_bits_to_f32(x).astype(np.float64)
    for t in range(5):
        gc, gs, dc, ds = ws[ids[t, 0]]
        Wgu, Wd = np_decode_golden(gc, gs), np_decode_golden(dc, ds)
        g, u = xf[t] @ Wgu[:64].T, xf[t] @ Wgu[64:].T
        want = alpha[t, 0] * ((g / (1 + np.exp(-g)) * u) @ Wd.T)
        assert np.max(np.abs(out[t] - want)) <= 1e-12 * max(1.0, np.max(np.abs(want)))


def test_layer_routed_is_linear_in_the_weights():
    cfg = wl.custom("rt2", 6, 64, 32, 4, 1, 2, seed=36)
    x = wl.tokens(cfg)
    W = oracle.OracleWeights(64, 32, 4, 1)
    for e in range(5):
        W.set_expert(e, *wl.expert_weights(cfg, e))
    rng = np.random.default_rng(36)
    ids = np.stack([rng.choice(4, 2, replace=False) for _ in range(6)]).astype(np.int32)
    w = rng.uniform(0.1, 1.0, (6, 2))
    shared = oracle.moe_layer_routed(W, x, ids, np.zeros_like(w))
    o1 = oracle.moe_layer_routed(W, x, ids, w) - shared
    o2 = oracle.moe_layer_routed(W, x, ids, 2 * w) - shared
    np.testing.assert_allclose(o2, 2 * o1, rtol=1e-12, atol=1e-12 * np.abs(o1).max())


def test_layer_routed_empty_slot_drops_its_term():
    # an id of -1 leaves the slot's term out of Eq. (1): column 1 empty on every
    # token equals the layer with k = 1 on column 0 alone, and the empty slot's
    # weight (NaN here) is never read
    cfg = wl.custom("rte", 6, 64, 32, 4, 1, 2, seed=38)
    x = wl.tokens(cfg)
    W = oracle.OracleWeights(64, 32, 4, 1)
    for e in range(5):
        W.set_expert(e, *wl.expert_weights(cfg, e))
    ids1 = np.array([[2], [0], [3], [3], [1], [0]], np.int32)
    w1 = np.array([[0.5], [1.25], [0.75], [2.0], [1.0], [0.25]])
    ids2 = np.concatenate([ids1, np.full((6, 1), -1, np.int32)], axis=1)
    w2 = np.concatenate([w1, np.full((6, 1), np.nan)], axis=1)
    np.testing.assert_array_equal(oracle.moe_layer_routed(W, x, ids2, w2), oracle.moe_layer_routed(W, x, ids1, w1))


def test_layer_routed_expert_subsets_sum_to_the_layer():
    # holders of disjoint expert subsets (the other subset's slots empty) each
    # add the shared expert once; their sum less one shared-only pass (every
    # slot empty) is the whole layer
    cfg = wl.custom("rts", 8, 64, 32, 6, 1, 3, seed=39)
    x = wl.tokens(cfg)
    W = oracle.OracleWeights(64, 32, 6, 1)
    for e in range(7):
        W.set_expert(e, *wl.expert_weights(cfg, e))
    rng = np.random.default_rng(39)
    ids = np.stack([rng.choice(6, 3, replace=False) for _ in range(8)]).astype(np.int32)
    w = rng.uniform(0.1, 1.0, (8, 3))
    full = oracle.moe_layer_routed(W, x, ids, w)
    lo = oracle.moe_layer_routed(W, x, np.where(ids < 3, ids, -1).astype(np.int32), w)
    hi = oracle.moe_layer_routed(W, x, np.where(ids >= 3, ids, -1).astype(np.int32), w)
    shared = oracle.moe_layer_routed(W, x, np.full_like(ids, -1), w)
    np.testing.assert_allclose(lo + hi - shared, full, rtol=1e-12, atol=1e-12 * np.abs(full).max())


def test_layer_routed_rejects_ids_out_of_range():
    cfg = wl.custom("rt3", 2, 64, 32, 3, 0, 1, seed=37)
    W = oracle.OracleWeights(64, 32, 3, 0)
    for e in range(3):
        W.set_expert(e, *wl.expert_weights(cfg, e))
    with pytest.raises(ValueError):
        oracle.moe_layer_routed(W, wl.tokens(cfg), np.array([[0], [3]], np.int32), np.ones((2, 1)))


# ------------------------------------------------------------------ group-32 INT4 pins
# "Cascadia: Resident 975B MoE Inference on Eleven AI PCs" §3.1 (packed 4-bit
# nibbles, one FP16 scale per 32-value group) and §3.5 (zero points).  Reading:
# w = s * (q - z), q the unsigned nibble, z the group's zero point (8 when none
# are stored), element 2j in the low nibble of byte j.

FP16_ONE = 0x3C00


def test_fp16_value_every_bit_pattern_matches_numpy():
    bits = np.arange(65536, dtype=np.uint32)
    want = bits.astype(np.uint16).view(np.float16).astype(np.float64)
    got = np.array([oracle.fp16_value(int(b)) for b in bits])
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    np.testing.assert_array_equal(got[~nan], want[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(want[~nan]))


def test_i4_unit_scale_is_code_minus_zero():
    for q in range(16):
        for z in range(16):
            assert oracle.i4_value(q, z, FP16_ONE) == q - z


def test_i4_value_is_exact_product():
    rng = np.random.default_rng(21)
    # normal, subnormal, negative and extreme FP16 scales
    sbits = np.concatenate([rng.integers(0, 0x7C00, 200), rng.integers(0x8000, 0xFC00, 200),
                            [0x0001, 0x03FF, 0x0400, 0x7BFF, 0xFBFF, 0x8001]]).astype(np.uint16)
    for b in sbits:
        s = Fraction(float(np.uint16(b).view(np.float16)))
        q, z = int(rng.integers(0, 16)), int(rng.integers(0, 16))
        assert Fraction(oracle.i4_value(q, z, int(b))) == (q - z) * s, (q, z, hex(b))


def test_i4_nibble_order_low_is_even():
    codes = np.full((1, 16), 0x88, np.uint8)  # every element q = 8 -> 0 with z = 8
    codes[0, 0] = 0x9A          # element 0: q = 10 -> 2, element 1: q = 9 -> 1
    codes[0, 7] = 0x08          # element 14: q = 8 -> 0, element 15: q = 0 -> -8
    out = oracle.i4_decode(codes, np.full((1, 1), FP16_ONE, np.uint16))
    assert out[0, 0] == 2.0 and out[0, 1] == 1.0
    assert out[0, 14] == 0.0 and out[0, 15] == -8.0
    assert np.count_nonzero(out) == 3


def test_i4_group_index_is_floor_k_over_32():
    codes = np.full((1, 48), 0x99, np.uint8)  # every q = 9
    scales = np.array([[0x3C00, 0x4000, 0x3400]], np.uint16)  # 1, 2, 0.25
    zeros = np.array([[8, 7, 13]], np.uint8)
    out = oracle.i4_decode(codes, scales, zeros)
    assert np.all(out[0, :32] == 1.0)
    assert np.all(out[0, 32:64] == 4.0)
    assert np.all(out[0, 64:] == -1.0)


def np_i4_decode(codes, scales, zeros):
    """Independent numpy decode of a group-32 INT4 matrix."""
    q = np.stack([codes & 0xF, codes >> 4], axis=-1).reshape(codes.shape[0], -1).astype(np.int64)
    z = np.repeat(zeros.astype(np.int64), 32, axis=1)
    s = np.repeat(scales.view(np.float16).astype(np.float64), 32, axis=1)
    return (q - z) * s


def test_i4_decode_matches_independent_numpy_random():
    rng = np.random.default_rng(22)
    codes, scales, zeros = wl.i4_matrix(rng, 9, 96, 2.0 ** -20, 2.0 ** 10, 0, 15, signed_scales=True)
    got = oracle.i4_decode(codes, scales, zeros).astype(np.float64)
    np.testing.assert_array_equal(got, np_i4_decode(codes, scales, zeros))
    # without stored zero points every zero point is 8
    np.testing.assert_array_equal(oracle.i4_decode(codes, scales), oracle.i4_decode(codes, scales, np.full_like(zeros, 8)))


@pytest.mark.parametrize("sbits,zero", [(0x7C00, 8), (0xFC00, 8), (0x7E00, 8), (0x7C01, 8), (FP16_ONE, 16),
                                        (FP16_ONE, 255)])
def test_i4_rejects_nonfinite_scale_and_zero_above_15(sbits, zero):
    scales = np.array([[FP16_ONE, sbits]], np.uint16)
    zeros = np.array([[8, zero]], np.uint8)
    with pytest.raises(ValueError):
        oracle.i4_decode(np.zeros((1, 32), np.uint8), scales, zeros)


def test_i4_accepts_zero_15_and_largest_scale():
    out = oracle.i4_decode(np.zeros((1, 16), np.uint8), np.array([[0xFBFF]], np.uint16), np.array([[15]], np.uint8))
    assert np.all(out == 15 * 65504.0)


def test_i4_size_identity():
    with open(os.path.join(GOLDEN, "int4g32_sizes.txt")) as f:
        rows = [l.split() for l in f if l.strip() and not l.startswith("#")]
    for r, c, z, b in rows:
        r, c, z, b = int(r), int(c), int(z), int(b)
        assert oracle.i4_bytes(r, c, bool(z)) == b
        assert Fraction(8 * b, r * c) == (Fraction(19, 4) if z else Fraction(9, 2))


def mx_as_i4(codes, scales):
    """An MXFP4 matrix with E8M0 = 126 (scale 1/2) and magnitudes up to 3 (codes
    0..5 and 8..13), written as group-32 INT4 with scale 1/4: q - z = 4 v."""
    assert np.all(scales == 126)
    v = np_decode_golden(codes, scales)            # multiples of 1/4 in [-1.5, 1.5]
    rng = np.random.default_rng(int(codes.sum()) % 1000)
    zeros = rng.integers(6, 10, size=scales.shape, dtype=np.uint8)
    q = (4 * v).astype(np.int64) + np.repeat(zeros.astype(np.int64), 32, axis=1)
    assert q.min() >= 0 and q.max() <= 15
    q = q.reshape(q.shape[0], -1, 2)
    i4 = (q[..., 0] | (q[..., 1] << 4)).astype(np.uint8)
    return i4, np.full(scales.shape, 0x3400, np.uint16), zeros


def small_mx(rng, rows, cols):
    # codes whose magnitude index is at most 5 (|v| <= 3), every E8M0 = 126
    lo = rng.integers(0, 6, (rows, cols // 2)) | (rng.integers(0, 2, (rows, cols // 2)) << 3)
    hi = rng.integers(0, 6, (rows, cols // 2)) | (rng.integers(0, 2, (rows, cols // 2)) << 3)
    return (lo | (hi << 4)).astype(np.uint8), np.full((rows, cols // 32), 126, np.uint8)


def test_i4_layer_equals_mxfp4_layer_on_equal_weights():
    # the same decoded weights in both formats give the same layer, bit for bit
    cfg = wl.custom("i4eq", 7, 96, 64, 6, 1, 2, seed=23)
    rng = np.random.default_rng(23)
    Wm = oracle.OracleWeights(96, 64, 6, 1)
    Wi = oracle.OracleWeights(96, 64, 6, 1, "int4g32")
    for e in range(7):
        gc, gs = small_mx(rng, 128, 96)
        dc, ds = small_mx(rng, 96, 64)
        Wm.set_expert(e, gc, gs, dc, ds)
        gi, gsi, gz = mx_as_i4(gc, gs)
        di, dsi, dz = mx_as_i4(dc, ds)
        np.testing.assert_array_equal(oracle.i4_decode(gi, gsi, gz), oracle.mx_decode(gc, gs))
        Wi.set_expert(e, gi, gsi, di, dsi, gz, dz)
    x, l = wl.tokens(cfg), wl.router_logits(cfg)
    a, ia, wa = oracle.moe_layer(Wm, x, l, 2)
    b, ib, wb = oracle.moe_layer(Wi, x, l, 2)
    np.testing.assert_array_equal(ia, ib)
    np.testing.assert_array_equal(a, b)


def test_i4_layer_brute_force_tiny():
    cfg = wl.custom("i4bf", 10, 64, 96, 5, 1, 3, seed=24)
    rng = np.random.default_rng(24)
    W = oracle.OracleWeights(64, 96, 5, 1, "int4g32")
    dec = []
    for e in range(6):
        gu = wl.i4_matrix(rng, 192, 64, 2.0 ** -7, 2.0 ** -3, 4, 12, signed_scales=True)
        dn = wl.i4_matrix(rng, 64, 96, 2.0 ** -7, 2.0 ** -3, 4, 12)
        W.set_expert(e, gu[0], gu[1], dn[0], dn[1], gu[2], dn[2])
        dec.append((np_i4_decode(*gu), np_i4_decode(*dn)))
    x, l = wl.tokens(cfg), wl.router_logits(cfg)
    out, ids, w = oracle.moe_layer(W, x, l, 3)
    xf = wl.bf16_bits_to_f32(x).astype(np.float64)
    want = np.zeros_like(out)
    for t in range(cfg.T):
        sel = brute_route(l[t].tolist(), 3)
        lv = np.array([float(l[t, e]) for e in sel])
        p = np.exp(lv - lv.max())
        p /= p.sum()
        for j, e in enumerate(list(sel) + [5]):
            Wgu, Wd = dec[e]
            g, u = xf[t] @ Wgu[:96].T, xf[t] @ Wgu[96:].T
            want[t] += (p[j] if j < 3 else 1.0) * ((g / (1 + np.exp(-g)) * u) @ Wd.T)
    assert np.max(np.abs(out - want)) / np.sqrt(np.mean(want ** 2)) <= 1e-12


def test_i4_dense_slices_equal_unsliced_and_textbook():
    H, I = 64, 128
    rng = np.random.default_rng(25)
    w = tuple(wl.i4_matrix(rng, r, c, 2.0 ** -7, 2.0 ** -4, 5, 11) for r, c in ((I, H), (I, H), (H, I)))
    x = wl.f32_to_bf16_bits(rng.standard_normal((3, H)).astype(np.float32))
    full = oracle.dense_ffn(w, x, 0, "int4g32")
    sliced = oracle.dense_ffn(w, x, 4, "int4g32")
    Wg, Wu, Wd = (np_i4_decode(*m) for m in w)
    xf = wl.bf16_bits_to_f32(x).astype(np.float64)
    g, u = xf @ Wg.T, xf @ Wu.T
    want = (g / (1 + np.exp(-g)) * u) @ Wd.T
    scale = np.sqrt(np.mean(want ** 2))
    assert np.max(np.abs(full - want)) / scale <= 1e-12
    assert np.max(np.abs(full - sliced)) / scale <= 1e-12


def onehot_i4(rows, cols, positions, q, scale, z):
    """INT4 matrix with one nonzero weight per row (code q at positions[r], code z
    elsewhere, so that every other weight is 0), FP16 scale `scale`, zero point z."""
    codes = np.full((rows, cols), z, np.uint8)
    for r, c in enumerate(positions):
        codes[r, c] = q
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    sbits = np.float16(scale).view(np.uint16)
    return packed, np.full((rows, cols // 32), sbits, np.uint16), np.full((rows, cols // 32), z, np.uint8)


def test_i4_onehot_expert_closed_form():
    # non-power-of-two FP16 scales: the weights are exactly (q - z) * float(fp16(scale))
    H, I = 64, 32
    rng = np.random.default_rng(26)
    a, b, dn = rng.integers(0, H, I), rng.integers(0, H, I), rng.integers(0, I, H)
    sg, su, sd = (float(np.float16(v)) for v in (0.3, -1.7, 0.0123))
    gc, gs, gz = onehot_i4(I, H, a, 11, 0.3, 9)     # gate row n = 2 * sg * e_{a_n}
    uc, us, uz = onehot_i4(I, H, b, 0, -1.7, 5)     # up row n = -5 * su * e_{b_n}
    dc, ds, dz = onehot_i4(H, I, dn, 15, 0.0123, 2)  # down row m = 13 * sd * e_{dn_m}
    W = oracle.OracleWeights(H, I, 1, 0, "int4g32")
    W.set_expert(0, np.concatenate([gc, uc]), np.concatenate([gs, us]), dc, ds, np.concatenate([gz, uz]), dz)
    x = wl.f32_to_bf16_bits(rng.standard_normal((3, H)).astype(np.float32))
    xf = wl.bf16_bits_to_f32(x).astype(np.float64)
    out, ids, w = oracle.moe_layer(W, x, np.zeros((3, 1), np.float32), 1)
    for t in range(3):
        h = [silu(2 * sg * xf[t, a[n]]) * (-5 * su) * xf[t, b[n]] for n in range(I)]
        want = [13 * sd * h[dn[m]] for m in range(H)]
        np.testing.assert_allclose(out[t], want, rtol=1e-14, atol=0)
