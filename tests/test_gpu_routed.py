"""GPU parity of the caller-routed layer and the sigmoid + bias router ("Cascadia:
Resident 975B MoE Inference on Eleven AI PCs" §3.1: routing enters the expert
computation as expert IDs and weights; sigmoid scores, bias-adjusted top-k
selection, weights normalised over the selected experts).

* moe_route_sigmoid: ids bit-exact against the oracle (FP64 keys on both sides),
  weights within 1e-6
* moe_forward_routed: outputs within the layer's bound against the oracle's layer
  for the same routing, on the single-kernel path (one, two and a few tokens)
  and the tensor-core path; bit-identical to moe_forward on moe_forward's own
  routing; an id out of range reports MOE_EDEVICE and runs as weight 0
"""
import numpy as np
import pytest
import torch

import oracle
from parity_util import NTHREADS, TOL, TOL_W, rel_err

from mxfp4_routed_expert_router_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _mods():
    from mxfp4_routed_expert_router_gb300 import binding, layer
    return binding, layer


def _sigmoid_case(T, E, k, seed, logits=None):
    rng = np.random.default_rng(seed)
    if logits is None:
        logits = (rng.standard_normal((T, E)) * 2).astype(np.float32)
    bias = (rng.standard_normal(E) * 0.3).astype(np.float32)
    scale = float(rng.uniform(0.5, 3.0))
    return logits, bias, scale


@pytest.mark.parametrize("T,E,k,seed", [(37, 200, 6, 1), (5, 1024, 8, 2), (64, 16, 16, 3), (9, 33, 1, 4)])
def test_route_sigmoid_matches_oracle(T, E, k, seed):
    B, _ = _mods()
    logits, bias, scale = _sigmoid_case(T, E, k, seed)
    ids = torch.full((T, k), -1, dtype=torch.int32, device="cuda")
    w = torch.full((T, k), -1.0, dtype=torch.float32, device="cuda")
    B.moe_route_sigmoid(torch.from_numpy(logits).cuda(), torch.from_numpy(bias).cuda(), T, E, k, scale, ids, w)
    torch.cuda.synchronize()
    rid, rw = oracle.route_sigmoid(logits, bias, k, scale)
    np.testing.assert_array_equal(ids.cpu().numpy(), rid)
    assert np.max(np.abs(w.cpu().numpy() - rw)) <= TOL_W * max(1.0, scale)


def test_route_sigmoid_ties_nan_and_no_bias():
    B, _ = _mods()
    rng = np.random.default_rng(5)
    vals = np.array([0.0, -0.0, 0.5, 0.5, -1.0, np.nan, 2.0], np.float32)
    T, E, k = 40, 24, 6
    logits = rng.choice(vals, size=(T, E)).astype(np.float32)
    ids = torch.empty((T, k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, k), dtype=torch.float32, device="cuda")
    B.moe_route_sigmoid(torch.from_numpy(logits).cuda(), None, T, E, k, 1.0, ids, w)
    torch.cuda.synchronize()
    rid, rw = oracle.route_sigmoid(logits, None, k, 1.0)
    np.testing.assert_array_equal(ids.cpu().numpy(), rid)
    got = w.cpu().numpy()
    fin = np.isfinite(rw)
    assert np.array_equal(np.isfinite(got), fin)
    assert np.max(np.abs(got[fin] - rw[fin])) <= TOL_W


def _random_routing(T, E, k, seed):
    rng = np.random.default_rng(seed)
    ids = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    w = rng.uniform(-0.5, 1.5, (T, k)).astype(np.float32)
    return ids, w


def _oracle_routed(cfg, x_bits, ids, w):
    W = oracle.OracleWeights(cfg.hidden, cfg.inter, cfg.n_experts, cfg.n_shared)
    for e in sorted(set(ids.ravel().tolist()) - {-1} | set(range(cfg.n_experts, cfg.n_groups))):
        W.set_expert(e, *wl.expert_weights(cfg, e))
    return oracle.moe_layer_routed(W, x_bits, ids, w.astype(np.float64), nthreads=NTHREADS)


ROUTED = [
    wl.custom("routed_T1_H7168_I2048_E8_S1_k4", 1, 7168, 2048, 8, 1, 4, seed=41),
    wl.custom("routed_T2_H320_I192_E16_S1_k3", 2, 320, 192, 16, 1, 3, seed=42),
    wl.custom("routed_T13_H288_I160_E32_S1_k4", 13, 288, 160, 32, 1, 4, seed=43),
    wl.custom("routed_T100_H288_I160_E16_S1_k4", 100, 288, 160, 16, 1, 4, seed=44),
]


@pytest.mark.parametrize("cfg", ROUTED, ids=lambda c: c.name)
def test_forward_routed_matches_oracle(cfg):
    _, layer = _mods()
    L = layer.MoeLayer(cfg)
    x = wl.tokens(cfg)
    ids, w = _random_routing(cfg.T, cfg.n_experts, cfg.k, cfg.seed)
    ids_d, w_d = torch.from_numpy(ids).cuda(), torch.from_numpy(w).cuda()
    rid = torch.full_like(ids_d, -1)
    rw = torch.full_like(w_d, -1.0)
    from mxfp4_routed_expert_router_gb300 import binding as B
    out = L.forward_routed(layer.bf16_tensor(x), ids_d, w_d, routing=B.routing_out(topk_ids=rid, topk_w=rw))
    L.sync()
    np.testing.assert_array_equal(rid.cpu().numpy(), ids)
    np.testing.assert_array_equal(rw.cpu().numpy(), w)
    ref = _oracle_routed(cfg, x, ids, w)
    assert rel_err(out.cpu().numpy(), ref) <= TOL
    L.free()


@pytest.mark.parametrize("cfg", [ROUTED[1], ROUTED[3]], ids=lambda c: c.name)
def test_forward_routed_equals_forward_on_its_routing(cfg):
    B, layer = _mods()
    L = layer.MoeLayer(cfg)
    x = layer.bf16_tensor(wl.tokens(cfg))
    lg = torch.from_numpy(wl.router_logits(cfg)).cuda()
    ids = torch.empty((cfg.T, cfg.k), dtype=torch.int32, device="cuda")
    w = torch.empty((cfg.T, cfg.k), dtype=torch.float32, device="cuda")
    a = L.forward(x, lg, cfg.k, routing=B.routing_out(topk_ids=ids, topk_w=w)).clone()
    b = L.forward_routed(x, ids, w).clone()
    L.sync()
    assert torch.equal(a, b)
    L.free()


@pytest.mark.parametrize("cfg", [ROUTED[1], ROUTED[3]], ids=lambda c: c.name)
def test_forward_routed_id_out_of_range(cfg):
    B, layer = _mods()
    L = layer.MoeLayer(cfg)
    x = wl.tokens(cfg)
    ids, w = _random_routing(cfg.T, cfg.n_experts, cfg.k, cfg.seed + 1)
    ids[0, 1] = cfg.n_experts          # out of range
    if cfg.T > 1:
        ids[cfg.T - 1, 0] = -3         # negative
    out = L.forward_routed(layer.bf16_tensor(x), torch.from_numpy(ids).cuda(), torch.from_numpy(w).cuda())
    with pytest.raises(B.MoeError) as ei:
        L.sync()
    assert ei.value.status == B.MOE_EDEVICE
    # the bad slots ran as expert 0 with weight 0
    ok_ids, ok_w = ids.copy(), w.copy()
    bad = (ids < 0) | (ids >= cfg.n_experts)
    ok_ids[bad] = 0
    ok_w[bad] = 0.0
    ref = _oracle_routed(cfg, x, ok_ids, ok_w)
    assert rel_err(out.cpu().numpy(), ref) <= TOL
    L.free()


# Empty slots (id -1): a holder of a subset of the experts runs the caller's
# routing with the slots of the other experts emptied; each empty slot adds
# nothing and its weight is never read (NaN here).  Cases for both paths: the
# single weight-streaming kernel (T*k <= 16 E, one of them with more than 2048
# slots) and the tensor-memory GEMMs with the chunked permutation (one of them
# over three chunks of 1024 slots).
EMPTY = [
    ROUTED[0],
    ROUTED[1],
    ROUTED[3],
    wl.custom("routed_T300_H288_I160_E160_S1_k8", 300, 288, 160, 160, 1, 8, seed=45),
    wl.custom("routed_T600_H288_I160_E16_S1_k4", 600, 288, 160, 16, 1, 4, seed=46),
]


@pytest.mark.parametrize("cfg", EMPTY, ids=lambda c: c.name)
def test_forward_routed_empty_slots(cfg):
    B, layer = _mods()
    L = layer.MoeLayer(cfg)
    x = wl.tokens(cfg)
    ids, w = _random_routing(cfg.T, cfg.n_experts, cfg.k, cfg.seed + 2)
    rng = np.random.default_rng(cfg.seed + 3)
    # the experts of the other holder (every third one) and a random eighth of
    # the slots are empty; token 0 has no routed slot left
    empty = (ids % 3 == 1) | (rng.random(ids.shape) < 0.125)
    empty[0, :] = True
    ids[empty] = -1
    w[empty] = np.nan
    T, k, E = cfg.T, cfg.k, cfg.n_experts
    dev = dict(device="cuda")
    rid = torch.full((T, k), -7, dtype=torch.int32, **dev)
    rw = torch.full((T, k), -1.0, dtype=torch.float32, **dev)
    off = torch.full((E + 1,), -7, dtype=torch.int32, **dev)
    ss = torch.full((T * k,), -7, dtype=torch.int32, **dev)
    sp = torch.full((T * k,), -7, dtype=torch.int32, **dev)
    out = L.forward_routed(layer.bf16_tensor(x), torch.from_numpy(ids).cuda(), torch.from_numpy(w).cuda(),
                           routing=B.routing_out(topk_ids=rid, topk_w=rw, expert_offsets=off, sorted_slot=ss,
                                                 slot_pos=sp))
    L.sync()
    np.testing.assert_array_equal(rid.cpu().numpy(), ids)
    np.testing.assert_array_equal(rw.cpu().numpy(), np.where(empty, np.float32(0), w))
    roff, rss, rsp = oracle.permute(ids, E)
    np.testing.assert_array_equal(off.cpu().numpy(), roff)
    np.testing.assert_array_equal(ss.cpu().numpy(), rss)
    np.testing.assert_array_equal(sp.cpu().numpy(), rsp)
    got = out.cpu().numpy()
    assert np.all(np.isfinite(got))
    ref = _oracle_routed(cfg, x, ids, w)
    assert rel_err(got, ref) <= TOL
    L.free()
