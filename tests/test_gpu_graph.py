"""GPU: forward calls captured into CUDA graphs (moe_graph_create / launch).

A replay equals the eager call bit for bit on the same inputs, picks up new
inputs written into the captured buffers, and matches the oracle within the
layer's bound.  A padded row bucket ("Cascadia: Resident 975B MoE Inference on
Eleven AI PCs" §3.2: pad the rows to a supported shape, then keep the real
row count; padded rows are routed to an expert a real row uses, with weight 0)
gives real rows that match the oracle run on the unpadded rows alone.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from parity_util import TOL, oracle_moe, oracle_moe_routed, rel_err

from mxfp4_routed_expert_router_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _mods():
    from mxfp4_routed_expert_router_gb300 import binding, layer
    return binding, layer


CASES = [
    wl.custom("graph_T1_H320_I192_E16_S1_k4", 1, 320, 192, 16, 1, 4, seed=51),     # single kernel, two-token class
    wl.custom("graph_T6_H320_I192_E16_S1_k4", 6, 320, 192, 16, 1, 4, seed=52),     # single kernel, local routing
    wl.custom("graph_T100_H288_I160_E16_S1_k4", 100, 288, 160, 16, 1, 4, seed=53),  # tensor-core path
]


@pytest.mark.parametrize("cfg", CASES, ids=lambda c: c.name)
def test_graph_replay_equals_eager_and_takes_new_inputs(cfg):
    B, layer = _mods()
    L = layer.MoeLayer(cfg)
    T, k = cfg.T, cfg.k
    x = layer.bf16_tensor(wl.tokens(cfg))
    lg = torch.from_numpy(wl.router_logits(cfg)).cuda()
    ref = L.forward(x, lg, k).clone()
    out = torch.full((T, cfg.hidden), float("nan"), dtype=torch.float32, device="cuda")
    ws, n = L.workspace(T, k)
    g = B.moe_graph_create(L.handle, x, lg, None, None, T, k, out, False, ws, n)
    try:
        for _ in range(3):
            B.moe_graph_launch(g)
        L.sync()
        assert torch.equal(out, ref)
        assert rel_err(out.cpu().numpy(), oracle_moe(cfg, wl.tokens(cfg), wl.router_logits(cfg), np.arange(T))) <= TOL
        # new inputs in the same buffers
        cfg2 = dataclasses.replace(cfg, seed=cfg.seed + 100, weight_seed=cfg.wseed)  # other tokens and logits, same layer
        x.copy_(layer.bf16_tensor(wl.tokens(cfg2)))
        lg.copy_(torch.from_numpy(wl.router_logits(cfg2)))
        B.moe_graph_launch(g)
        L.sync()
        got = out.clone()
        ref2 = L.forward(x, lg, k).clone()
        L.sync()
        assert torch.equal(got, ref2)
        assert rel_err(got.cpu().numpy(),
                       oracle_moe(cfg2, wl.tokens(cfg2), wl.router_logits(cfg2), np.arange(T))) <= TOL
    finally:
        B.moe_graph_free(g)
    L.free()


@pytest.mark.parametrize("T,Tb,seed", [
    (3, 4, 54),      # single kernel
    (100, 128, 55),  # tensor-core path
])
def test_graph_padded_bucket_with_caller_routing(T, Tb, seed):
    B, layer = _mods()
    E, k = 16, 4
    cfg = wl.custom(f"graph_bucket_T{T}_H320_I192_E16_S1_k4", T, 320, 192, E, 1, k, seed=seed)
    L = layer.MoeLayer(cfg)
    rng = np.random.default_rng(seed)
    ids = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    w = rng.uniform(0.1, 1.0, (T, k)).astype(np.float32)
    x = wl.tokens(cfg)
    ref = L.forward_routed(layer.bf16_tensor(x), torch.from_numpy(ids).cuda(), torch.from_numpy(w).cuda()).clone()
    L.sync()
    # bucket of Tb rows: every padded row repeats row 0's experts with weight 0
    pad = Tb - T
    xb = torch.zeros((Tb, cfg.hidden), dtype=torch.bfloat16, device="cuda")
    xb[:T] = layer.bf16_tensor(x)
    idb = torch.from_numpy(np.concatenate([ids, np.repeat(ids[:1], pad, axis=0)])).cuda()
    wb = torch.from_numpy(np.concatenate([w, np.zeros((pad, k), np.float32)])).cuda()
    out = torch.empty((Tb, cfg.hidden), dtype=torch.float32, device="cuda")
    ws, n = L.workspace(Tb, k)
    g = B.moe_graph_create(L.handle, xb, None, idb, wb, Tb, k, out, False, ws, n)
    try:
        B.moe_graph_launch(g)
        L.sync()
        real = out[:T].cpu().numpy()
        assert rel_err(real, ref.cpu().numpy()) <= TOL
        # the real rows against the oracle on the unpadded rows alone
        assert rel_err(real, oracle_moe_routed(cfg, x, ids, w.astype(np.float64))) <= TOL
    finally:
        B.moe_graph_free(g)
    L.free()


def test_graph_with_host_copies():
    # one launch runs the whole step: x and logits in from pinned host memory, out back
    B, layer = _mods()
    cfg = CASES[0]
    L = layer.MoeLayer(cfg)
    T, k = cfg.T, cfg.k
    x_bits = wl.tokens(cfg)
    lg_np = wl.router_logits(cfg)
    ref = L.forward(layer.bf16_tensor(x_bits), torch.from_numpy(lg_np).cuda(), k).clone()
    L.sync()
    hx = torch.from_numpy(x_bits.view(np.int16)).view(torch.bfloat16).pin_memory()
    hl = torch.from_numpy(lg_np).pin_memory()
    hout = torch.full((T, cfg.hidden), float("nan"), dtype=torch.float32).pin_memory()
    x = torch.empty((T, cfg.hidden), dtype=torch.bfloat16, device="cuda")
    lg = torch.empty((T, cfg.n_experts), dtype=torch.float32, device="cuda")
    out = torch.empty((T, cfg.hidden), dtype=torch.float32, device="cuda")
    ws, n = L.workspace(T, k)
    g = B.moe_graph_create(L.handle, x, lg, None, None, T, k, out, False, ws, n, x_host=hx, logits_host=hl,
                           out_host=hout)
    try:
        B.moe_graph_launch(g)
        L.sync()
        assert torch.equal(hout, ref.cpu())
        assert rel_err(hout.numpy(), oracle_moe(cfg, x_bits, lg_np, np.arange(T))) <= TOL
        # the routing this layer runs with, bit for bit against the oracle
        ids = torch.empty((T, k), dtype=torch.int32, device="cuda")
        L.forward(x, lg, k, routing=B.routing_out(topk_ids=ids))
        L.sync()
        np.testing.assert_array_equal(ids.cpu().numpy(), oracle.route(lg_np, k)[0])
        # the next step's inputs are written into the pinned buffers only
        cfg2 = dataclasses.replace(cfg, seed=cfg.seed + 100, weight_seed=cfg.wseed)
        hx.copy_(torch.from_numpy(wl.tokens(cfg2).view(np.int16)).view(torch.bfloat16))
        hl.copy_(torch.from_numpy(wl.router_logits(cfg2)))
        B.moe_graph_launch(g)
        L.sync()
        ref2 = L.forward(hx.cuda(), hl.cuda(), k).clone()
        L.sync()
        assert torch.equal(hout, ref2.cpu())
        assert rel_err(hout.numpy(),
                       oracle_moe(cfg2, wl.tokens(cfg2), wl.router_logits(cfg2), np.arange(T))) <= TOL
    finally:
        B.moe_graph_free(g)
    L.free()


def test_graph_dense_slices():
    B, layer = _mods()
    cfg = wl.dense(1, "mxfp4")
    L = layer.MoeLayer(cfg)
    x = layer.bf16_tensor(wl.tokens(cfg))
    ref = L.forward(x, None).clone()
    out = torch.empty_like(ref)
    ws, n = L.workspace(1, 0)
    g = B.moe_graph_create(L.handle, x, None, None, None, 1, 0, out, False, ws, n)
    try:
        B.moe_graph_launch(g)
        L.sync()
        assert torch.equal(out, ref)
    finally:
        B.moe_graph_free(g)
    L.free()


def test_graph_rejects_both_routings():
    B, layer = _mods()
    cfg = CASES[0]
    L = layer.MoeLayer(cfg)
    x = layer.bf16_tensor(wl.tokens(cfg))
    lg = torch.from_numpy(wl.router_logits(cfg)).cuda()
    ids = torch.zeros((1, 4), dtype=torch.int32, device="cuda")
    w = torch.zeros((1, 4), dtype=torch.float32, device="cuda")
    out = torch.empty((1, cfg.hidden), dtype=torch.float32, device="cuda")
    ws, n = L.workspace(1, 4)
    with pytest.raises(B.MoeError):
        B.moe_graph_create(L.handle, x, lg, ids, w, 1, 4, out, False, ws, n)
    with pytest.raises(B.MoeError):
        B.moe_graph_create(L.handle, x, None, None, None, 1, 4, out, False, ws, n)
    L.free()
