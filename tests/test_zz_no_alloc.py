"""moe_route_static: routing and grouping with the library's fixed device
scratch and no allocation.  Its results must equal those moe_forward writes
through MoeRoutingOut on the same logits, and match the oracle's routing and
stable permutation bit for bit (weights within 1e-6); its device-side error
flag, read by moe_route_static_status, stays clear.

Named to be collected last, so the GPU test runs both after every other test
in the session and (run on its own) in a fresh process.
"""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
from parity_util import TOL_W
from mxfp4_routed_expert_router_gb300 import workloads as wl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "mxfp4_routed_expert_router_gb300", "csrc", "route_static.cu")
MAX_SLOTS = 65536
MAX_EXPERTS = 1024


def _lib():
    from mxfp4_routed_expert_router_gb300 import binding
    return binding


def test_limits_match_header():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    assert re.search(r"#define MOE_ROUTE_STATIC_MAX_EXPERTS\s+%d\b" % MAX_EXPERTS, src)
    assert re.search(r"#define MOE_ROUTE_STATIC_MAX_SLOTS\s+%d\b" % MAX_SLOTS, src)


def test_source_calls_no_allocator():
    code = re.sub(r"//[^\n]*|/\*.*?\*/", "", open(SRC).read(), flags=re.S)
    banned = r"\b(cudaMalloc\w*|cudaFree\w*|cudaHostAlloc|cuMemAlloc\w*|cuMemCreate|cuMemFree\w*|malloc|calloc|realloc)\s*\("
    assert not re.search(banned, code)
    assert not re.search(r"\bnew\s+[A-Za-z_]", code)
    assert "static __device__ __align__(256)" in code
    assert "cudaGetSymbolAddress" in code


def test_sizes_beyond_the_scratch_are_rejected_before_any_launch():
    B = _lib()
    L = B.lib
    # these are refused by the host-side checks, before any CUDA call
    assert L.moe_route_static(None, MAX_SLOTS // 4 + 1, 64, 4, None, None, None, None, None, None) == B.MOE_EINVAL
    assert "fixed scratch limit" in B.moe_last_error()
    assert L.moe_route_static(None, 8, MAX_EXPERTS + 1, 4, None, None, None, None, None, None) == B.MOE_EINVAL
    assert L.moe_route_static(None, 8, 64, 0, None, None, None, None, None, None) == B.MOE_EINVAL
    assert L.moe_route_static(None, 8, 4, 5, None, None, None, None, None, None) == B.MOE_EINVAL
    assert L.moe_route_static(None, -1, 64, 4, None, None, None, None, None, None) == B.MOE_EINVAL
    assert L.moe_route_static(None, 8, 64, 4, None, None, None, None, None, None) == B.MOE_EINVAL
    assert "NULL" in B.moe_last_error()
    assert L.moe_route_static(None, 0, 64, 4, None, None, None, None, None, None) == B.MOE_OK


def _routing_buffers(torch, T, E, k):
    return (torch.full((T, k), -7, dtype=torch.int32, device="cuda"),
            torch.full((T, k), -7.0, dtype=torch.float32, device="cuda"),
            torch.full((E + 1,), -7, dtype=torch.int32, device="cuda"),
            torch.full((T * k,), -7, dtype=torch.int32, device="cuda"),
            torch.full((T * k,), -7, dtype=torch.int32, device="cuda"))


def _forward_routing(torch, B, L, cfg, x_bits, logits, k):
    from mxfp4_routed_expert_router_gb300 import layer
    T = x_bits.shape[0]
    bufs = _routing_buffers(torch, T, cfg.n_experts, k)
    L.forward(layer.bf16_tensor(x_bits), torch.from_numpy(logits).cuda(), k, routing=B.routing_out(*bufs))
    L.sync()
    return [b.cpu().numpy() for b in bufs]


def _assert_oracle(static, logits, E, k):
    ids, w, off, ss, sp = static
    rid, rw = oracle.route(logits, k)
    np.testing.assert_array_equal(ids, rid)
    assert np.max(np.abs(w - rw)) <= TOL_W
    roff, rss, rsp = oracle.permute(rid, E)
    np.testing.assert_array_equal(off, roff)
    np.testing.assert_array_equal(ss, rss)
    np.testing.assert_array_equal(sp, rsp)


def _assert_same(static, ref):
    ids, w, off, ss, sp = static
    rids, rw, roff, rss, rsp = ref
    np.testing.assert_array_equal(ids, rids)
    assert np.max(np.abs(w - rw)) <= TOL_W
    np.testing.assert_array_equal(off, roff)
    np.testing.assert_array_equal(ss, rss)
    np.testing.assert_array_equal(sp, rsp)


@pytest.mark.gpu
def test_route_static_matches_forward_routing_two_calls_in_a_row():
    import torch
    from mxfp4_routed_expert_router_gb300 import layer
    B = _lib()
    E, k = 64, 4
    # the larger call first: the second, smaller one must not see its counts
    cases = [wl.custom("no_alloc_a", 517, 256, 128, E, 0, k, seed=41, logits="zipf"),
             wl.custom("no_alloc_b", 9, 256, 128, E, 0, k, seed=42)]
    L = layer.MoeLayer(cases[0], k_max=k)
    inputs = [(wl.tokens(c), wl.router_logits(c)) for c in cases]
    refs = [_forward_routing(torch, B, L, cases[0], x, lg, k) for x, lg in inputs]

    outs = []
    for (x, lg), c in zip(inputs, cases):
        bufs = _routing_buffers(torch, c.T, E, k)
        B.moe_route_static(torch.from_numpy(lg).cuda(), c.T, E, k, *bufs)
        outs.append(bufs)
    B.moe_route_static_status()
    for bufs, ref, (x, lg) in zip(outs, refs, inputs):
        got = [b.cpu().numpy() for b in bufs]
        _assert_same(got, ref)
        _assert_oracle(got, lg, E, k)
    L.free()


@pytest.mark.gpu
def test_route_static_at_the_slot_limit():
    import torch
    from mxfp4_routed_expert_router_gb300 import layer
    B = _lib()
    E, k = 128, 4
    T = MAX_SLOTS // k
    cfg = wl.custom("no_alloc_max", T, 256, 128, E, 0, k, seed=43, logits="biased")
    L = layer.MoeLayer(cfg, k_max=k)
    x, lg = wl.tokens(cfg), wl.router_logits(cfg)
    ref = _forward_routing(torch, B, L, cfg, x, lg, k)
    L.free()
    lg_d = torch.from_numpy(lg).cuda()
    for _ in range(2):
        bufs = _routing_buffers(torch, T, E, k)
        B.moe_route_static(lg_d, T, E, k, *bufs)
        B.moe_route_static_status()
        got = [b.cpu().numpy() for b in bufs]
        _assert_same(got, ref)
        _assert_oracle(got, lg, E, k)
    with pytest.raises(B.MoeError) as e:
        B.moe_route_static(lg_d, T + 1, E, k, *_routing_buffers(torch, 1, E, k))
    assert e.value.status == B.MOE_EINVAL and "fixed scratch limit" in str(e.value)
