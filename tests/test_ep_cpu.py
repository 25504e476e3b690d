"""Expert parallelism, host side: the expert ranges, the routing a holder of a
range runs (its own indices, -1 elsewhere) and, through the oracle, that the
holders' partial layers add up to the layer -- in one process and over two
gloo ranks with an all-reduce.  The oracle's -1 empty slot leaves a term out of
Eq. (1) of "Cascadia: Resident 975B MoE Inference on Eleven AI PCs" §3.3, so
the partials of disjoint expert ranges (the shared experts on rank 0 only)
sum to the whole sum."""
import multiprocessing as mp
import socket

import numpy as np
import pytest

import oracle
from mxfp4_routed_expert_router_gb300 import ep
from mxfp4_routed_expert_router_gb300 import workloads as wl

CFG = wl.custom("ep_T9_H64_I64_E7_S1_k3", 9, 64, 64, 7, 1, 3, seed=91)


@pytest.mark.parametrize("E,world", [(7, 1), (7, 2), (7, 3), (7, 7), (256, 8), (10, 4)])
def test_expert_ranges_tile_the_experts(E, world):
    r = ep.expert_ranges(E, world)
    assert len(r) == world and r[0][0] == 0 and r[-1][1] == E
    assert all(a[1] == b[0] for a, b in zip(r, r[1:]))
    sizes = [e1 - e0 for e0, e1 in r]
    assert min(sizes) >= 1 and max(sizes) - min(sizes) <= 1 and sizes == sorted(sizes, reverse=True)


@pytest.mark.parametrize("E,world", [(4, 5), (4, 0)])
def test_expert_ranges_reject(E, world):
    with pytest.raises(ValueError):
        ep.expert_ranges(E, world)


def test_local_routing_maps_own_experts_and_empties_the_rest():
    ids = np.array([[0, 3, 6], [2, -1, 5], [4, 4, 1]], np.int32)
    np.testing.assert_array_equal(ep.local_routing(ids, 2, 5), [[-1, 1, -1], [0, -1, -1], [2, 2, -1]])
    np.testing.assert_array_equal(ep.local_routing(ids, 0, 7), ids)
    # every non-empty slot is held by exactly one range
    held = sum((ep.local_routing(ids, e0, e1) >= 0).astype(int) for e0, e1 in ep.expert_ranges(7, 3))
    np.testing.assert_array_equal(held, (ids >= 0).astype(int))


def test_rank_groups_put_the_shared_experts_on_rank_0():
    assert ep.rank_groups(CFG, 0, 3) == [0, 1, 2, 7]
    assert ep.rank_groups(CFG, 1, 3) == [3, 4]
    assert ep.rank_groups(CFG, 2, 3) == [5, 6]


def _routing(cfg):
    ids, w = oracle.route(wl.router_logits(cfg), cfg.k)
    return ids, w


def _oracle_partial(cfg, rank, world, x, ids, w):
    e0, e1 = ep.expert_ranges(cfg.n_experts, world)[rank]
    groups = ep.rank_groups(cfg, rank, world)
    W = oracle.OracleWeights(cfg.hidden, cfg.inter, e1 - e0, len(groups) - (e1 - e0))
    for i, g in enumerate(groups):
        W.set_expert(i, *wl.expert_weights(cfg, g))
    return oracle.moe_layer_routed(W, x, ep.local_routing(ids, e0, e1), w)


def _oracle_full(cfg, x, ids, w):
    W = oracle.OracleWeights(cfg.hidden, cfg.inter, cfg.n_experts, cfg.n_shared)
    for g in range(cfg.n_groups):
        W.set_expert(g, *wl.expert_weights(cfg, g))
    return oracle.moe_layer_routed(W, x, ids, w)


@pytest.mark.parametrize("world", [2, 3, 7])
def test_partial_layers_sum_to_the_layer_single_process(world):
    x = wl.tokens(CFG)
    ids, w = _routing(CFG)
    full = _oracle_full(CFG, x, ids, w)
    acc = sum(_oracle_partial(CFG, r, world, x, ids, w) for r in range(world))
    rms = np.sqrt(np.mean(full ** 2))
    assert np.max(np.abs(acc - full)) <= 1e-12 * rms


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _ep_rank(rank, world, port, q):
    import torch
    import torch.distributed as dist
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        x = wl.tokens(CFG)
        ids, w = _routing(CFG)
        part = _oracle_partial(CFG, rank, world, x, ids, w)
        t = torch.from_numpy(part.copy())
        dist.all_reduce(t, op=dist.ReduceOp.SUM)
        q.put((rank, ep.expert_ranges(CFG.n_experts, world)[rank], part, t.numpy()))
    finally:
        dist.destroy_process_group()


def test_two_rank_all_reduce_gives_the_layer_over_gloo():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_ep_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = {}
    for _ in procs:
        rank, rng, part, reduced = q.get(timeout=300)
        got[rank] = (rng, part, reduced)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [got[r][0] for r in range(world)] == [(0, 4), (4, 7)]
    x = wl.tokens(CFG)
    ids, w = _routing(CFG)
    full = _oracle_full(CFG, x, ids, w)
    rms = np.sqrt(np.mean(full ** 2))
    for r in range(world):
        # every rank holds the same reduced output, equal to the full layer
        assert np.max(np.abs(got[r][2] - full)) <= 1e-12 * rms
        # and no rank's partial alone is the layer
        assert np.max(np.abs(got[r][1] - full)) > 1e-3 * rms
