"""Tensor parallelism over the intermediate dimension, on the CPU.

The split rests on the sum-over-slices identity of the dense FFN ("Cascadia:
Resident 975B MoE Inference on Eleven AI PCs" §3.4, Eq. 2): every feature n of
an expert's SwiGLU block uses gate row n, up row n and down column n only, so
the layer output is the sum of the layers restricted to disjoint feature
ranges.  These tests check the host logic that cuts the weights (byte ranges
that tile every array exactly) and, over two gloo ranks, that the oracle's
per-rank partial layers reduced by an all-reduce give the full layer."""
import multiprocessing as mp
import socket

import numpy as np
import pytest

import oracle
from mxfp4_routed_expert_router_gb300 import tp
from mxfp4_routed_expert_router_gb300 import workloads as wl

CFG = wl.custom("tp_T24_H256_I224_E8_S1_k3", 24, 256, 224, 8, 1, 3, seed=81)


@pytest.mark.parametrize("inter,world", [(2048, 1), (2048, 2), (2048, 4), (2048, 8), (224, 2), (224, 3), (96, 3),
                                         (2048, 3), (18432, 8)])
def test_shard_ranges_tile_the_features(inter, world):
    r = tp.shard_ranges(inter, world)
    assert len(r) == world and r[0][0] == 0 and r[-1][1] == inter
    for (a0, a1), (b0, _) in zip(r, r[1:]):
        assert a1 == b0
    widths = [f1 - f0 for f0, f1 in r]
    assert all(w > 0 and w % 32 == 0 for w in widths)
    assert max(widths) - min(widths) <= 32
    assert widths == sorted(widths, reverse=True)


@pytest.mark.parametrize("inter,world", [(100, 2), (64, 3), (2048, 0)])
def test_shard_ranges_reject(inter, world):
    with pytest.raises(ValueError):
        tp.shard_ranges(inter, world)


def test_shard_mx_expert_rejects_unaligned_ranges():
    gc, gs, dc, ds = wl.expert_weights(CFG, 0)
    for f0, f1 in ((16, 64), (0, 48), (64, 64), (0, 256)):
        with pytest.raises(ValueError):
            tp.shard_mx_expert(gc, gs, dc, ds, CFG.inter, f0, f1)


@pytest.mark.parametrize("world", [2, 3])
def test_shards_tile_every_weight_byte(world):
    """Each rank's arrays are exactly the expected byte ranges of the full
    arrays, and the ranks' ranges together cover every byte once."""
    H, I = CFG.hidden, CFG.inter
    gc, gs, dc, ds = wl.expert_weights(CFG, 5)
    seen = [np.zeros(a.shape, np.int32) for a in (gc, gs, dc, ds)]
    total = 0
    for f0, f1 in tp.shard_ranges(I, world):
        sg, ss, sdc, sds = tp.shard_mx_expert(gc, gs, dc, ds, I, f0, f1)
        w = f1 - f0
        assert sg.shape == (2 * w, H // 2) and ss.shape == (2 * w, H // 32)
        assert sdc.shape == (H, w // 2) and sds.shape == (H, w // 32)
        assert all(a.flags.c_contiguous for a in (sg, ss, sdc, sds))
        # gate rows first, then up rows, both in feature order
        assert np.array_equal(sg[:w], gc[f0:f1]) and np.array_equal(sg[w:], gc[I + f0:I + f1])
        assert np.array_equal(ss[:w], gs[f0:f1]) and np.array_equal(ss[w:], gs[I + f0:I + f1])
        # down: code bytes [f0/2, f1/2) and scale bytes [f0/32, f1/32) of every row
        assert np.array_equal(sdc, dc[:, f0 // 2:f1 // 2]) and np.array_equal(sds, ds[:, f0 // 32:f1 // 32])
        seen[0][f0:f1] += 1
        seen[0][I + f0:I + f1] += 1
        seen[1][f0:f1] += 1
        seen[1][I + f0:I + f1] += 1
        seen[2][:, f0 // 2:f1 // 2] += 1
        seen[3][:, f0 // 32:f1 // 32] += 1
        total += sum(a.nbytes for a in (sg, ss, sdc, sds))
    assert all(np.all(s == 1) for s in seen)
    assert total == sum(a.nbytes for a in (gc, gs, dc, ds)) == oracle.mx_bytes(2 * I, H) + oracle.mx_bytes(H, I)


def _oracle_full(cfg, x, logits):
    W = oracle.OracleWeights(cfg.hidden, cfg.inter, cfg.n_experts, cfg.n_shared)
    for e in range(cfg.n_groups):
        W.set_expert(e, *wl.expert_weights(cfg, e))
    return oracle.moe_layer(W, x, logits, cfg.k)


def _oracle_partial(cfg, f0, f1, x, logits):
    sc = tp.shard_config(cfg, f0, f1)
    W = oracle.OracleWeights(sc.hidden, sc.inter, sc.n_experts, sc.n_shared)
    for e, w in enumerate(tp.shard_weights(cfg, f0, f1)):
        W.set_expert(e, *w)
    return oracle.moe_layer(W, x, logits, cfg.k)


def test_partial_layers_sum_to_the_layer_single_process():
    x, logits = wl.tokens(CFG), wl.router_logits(CFG)
    full, ids, w = _oracle_full(CFG, x, logits)
    acc = np.zeros_like(full)
    for f0, f1 in tp.shard_ranges(CFG.inter, 3):
        part, pids, pw = _oracle_partial(CFG, f0, f1, x, logits)
        assert np.array_equal(pids, ids) and np.array_equal(pw, w)
        acc += part
    rms = np.sqrt(np.mean(full ** 2))
    assert np.max(np.abs(acc - full)) <= 1e-12 * rms


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _tp_rank(rank, world, port, q):
    import torch
    import torch.distributed as dist
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        f0, f1 = tp.shard_ranges(CFG.inter, world)[rank]
        x, logits = wl.tokens(CFG), wl.router_logits(CFG)
        part, ids, _ = _oracle_partial(CFG, f0, f1, x, logits)
        t = torch.from_numpy(part.copy())
        dist.all_reduce(t, op=dist.ReduceOp.SUM)
        q.put((rank, (f0, f1), part, t.numpy(), ids))
    finally:
        dist.destroy_process_group()


def test_two_rank_all_reduce_gives_the_layer_over_gloo():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_tp_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = {}
    for _ in procs:
        rank, rng, part, reduced, ids = q.get(timeout=300)
        got[rank] = (rng, part, reduced, ids)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [got[r][0] for r in range(world)] == [(0, 128), (128, 224)]
    x, logits = wl.tokens(CFG), wl.router_logits(CFG)
    full, ids, _ = _oracle_full(CFG, x, logits)
    rms = np.sqrt(np.mean(full ** 2))
    for r in range(world):
        assert np.array_equal(got[r][3], ids)
        # every rank holds the same reduced output, equal to the full layer
        assert np.max(np.abs(got[r][2] - full)) <= 1e-12 * rms
        # and no rank's partial alone is the layer
        assert np.max(np.abs(got[r][1] - full)) > 1e-3 * rms
