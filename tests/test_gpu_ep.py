"""Expert-parallel shards of a routed MXFP4 layer, on one GPU.

Each rank's handle holds a contiguous range of the routed experts (rank 0 also
the shared ones) and is told its range (moe_set_expert_range); it is given the
layer's whole routing in global expert ids, runs the slots of its own experts
and leaves the others empty.  On one GPU the ranks run one after the other:
every rank's routing copy must be the host mapping (its own indices, -1
elsewhere), its partial output the oracle's partial layer, and the sum of the
partials the oracle's whole layer (Eq. (1) of "Cascadia: Resident 975B MoE
Inference on Eleven AI PCs" §3.3 is a sum over experts).  Between GPUs that sum
is one all-reduce, which the gloo test on the CPU covers."""
import numpy as np
import pytest
import torch

import oracle
from parity_util import NTHREADS, TOL, rel_err

from mxfp4_routed_expert_router_gb300 import ep
from mxfp4_routed_expert_router_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

CASES = [
    (wl.custom("ep_T1_H7168_I2048_E16_S1_k8", 1, 7168, 2048, 16, 1, 8, seed=92), 2),    # single-kernel decode
    (wl.custom("ep_T5_H320_I192_E12_S1_k4", 5, 320, 192, 12, 1, 4, seed=93), 5),        # 2-3 experts a rank < k
    (wl.custom("ep_T600_H288_I160_E16_S1_k4", 600, 288, 160, 16, 1, 4, seed=94), 2),    # tensor-core path
    (wl.custom("ep_T300_H512_I256_E32_S2_k6", 300, 512, 256, 32, 2, 6, seed=95), 3),    # two shared experts
]


def _routing(cfg):
    ids, w = oracle.route(wl.router_logits(cfg), cfg.k)
    return ids, w.astype(np.float32)


def _oracle(cfg, groups, n_routed, x, ids, w):
    W = oracle.OracleWeights(cfg.hidden, cfg.inter, n_routed, len(groups) - n_routed)
    used = set(ids.ravel().tolist()) - {-1}
    for i, g in enumerate(groups):
        if i in used or i >= n_routed:
            W.set_expert(i, *wl.expert_weights(cfg, g))
    return oracle.moe_layer_routed(W, x, ids, w.astype(np.float64), nthreads=NTHREADS)


@pytest.mark.parametrize("cfg,world", CASES, ids=[c.name for c, _ in CASES])
def test_expert_shards_sum_to_the_layer(cfg, world):
    from mxfp4_routed_expert_router_gb300 import binding as B
    from mxfp4_routed_expert_router_gb300.layer import bf16_tensor

    x_bits = wl.tokens(cfg)
    ids, w = _routing(cfg)
    x, ids_d, w_d = bf16_tensor(x_bits), torch.from_numpy(ids).cuda(), torch.from_numpy(w).cuda()
    full = _oracle(cfg, list(range(cfg.n_groups)), cfg.n_experts, x_bits, ids, w)
    rms = np.sqrt(np.mean(full ** 2))
    total = torch.zeros((cfg.T, cfg.hidden), dtype=torch.float32, device="cuda")
    for rank in range(world):
        r = ep.ExpertParallelMoe(cfg, rank, world)
        try:
            rid = torch.full_like(ids_d, -7)
            part = r.forward_routed(x, ids_d, w_d, routing=B.routing_out(topk_ids=rid))
            r.sync()
            lid = ep.local_routing(ids, r.e0, r.e1)
            np.testing.assert_array_equal(rid.cpu().numpy(), lid)
            ref = _oracle(cfg, ep.rank_groups(cfg, rank, world), r.e1 - r.e0, x_bits, lid, w)
            assert np.max(np.abs(part.cpu().numpy() - ref)) / rms <= TOL, (rank, r.e0, r.e1)
            total += part
        finally:
            r.free()
    torch.cuda.synchronize()
    assert rel_err(total.cpu().numpy(), full) <= TOL


def test_expert_range_checks_and_global_ids():
    from mxfp4_routed_expert_router_gb300 import binding as B
    from mxfp4_routed_expert_router_gb300.layer import bf16_tensor

    cfg = CASES[1][0]
    r = ep.ExpertParallelMoe(cfg, 1, 4)     # experts [3, 6) of 12
    try:
        assert (r.e0, r.e1) == (3, 6)
        with pytest.raises(B.MoeError) as ei:
            B.moe_set_expert_range(r.handle, 10, cfg.n_experts)   # [10, 13) is not a part of [0, 12)
        assert ei.value.status == B.MOE_EINVAL
        with pytest.raises(B.MoeError) as ei:
            B.moe_set_expert_range(r.handle, -1, cfg.n_experts)
        assert ei.value.status == B.MOE_EINVAL
        # routing over the handle's own experts is refused on a ranged handle
        x = bf16_tensor(wl.tokens(cfg))
        lg = torch.zeros((cfg.T, 3), dtype=torch.float32, device="cuda")
        n = B.moe_workspace_bytes(r.handle, cfg.T, 2)
        ws = torch.empty(n, dtype=torch.uint8, device="cuda")
        out = torch.empty((cfg.T, cfg.hidden), dtype=torch.float32, device="cuda")
        with pytest.raises(B.MoeError) as ei:
            B.moe_forward(r.handle, x, lg, cfg.T, 2, out, False, ws, n)
        assert ei.value.status == B.MOE_EINVAL
        # an id beyond the layer's experts is a device-side error; the slot runs
        # as the handle's expert 0 with weight 0 and the rest of the layer is kept
        ids, w = _routing(cfg)
        ids[0, 0] = cfg.n_experts
        part = r.forward_routed(x, torch.from_numpy(ids).cuda(), torch.from_numpy(w).cuda())
        with pytest.raises(B.MoeError) as ei:
            r.sync()
        assert ei.value.status == B.MOE_EDEVICE
        lid = ep.local_routing(ids, 3, 6)
        lw = w.copy()
        lid[0, 0], lw[0, 0] = 0, 0.0
        ref = _oracle(cfg, ep.rank_groups(cfg, 1, 4), 3, wl.tokens(cfg), lid, lw)
        full = _oracle(cfg, list(range(cfg.n_groups)), cfg.n_experts, wl.tokens(cfg), *_routing(cfg))
        assert np.max(np.abs(part.cpu().numpy() - ref)) / np.sqrt(np.mean(full ** 2)) <= TOL
    finally:
        r.free()
