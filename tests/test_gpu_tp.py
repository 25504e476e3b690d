"""Tensor-parallel shards of a routed MXFP4 layer, on one GPU.

Each rank's handle holds the intermediate features [f0, f1) of every expert
(gate rows, up rows and down columns with their E8M0 scales) and runs the whole
layer on that slice.  On one GPU the ranks run one after the other; their
partial outputs must each match the oracle's partial layer, and their sum the
oracle's full layer (the sum-over-slices identity of "Cascadia: Resident 975B
MoE Inference on Eleven AI PCs" §3.4, Eq. 2).  Between GPUs that sum is one
all-reduce, which the gloo test on the CPU covers."""
import numpy as np
import pytest
import torch

import oracle
from parity_util import NTHREADS, TOL, oracle_moe, rel_err

from mxfp4_routed_expert_router_gb300 import tp
from mxfp4_routed_expert_router_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

CASES = [
    (wl.custom("tp_T1_H7168_I2048_E16_S1_k8", 1, 7168, 2048, 16, 1, 8, seed=82), 2),   # single-kernel decode
    (wl.custom("tp_T24_H256_I224_E8_S1_k3", 24, 256, 224, 8, 1, 3, seed=81), 3),       # uneven shards 96/64/64
    (wl.custom("tp_T300_H512_I256_E32_S2_k6", 300, 512, 256, 32, 2, 6, seed=83), 2),   # tensor-core path
]


def _oracle_partial(cfg, f0, f1, x, logits):
    sc = tp.shard_config(cfg, f0, f1)
    ids, _ = oracle.route(logits, cfg.k)
    needed = set(np.unique(ids).tolist()) | set(range(cfg.n_experts, cfg.n_groups))
    W = oracle.OracleWeights(sc.hidden, sc.inter, sc.n_experts, sc.n_shared)
    for e in sorted(needed):
        W.set_expert(e, *tp.shard_mx_expert(*wl.expert_weights(cfg, e), cfg.inter, f0, f1))
    return oracle.moe_layer(W, x, logits, cfg.k, nthreads=NTHREADS)[0]


@pytest.mark.parametrize("cfg,world", CASES, ids=[c.name for c, _ in CASES])
def test_shards_sum_to_the_layer(cfg, world):
    from mxfp4_routed_expert_router_gb300.layer import bf16_tensor

    x_bits, logits = wl.tokens(cfg), wl.router_logits(cfg)
    x, lg = bf16_tensor(x_bits), torch.from_numpy(logits).cuda()
    total = torch.zeros((cfg.T, cfg.hidden), dtype=torch.float32, device="cuda")
    for rank in range(world):
        r = tp.TensorParallelMoe(cfg, rank, world)
        try:
            part = r.forward(x, lg)
            torch.cuda.synchronize()
            ref = _oracle_partial(cfg, r.f0, r.f1, x_bits, logits)
            assert rel_err(part.cpu().numpy(), ref) <= TOL, (rank, r.f0, r.f1)
            total += part
        finally:
            r.free()
    torch.cuda.synchronize()
    full = oracle_moe(cfg, x_bits, logits, np.arange(cfg.T))
    assert rel_err(total.cpu().numpy(), full) <= TOL
