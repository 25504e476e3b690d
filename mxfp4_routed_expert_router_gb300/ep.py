"""Expert parallelism of the routed MoE layer.

Eq. (1) of "Cascadia: Resident 975B MoE Inference on Eleven AI PCs" §3.3
writes a token's output as a sum over the experts selected for it, each term
its routing weight times that expert's SwiGLU FFN of the token.  The sum splits
over any partition of the experts: rank r holds the routed experts
[e0_r, e1_r) (contiguous, as equal as possible) and rank 0 also the shared
experts (weight 1, added once).  Every rank is given every token row and the
whole routing (the layer's global expert ids and weights), runs the slots of
the experts it holds -- the library turns the others into empty slots
(moe_set_expert_range) -- and the ranks' FP32 partial outputs add up to the
layer: one all-reduce of [T, H] per layer (or a reduce-scatter when each rank
keeps only its own tokens afterwards).

This is the all-gather / local experts / reduce form of expert parallelism;
the all-to-all form (each rank receives only the token rows routed to its
experts) moves fewer bytes when T is large and is not built here.

This module is host logic only: it computes the ranges, picks the rank's
weights, and wraps one rank's library handle; the id mapping, the grouping and
every step of the layer run in libmoe_gb300.so, and the sum across ranks is
torch.distributed's all-reduce (NCCL between GPUs).  The tests run the ranks
one after another on a single device and the all-reduce over gloo on the CPU.
"""
from __future__ import annotations

from typing import List, Tuple

import numpy as np

from . import workloads as wl


def expert_ranges(n_experts: int, world: int) -> List[Tuple[int, int]]:
    """[e0, e1) of every rank: contiguous, covering [0, n_experts), at least one
    expert each, as equal as possible (earlier ranks take the extra ones)."""
    if world < 1 or world > n_experts:
        raise ValueError(f"cannot split {n_experts} experts over {world} ranks")
    base, extra = divmod(n_experts, world)
    out, e0 = [], 0
    for r in range(world):
        n = base + (1 if r < extra else 0)
        out.append((e0, e0 + n))
        e0 += n
    return out


def local_routing(ids: np.ndarray, e0: int, e1: int) -> np.ndarray:
    """The routing a holder of experts [e0, e1) runs, in its own expert
    indices: id - e0 for its experts, -1 (an empty slot) for every other id.
    The library does this mapping on the device; this host copy is for
    checking it."""
    ids = np.asarray(ids, np.int32)
    return np.where((ids >= e0) & (ids < e1), ids - e0, -1).astype(np.int32)


def rank_groups(cfg: wl.LayerConfig, rank: int, world: int) -> List[int]:
    """The layer's expert groups rank `rank` holds, in the order its handle
    numbers them: its routed experts, then (rank 0 only) the shared ones."""
    e0, e1 = expert_ranges(cfg.n_experts, world)[rank]
    shared = list(range(cfg.n_experts, cfg.n_groups)) if rank == 0 else []
    return list(range(e0, e1)) + shared


class ExpertParallelMoe:
    """One rank of a routed layer whose experts are split over the ranks.

    forward_routed() runs the rank's experts on the layer's routing and, when a
    process group is given, sums the partial outputs across ranks in place
    (torch.distributed all-reduce); without one it returns the rank's partial
    output."""

    def __init__(self, cfg: wl.LayerConfig, rank: int, world: int, device: str = "cuda", k_max=None):
        from . import binding as B
        from .layer import u8_tensor, u16_tensor

        if cfg.dense:
            raise ValueError("expert parallelism splits a routed layer")
        self.cfg, self.rank, self.world = cfg, rank, world
        self.e0, self.e1 = expert_ranges(cfg.n_experts, world)[rank]
        self.device = device
        fmt = {"bf16": B.MOE_W_BF16, "mxfp4": B.MOE_W_MXFP4, "int4g32": B.MOE_W_INT4G32}[cfg.weight_format]
        gate_up, down = [], []
        for g in rank_groups(cfg, rank, world):
            w = wl.expert_weights(cfg, g)
            if fmt == B.MOE_W_INT4G32:
                gc, gs, dc, ds, gz, dz = w
                gate_up.append((u8_tensor(gc, device), u16_tensor(gs, device), u8_tensor(gz, device)))
                down.append((u8_tensor(dc, device), u16_tensor(ds, device), u8_tensor(dz, device)))
            else:
                gc, gs, dc, ds = w
                gate_up.append((u8_tensor(gc, device), u8_tensor(gs, device)))
                down.append((u8_tensor(dc, device), u8_tensor(ds, device)))
        c = B.MoeConfig(hidden=cfg.hidden, inter=cfg.inter, n_experts=self.e1 - self.e0,
                        n_shared=cfg.n_shared if rank == 0 else 0, k_max=k_max or cfg.k, n_slices=0, fmt=fmt)
        self.B = B
        self.handle = B.moe_load_weights(c, gate_up, down)
        B.moe_set_expert_range(self.handle, self.e0, cfg.n_experts)
        self._ws = None

    def forward_routed(self, x, topk_ids, topk_w, group=None, routing=None, stream=None):
        """x [T, H] BF16, topk_ids [T, k] int32 (the layer's expert ids or -1),
        topk_w [T, k] float32, all on this rank's device."""
        import torch

        B = self.B
        T, k = topk_ids.shape
        n = B.moe_workspace_bytes(self.handle, T, k)
        if self._ws is None or self._ws.numel() < n:
            self._ws = torch.empty(max(n, 256), dtype=torch.uint8, device=self.device)
        out = torch.empty((T, self.cfg.hidden), dtype=torch.float32, device=self.device)
        B.moe_forward_routed(self.handle, x, topk_ids, topk_w, T, k, out, False, self._ws, n, routing, stream)
        if group is not None:
            import torch.distributed as dist
            dist.all_reduce(out, op=dist.ReduceOp.SUM, group=group)
        return out

    def sync(self, stream=None):
        self.B.moe_sync_status(self.handle, stream)

    def free(self):
        if self.handle:
            self.B.moe_free(self.handle)
            self.handle = None
        self._ws = None
