"""A device-resident MoE (or dense) layer: synthetic weights uploaded with torch,
handed to the C-ABI library, plus a reusable workspace.

torch is used only for device memory and streams; every step of the layer runs
in libmoe_gb300.so through ``binding``.
"""
from __future__ import annotations

import concurrent.futures as cf
from typing import Optional

import numpy as np
import torch

from . import binding as B
from . import workloads as wl


def bf16_tensor(bits: np.ndarray, device="cuda") -> torch.Tensor:
    """BF16 bit patterns (uint16 numpy) -> torch.bfloat16 tensor on `device`."""
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
    return t.to(device) if device != "cpu" else t


def u8_tensor(a: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def u16_tensor(a: np.ndarray, device="cuda") -> torch.Tensor:
    """16-bit patterns (e.g. FP16 scale bits) as an int16 tensor, bits unchanged."""
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint16).view(np.int16)).to(device)


class MoeLayer:
    """Owns a library handle for one synthetic layer configuration."""

    def __init__(self, cfg: wl.LayerConfig, device: str = "cuda", k_max: Optional[int] = None, stream=None):
        self.cfg = cfg
        self.device = torch.device(device)
        self.dense = cfg.dense
        self._ws = None
        self.handle = None
        fmt = {"bf16": B.MOE_W_BF16, "mxfp4": B.MOE_W_MXFP4, "int4g32": B.MOE_W_INT4G32}[cfg.weight_format]
        if cfg.dense:
            c = B.MoeConfig(hidden=cfg.hidden, inter=cfg.inter, n_experts=cfg.n_slices, n_shared=0, k_max=0,
                            n_slices=cfg.n_slices, fmt=fmt)
            g, u, d = wl.dense_weights(cfg)
            if fmt == B.MOE_W_BF16:
                staged = [(bf16_tensor(a, device), None) for a in (g, u, d)]
            elif fmt == B.MOE_W_INT4G32:
                staged = [(u8_tensor(a[0], device), u16_tensor(a[1], device), u8_tensor(a[2], device))
                          for a in (g, u, d)]
            else:
                staged = [(u8_tensor(a[0], device), u8_tensor(a[1], device)) for a in (g, u, d)]
            gate_up, down = staged[:2], staged[2:]
        else:
            c = B.MoeConfig(hidden=cfg.hidden, inter=cfg.inter, n_experts=cfg.n_experts, n_shared=cfg.n_shared,
                            k_max=k_max or cfg.k, n_slices=0, fmt=fmt)
            gate_up, down = [], []

            def gen(e):
                return wl.expert_weights(cfg, e)

            with cf.ThreadPoolExecutor(max_workers=8) as ex:
                for w in ex.map(gen, range(cfg.n_groups)):
                    if fmt == B.MOE_W_INT4G32:
                        gc, gs, dc, ds, gz, dz = w
                        gate_up.append((u8_tensor(gc, device), u16_tensor(gs, device), u8_tensor(gz, device)))
                        down.append((u8_tensor(dc, device), u16_tensor(ds, device), u8_tensor(dz, device)))
                    else:
                        gc, gs, dc, ds = w
                        gate_up.append((u8_tensor(gc, device), u8_tensor(gs, device)))
                        down.append((u8_tensor(dc, device), u8_tensor(ds, device)))
        self.config = c
        self.handle = B.moe_load_weights(c, gate_up, down, stream)
        del gate_up, down

    def workspace(self, T: int, k: int) -> tuple:
        n = B.moe_workspace_bytes(self.handle, T, 0 if self.dense else k)
        if self._ws is None or self._ws.numel() < n:
            self._ws = torch.empty(max(n, 256), dtype=torch.uint8, device=self.device)
        return self._ws, n

    def forward(self, x: torch.Tensor, logits: Optional[torch.Tensor], k: Optional[int] = None,
                out: Optional[torch.Tensor] = None, accumulate: bool = False, routing=None, stream=None):
        T = x.shape[0]
        if out is None:
            out = torch.empty((T, self.cfg.hidden), dtype=torch.float32, device=self.device)
        if self.dense:
            ws, n = self.workspace(T, 0)
            B.moe_dense_sliced_forward(self.handle, x, T, out, accumulate, ws, n, stream)
        else:
            k = k or self.cfg.k
            ws, n = self.workspace(T, k)
            B.moe_forward(self.handle, x, logits, T, k, out, accumulate, ws, n, routing, stream)
        return out

    def forward_routed(self, x: torch.Tensor, topk_ids: torch.Tensor, topk_w: torch.Tensor,
                       out: Optional[torch.Tensor] = None, accumulate: bool = False, routing=None, stream=None):
        """The layer for routing given as expert ids (int32 [T, k]) and weights (float32 [T, k]).
        An id of -1 is an empty slot (it adds nothing; its weight is not read)."""
        T, k = topk_ids.shape
        if out is None:
            out = torch.empty((T, self.cfg.hidden), dtype=torch.float32, device=self.device)
        ws, n = self.workspace(T, k)
        B.moe_forward_routed(self.handle, x, topk_ids, topk_w, T, k, out, accumulate, ws, n, routing, stream)
        return out

    def sync(self, stream=None):
        B.moe_sync_status(self.handle, stream)

    def free(self):
        if self.handle:
            B.moe_free(self.handle)
            self.handle = None
        self._ws = None

    def __del__(self):
        try:
            self.free()
        except Exception:
            pass
