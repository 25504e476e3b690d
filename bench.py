#!/usr/bin/env python
"""Benchmark of the GB300 MXFP4 routed-expert MoE layer.

One step = one full forward pass of the layer (routing, grouping, gate|up GEMM
with SwiGLU, down GEMM, combine) on one batch of seeded synthetic input, with
inputs resident in HBM.  Default workload: the decode layer, T=1 token,
H=7168, I=2048, 256 routed MXFP4 experts + 1 shared, top-8.

Timing: W warm-up steps, then K steps, each timed with CUDA events on the
launching stream; the L2 cache (129 MB) is flushed between steps by writing a
512 MB buffer outside the timed events.  Per-stage CUDA events recorded by the
library on the same stream give the dominant kernel's duration for the roofline.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                       [--workload decode_T1|sweep_T15|...|prefill_T8192|dense_bf16_T4096|...]
Under torchrun each rank runs an independent replica of the layer on its own
GPU (the layer is not sharded); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from mxfp4_routed_expert_router_gb300 import workloads as wl  # noqa: E402

METRIC = "MoE-layer tokens/s; decode weight-stream HBM GB/s; prefill tensor TFLOPS vs peak"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# GB300 datasheet figures, reported beside the measured ones: HBM3e 7.9 TB/s,
# dense BF16 tensor 2.25 PFLOP/s
NOMINAL_PEAKS = {"hbm_gbs": 7900.0, "bf16_tflops": 2250.0}
L2_FLUSH_BYTES = 512 << 20
MX_BYTES_PER_WEIGHT = 17 / 32   # 4 bits of code + 8 bits of scale per 32 weights
# stored bytes per weight of each format: group-32 INT4 carries a 16-bit scale
# and an 8-bit zero point per 32 weights
BYTES_PER_WEIGHT = {"mxfp4": MX_BYTES_PER_WEIGHT, "int4g32": 19 / 32, "bf16": 2.0}


def workload(name: str) -> wl.LayerConfig:
    if name == "tiny":
        return wl.tiny()
    kind, _, rest = name.rpartition("_T")
    T = int(rest)
    if kind == "decode":
        return wl.decode(T)
    if kind == "sweep":
        return wl.sweep(T)
    if kind == "prefill":
        return wl.prefill(T)
    if kind in ("dense_bf16", "dense_mxfp4", "dense_int4g32"):
        return wl.dense(T, kind.split("_")[1])
    raise SystemExit(f"unknown workload {name}")


def describe(cfg: wl.LayerConfig) -> str:
    if cfg.dense:
        return (f"{cfg.name}: dense SwiGLU FFN T={cfg.T}, H={cfg.hidden}, I={cfg.inter} as {cfg.n_slices} "
                f"all-active slices of {cfg.inter // cfg.n_slices}, {cfg.weight_format.upper()} weights")
    fmt = {"mxfp4": "MXFP4", "int4g32": "group-32 INT4", "bf16": "BF16"}[cfg.weight_format]
    return (f"{cfg.name}: MoE layer T={cfg.T}, H={cfg.hidden}, I={cfg.inter}, E={cfg.n_experts} routed + "
            f"{cfg.n_shared} shared {fmt} experts, top-{cfg.k}, logits {cfg.logits}")


def read_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained")}, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ------------------------------------------------------------------ algorithmic work

def work_model(cfg: wl.LayerConfig, groups_active: int):
    """Algorithmic bytes and flops of the two GEMM kernels for one call.

    groups_active: expert groups with at least one token (routed experts hit by
    the batch, plus shared experts / dense slices).  Weight bytes are counted
    once per active group in their stored format (MXFP4: 17/32 byte per weight,
    group-32 INT4 with zero points: 19/32);
    flops are 2 per multiply-add over every (position, weight) pair.
    """
    H, T = cfg.hidden, cfg.T
    if cfg.dense:
        I = cfg.inter // cfg.n_slices
        P = T * cfg.n_slices
    else:
        I = cfg.inter
        P = T * cfg.k + T * cfg.n_shared
    wb = BYTES_PER_WEIGHT[cfg.weight_format]
    gu_w = groups_active * 2 * I * H * wb
    dn_w = groups_active * H * I * wb
    gate_up = {"bytes": gu_w + T * H * 2 + P * I * 4, "flops": 2.0 * P * 2 * I * H,
               "weight_bytes": gu_w, "per_unit": 2 * I * H * wb}
    down = {"bytes": dn_w + P * I * 4 + P * H * 4, "flops": 2.0 * P * H * I, "weight_bytes": dn_w,
            "per_unit": H * I * wb}
    # the single-kernel layer of decode-sized batches: h and y stay on chip / in
    # L2, so its algorithmic traffic is the weights, x, the logits and out
    E = 0 if cfg.dense else cfg.n_experts
    layer = {"bytes": gu_w + dn_w + T * H * 2 + T * E * 4 + T * H * 4, "flops": gate_up["flops"] + down["flops"],
             "weight_bytes": gu_w + dn_w, "per_unit": 3 * I * H * wb}
    return gate_up, down, layer


# ------------------------------------------------------------------ clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.proc.wait(5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if not self.proc or not self.path or not os.path.exists(self.path):
            return None
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return None
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = sorted({names[i] for _, _, r in rows for i, v in enumerate(r) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


def tc_fp16_operands(cfg) -> bool:
    """Whether the tensor-memory GEMMs take FP16 operands for this layer: the
    library decodes MXFP4 weights exactly to FP16 against a per-row exponent
    base when no row's E8M0 exponents span more than 23 (the seeded exponents
    are uniform in [e8m0_lo, e8m0_hi], so a range of at most 23 guarantees it),
    and group-32 INT4 weights always to FP16 hi + lo pairs.  BF16 weights, and
    MXFP4 rows of a wider span, run with BF16 operands."""
    if cfg.weight_format == "int4g32":
        return True
    return cfg.weight_format == "mxfp4" and cfg.e8m0_hi - cfg.e8m0_lo <= 23


def kernels_per_step(cfg, streaming: bool) -> int:
    """Kernels of this library launched by one forward call.

    The single-kernel layer launches one kernel.  Otherwise: the router and the
    two kernels of the chunked permutation (routed) or the dense plan (dense);
    the token preparation (FP16 operands) or the row gather (BF16 operands);
    gate|up and down; then the combine."""
    if streaming:
        return 1
    return (1 if cfg.dense else 3) + 3 + 1


def operand_dtype(cfg, streaming: bool) -> str:
    """Operand type of the layer's products (FP32 accumulation throughout): the
    single-kernel layer decodes MXFP4 and INT4 weights to FP16; the tensor-memory
    GEMMs take FP16 or BF16 operands as tc_fp16_operands says."""
    if streaming:
        return "f16" if cfg.weight_format in ("mxfp4", "int4g32") else "bf16"
    return "f16" if tc_fp16_operands(cfg) else "bf16"


def roofline_entry(dom: dict, dom_ms: float, peaks: dict, peak_src: str, dtype: str = "bf16") -> dict:
    """Roofline of a kernel from its algorithmic bytes and flops and its time:
    the bound is whichever minimum time is longer at the measured peaks; the
    fraction is also given against the datasheet peak (frac_nominal).  FP16
    and BF16 products have the same dense tensor rate (2.25 PFLOP/s nominal
    each), so an FP16 contraction takes the measured BF16 peak times 1."""
    tensor_bound = dom["flops"] / (peaks["bf16_tflops"] * 1e12) > dom["bytes"] / (peaks["hbm_gbs"] * 1e9)
    if tensor_bound:
        achieved = dom["flops"] / (dom_ms * 1e-3) / 1e12
        return {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                "frac": achieved / peaks["bf16_tflops"],
                "peak_source": (f"bf16 burst, of {peak_src}" if dtype == "bf16" else
                                f"{dtype}: bf16 burst x 1 (equal nominal rates), of {peak_src}"),
                "frac_nominal": achieved / NOMINAL_PEAKS["bf16_tflops"]}
    achieved = dom["bytes"] / (dom_ms * 1e-3) / 1e9
    return {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": achieved / peaks["hbm_gbs"], "peak_source": f"copy bandwidth, of {peak_src}",
            "frac_nominal": achieved / NOMINAL_PEAKS["hbm_gbs"]}


# ------------------------------------------------------------------ traffic (ncu)

def ncu_traffic(kernel_key: str):
    """Per-launch DRAM traffic of a kernel from the committed ncu summary, or
    None when the kernel's source changed since that capture."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    ent = d.get(kernel_key)
    if not ent:
        return None
    src = os.path.join(ROOT, ent["source"])
    if not os.path.exists(src) or hashlib.sha256(open(src, "rb").read()).hexdigest() != ent["source_sha256"]:
        return None
    return float(ent["bytes_per_launch"]) * float(ent.get("scale_to_workload", 1.0))


# ------------------------------------------------------------------ ranks

def max_over_ranks(value: float, dist, device=None) -> float:
    """The largest value over all ranks: a job's step time is its slowest rank's."""
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(world: int, tokens_per_rank: int, ms: float) -> float:
    """Whole-job throughput of N independent replicas (weak scaling): every
    rank's tokens over the slowest rank's step time."""
    return world * tokens_per_rank / (ms * 1e-3)


# ------------------------------------------------------------------ our arm

# Workloads measured beside the headline one, on the same loaded layer (the
# decode, sweep and prefill workloads share their expert weights): the metric
# also asks for the sweep's weight-stream GB/s and prefill's tensor TFLOP/s.
EXTRA_WORKLOADS = ("sweep_T15", "sweep_T88", "sweep_T176", "prefill_T8192")


def same_layer(a: wl.LayerConfig, b: wl.LayerConfig) -> bool:
    keys = ("hidden", "inter", "n_experts", "n_shared", "k", "wseed", "e8m0_lo", "e8m0_hi", "dense", "n_slices",
            "weight_format")
    return all(getattr(a, k) == getattr(b, k) for k in keys)


def dominant_kernel(cfg, stage_ms, groups):
    """The dominant kernel of a workload and its roofline inputs: the
    single-kernel layer when the batch ran through it (profile stage 5), else
    the longer of the two GEMM stages."""
    gate_up, down, layer_w = work_model(cfg, groups)
    if stage_ms.get("layer", 0.0) > stage_ms["gate_up"] + stage_ms["down"]:
        return "layer", layer_w
    name = "gate_up" if stage_ms["gate_up"] >= stage_ms["down"] else "down"
    return name, gate_up if name == "gate_up" else down


class Workload:
    """Device-resident inputs of one workload on a loaded layer, and its timed steps."""

    def __init__(self, L, cfg, dev):
        import torch

        from mxfp4_routed_expert_router_gb300 import binding as B
        from mxfp4_routed_expert_router_gb300.layer import bf16_tensor

        self.L, self.cfg, self.dev, self.B = L, cfg, dev, B
        self.x_bits = wl.tokens(cfg)
        self.x = bf16_tensor(self.x_bits, str(dev))
        self.logits_np = None if cfg.dense else wl.router_logits(cfg)
        self.logits = None if cfg.dense else torch.from_numpy(self.logits_np).to(dev)
        self.out = torch.empty((cfg.T, cfg.hidden), dtype=torch.float32, device=dev)

    def step(self, routing=None):
        self.L.forward(self.x, self.logits, self.cfg.k, out=self.out, routing=routing)

    def active_groups(self):
        """Distinct active expert groups of this batch (the unit of the weight stream)."""
        import torch
        cfg = self.cfg
        if cfg.dense:
            return cfg.n_slices
        ids = torch.empty((cfg.T, cfg.k), dtype=torch.int32, device=self.dev)
        self.step(self.B.routing_out(topk_ids=ids))
        self.L.sync()
        return int(torch.unique(ids).numel()) + cfg.n_shared

    def timed(self, steps, warmup, flush, stream, dist=None):
        """Mean device ms per step over `steps` steps (CUDA events on the launching
        stream, L2 flushed before each step outside the events) and the SM clocks
        sampled meanwhile."""
        import torch
        for _ in range(warmup):
            self.step()
        self.L.sync()
        if dist:
            dist.barrier()
        torch.cuda.synchronize(self.dev)
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        with ClockSampler(self.dev.index) as clk:
            for i in range(steps):
                flush.zero_()
                starts[i].record(stream)
                self.step()
                ends[i].record(stream)
            torch.cuda.synchronize(self.dev)
        if dist:
            dist.barrier()
        torch.cuda.synchronize(self.dev)
        times = [s.elapsed_time(e) for s, e in zip(starts, ends)]
        ms = sum(times) / len(times)
        if dist:
            ms = max_over_ranks(ms, dist, self.dev)
        self.L.sync()
        return ms, clk.summary()

    def stages(self, n, flush):
        """Per-stage device time from the library's own events on the same stream,
        in separate (untimed) steps so that the events do not perturb the timed ones."""
        B = self.B
        B.moe_profile_enable(self.L.handle, True)
        st = []
        for _ in range(n):
            flush.zero_()
            self.step()
            st.append(B.moe_profile_read(self.L.handle))
        B.moe_profile_enable(self.L.handle, False)
        self.L.sync()
        return {k: sum(s[k] for s in st) / len(st) for k in st[0]}


def summarize_extra(cfg, ms, clocks, stage_ms, groups, peaks, peak_src):
    """Per-workload numbers of a workload measured beside the headline one."""
    gate_up, down, layer_w = work_model(cfg, groups)
    weight_bytes = gate_up["weight_bytes"] + down["weight_bytes"]
    flops = gate_up["flops"] + down["flops"]
    dom_name, dom = dominant_kernel(cfg, stage_ms, groups)
    r = {"workload": describe(cfg), "T": cfg.T, "ms_per_step": ms, "tokens_per_s": cfg.T / (ms * 1e-3),
         "active_groups": groups, "weight_GBps": weight_bytes / (ms * 1e-3) / 1e9,
         "layer_TFLOPs": flops / (ms * 1e-3) / 1e12, "clocks": clocks,
         "stages_ms": {"layer": stage_ms["layer"]} if dom_name == "layer" else stage_ms}
    roof = roofline_entry(dom, stage_ms[dom_name], peaks, peak_src, operand_dtype(cfg, dom_name == "layer"))
    roof["kernel"] = "single-kernel MoE layer" if dom_name == "layer" else f"{dom_name} GEMM"
    roof["kernel_ms"] = stage_ms[dom_name]
    roof["traffic"] = ncu_traffic(f"{dom_name}:{cfg.name}")
    r["roofline"] = roof
    if dom_name == "layer":
        # HBM-bound: the weight stream over the step, as a fraction of the copy peak
        r["weight_stream_frac"] = r["weight_GBps"] / peaks["hbm_gbs"]
    else:
        # tensor-bound: each GEMM, and the whole step, against the bf16 tensor peak
        tp = peaks["bf16_tflops"]
        r["gate_up"] = {"ms": stage_ms["gate_up"], "TFLOPs": gate_up["flops"] / (stage_ms["gate_up"] * 1e-3) / 1e12}
        r["down"] = {"ms": stage_ms["down"], "TFLOPs": down["flops"] / (stage_ms["down"] * 1e-3) / 1e12}
        for kk in ("gate_up", "down"):
            r[kk]["tensor_frac"] = r[kk]["TFLOPs"] / tp
        r["layer_tensor_frac"] = r["layer_TFLOPs"] / tp
    r["peak_source"] = f"copy bandwidth / bf16 burst, of {peak_src}"
    return r


def bench_config(cfg: wl.LayerConfig, groups: int, world: int) -> dict:
    """The `config` object of the JSON line (the same for both arms)."""
    tokens_per_expert = (cfg.T * cfg.k) / max(1, groups - cfg.n_shared) if not cfg.dense else cfg.T
    return {"workload": describe(cfg), "weights": cfg.weight_format, "T": cfg.T, "hidden": cfg.hidden,
            "inter": cfg.inter, "experts": cfg.n_experts, "shared": cfg.n_shared, "top_k": cfg.k,
            "active_groups": groups, "tokens_per_routed_expert": tokens_per_expert,
            "l2": "flushed between steps (512 MB write outside the timed events)",
            "parallelism": f"replicas x{world}"}


def run_ours(args, cfg, rank, world):
    import torch

    from mxfp4_routed_expert_router_gb300 import binding as B
    from mxfp4_routed_expert_router_gb300.layer import MoeLayer

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    L = MoeLayer(cfg, device=str(dev))
    W = Workload(L, cfg, dev)
    x, logits, out, x_bits = W.x, W.logits, W.out, W.x_bits
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    for _ in range(args.warmup):
        W.step()
    L.sync()
    groups = W.active_groups()

    dist = None
    if world > 1:
        import torch.distributed as dist
    ms, clocks = W.timed(args.steps, 0, flush, stream, dist)
    stage_ms = W.stages(max(3, min(args.steps, 10)), flush)

    # end to end through the public API with host buffers: pinned x/logits in,
    # out back to pinned host memory, copies inside the timed region
    hx = torch.from_numpy(x_bits.view(np.int16)).view(torch.bfloat16).pin_memory()
    hl = None if cfg.dense else torch.from_numpy(W.logits_np).pin_memory()
    hout = torch.empty((cfg.T, cfg.hidden), dtype=torch.float32).pin_memory()
    e2e_times = []
    for i in range(max(3, min(args.steps, 20))):
        flush.zero_()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(stream)
        x.copy_(hx, non_blocking=True)
        if hl is not None:
            logits.copy_(hl, non_blocking=True)
        L.forward(x, logits, cfg.k, out=out)
        hout.copy_(out, non_blocking=True)
        e.record(stream)
        e.synchronize()
        e2e_times.append(s.elapsed_time(e))
    e2e_ms = sum(e2e_times) / len(e2e_times)

    # the same step replayed from a CUDA graph of the call (moe_graph_create):
    # device time per replay, L2 flushed between replays like the timed steps
    ws, nws = L.workspace(cfg.T, 0 if cfg.dense else cfg.k)
    graph = B.moe_graph_create(L.handle, x, logits, None, None, cfg.T, 0 if cfg.dense else cfg.k, out, False, ws,
                               nws)
    g_times = []
    try:
        for i in range(args.warmup + max(3, min(args.steps, 20))):
            flush.zero_()
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record(stream)
            B.moe_graph_launch(graph, stream)
            e.record(stream)
            e.synchronize()
            if i >= args.warmup:
                g_times.append(s.elapsed_time(e))
    finally:
        B.moe_graph_free(graph)
    graph_ms = sum(g_times) / len(g_times)

    h2d = x_bits.nbytes + (0 if cfg.dense else cfg.T * cfg.n_experts * 4)
    d2h = cfg.T * cfg.hidden * 4

    gate_up, down, layer_w = work_model(cfg, groups)
    peaks, peak_src = read_peaks()
    dom_name, dom = dominant_kernel(cfg, stage_ms, groups)
    dom_ms = stage_ms[dom_name]
    if dom_name == "layer":
        # the single kernel runs every stage; the other marks are empty
        stage_ms = {"layer": stage_ms["layer"]}
    roof = roofline_entry(dom, dom_ms, peaks, peak_src, operand_dtype(cfg, dom_name == "layer"))
    roof["kernel"] = "single-kernel MoE layer" if dom_name == "layer" else f"{dom_name} GEMM"
    roof["traffic"] = ncu_traffic(f"{dom_name}:{cfg.name}")
    roof["algorithmic_bytes"] = dom["bytes"]
    roof["algorithmic_flops"] = dom["flops"]
    roof["kernel_ms"] = dom_ms
    streaming = dom_name == "layer"
    launches_per_step = kernels_per_step(cfg, streaming)
    dtype = operand_dtype(cfg, streaming)
    weight_bytes = gate_up["weight_bytes"] + down["weight_bytes"]
    value = job_tokens_per_s(world, cfg.T, ms)
    res = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": dtype, "data": "synthetic (seeded; random MXFP4 codes and E8M0 scales)",
        "config": bench_config(cfg, groups, world),
        "weight_stream_GBps": weight_bytes / (ms * 1e-3) / 1e9,
        "layer_TFLOPs": (gate_up["flops"] + down["flops"]) / (ms * 1e-3) / 1e12,
        "stages_ms": stage_ms,
        "roofline": roof,
        "e2e": {"value": world * cfg.T / (e2e_ms * 1e-3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
        "graph": {"value": world * cfg.T / (graph_ms * 1e-3), "unit": "tokens/s", "ms_per_step": graph_ms,
                  "note": "the same call replayed from a CUDA graph (moe_graph_create / moe_graph_launch)"},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
    }
    del W

    # the other workloads of the metric on the same layer, each with its own
    # timed steps, L2 flush, stage events and clock record
    extras = {}
    names = [] if args.extra == "none" else [n for n in args.extra.split(",") if n]
    for name in names:
        ecfg = workload(name)
        if ecfg.name == cfg.name or not same_layer(ecfg, cfg):
            continue
        EW = Workload(L, ecfg, dev)
        EW.step()
        egroups = EW.active_groups()
        esteps = max(3, min(args.steps, 10))
        ems, eclk = EW.timed(esteps, args.warmup, flush, stream, dist)
        est = EW.stages(3, flush)
        e_ent = summarize_extra(ecfg, ems, eclk, est, egroups, peaks, peak_src)
        e_ent["tokens_per_s"] = job_tokens_per_s(world, ecfg.T, ems)
        e_ent["steps"] = esteps
        e_ent["gpu_launches"] = esteps * kernels_per_step(ecfg, e_ent["roofline"]["kernel"] == "single-kernel MoE layer")
        e_ent["dtype"] = operand_dtype(ecfg, e_ent["roofline"]["kernel"] == "single-kernel MoE layer")
        extras[name] = e_ent
        del EW
    if extras:
        res["workloads"] = extras
    L.free()
    return res


# ------------------------------------------------------------------ the oracle (CPU)

_DENSE_CACHE = {}


def oracle_sample(cfg: wl.LayerConfig, budget_s: float, max_tokens: int = None, cores=None):
    """Time the CPU oracle, as it stands, on a bounded token sample of the workload.

    cores: the host CPUs the oracle may run on (its threads inherit the calling
    thread's affinity; default: every CPU this process may use); it is given
    one thread per core.  Returns (tokens processed, seconds, threads used,
    description).  The oracle runs the (token, expert) jobs of one expert in
    parallel, one expert after another, so the threads it actually uses are
    bounded by the largest number of jobs of one expert in the sample."""
    import oracle

    oracle.build()
    x_bits = wl.tokens(cfg)
    all_cores = sorted(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else None
    cores = sorted(cores) if cores is not None else all_cores
    nthreads = len(cores) if cores else (os.cpu_count() or 1)
    sample = wl.sample_tokens(cfg.T, max_tokens or cfg.T)
    done, secs, rounds = 0, 0.0, 0
    if cfg.dense:
        if cfg.name not in _DENSE_CACHE:
            _DENSE_CACHE.clear()
            _DENSE_CACHE[cfg.name] = wl.dense_weights(cfg)
        weights = _DENSE_CACHE[cfg.name]
    else:
        lg = wl.router_logits(cfg)
    if cores and all_cores and cores != all_cores:
        os.sched_setaffinity(0, cores)
    try:
        while secs < budget_s or rounds == 0:
            t0 = time.perf_counter()
            if cfg.dense:
                oracle.dense_ffn(weights, x_bits[sample], cfg.n_slices, cfg.weight_format)
            else:
                ids, _ = oracle.route(lg[sample], cfg.k)
                needed = sorted(set(ids.ravel().tolist()) | set(range(cfg.n_experts, cfg.n_groups)))
                W = oracle.OracleWeights(cfg.hidden, cfg.inter, cfg.n_experts, cfg.n_shared, cfg.weight_format)
                for e in needed:
                    W.set_expert(e, *wl.expert_weights(cfg, e))
                t0 = time.perf_counter()  # weight generation is input synthesis, not oracle work
                oracle.moe_layer(W, x_bits[sample], lg[sample], cfg.k, nthreads=nthreads)
            secs += time.perf_counter() - t0
            done += len(sample)
            rounds += 1
    finally:
        if cores and all_cores and cores != all_cores:
            os.sched_setaffinity(0, all_cores)
    if cfg.dense:
        used = 1
    else:
        ids, _ = oracle.route(lg[sample], cfg.k)
        jobs = np.bincount(ids.ravel(), minlength=cfg.n_experts).tolist() + [len(sample)] * cfg.n_shared
        used = max(min(nthreads, int(c)) for c in jobs if c > 0)
    desc = (f"{len(sample)} of {cfg.T} tokens per round x {rounds} rounds "
            f"({'dense FFN' if cfg.dense else 'full routing + every selected and shared expert'}, "
            f"weights decoded per round)")
    return done, secs, used, desc


def cpu_baseline_entry(cfg, budget_s: float) -> dict:
    """The oracle on the host's cores and, beside it, on one core."""
    avail = sorted(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else list(range(os.cpu_count() or 1))
    ntok = oracle_budget_tokens(cfg)
    done, secs, used, desc = oracle_sample(cfg, budget_s, ntok, avail)
    d1, s1, _, desc1 = oracle_sample(cfg, budget_s / 2, ntok, avail[:1])
    return {"value": done / secs, "unit": "tokens/s", "cores": used, "kind": "oracle",
            "sample": desc + f"; {secs:.1f} s of CPU work",
            "host_cores": os.cpu_count(), "cores_available": len(avail),
            "threads_given": len(avail),
            "pinning": "the oracle's threads inherit this process's CPU affinity (all available cores); "
                       "threads are not bound one to a core",
            "single_core": {"value": d1 / s1, "unit": "tokens/s", "cores": 1,
                            "pinning": f"bound to CPU {avail[0]}", "sample": desc1 + f"; {s1:.1f} s of CPU work"}}


def oracle_budget_tokens(cfg):
    if cfg.dense:
        return 1 if cfg.T == 1 else 2
    return min(cfg.T, 2)


def run_reference(args, cfg, rank, world):
    if rank != 0:
        return None
    import oracle

    times = []
    sample_desc = ""
    used = 1
    ntok = oracle_budget_tokens(cfg)
    for _ in range(args.warmup if args.warmup < 1 else 1):
        oracle_sample(cfg, 0.0, ntok)
    for _ in range(args.steps):
        done, secs, used, sample_desc = oracle_sample(cfg, 0.0, ntok)
        times.append(secs / done)   # seconds per token
    per_tok = sum(times) / len(times)
    value = 1.0 / per_tok
    if cfg.dense:
        groups = cfg.n_slices
    else:
        ids, _ = oracle.route(wl.router_logits(cfg), cfg.k)
        groups = len(np.unique(ids)) + cfg.n_shared
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": per_tok * 1e3 * cfg.T,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded)", "config": bench_config(cfg, groups, 1),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": used, "kind": "oracle",
                         "sample": sample_desc, "host_cores": os.cpu_count()},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="decode_T1")
    ap.add_argument("--cpu-baseline-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--weights", default="mxfp4", choices=["mxfp4", "int4g32"],
                    help="weight format of a routed workload")
    ap.add_argument("--extra", default=",".join(EXTRA_WORKLOADS),
                    help="comma-separated workloads measured beside the main one on the same layer ('none': skip)")
    ap.add_argument("--experts", type=int, default=0,
                    help="profiling aid: routed experts of a smaller layer with the same shapes per expert")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    cfg = workload(args.workload)
    import dataclasses
    if args.weights != "mxfp4" and not cfg.dense:
        cfg = dataclasses.replace(cfg, name=f"{cfg.name}_{args.weights}", weight_format=args.weights)
    if args.experts:
        cfg = dataclasses.replace(cfg, name=f"{cfg.name}_E{args.experts}", n_experts=args.experts)
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))

    if args.impl == "reference":
        res = run_reference(args, cfg, rank, world)
        if res is not None:
            print(json.dumps(res))
        return

    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        dist.init_process_group("nccl")
    res = run_ours(args, cfg, rank, world)
    if rank == 0:
        if not args.no_cpu_baseline:
            res["cpu_baseline"] = cpu_baseline_entry(cfg, args.cpu_baseline_seconds)
        print(json.dumps(res))
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
