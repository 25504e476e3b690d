"""CPU tests of bench.py's host logic: the algorithmic-byte model behind the
roofline, the ncu traffic captures keyed by their kernel sources, the
max-over-ranks step time of an N-rank run (world size 2 over gloo), the
reference arm's JSON line, and the ranks that stay silent."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_algorithmic_bytes_of_decode():
    # MXFP4 costs 17/32 byte per weight (4-bit codes + one E8M0 byte per 32):
    # an expert (gate|up [4096, 7168] and down [7168, 2048]) is 23,396,352 bytes
    cfg = bench.workload("decode_T1")
    gu, dn, layer = bench.work_model(cfg, 9)
    assert gu["per_unit"] + dn["per_unit"] == 23_396_352
    assert layer["weight_bytes"] == 9 * 23_396_352
    # plus x (BF16), the logits (FP32 [1][256]) and out (FP32)
    assert layer["bytes"] == 9 * 23_396_352 + 7168 * 2 + 256 * 4 + 7168 * 4
    # two flops per multiply-add over every (position, weight) pair: 9 positions
    assert layer["flops"] == 2 * 9 * 3 * 2048 * 7168


def test_algorithmic_bytes_of_int4_decode():
    # group-32 INT4 with FP16 scales and zero points costs 19/32 byte per weight:
    # an expert is 3 * 8,716,288 = 26,148,864 bytes
    import dataclasses
    cfg = dataclasses.replace(bench.workload("decode_T1"), weight_format="int4g32")
    gu, dn, layer = bench.work_model(cfg, 9)
    assert gu["per_unit"] + dn["per_unit"] == 26_148_864
    assert layer["weight_bytes"] == 9 * 26_148_864
    dense = bench.work_model(bench.workload("dense_int4g32_T1"), 9)[2]
    assert dense["weight_bytes"] == 3 * 7168 * 18432 * 19 / 32


def test_roofline_bound_and_fractions():
    peaks = {"hbm_gbs": 6714.6, "bf16_tflops": 1937.1, "bf16_tflops_sustained": 1741.4}
    _, _, layer = bench.work_model(bench.workload("decode_T1"), 9)
    r = bench.roofline_entry(layer, 0.0705, peaks, "measured")
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert r["achieved"] == pytest.approx(layer["bytes"] / 70.5e-6 / 1e9)
    assert r["frac"] == pytest.approx(r["achieved"] / 6714.6)
    assert r["frac_nominal"] == pytest.approx(r["achieved"] / 7900.0)
    # prefill gate|up: 73,728 token positions over 257 groups is a dense contraction
    gu, _, _ = bench.work_model(bench.workload("prefill_T8192"), 257)
    r = bench.roofline_entry(gu, 5.5, peaks, "measured")
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert r["frac"] == pytest.approx(gu["flops"] / 5.5e-3 / 1e12 / 1937.1)
    assert r["frac_nominal"] == pytest.approx(gu["flops"] / 5.5e-3 / 1e12 / 2250.0)


def test_traffic_entries_match_their_sources_and_go_stale_on_change(tmp_path, monkeypatch):
    # every committed capture is keyed by the sha256 of the kernel source it was
    # taken on; a changed source yields no traffic rather than a stale figure
    import hashlib
    import shutil
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        entries = json.load(f)
    for key, ent in entries.items():
        with open(os.path.join(ROOT, ent["source"]), "rb") as f:
            assert hashlib.sha256(f.read()).hexdigest() == ent["source_sha256"], key
        assert ent["bytes_per_launch"] == ent["dram_bytes_read"] + ent["dram_bytes_write"], key
        assert bench.ncu_traffic(key) == pytest.approx(ent["bytes_per_launch"] * ent.get("scale_to_workload", 1.0))
    assert bench.ncu_traffic("layer:no_such_workload") is None
    fake = tmp_path / "repo"
    shutil.copytree(os.path.join(ROOT, "profiles"), fake / "profiles")
    src = entries["layer:decode_T1"]["source"]
    (fake / os.path.dirname(src)).mkdir(parents=True)
    shutil.copy(os.path.join(ROOT, src), fake / src)
    monkeypatch.setattr(bench, "ROOT", str(fake))
    assert bench.ncu_traffic("layer:decode_T1") is not None
    with open(fake / src, "a") as f:
        f.write("\n// edited\n")
    assert bench.ncu_traffic("layer:decode_T1") is None


def test_extra_workload_roofline_carries_traffic():
    peaks = {"hbm_gbs": 6714.6, "bf16_tflops": 1937.1}
    stage = {"routing": 0.01, "grouping": 0.02, "gate_up": 4.3, "down": 2.45, "combine": 0.3, "layer": 0.0}
    r = bench.summarize_extra(bench.workload("prefill_T8192"), 7.3, {}, stage, 257, peaks, "measured")
    assert r["roofline"]["kernel"] == "gate_up GEMM"
    assert r["roofline"]["traffic"] == bench.ncu_traffic("gate_up:prefill_T8192")
    stage = {"routing": 0.0, "grouping": 0.0, "gate_up": 0.0, "down": 0.0, "combine": 0.0, "layer": 1.48}
    r = bench.summarize_extra(bench.workload("sweep_T88"), 1.48, {}, stage, 187, peaks, "measured")
    assert r["roofline"]["kernel"] == "single-kernel MoE layer" and r["roofline"]["traffic"] is None


def test_job_throughput_is_weak_scaling():
    assert bench.job_tokens_per_s(1, 1, 0.1) == pytest.approx(10_000.0)
    assert bench.job_tokens_per_s(4, 8, 2.0) == pytest.approx(16_000.0)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, values, q):
    import torch.distributed as dist
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        q.put((rank, bench.max_over_ranks(values[rank], dist)))
    finally:
        dist.destroy_process_group()


def test_step_time_is_the_slowest_rank_over_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    values = [0.0712, 0.0901]
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, values, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert got == {0: max(values), 1: max(values)}


def _bench(args, env_extra=None):
    env = dict(os.environ, **(env_extra or {}))
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], capture_output=True, text=True,
                          timeout=600, env=env, cwd=ROOT)


def test_reference_arm_prints_one_contract_line():
    r = _bench(["--impl", "reference", "--workload", "tiny", "--steps", "1", "--warmup", "3"])
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["unit"] == "tokens/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]
    assert d["config"]["workload"].startswith("tiny")


def test_reference_arm_with_int4_weights():
    r = _bench(["--impl", "reference", "--workload", "tiny", "--weights", "int4g32", "--steps", "1", "--warmup", "3"])
    assert r.returncode == 0, r.stderr[-2000:]
    d = json.loads(r.stdout.strip().splitlines()[-1])
    assert d["impl"] == "reference" and d["value"] > 0
    assert d["config"]["workload"].startswith("tiny_int4g32") and "group-32 INT4" in d["config"]["workload"]


def test_reference_arm_is_silent_on_other_ranks():
    r = _bench(["--impl", "reference", "--workload", "tiny", "--steps", "1", "--warmup", "3"],
               {"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"})
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""
