"""Host logic of the benchmark's multi-rank path, on the CPU: the
max-over-ranks reduction with two gloo ranks, and the reference arm's rule
that only rank 0 works and prints."""
from __future__ import annotations

import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        # each rank reports its own step and kernel times; the job takes the slowest
        got = bench.max_over_ranks([1.0 + rank, 5.0 - rank, 0.25 * (rank + 1)], "cpu", world)
        out.put((rank, got))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert res[0] == res[1] == [2.0, 5.0, 0.5]


def test_max_over_ranks_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks([3, 1.5], "cpu", 1) == [3.0, 1.5]


def test_reference_arm_other_ranks_exit_without_output():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1", MASTER_ADDR="127.0.0.1",
               MASTER_PORT=str(_free_port()))
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "3",
                        "--warmup", "3"], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""


def test_reference_arm_prints_the_contract_line():
    """Rank 0 of the reference arm (the oracle on the host cores) prints one
    JSON line with the benchmark's keys, its own cpu_baseline and an e2e
    object that moves no bytes between host and device."""
    import json
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK")}
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0"], env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [x for x in r.stdout.splitlines() if x.strip()]
    assert len(lines) == 1
    line = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["steps"] == 1 and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["cpu_baseline"]["cores"] >= 1 and line["cpu_baseline"]["sample"]
    e2e = line["e2e"]
    assert e2e["value"] == line["value"] and e2e["unit"] == line["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0
    assert "workload" in line["config"]


def test_clock_summary_skips_idle_samples_and_collects_reasons():
    """The clocks object describes the GPU under load: samples taken while
    the GPU-idle reason is active (host work between timed parts, when the
    SM clock drops) are left out; throttle reasons are collected from the
    rest."""
    sys.path.insert(0, ROOT)
    import bench

    def row(clk, idle, cap="Not Active", thermal="Not Active"):
        return ["0", str(clk), "2070", "300.0", "0x0", "Not Active", "Not Active", thermal, cap, idle]

    rows = [row(120, "Active")] * 50 + [row(2070, "Not Active")] * 5 + [row(1965, "Not Active", cap="Active")] * 2
    got = bench.summarize_clocks(rows + [["garbage"]])
    assert got["samples"] == 7 and got["samples_total"] == 57
    assert got["sm_mhz"] == 2070 and got["sm_max_mhz"] == 2070
    assert got["reasons"] == ["sw_power_cap"]
    none = bench.summarize_clocks([row(120, "Active")] * 3)
    assert none["samples"] == 0 and none["sm_mhz"] is None
