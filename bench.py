#!/usr/bin/env python
"""Benchmark of paged attention over an fp8 KV cache on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Headline workload: serving batch decode -- 64 requests with KV lengths
uniform in [512, 4096], 32 query / 8 KV heads, head_dim 128, page 16, bf16
query and output, e4m3fn KV cache with per-tensor scales (seeded, synthetic).
A step is one pass of the decode hot path over that batch: the split-KV
decode kernel and the LSE merge kernel, one pafp8_run (the plan is built once,
outside the timed region; the end-to-end figure re-plans every step).  The
decode kernel's own time, for its roofline, comes from a second loop that
runs it alone.

value = algorithmic bytes per step / device time per step, where the bytes
count the fp8 K and V rows the requests own at 1 byte per element, plus q, o,
lse and the page indices.  Split-KV partial states are not counted.

Timing: W warm-up steps, then exactly K timed steps between a barrier and a
device synchronize; reading a 256 MiB buffer evicts L2 between the timed
steps, outside the CUDA events that time each step on the launching stream
(a read rather than a write, so no dirty lines are written back during the
next step).
Under torchrun every rank runs the same workload on its own GPU (replicas, no
collective on the data path) and rank 0 prints the max time over ranks.

Output (rank 0): one JSON line with the full record of every timed part
(the other decode and prefill workloads, the 2-byte caches, the KV append,
POD), then the headline JSON line, last and compact: the serving decode
step, its roofline, the end-to-end figure with its breakdown, the clocks, a
roofline entry for each of the five named workloads ("configs") and the CPU
oracle baseline.

--impl reference times the CPU oracle (fp64, all host cores) on a bounded
sample of the same workload, as the reference arm.
"""
from __future__ import annotations

import argparse
import csv
import hashlib
import io
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "paged fp8-KV decode HBM GB/s (% of peak); causal prefill TFLOPS (% of peak)"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
L2_FLUSH_BYTES = 256 << 20

# DRAM bytes (read + write) per launch of the decode kernel on the serving
# workload, from one ncu capture of the kernel source with this SHA-256; a
# changed kernel reports null until it is captured again.
NCU_TRAFFIC = {
    "8c94b805d7f854b2a685a89adaf643807277c06c16f5fca2b27cb39f45c3fc53": 309745408,
}
# The same for the prefill kernels, per workload index, keyed by the SHA-256
# of their sources (prefill.cuh, then prefill_pair.cuh).
NCU_TRAFFIC_PREFILL = {
    "8a8b8f6abc782551a2f5f796339847147b0b8e84b8d94dfafe4ad22d16bf1a66": {4: 168300544, 5: 190012928, 7: 259149824},
}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=100)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--mode", choices=["all", "decode", "prefill", "append", "pod"], default="all",
                    help="which parts to time (profiling runs use one)")
    ap.add_argument("--prefill-steps", type=int, default=30)
    return ap.parse_args()


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(values, device, world: int):
    """Each value's maximum over all ranks (the slowest rank decides a
    whole-job time); the values themselves at world size 1."""
    if world == 1:
        return [float(v) for v in values]
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t]


def decode_bytes(b) -> int:
    """Algorithmic bytes of one decode pass over batch b."""
    qb = 1 if b.q_dtype in ("e4m3fn", "e5m2") else 2
    kv = b.kv_bytes()
    q = b.nnz_qo * b.num_qo_heads * b.head_dim * qb
    o = b.nnz_qo * b.num_qo_heads * b.head_dim * 2
    lse = b.nnz_qo * b.num_qo_heads * 4
    idx = 4 * int(b.kv_indptr[-1])
    return kv + q + o + lse + idx


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def measured_bf16_tflops():
    """Dense bf16 tensor peak (burst, for a kernel timed alone)."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["bf16_tflops"]), "measured"
    except Exception:
        return FALLBACK_BF16_TFLOPS, "fallback"


def time_prefill(index, dev, steps, warmup):
    """Device time of the prefill kernel on named workload `index`; returns
    a dict with TFLOPS over the admitted causal pairs and its roofline."""
    import torch

    import paged_attention_fp8_gb300 as pa
    from paged_attention_fp8_gb300.workloads import TORCH_DTYPES, WORKLOADS, workload

    b = workload(index)
    flops = b.causal_flops()
    q = b.q.to(dev)
    k = b.k_cache.to(dev)
    v = b.v_cache.to(dev)
    idx = b.kv_indices.to(dev)
    plan = pa.Plan(mode="prefill", num_qo_heads=b.num_qo_heads, num_kv_heads=b.num_kv_heads,
                   num_pages=b.num_pages, kv_indptr=b.kv_indptr, last_page_len=b.last_page_len,
                   qo_indptr=b.qo_indptr, q_dtype=b.q_dtype, kv_dtype=b.kv_dtype, o_dtype=b.o_dtype,
                   sm_scale=b.sm_scale)
    ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device=dev)
    plan.upload(ws)
    o = torch.empty(b.nnz_qo, b.num_qo_heads, b.head_dim, dtype=TORCH_DTYPES[b.o_dtype], device=dev)
    lse = torch.empty(b.nnz_qo, b.num_qo_heads, dtype=torch.float32, device=dev)
    flush = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    kw = dict(q_scale=b.q_scale, k_scale=b.k_scale, v_scale=b.v_scale)
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        flush.sum()
        plan.run(q, k, v, idx, o, lse, ws, **kw)
    torch.cuda.synchronize()
    plan.device_status(ws)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
    for i in range(steps):
        flush.sum()
        ev[i][0].record(stream)
        plan.run(q, k, v, idx, o, lse, ws, **kw)
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    plan.device_status(ws)
    ms = statistics.mean(e[0].elapsed_time(e[1]) for e in ev)
    tflops = flops / (ms * 1e-3) / 1e12
    p16, kind = measured_bf16_tflops()
    traffic = NCU_TRAFFIC_PREFILL.get(kernel_sha("prefill.cuh", "prefill_pair.cuh"), {}).get(index)
    fp8 = b.q_dtype in ("e4m3fn", "e5m2")
    out = {"workload": WORKLOADS[index], "value": round(tflops, 2), "unit": "TFLOP/s",
           "ms_per_launch": round(ms, 5), "flops": flops, "launches": steps,
           "mma": ("QK^T fp8 kind::f8f6f4, PV f16 kind::f16" if fp8 else
                   "bf16 kind::f16 on CTA pairs (cta_group::2, M 256; 2-byte cache, V read as the MN-major operand)"
                   if b.kv_dtype in ("f16", "bf16")
                   else "f16 kind::f16 (fp8 KV dequantized)")}
    if fp8:
        p8 = 2.0 * p16  # another dtype's measured peak x the nominal fp8/bf16 ratio
        blended = 2.0 / (1.0 / p8 + 1.0 / p16)
        out["roofline"] = {"bound": "tensor", "achieved": round(tflops, 2), "peak": round(blended, 1),
                           "unit": "TFLOP/s", "frac": round(tflops / blended, 4), "traffic": traffic,
                           "peak_kind": f"{kind} bf16 x nominal fp8 ratio 2, blended for half the flops at each rate",
                           "frac_of_dense_bf16": round(tflops / p16, 4)}
    else:
        out["roofline"] = {"bound": "tensor", "achieved": round(tflops, 2), "peak": p16, "unit": "TFLOP/s",
                           "frac": round(tflops / p16, 4), "traffic": traffic, "peak_kind": f"{kind} dense bf16"}
    del q, k, v, idx, o, lse, ws, flush
    torch.cuda.empty_cache()
    return out


def time_decode(index, dev, steps, warmup):
    """Device time of one decode step (the decode kernel and its split-KV
    merge, one pafp8_run) on named workload `index`, L2 evicted before each
    step, plus the decode kernel alone (stage 1, a second loop); GB/s over
    the algorithmic bytes (KV at its element size, q, o, lse, page ids)."""
    import torch

    import paged_attention_fp8_gb300 as pa
    from paged_attention_fp8_gb300.workloads import TORCH_DTYPES, WORKLOADS, workload

    b = workload(index)
    nbytes = decode_bytes(b)
    q, k, v, idx = b.q.to(dev), b.k_cache.to(dev), b.v_cache.to(dev), b.kv_indices.to(dev)
    plan = pa.Plan(mode="decode", num_qo_heads=b.num_qo_heads, num_kv_heads=b.num_kv_heads,
                   num_pages=b.num_pages, kv_indptr=b.kv_indptr, last_page_len=b.last_page_len,
                   q_dtype=b.q_dtype, kv_dtype=b.kv_dtype, o_dtype=b.o_dtype, sm_scale=b.sm_scale)
    meta = plan.metadata()
    ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device=dev)
    plan.upload(ws)
    o = torch.empty(b.nnz_qo, b.num_qo_heads, b.head_dim, dtype=TORCH_DTYPES[b.o_dtype], device=dev)
    lse = torch.empty(b.nnz_qo, b.num_qo_heads, dtype=torch.float32, device=dev)
    flush = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    kw = dict(q_scale=b.q_scale, k_scale=b.k_scale, v_scale=b.v_scale)
    stream = torch.cuda.current_stream()

    def loop(stage):
        for _ in range(warmup):
            flush.sum()
            plan.run_stage(stage, q, k, v, idx, o, lse, ws, **kw)
        torch.cuda.synchronize()
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
        for i in range(steps):
            flush.sum()
            ev[i][0].record(stream)
            plan.run_stage(stage, q, k, v, idx, o, lse, ws, **kw)
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        plan.device_status(ws)
        return statistics.mean(e[0].elapsed_time(e[1]) for e in ev)

    ms = loop(0)
    ms_dec = loop(1)
    gbs = nbytes / (ms * 1e-3) / 1e9
    peak, kind = measured_peaks()
    del q, k, v, idx, o, lse, ws, flush
    torch.cuda.empty_cache()
    return {"workload": WORKLOADS[index], "value": round(gbs, 1), "unit": "GB/s", "ms_per_step": round(ms, 5),
            "bytes_per_step": nbytes, "steps": steps, "num_ctas": int(meta[6]), "merge_rows": int(meta[9]),
            "decode_kernel_ms": round(ms_dec, 5),
            "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peak, "unit": "GB/s",
                         "frac": round(gbs / peak, 4), "peak_kind": kind,
                         "kernel_frac": round(nbytes / (ms_dec * 1e-3) / 1e9 / peak, 4),
                         "note": "whole step (decode + merge kernels); kernel_frac: the decode kernel alone"}}


def append_bytes(a) -> int:
    """Algorithmic bytes of one KV append: the new K and V rows read, their
    fp8 codes written, and each token's request index and position."""
    el = a.nnz * a.base.num_kv_heads * a.base.head_dim
    return 2 * el * a.k_new.element_size() + 2 * el + 8 * a.nnz


def time_append(index, dev, steps, warmup):
    """Device time of one pafp8_append_kv launch on a named append workload
    (inputs resident, L2 evicted before each timed sample); GB/s over its
    algorithmic bytes.  The one-token-per-request workload is timed as 20
    back-to-back launches per sample (a single launch of it is shorter than
    the host's launch call): the 20 launches are captured once in a CUDA
    graph and each sample replays it."""
    import torch

    import paged_attention_fp8_gb300 as pa
    from paged_attention_fp8_gb300.workloads import APPEND_WORKLOADS, append_workload

    a = append_workload(index)
    b = a.base
    nbytes = append_bytes(a)
    kn, vn = a.k_new.to(dev), a.v_new.to(dev)
    bi, ps = a.batch_indices.to(dev), a.positions.to(dev)
    ip, ix = b.kv_indptr.to(dev), b.kv_indices.to(dev)
    kc, vc = b.k_cache.to(dev), b.v_cache.to(dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    flush = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    def launch():  # on torch's current stream (the capture stream inside a graph capture)
        pa.pafp8_append_kv(kn, vn, bi, ps, ip, ix, kc, vc, k_scale=b.k_scale, v_scale=b.v_scale, status=st)

    reps = 20 if a.nnz < 1024 else 1
    for _ in range(warmup):
        flush.sum()
        launch()
    torch.cuda.synchronize()
    sample = launch
    if reps > 1:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for _ in range(reps):
                launch()
        sample = graph.replay
        for _ in range(warmup):
            sample()
        torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
    for i in range(steps):
        flush.sum()
        # A ~50 us device-side wait after the eviction keeps the host's launch
        # call ahead of the GPU, so the events bracket the append work alone
        # (a ~10 us launch is shorter than the host's launch path).
        torch.cuda._sleep(100_000)
        ev[i][0].record(stream)
        sample()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    if int(st.item()) != 0:
        raise RuntimeError("append skipped tokens on a well-formed workload")
    ms = statistics.median(e[0].elapsed_time(e[1]) for e in ev) / reps
    gbs = nbytes / (ms * 1e-3) / 1e9
    peak, kind = measured_peaks()
    del kn, vn, bi, ps, ip, ix, kc, vc, st, flush
    torch.cuda.empty_cache()
    return {"workload": APPEND_WORKLOADS[index], "tokens": a.nnz, "value": round(gbs, 1), "unit": "GB/s",
            "us_per_launch": round(ms * 1e3, 2), "bytes_per_launch": nbytes, "launches": steps * reps,
            "launches_per_sample": reps,
            "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peak, "unit": "GB/s",
                         "frac": round(gbs / peak, 4), "peak_kind": kind}}


def kernel_sha(*names: str) -> str:
    """SHA-256 of the named kernel sources, concatenated in order."""
    h = hashlib.sha256()
    for name in names:
        with open(os.path.join(ROOT, "paged_attention_fp8_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running.
    The summary covers the samples taken under load (the GPU-idle reason not
    active); idle stretches (host work between the timed parts) drop the SM
    clock and say nothing about the timed kernels."""

    FIELDS = ["index", "clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap",
              "clocks_event_reasons.gpu_idle"]

    def __init__(self, gpu_id: str):
        self.proc = None
        self.file = tempfile.NamedTemporaryFile(mode="w+", suffix=".csv", delete=False)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", gpu_id, "--query-gpu=" + ",".join(self.FIELDS),
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=self.file, stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        rows = [r for r in csv.reader(io.StringIO(self.file.read())) if len(r) == len(self.FIELDS)]
        self.file.close()
        os.unlink(self.file.name)
        return summarize_clocks(rows)


def summarize_clocks(rows):
    """Median SM clock, max clock and the throttle reasons seen, over the
    samples taken under load (rows of ClockSampler.FIELDS)."""
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    sm, mx, reasons, total = [], [], set(), 0
    for r in rows:
        if len(r) != len(ClockSampler.FIELDS):
            continue
        try:
            clk, cmax = float(r[1]), float(r[2])
        except ValueError:
            continue
        total += 1
        if r[9].strip().lower() == "active":  # idle GPU: not a timed stretch
            continue
        sm.append(clk)
        mx.append(cmax)
        for n, v in zip(names, r[5:9]):
            if v.strip().lower() == "active":
                reasons.add(n)
    if not sm:
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "samples_total": total}
    return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
            "samples": len(sm), "samples_total": total}


def gpu_id_for(torch, dev) -> str:
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return str(dev.index or 0)


def oracle_decode_sample(b, n: int):
    """Run the oracle on the first n requests (every query head); returns
    (seconds, algorithmic bytes of the sample, threads used)."""
    import numpy as np

    import oracle
    from paged_attention_fp8_gb300.workloads import raw_numpy

    raw = getattr(b, "_raw_cache", None)
    if raw is None:
        raw = dict(q=raw_numpy(b.q), k=raw_numpy(b.k_cache), v=raw_numpy(b.v_cache))
        b._raw_cache = raw
    rows = np.repeat(np.arange(n), b.num_qo_heads)
    heads = np.tile(np.arange(b.num_qo_heads), n)
    t0 = time.perf_counter()
    oracle.paged_attention(q=raw["q"], q_dtype=b.q_dtype, k_cache=raw["k"], v_cache=raw["v"],
                           kv_dtype=b.kv_dtype, qo_indptr=b.qo_indptr.numpy(),
                           kv_indptr=b.kv_indptr.numpy(), kv_indices=b.kv_indices.numpy(),
                           last_page_len=b.last_page_len.numpy(), num_qo_heads=b.num_qo_heads,
                           num_kv_heads=b.num_kv_heads, q_scale=b.q_scale, k_scale=b.k_scale,
                           v_scale=b.v_scale, sm_scale=b.sm_scale, causal=False, rows=rows,
                           heads=heads)
    dt = time.perf_counter() - t0
    kv_tokens = sum(b.kv_lens[:n])
    by = 2 * kv_tokens * b.num_kv_heads * b.head_dim + n * b.num_qo_heads * b.head_dim * 6 + \
        4 * int(b.kv_indptr[n])
    return dt, by, oracle.num_threads()


def oracle_sample_size(b, budget_s: float) -> int:
    """Requests per oracle sample so that one sample takes about budget_s."""
    dt, by, _ = oracle_decode_sample(b, 1)
    per_req = max(dt, 1e-4)
    return max(1, min(b.batch, int(budget_s / per_req)))


def oracle_prefill_sample(b, nrows: int):
    """Run the oracle on the last nrows new query rows of request 0 (every
    query head; the rows with the most admitted keys); returns (seconds, FLOPs
    over the admitted causal pairs, threads used)."""
    import numpy as np

    import oracle
    from paged_attention_fp8_gb300.workloads import raw_numpy

    qo, kv = b.qo_lens[0], b.kv_lens[0]
    nrows = max(1, min(nrows, qo))
    first = qo - nrows
    rows = np.repeat(np.arange(first, qo), b.num_qo_heads)
    heads = np.tile(np.arange(b.num_qo_heads), nrows)
    raw = getattr(b, "_raw_cache", None)
    if raw is None:
        raw = dict(q=raw_numpy(b.q), k=raw_numpy(b.k_cache), v=raw_numpy(b.v_cache))
        b._raw_cache = raw
    t0 = time.perf_counter()
    oracle.paged_attention(q=raw["q"], q_dtype=b.q_dtype, k_cache=raw["k"], v_cache=raw["v"],
                           kv_dtype=b.kv_dtype, qo_indptr=b.qo_indptr.numpy(),
                           kv_indptr=b.kv_indptr.numpy(), kv_indices=b.kv_indices.numpy(),
                           last_page_len=b.last_page_len.numpy(), num_qo_heads=b.num_qo_heads,
                           num_kv_heads=b.num_kv_heads, q_scale=b.q_scale, k_scale=b.k_scale,
                           v_scale=b.v_scale, sm_scale=b.sm_scale, causal=True, rows=rows,
                           heads=heads)
    dt = time.perf_counter() - t0
    keys = sum(kv - qo + i + 1 for i in range(first, qo))  # admitted keys of the sampled rows
    return dt, 4 * b.head_dim * b.num_qo_heads * keys, oracle.num_threads()


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.split(":")[0].strip() in ("Model name", "Model"):
                v = line.split(":", 1)[1].strip()
                if v and not v.isdigit():
                    return v
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu model")):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.machine()


def cpu_baseline(b_decode, b_prefill, budget_s: float = 6.0):
    """The oracle timed on this host's cores: the serving decode sample on
    every core and on one, and a prefill sample on every core.  Each sample
    is sized to about budget_s."""
    import oracle

    cores = oracle.num_threads()
    n = oracle_sample_size(b_decode, budget_s)
    dt, by, _ = oracle_decode_sample(b_decode, n)
    oracle.set_num_threads(1)
    try:
        n1 = max(1, min(n, int(budget_s / max(dt / n * cores, 1e-4))))
        dt1, by1, _ = oracle_decode_sample(b_decode, n1)
        rows1 = 8
        tp, fp, _ = oracle_prefill_sample(b_prefill, rows1)
    finally:
        oracle.set_num_threads(cores)
    rows = max(8, min(b_prefill.qo_lens[0], int(rows1 * budget_s / max(tp / cores, 1e-4))))
    tpa, fpa, _ = oracle_prefill_sample(b_prefill, rows)
    return {"value": round(by / dt / 1e9, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"serving decode: first {n} of {b_decode.batch} requests, every query head ({dt:.2f} s, fp64)",
            "value_1_thread": round(by1 / dt1 / 1e9, 4),
            "sample_1_thread": f"first {n1} requests ({dt1:.2f} s)",
            "prefill_tflops": round(fpa / tpa / 1e12, 5),
            "prefill_tflops_1_thread": round(fp / tp / 1e12, 6),
            "prefill_sample": f"ragged prefill: last {rows} (1 thread: {rows1}) rows of request 0, every query head "
                              f"({tpa:.2f} s / {tp:.2f} s)",
            "cpu": cpu_model()}


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    from paged_attention_fp8_gb300.workloads import WORKLOADS, workload

    b = workload(2)
    # Every step is the same bounded sample, sized so the whole run takes a
    # couple of minutes at most.
    budget = max(0.01, min(10.0, 120.0 / max(1, args.steps + args.warmup)))
    n = oracle_sample_size(b, budget)
    times, rates = [], []
    cores = 1
    for i in range(args.warmup + args.steps):
        dt, by, cores = oracle_decode_sample(b, n)
        if i >= args.warmup:
            rates.append(by / dt / 1e9)
            times.append(dt)
    value = statistics.median(rates)
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * statistics.median(times), 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOADS[2], "batch": b.batch, "num_qo_heads": b.num_qo_heads,
                   "num_kv_heads": b.num_kv_heads, "head_dim": b.head_dim, "page_size": b.page_size,
                   "kv_dtype": b.kv_dtype, "q_dtype": b.q_dtype, "o_dtype": b.o_dtype,
                   "parallelism": f"replicas{args.gpus}"},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": f"first {n} of {b.batch} requests, every query head, per step"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# (prefill CTAs, decode CTAs) pairs timed; None = every SM.
POD_SPLITS = ((-12, 12), (-16, 16), (-20, 20), (-24, 24), (-32, 32), (None, None), (None, 24), (-24, None),
              (None, 64))


def time_pod(dev, steps, warmup):
    """Prefill and decode over one pool (POD workload 10): device time of
    the two phases run one after the other, each on the whole GPU, against
    pafp8_run_pod with the SMs split between them, over a few splits."""
    import torch

    import paged_attention_fp8_gb300 as pa
    from paged_attention_fp8_gb300.workloads import POD_WORKLOADS, TORCH_DTYPES, pod_workload

    pb = pod_workload(10)
    pre, dec = pb.prefill, pb.decode
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    k = pre.k_cache.to(dev)
    v = pre.v_cache.to(dev)
    kw = dict(q_scale=pre.q_scale, k_scale=pre.k_scale, v_scale=pre.v_scale)

    def side(b, ctas):
        plan = pa.Plan(mode=b.mode, num_qo_heads=b.num_qo_heads, num_kv_heads=b.num_kv_heads,
                       num_pages=b.num_pages, kv_indptr=b.kv_indptr, last_page_len=b.last_page_len,
                       qo_indptr=b.qo_indptr if b.mode == "prefill" else None, q_dtype=b.q_dtype,
                       kv_dtype=b.kv_dtype, o_dtype=b.o_dtype, sm_scale=b.sm_scale, num_ctas=ctas)
        ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device=dev)
        plan.upload(ws)
        return plan, ws

    t = {}
    for name, b in (("p", pre), ("d", dec)):
        t[name] = dict(q=b.q.to(dev), idx=b.kv_indices.to(dev),
                       o=torch.empty(b.nnz_qo, b.num_qo_heads, b.head_dim, dtype=TORCH_DTYPES[b.o_dtype],
                                     device=dev),
                       lse=torch.empty(b.nnz_qo, b.num_qo_heads, dtype=torch.float32, device=dev))
    flush = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    def timed(call, plans):
        for _ in range(warmup):
            flush.sum()
            call()
        torch.cuda.synchronize()
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
        for i in range(steps):
            flush.sum()
            ev[i][0].record(stream)
            call()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        for plan, ws in plans:
            plan.device_status(ws)
        return statistics.median(e[0].elapsed_time(e[1]) for e in ev) * 1e3

    P, D = t["p"], t["d"]
    pp, pw = side(pre, 0)
    dp, dw = side(dec, 0)

    def sequential():
        pp.run(P["q"], k, v, P["idx"], P["o"], P["lse"], pw, **kw)
        dp.run(D["q"], k, v, D["idx"], D["o"], D["lse"], dw, **kw)
    seq_us = timed(sequential, [(pp, pw), (dp, dw)])
    sweep = {}
    for sp, sd in POD_SPLITS:
        npre = sms if sp is None else sms + sp
        ndec = sms if sd is None else sd
        pp2, pw2 = side(pre, npre)
        dp2, dw2 = side(dec, ndec)

        def pod():
            pa.pafp8_run_pod(pp2.handle, P["q"], P["idx"], P["o"], P["lse"], pw2, dp2.handle, D["q"], D["idx"],
                             D["o"], D["lse"], dw2, k, v, **kw)
        sweep[(npre, ndec)] = timed(pod, [(pp2, pw2), (dp2, dw2)])
        del pp2, pw2, dp2, dw2
    best = min(sweep, key=lambda x: sweep[x])
    out = {"workload": POD_WORKLOADS[10], "unit": "us per step", "higher_is_better": False,
           "sequential_us": round(seq_us, 2), "value": round(sweep[best], 2),
           "prefill_ctas": best[0], "decode_ctas": best[1], "gain": round(seq_us / sweep[best], 4),
           "sweep_us": {f"{a}+{b}": round(y, 2) for (a, b), y in sweep.items()},
           "prefill_tflops": round(pre.causal_flops() / (sweep[best] * 1e-6) / 1e12, 2),
           "decode_kv_gbs": round(decode_bytes(dec) / (sweep[best] * 1e-6) / 1e9, 2),
           "steps": steps,
           "note": "sequential = pafp8_run of the prefill then of the decode, each on every SM; value = "
                   "pafp8_run_pod with the plans' CTA counts of the best entry of sweep_us (keys: prefill "
                   "CTAs + decode CTAs; a sum above the SM count leaves the later CTAs waiting for SMs); "
                   "prefill_tflops and decode_kv_gbs are each phase's work over the whole POD step"}
    del k, v, t, P, D, flush, pp, pw, dp, dw
    torch.cuda.empty_cache()
    return out


def run_ours(args):
    import torch
    import torch.distributed as dist

    import paged_attention_fp8_gb300 as pa
    from paged_attention_fp8_gb300 import build as pbuild
    from paged_attention_fp8_gb300.workloads import TORCH_DTYPES, WORKLOADS, workload

    world, rank, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pbuild.build()
    # nvidia-smi samples from here to the end of the run (every timed part).
    sampler = ClockSampler(gpu_id_for(torch, dev)) if rank == 0 and args.mode in ("all", "decode") else None

    if args.mode == "prefill":
        res = {str(i): time_prefill(i, dev, args.prefill_steps, max(3, args.warmup)) for i in (4, 5, 7)}
        if rank == 0:
            print(json.dumps({"mode": "prefill", "prefill": res}), flush=True)
        if world > 1:
            dist.destroy_process_group()
        return

    if args.mode == "pod":
        res = time_pod(dev, args.prefill_steps, max(3, args.warmup))
        if rank == 0:
            print(json.dumps({"mode": "pod", "pod": res}), flush=True)
        if world > 1:
            dist.destroy_process_group()
        return

    if args.mode == "append":
        res = {str(i): time_append(i, dev, min(args.steps, 200), max(3, args.warmup)) for i in (8, 9)}
        if rank == 0:
            print(json.dumps({"mode": "append", "append_kv": res}), flush=True)
        if world > 1:
            dist.destroy_process_group()
        return

    b = workload(2)
    nbytes = decode_bytes(b)
    q = b.q.to(dev)
    k = b.k_cache.to(dev)
    v = b.v_cache.to(dev)
    idx = b.kv_indices.to(dev)
    plan = pa.Plan(mode="decode", num_qo_heads=b.num_qo_heads, num_kv_heads=b.num_kv_heads,
                   num_pages=b.num_pages, kv_indptr=b.kv_indptr, last_page_len=b.last_page_len,
                   q_dtype=b.q_dtype, kv_dtype=b.kv_dtype, o_dtype=b.o_dtype, sm_scale=b.sm_scale)
    meta = plan.metadata()
    num_ctas, num_merge = int(meta[6]), int(meta[9])
    ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device=dev)
    plan.upload(ws)
    o = torch.empty(b.batch, b.num_qo_heads, b.head_dim, dtype=TORCH_DTYPES[b.o_dtype], device=dev)
    lse = torch.empty(b.batch, b.num_qo_heads, dtype=torch.float32, device=dev)
    flush = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    scales = dict(q_scale=b.q_scale, k_scale=b.k_scale, v_scale=b.v_scale)
    stream = torch.cuda.current_stream()

    def step(ev=None, stage=0):
        if ev is not None:
            ev[0].record(stream)
        plan.run_stage(stage, q, k, v, idx, o, lse, ws, **scales)
        if ev is not None:
            ev[1].record(stream)

    for _ in range(args.warmup):
        flush.sum()
        step()
    torch.cuda.synchronize()
    plan.device_status(ws)

    launches_per_step = (1 if num_ctas > 0 else 0) + (1 if num_merge > 0 else 0)
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(args.steps):
        flush.sum()
        step(events[i])
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    wall = time.perf_counter() - t0
    plan.device_status(ws)
    step_ms = [e[0].elapsed_time(e[1]) for e in events]
    ms_step = statistics.mean(step_ms)
    # The decode kernel alone (stage 1), for its roofline: a second timed
    # loop, since an event between the two kernels of a step would also
    # separate the merge kernel from its programmatic launch.
    torch.cuda.synchronize()
    for i in range(args.steps):
        flush.sum()
        step(events[i], stage=1)
    torch.cuda.synchronize()
    dec_ms = [e[0].elapsed_time(e[1]) for e in events]
    ms_dec = statistics.mean(dec_ms)
    ms_step, ms_dec = max_over_ranks([ms_step, ms_dec], dev, world)

    # ---- end to end through the public API, every step: re-plan on the host,
    # then one pafp8_run_host call: it uploads the plan, copies the step's
    # inputs (q and kv_indices, pinned host memory) into the staging part of
    # the workspace, runs, and copies the result (o and lse) back into pinned
    # host memory; the host then waits for that result.  Two steps are in
    # flight, each with its own workspace, output buffers and stream: the host
    # plans and launches step i + 1 while the GPU runs step i (and its copies
    # overlap step i's kernels), then waits for step i's result.  The KV cache
    # stays resident in HBM: it is the state a decode step reads, not an input.
    q_h = b.q.contiguous().pin_memory()
    idx_h = b.kv_indices.contiguous().pin_memory()
    qb, ib = q_h.numel() * q_h.element_size(), idx_h.numel() * 4
    ob, lb = o.numel() * o.element_size(), lse.numel() * 4
    host_ws = plan.host_workspace_bytes(b.q_dtype)
    bufs = [dict(ws=torch.empty(host_ws, dtype=torch.uint8, device=dev),
                 o_h=torch.empty(tuple(o.shape), dtype=o.dtype).pin_memory(),
                 lse_h=torch.empty(tuple(lse.shape), dtype=torch.float32).pin_memory(),
                 stream=torch.cuda.Stream(), ev=torch.cuda.Event(), plan=None) for _ in range(2)]
    indptr_h, last_h = b.kv_indptr, b.last_page_len
    h2d = qb + ib + int(meta.size) * 4
    d2h = ob + lb
    e2e_steps = max(1, min(args.e2e_steps, args.steps))

    def new_plan():
        return pa.Plan(mode="decode", num_qo_heads=b.num_qo_heads, num_kv_heads=b.num_kv_heads,
                       num_pages=b.num_pages, kv_indptr=indptr_h, last_page_len=last_h,
                       q_dtype=b.q_dtype, kv_dtype=b.kv_dtype, o_dtype=b.o_dtype, sm_scale=b.sm_scale)

    def launch(x):
        # x's buffers were last used two steps ago, whose result the host has
        # already waited for.
        x["plan"] = new_plan()
        x["plan"].run_host(q_h, k, v, idx_h, x["o_h"], x["lse_h"], x["ws"], stream=x["stream"], **scales)
        x["ev"].record(x["stream"])

    def e2e_loop(n, in_flight):
        for i in range(n):
            launch(bufs[i % in_flight])
            if in_flight == 1 or i > 0:
                bufs[(i - in_flight + 1) % in_flight]["ev"].synchronize()  # that step's result is on the host
        torch.cuda.synchronize()

    e2e = {}
    for in_flight in (1, 2):
        e2e_loop(3, in_flight)
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        t1 = time.perf_counter()
        e2e_loop(e2e_steps, in_flight)
        e2e[in_flight] = (time.perf_counter() - t1) / e2e_steps
    for x in bufs:
        x["plan"].device_status(x["ws"], stream=x["stream"])
    e2e_s, e2e_serial_s = max_over_ranks([e2e[2], e2e[1]], dev, world)
    # Where a step's time goes, one step at a time (medians over the e2e
    # steps): planning on the host, the run_host call (host time to enqueue
    # the upload, copies and kernels), and the wait until the result is on
    # the host.
    x0 = bufs[0]
    parts = {"plan": [], "run_host_call": [], "wait": []}
    for _ in range(e2e_steps):
        t = time.perf_counter()
        p2 = new_plan()
        parts["plan"].append(time.perf_counter() - t)
        t = time.perf_counter()
        p2.run_host(q_h, k, v, idx_h, x0["o_h"], x0["lse_h"], x0["ws"], stream=x0["stream"], **scales)
        parts["run_host_call"].append(time.perf_counter() - t)
        t = time.perf_counter()
        x0["stream"].synchronize()
        parts["wait"].append(time.perf_counter() - t)
    breakdown = {k2: round(statistics.median(v2) * 1e6, 1) for k2, v2 in parts.items()}
    del flush, bufs
    torch.cuda.empty_cache()

    detail = {}
    if args.mode == "all":
        w = max(3, min(args.warmup, 20))
        dsteps = min(max(args.steps, 20), 200)
        for i in (1, 3, 6):
            detail[i] = time_decode(i, dev, dsteps, w)
        for i in (4, 5, 7):
            detail[i] = time_prefill(i, dev, args.prefill_steps, max(3, min(args.warmup, 10)))
        append_res = {i: time_append(i, dev, min(args.steps, 200), w) for i in (8, 9)}
        pod_res = time_pod(dev, args.prefill_steps, max(3, min(args.warmup, 10)))

    if rank != 0:
        dist.destroy_process_group()
        return
    clocks = sampler.stop() if sampler else None

    peak, peak_kind = measured_peaks()
    achieved = nbytes / (ms_dec * 1e-3) / 1e9
    traffic = NCU_TRAFFIC.get(kernel_sha("decode.cu"))
    value = world * nbytes / (ms_step * 1e-3) / 1e9
    step_roof = {"bound": "hbm", "achieved": round(nbytes / (ms_step * 1e-3) / 1e9, 1), "peak": peak,
                 "unit": "GB/s", "frac": round(nbytes / (ms_step * 1e-3) / 1e9 / peak, 4)}
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(b, workload(4))

    def brief(d):
        r = d["roofline"]
        out = {"us": round(1e3 * d.get("ms_per_step", d.get("ms_per_launch", 0.0)), 2), "value": d["value"],
               "unit": d["unit"],
               "roofline": {"bound": r["bound"], "achieved": r["achieved"], "peak": r["peak"], "unit": r["unit"],
                            "frac": r["frac"], "traffic": r.get("traffic")}}
        if "kernel_frac" in r:
            out["roofline"]["kernel_frac"] = r["kernel_frac"]
        if "frac_of_dense_bf16" in r:
            out["roofline"]["frac_of_dense_bf16"] = r["frac_of_dense_bf16"]
        return out

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": f"{b.kv_dtype} KV -> f16 MMA, f32 accumulate ({b.q_dtype} q, {b.o_dtype} o)",
        "data": "synthetic",
        "config": {"workload": WORKLOADS[2], "bytes_per_step": nbytes, "parallelism": f"replicas{world}",
                   "l2": "evicted between timed steps by a 256 MiB read outside the events; KV 303 MB > L2",
                   "timed_region_s": round(wall, 4)},
        "roofline": {"bound": "hbm", "kernel": "decode_kernel", "achieved": round(achieved, 1),
                     "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "peak_kind": peak_kind, "traffic": traffic, "step_frac": step_roof["frac"]},
        "e2e": {"value": round(world * nbytes / e2e_s / 1e9, 2), "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_s * 1e3, 4),
                "in_flight": 2, "serial_ms_per_step": round(e2e_serial_s * 1e3, 4), "breakdown_us": breakdown},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
    }
    if args.mode == "all":
        line["configs"] = {
            "1_tiny_decode": brief(detail[1]),
            "2_serving_decode": {"us": round(ms_step * 1e3, 2), "value": round(value / world, 1), "unit": "GB/s",
                                 "roofline": dict(step_roof, traffic=traffic,
                                                  kernel_frac=round(achieved / peak, 4))},
            "3_long_context_decode": brief(detail[3]),
            "4_ragged_prefill": brief(detail[4]),
            "5_fp8_prefill": brief(detail[5]),
        }
    if cpu is not None:
        line["cpu_baseline"] = cpu
    # The full records first (one JSON line), the headline line last.
    if args.mode == "all":
        full = {"detail": True, "decode": {str(i): detail[i] for i in (1, 3, 6)},
                "prefill": {str(i): detail[i] for i in (4, 5, 7)},
                "append_kv": {"prefill_tokens": append_res[8], "decode_step": append_res[9]},
                "pod": pod_res}
        print(json.dumps(full), flush=True)
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def main():
    args = parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
