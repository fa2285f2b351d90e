"""Run-call modes: PAFP8_DEBUG (a launching call synchronizes and returns the
kernels' status), pafp8_run captured into a CUDA graph (bit-identical
replays) and pafp8_run_host (host buffers in and out), for decode and
prefill."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import paged_attention_fp8_gb300 as pa
from common import oracle_on
from gpu_common import DeviceBatch, assert_close
from paged_attention_fp8_gb300.workloads import make_batch, with_layout, workload

pytestmark = pytest.mark.gpu


def test_debug_mode_reports_a_bad_page_at_the_call(cuda_device, monkeypatch):
    b = workload(1)
    b.kv_indices = b.kv_indices.clone()
    b.kv_indices[3] = b.num_pages + 5
    db = DeviceBatch(b, cuda_device)
    monkeypatch.setenv("PAFP8_DEBUG", "1")
    with pytest.raises(pa.Pafp8Error) as ei:
        db.run()
    assert ei.value.status == 7  # PAFP8_ERR_BOUNDS, from the run call itself
    db.plan.device_status(db.ws)  # the status word was read and cleared


def test_debug_mode_is_silent_on_good_input(cuda_device, monkeypatch):
    b = make_batch([1, 40, 300], [1, 20, 129], num_qo_heads=8, num_kv_heads=2, seed=3)
    db = DeviceBatch(b, cuda_device, num_ctas=7)
    monkeypatch.setenv("PAFP8_DEBUG", "1")
    db.run()
    monkeypatch.setenv("PAFP8_DEBUG", "0")
    o, lse = db.result()
    ro, rl = oracle_on(b)
    assert_close(o, lse, ro, rl, "prefill under PAFP8_DEBUG")


@pytest.mark.parametrize("mode", ["decode", "prefill", "decode_head64_hnd32", "prefill_head64_hnd32"])
def test_run_replays_from_a_cuda_graph(cuda_device, mode):
    extra = dict(head_dim=64, page_size=32, pool_pages=200) if mode.endswith("hnd32") else {}
    if mode.startswith("decode"):
        b = make_batch([0, 17, 900, 2500], num_qo_heads=32, num_kv_heads=8, seed=31, **extra)
    else:
        b = make_batch([40, 300, 700], [40, 129, 256], num_qo_heads=32, num_kv_heads=8, seed=32, **extra)
    if mode.endswith("hnd32"):
        b = with_layout(b, "HND")
    db = DeviceBatch(b, cuda_device, num_ctas=24)
    db.run()
    o1, l1 = db.result()
    db.o.zero_()
    db.lse.zero_()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            db.run()
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    o2, l2 = db.result()
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


@pytest.mark.parametrize("mode", ["decode", "prefill_fp8"])
def test_run_host_matches_run(cuda_device, mode):
    """pafp8_run_host (q, kv_indices, o and lse in pinned host memory) gives
    pafp8_run's outputs bit for bit, within the oracle's bound."""
    if mode == "decode":
        b = make_batch([0, 17, 900, 2500], num_qo_heads=32, num_kv_heads=8, seed=33)
    else:
        b = make_batch([40, 300, 700], [40, 129, 256], num_qo_heads=32, num_kv_heads=8, q_dtype="e4m3fn",
                       kv_dtype="e4m3fn", seed=34)
    db = DeviceBatch(b, cuda_device, num_ctas=24)
    db.run()
    o1, l1 = db.result()
    ws = torch.empty(db.plan.host_workspace_bytes(b.q_dtype), dtype=torch.uint8, device=cuda_device)
    q_h = b.q.contiguous().pin_memory()
    idx_h = b.kv_indices.contiguous().pin_memory()
    o_h = torch.full(tuple(db.o.shape), float("nan"), dtype=db.o.dtype).pin_memory()
    lse_h = torch.full(tuple(db.lse.shape), float("nan"), dtype=torch.float32).pin_memory()
    db.plan.run_host(q_h, db.k, db.v, idx_h, o_h, lse_h, ws, q_scale=b.q_scale, k_scale=b.k_scale,
                     v_scale=b.v_scale)
    torch.cuda.synchronize()
    db.plan.device_status(ws)
    o2, l2 = o_h.double().numpy(), lse_h.double().numpy()
    assert np.array_equal(o2, o1) and np.array_equal(l2, l1)
    ro, rl = oracle_on(b)
    assert_close(o2, l2, ro, rl, f"run_host {mode}")
