"""The no-allocation decode entry point against the workspace entry point and
the oracle.

Some callers of this library may not allocate device memory at all, e.g. a
plugin or enqueue callback inside an inference engine that owns every device
buffer and forbids cudaMalloc because it can synchronize the device.  For
them pafp8_run_decode_noalloc keeps the plan metadata and the split-KV
partial states in a scratch array built into the library.  This file is
collected last so that a run stopping at the first failure has already run
every other test; it passes both alone and after the others.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import paged_attention_fp8_gb300 as pa
from common import oracle_on
from gpu_common import DeviceBatch, assert_close
from paged_attention_fp8_gb300.workloads import make_batch, with_layout, workload

pytestmark = pytest.mark.gpu


def _noalloc(db: DeviceBatch, o, lse):
    b = db.batch
    pa.pafp8_run_decode_noalloc(db.plan.handle, db.q, db.k, db.v, db.kv_indices, o, lse,
                                q_scale=b.q_scale, k_scale=b.k_scale, v_scale=b.v_scale)


def _ragged_batch():
    return make_batch([0, 1, 17, 300, 2500, 0, 64], num_qo_heads=32, num_kv_heads=8, seed=77)


def _check_twice(db: DeviceBatch, ref_o, ref_lse, what: str):
    o = torch.empty_like(db.o)
    lse = torch.empty_like(db.lse)
    for _ in range(2):  # the scratch keeps the last call's bytes: run twice
        o.fill_(float("nan"))
        lse.fill_(float("nan"))
        _noalloc(db, o, lse)
        torch.cuda.synchronize()
        assert_close(o.double().cpu().numpy(), lse.double().cpu().numpy(), ref_o, ref_lse, what)


@pytest.mark.parametrize("which", ["serving", "ragged_empty"])
def test_noalloc_matches_workspace_entry_point_twice(cuda_device, which):
    if which == "serving":
        db = DeviceBatch(workload(2), cuda_device)  # split-KV with merge over every SM
    else:
        db = DeviceBatch(_ragged_batch(), cuda_device, num_ctas=24)
    db.run()
    ref_o, ref_lse = db.result()
    _check_twice(db, ref_o, ref_lse, f"no-alloc {which} vs pafp8_run")


@pytest.mark.parametrize("shape", ["head64", "hnd_page32", "head64_hnd_page64_fp8q"])
def test_noalloc_other_shapes_against_the_oracle(cuda_device, shape):
    """head_dim 64, head-major caches and large pages through the no-allocation
    call: the same bytes as the workspace entry point, and the oracle."""
    d = 64 if "head64" in shape else 128
    P = 64 if "page64" in shape else (32 if "page32" in shape else 16)
    q = "e4m3fn" if shape.endswith("fp8q") else "bf16"
    b = make_batch([0, 1, 33, 400, 2100], num_qo_heads=16, num_kv_heads=4, head_dim=d, page_size=P, q_dtype=q,
                   seed=223, pool_pages=3000 // P)
    if "hnd" in shape:
        b = with_layout(b, "HND")
    db = DeviceBatch(b, cuda_device, num_ctas=20)
    db.run()
    ref = db.result()
    ro, rl = oracle_on(b)
    _check_twice(db, ro, rl, f"no-alloc {shape} vs oracle")
    o = torch.empty_like(db.o)
    lse = torch.empty_like(db.lse)
    _noalloc(db, o, lse)
    torch.cuda.synchronize()
    assert np.array_equal(o.double().cpu().numpy(), ref[0]) and np.array_equal(lse.double().cpu().numpy(), ref[1])


def test_noalloc_serving_workload_against_the_oracle(cuda_device):
    """The serving decode batch (64 requests, split-KV over every SM) through
    the no-allocation call, compared with the fp64 oracle on every output."""
    b = workload(2)
    db = DeviceBatch(b, cuda_device)
    ro, rl = oracle_on(b)
    _check_twice(db, ro, rl, "no-alloc serving vs oracle")


def test_noalloc_plans_back_to_back(cuda_device):
    """A large plan, then a small one with a different partition, then the
    large one again: each call loads its own metadata into the shared scratch,
    so stale bytes from the previous plan never reach a result."""
    big = DeviceBatch(workload(2), cuda_device)
    small = DeviceBatch(_ragged_batch(), cuda_device, num_ctas=24)
    refs = {}
    for name, db in (("serving", big), ("ragged", small)):
        db.run()
        refs[name] = db.result()
    for name, db in (("serving", big), ("ragged", small), ("serving", big)):
        o = torch.full_like(db.o, float("nan"))
        lse = torch.full_like(db.lse, float("nan"))
        _noalloc(db, o, lse)
        torch.cuda.synchronize()
        assert_close(o.double().cpu().numpy(), lse.double().cpu().numpy(), *refs[name],
                     f"no-alloc {name} after the other plan")


def test_noalloc_debug_mode_reports_a_bad_page(cuda_device, monkeypatch):
    """With PAFP8_DEBUG set the call synchronizes and returns the kernels'
    status: a page index outside the pool comes back as PAFP8_ERR_BOUNDS."""
    b = workload(1)
    b.kv_indices = b.kv_indices.clone()
    b.kv_indices[3] = b.num_pages + 5
    db = DeviceBatch(b, cuda_device)
    monkeypatch.setenv("PAFP8_DEBUG", "1")
    with pytest.raises(pa.Pafp8Error) as ei:
        _noalloc(db, db.o, db.lse)
    assert ei.value.status == 7  # PAFP8_ERR_BOUNDS
    good = DeviceBatch(workload(1), cuda_device)
    _noalloc(good, good.o, good.lse)  # the status word was cleared: a good call is OK
    monkeypatch.setenv("PAFP8_DEBUG", "0")
    torch.cuda.synchronize()
    ro, rl = oracle_on(workload(1))
    assert_close(good.o.double().cpu().numpy(), good.lse.double().cpu().numpy(), ro, rl,
                 "no-alloc after a reported bad page")


def test_noalloc_refuses_plan_beyond_its_scratch(cuda_device):
    """One-page splits of a long batch need far more partial-state scratch
    than the built-in array holds: refused with a sentence, nothing launched."""
    B, Hq, Hkv, pages = 8, 64, 8, 2048  # 8 requests x 32768 tokens
    indptr = np.arange(B + 1, dtype=np.int32) * pages
    last = np.full(B, 16, dtype=np.int32)
    plan = pa.Plan(mode="decode", num_qo_heads=Hq, num_kv_heads=Hkv, num_pages=B * pages,
                   kv_indptr=indptr, last_page_len=last, q_dtype="f16", kv_dtype="e5m2",
                   o_dtype="f16", fixed_split_pages=1)
    assert plan.workspace_bytes > (16 << 20)
    q = torch.zeros(B, Hq, 128, dtype=torch.float16, device=cuda_device)
    o = torch.empty_like(q)
    lse = torch.empty(B, Hq, dtype=torch.float32, device=cuda_device)
    kv = torch.zeros(16, dtype=torch.uint8, device=cuda_device).view(torch.float8_e5m2)
    idx = torch.zeros(16, dtype=torch.int32, device=cuda_device)
    with pytest.raises(pa.Pafp8Error) as ei:
        pa.pafp8_run_decode_noalloc(plan.handle, q, kv, kv, idx, o, lse)
    assert ei.value.status == 4 and "built-in scratch" in str(ei.value)
