"""The no-allocation decode entry point against the workspace entry point.

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
from gpu_common import DeviceBatch, assert_close
from paged_attention_fp8_gb300.workloads import make_batch, workload

pytestmark = pytest.mark.gpu


def _noalloc(db: DeviceBatch, o, lse):
    b = db.batch
    pa.pafp8_run_decode_noalloc(db.plan.handle, db.q, db.k, db.v, db.kv_indices, o, lse,
                                q_scale=b.q_scale, k_scale=b.k_scale, v_scale=b.v_scale)


@pytest.mark.parametrize("which", ["serving", "ragged_empty"])
def test_noalloc_matches_workspace_entry_point_twice(cuda_device, which):
    if which == "serving":
        b = workload(2)  # split-KV with merge over every SM
        db = DeviceBatch(b, cuda_device)
    else:
        b = make_batch([0, 1, 17, 300, 2500, 0, 64], num_qo_heads=32, num_kv_heads=8, seed=77)
        db = DeviceBatch(b, cuda_device, num_ctas=24)
    db.run()
    ref_o, ref_lse = db.result()
    o = torch.empty_like(db.o)
    lse = torch.empty_like(db.lse)
    for _ in range(2):  # the scratch keeps the last call's bytes: run twice
        o.fill_(float("nan"))
        lse.fill_(float("nan"))
        _noalloc(db, o, lse)
        torch.cuda.synchronize()
        assert_close(o.double().cpu().numpy(), lse.double().cpu().numpy(), ref_o, ref_lse,
                     f"no-alloc {which}")


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
