"""Running a seeded PagedBatch through libpafp8 on the GPU (tests only)."""
from __future__ import annotations

import numpy as np
import torch

import paged_attention_fp8_gb300 as pa
from paged_attention_fp8_gb300.workloads import TORCH_DTYPES, PagedBatch

# Parity bar: |o - ref| <= ATOL + RTOL * |ref| on the 16-bit outputs,
# |lse - ref| <= LSE_ATOL.
ATOL, RTOL, LSE_ATOL = 2e-2, 2e-2, 1e-3


class DeviceBatch:
    """Device copies of a batch's inputs plus a planned, uploaded workspace."""

    def __init__(self, batch: PagedBatch, device, **plan_kw):
        self.batch = batch
        self.device = device
        self.q = batch.q.to(device)
        self.k = batch.k_cache.to(device)
        self.v = batch.v_cache.to(device)
        self.kv_indices = batch.kv_indices.to(device)
        self.plan = pa.Plan(mode=batch.mode, num_qo_heads=batch.num_qo_heads,
                            num_kv_heads=batch.num_kv_heads, num_pages=batch.num_pages,
                            kv_indptr=batch.kv_indptr, last_page_len=batch.last_page_len,
                            qo_indptr=batch.qo_indptr if batch.mode == "prefill" else None,
                            q_dtype=batch.q_dtype, kv_dtype=batch.kv_dtype, o_dtype=batch.o_dtype,
                            sm_scale=batch.sm_scale, kv_layout=batch.kv_layout, page_size=batch.page_size,
                            head_dim=batch.head_dim,
                            **plan_kw)
        self.ws = torch.empty(self.plan.workspace_bytes, dtype=torch.uint8, device=device)
        self.plan.upload(self.ws)
        n = batch.nnz_qo
        self.o = torch.empty(n, batch.num_qo_heads, batch.head_dim, dtype=TORCH_DTYPES[batch.o_dtype],
                             device=device)
        self.lse = torch.empty(n, batch.num_qo_heads, dtype=torch.float32, device=device)

    def run(self, stage=None):
        kw = dict(q_scale=self.batch.q_scale, k_scale=self.batch.k_scale, v_scale=self.batch.v_scale)
        if stage is None:
            self.plan.run(self.q, self.k, self.v, self.kv_indices, self.o, self.lse, self.ws, **kw)
        else:
            self.plan.run_stage(stage, self.q, self.k, self.v, self.kv_indices, self.o, self.lse,
                                self.ws, **kw)

    def result(self):
        self.plan.device_status(self.ws)
        return self.o.double().cpu().numpy(), self.lse.double().cpu().numpy()


def run_gpu(batch: PagedBatch, device, **plan_kw):
    db = DeviceBatch(batch, device, **plan_kw)
    db.run()
    return db.result()


def assert_close(o, lse, ref_o, ref_lse, what=""):
    assert np.all(np.isfinite(o)), f"{what}: non-finite output"
    err = np.abs(o - ref_o) - (ATOL + RTOL * np.abs(ref_o))
    worst = np.unravel_index(np.argmax(err), err.shape)
    assert err.max() <= 0, (f"{what}: |o - ref| exceeds {ATOL} + {RTOL}|ref| at {worst}: "
                            f"got {o[worst]}, ref {ref_o[worst]}")
    fin = np.isfinite(ref_lse)
    assert np.array_equal(fin, np.isfinite(lse)), f"{what}: lse finiteness differs"
    if fin.any():
        dl = np.abs(lse[fin] - ref_lse[fin]).max()
        assert dl <= LSE_ATOL, f"{what}: |lse - ref| = {dl}"
    assert np.array_equal(np.isneginf(ref_lse), np.isneginf(lse))
