"""Glue between the seeded workloads and the CPU oracle (tests only)."""
from __future__ import annotations

import numpy as np

import oracle
from paged_attention_fp8_gb300.workloads import PagedBatch, raw_numpy


def oracle_on(batch: PagedBatch, rows=None, heads=None, **over):
    """Run the oracle on a PagedBatch.  Without a selection the result is
    reshaped to o [nnz_qo, Hq, D], lse [nnz_qo, Hq]."""
    kw = dict(
        q=raw_numpy(over.pop("q", batch.q)), q_dtype=over.pop("q_dtype", batch.q_dtype),
        k_cache=raw_numpy(over.pop("k_cache", batch.k_cache)),
        v_cache=raw_numpy(over.pop("v_cache", batch.v_cache)),
        kv_dtype=over.pop("kv_dtype", batch.kv_dtype),
        qo_indptr=over.pop("qo_indptr", batch.qo_indptr).numpy(),
        kv_indptr=over.pop("kv_indptr", batch.kv_indptr).numpy(),
        kv_indices=over.pop("kv_indices", batch.kv_indices).numpy(),
        last_page_len=over.pop("last_page_len", batch.last_page_len).numpy(),
        num_qo_heads=batch.num_qo_heads, num_kv_heads=batch.num_kv_heads,
        q_scale=over.pop("q_scale", batch.q_scale), k_scale=over.pop("k_scale", batch.k_scale),
        v_scale=over.pop("v_scale", batch.v_scale), sm_scale=over.pop("sm_scale", batch.sm_scale),
        causal=over.pop("causal", batch.causal), rows=rows, heads=heads,
        kv_layout=over.pop("kv_layout", batch.kv_layout))
    if over:
        raise TypeError(f"unknown overrides {sorted(over)}")
    o, lse = oracle.paged_attention(**kw)
    if rows is None:
        n = int(batch.qo_indptr[-1])
        return o.reshape(n, batch.num_qo_heads, batch.head_dim), lse.reshape(n, batch.num_qo_heads)
    return o, lse


def max_rel_excess(got: np.ndarray, ref: np.ndarray, atol: float, rtol: float) -> float:
    """max(|got-ref| - (atol + rtol*|ref|)); <= 0 means within tolerance."""
    return float(np.max(np.abs(got - ref) - (atol + rtol * np.abs(ref))))
