"""Brute-force attention for tiny inputs, written independently of the oracle.

It shares nothing with ``oracle/``: element codes are decoded by torch's own
dtype casts (a second, independent decoder), the page table is walked with
Python loops, and the softmax is the explicit exp / sum with no running
max or rescaling.  Only for inputs of a few hundred keys at most.
"""
from __future__ import annotations

import math

import numpy as np
import torch


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.to(torch.float64).numpy()


def attention(batch, *, q=None, k_cache=None, v_cache=None, k_scale=None, v_scale=None,
              q_scale=None, sm_scale=None, causal=None):
    """Outputs for every (row, head) of a ``PagedBatch`` (fields overridable).
    Returns o [nnz_qo, Hq, D] and lse [nnz_qo, Hq] as fp64 numpy arrays."""
    q = batch.q if q is None else q
    k_cache = batch.k_cache if k_cache is None else k_cache
    v_cache = batch.v_cache if v_cache is None else v_cache
    k_scale = batch.k_scale if k_scale is None else k_scale
    v_scale = batch.v_scale if v_scale is None else v_scale
    q_scale = batch.q_scale if q_scale is None else q_scale
    sm_scale = batch.sm_scale if sm_scale is None else sm_scale
    causal = batch.causal if causal is None else causal

    qd = to_f64(q) * q_scale
    kd = to_f64(k_cache) * k_scale
    vd = to_f64(v_cache) * v_scale
    Hq, Hkv, D, P = batch.num_qo_heads, batch.num_kv_heads, batch.head_dim, batch.page_size
    group = Hq // Hkv
    qo_indptr = batch.qo_indptr.tolist()
    kv_indptr = batch.kv_indptr.tolist()
    kv_indices = batch.kv_indices.tolist()
    nnz = qo_indptr[-1]
    o = np.zeros((nnz, Hq, D))
    lse = np.full((nnz, Hq), -np.inf)
    for b in range(len(kv_indptr) - 1):
        kv_len = batch.kv_lens[b]
        qo_len = qo_indptr[b + 1] - qo_indptr[b]
        pages = kv_indices[kv_indptr[b]:kv_indptr[b + 1]]
        # Dense copies of this request's rows, token by token.
        K = np.zeros((kv_len, Hkv, D))
        V = np.zeros((kv_len, Hkv, D))
        for t in range(kv_len):
            K[t] = kd[pages[t // P], t % P]
            V[t] = vd[pages[t // P], t % P]
        for i in range(qo_len):
            r = qo_indptr[b] + i
            for h in range(Hq):
                hk = h // group
                keys = [j for j in range(kv_len) if (not causal) or j <= i + kv_len - qo_len]
                if not keys:
                    continue
                logits = np.array([sm_scale * float(np.dot(qd[r, h], K[j, hk])) for j in keys])
                w = np.exp(logits)  # tiny inputs: no overflow for the values used
                tot = w.sum()
                o[r, h] = sum(w[n] / tot * V[j, hk] for n, j in enumerate(keys))
                lse[r, h] = math.log(tot)
    return o, lse
