"""The POD workload's shared page pool (host side, no GPU): the decode
requests' pages lie past the prefill pool and hold the decode batch's own
codes, so the oracle gives the same decode result on the shared pool as on
the decode batch's own pool read with the shared scales."""
from __future__ import annotations

import dataclasses

import numpy as np

from common import oracle_on
from paged_attention_fp8_gb300.workloads import make_batch, pod_batch, pod_workload


def test_pod_pool_is_disjoint_and_shared():
    pb = pod_workload(10, scale_down=16)
    pre, dec = pb.prefill, pb.decode
    assert pre.k_cache is dec.k_cache and pre.v_cache is dec.v_cache
    assert pre.num_pages == dec.num_pages == pre.k_cache.shape[0]
    pp = set(pre.kv_indices.tolist())
    dp = set(dec.kv_indices.tolist())
    assert not pp & dp
    assert max(pp) < min(dp) and max(dp) < pre.num_pages
    assert (pre.k_scale, pre.v_scale) == (dec.k_scale, dec.v_scale)


def test_pod_decode_reads_its_own_codes():
    pre = make_batch([40, 90], [8, 90], num_qo_heads=8, num_kv_heads=2, seed=5, pool_pages=12)
    dec = make_batch([0, 1, 33, 70], num_qo_heads=8, num_kv_heads=2, seed=6, pool_pages=10)
    pb = pod_batch(pre, dec)
    o, lse = oracle_on(pb.decode)
    own = dataclasses.replace(dec, k_scale=pre.k_scale, v_scale=pre.v_scale)
    ro, rl = oracle_on(own)
    assert np.array_equal(o, ro) and np.array_equal(lse, rl, equal_nan=True)
    o, lse = oracle_on(pb.prefill)
    ro, rl = oracle_on(pre)
    assert np.array_equal(o, ro) and np.array_equal(lse, rl, equal_nan=True)
