"""HND (head-major) caches: the same kernels read them through differently
strided tensor maps, so every result must equal the NHD run bit for bit,
and the oracle (its own HND gather) agrees within the parity bound.  Pages
of 16 m tokens too: in HND the 16-token sub-page j of a page is token slots
16 j .. 16 j + 15 of each head's run of page_size slots."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import paged_attention_fp8_gb300 as pa
from common import oracle_on
from gpu_common import assert_close, run_gpu
from paged_attention_fp8_gb300.workloads import make_batch, new_tokens, raw_numpy, with_layout, workload

pytestmark = pytest.mark.gpu


def _both(b, dev, **kw):
    o1, l1 = run_gpu(b, dev, **kw)
    h = with_layout(b, "HND")
    o2, l2 = run_gpu(h, dev, **kw)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2), "HND differs from NHD"
    return h, o2, l2


@pytest.mark.parametrize("kv,q", [("e4m3fn", "bf16"), ("e5m2", "f16"), ("bf16", "bf16"), ("f16", "bf16")])
def test_decode_hnd(cuda_device, kv, q):
    b = make_batch([1, 17, 300, 1000, 2049], num_qo_heads=16, num_kv_heads=4, q_dtype=q, kv_dtype=kv,
                   seed=71, pool_pages=300)
    h, o, l = _both(b, cuda_device, num_ctas=9)
    ro, rl = oracle_on(h)
    assert_close(o, l, ro, rl, f"decode HND {q}/{kv}")


@pytest.mark.parametrize("q,kv", [("bf16", "e4m3fn"), ("e4m3fn", "e4m3fn"), ("bf16", "bf16")])
def test_prefill_hnd(cuda_device, q, kv):
    b = make_batch([300, 129, 77], [200, 129, 77], num_qo_heads=16, num_kv_heads=4, q_dtype=q, kv_dtype=kv,
                   seed=73, pool_pages=60)
    h, o, l = _both(b, cuda_device, num_ctas=7)
    ro, rl = oracle_on(h)
    assert_close(o, l, ro, rl, f"prefill HND {q}/{kv}")


def test_serving_decode_hnd_full_size(cuda_device):
    _both(workload(2), cuda_device)


@pytest.mark.parametrize("fmt", ["e4m3fn", "e5m2"])
def test_append_hnd(cuda_device, fmt):
    base = with_layout(make_batch([40, 129, 300], [40, 1, 77], num_qo_heads=8, num_kv_heads=4, kv_dtype=fmt,
                                  seed=79, pool_pages=40), "HND")
    a = new_tokens(base, src_dtype="bf16", seed=6)
    dev = cuda_device
    kc, vc = base.k_cache.to(dev), base.v_cache.to(dev)
    pa.pafp8_append_kv(a.k_new.to(dev), a.v_new.to(dev), a.batch_indices.to(dev), a.positions.to(dev),
                       base.kv_indptr.to(dev), base.kv_indices.to(dev), kc, vc, k_scale=base.k_scale,
                       v_scale=base.v_scale, kv_layout="HND")
    torch.cuda.synchronize()
    rk, rv, skipped = oracle.append_kv(
        fmt=fmt, k_new=oracle.as_f32(raw_numpy(a.k_new), "bf16"), v_new=oracle.as_f32(raw_numpy(a.v_new), "bf16"),
        batch_indices=a.batch_indices.numpy(), positions=a.positions.numpy(), kv_indptr=base.kv_indptr.numpy(),
        kv_indices=base.kv_indices.numpy(), k_cache=raw_numpy(base.k_cache), v_cache=raw_numpy(base.v_cache),
        k_scale=base.k_scale, v_scale=base.v_scale, kv_layout="HND")
    assert skipped == 0
    assert np.array_equal(raw_numpy(kc), rk) and np.array_equal(raw_numpy(vc), rv)


@pytest.mark.parametrize("P", [32, 64, 128])
@pytest.mark.parametrize("kv,q,d", [("e4m3fn", "bf16", 128), ("bf16", "bf16", 128), ("e5m2", "f16", 64),
                                    ("e4m3fn", "e4m3fn", 64)])
def test_decode_hnd_large_pages(cuda_device, P, kv, q, d):
    b = make_batch([1, 15, 33, 300, 2049], num_qo_heads=16, num_kv_heads=4, head_dim=d, q_dtype=q, kv_dtype=kv,
                   page_size=P, seed=181 + P, pool_pages=4200 // P)
    h, o, l = _both(b, cuda_device, num_ctas=11)
    ro, rl = oracle_on(h)
    assert_close(o, l, ro, rl, f"decode HND page_size {P} {q}/{kv} head_dim {d}")


@pytest.mark.parametrize("P", [32, 64])
@pytest.mark.parametrize("q,kv,d", [("bf16", "e4m3fn", 128), ("e4m3fn", "e4m3fn", 128), ("bf16", "bf16", 128),
                                    ("f16", "e5m2", 64), ("e4m3fn", "e4m3fn", 64), ("f16", "f16", 64)])
def test_prefill_hnd_large_pages(cuda_device, P, q, kv, d):
    b = make_batch([300, 129, 77], [200, 129, 50], num_qo_heads=16, num_kv_heads=4, head_dim=d, q_dtype=q,
                   kv_dtype=kv, page_size=P, seed=191 + P, pool_pages=1200 // P)
    h, o, l = _both(b, cuda_device, num_ctas=7)
    ro, rl = oracle_on(h)
    assert_close(o, l, ro, rl, f"prefill HND page_size {P} {q}/{kv} head_dim {d}")


@pytest.mark.parametrize("P,d", [(32, 128), (64, 64)])
def test_append_hnd_large_pages(cuda_device, P, d):
    base = with_layout(make_batch([40, 129, 300], [40, 1, 77], num_qo_heads=8, num_kv_heads=4, head_dim=d,
                                  page_size=P, seed=197 + P, pool_pages=800 // P), "HND")
    a = new_tokens(base, src_dtype="bf16", seed=7)
    dev = cuda_device
    kc, vc = base.k_cache.to(dev), base.v_cache.to(dev)
    pa.pafp8_append_kv(a.k_new.to(dev), a.v_new.to(dev), a.batch_indices.to(dev), a.positions.to(dev),
                       base.kv_indptr.to(dev), base.kv_indices.to(dev), kc, vc, k_scale=base.k_scale,
                       v_scale=base.v_scale, kv_layout="HND")
    torch.cuda.synchronize()
    rk, rv, skipped = oracle.append_kv(
        fmt="e4m3fn", k_new=oracle.as_f32(raw_numpy(a.k_new), "bf16"), v_new=oracle.as_f32(raw_numpy(a.v_new), "bf16"),
        batch_indices=a.batch_indices.numpy(), positions=a.positions.numpy(), kv_indptr=base.kv_indptr.numpy(),
        kv_indices=base.kv_indices.numpy(), k_cache=raw_numpy(base.k_cache), v_cache=raw_numpy(base.v_cache),
        k_scale=base.k_scale, v_scale=base.v_scale, kv_layout="HND")
    assert skipped == 0
    assert np.array_equal(raw_numpy(kc), rk) and np.array_equal(raw_numpy(vc), rv)
