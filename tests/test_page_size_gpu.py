"""Pages of 32, 64 and 128 tokens (NHD): against the oracle, which reads any
page size directly, and bit for bit against the same cache bytes described
as a table of 16-token pages (a page of 16 m tokens is m consecutive 16-token
pages), for decode, prefill and the append."""
from __future__ import annotations

import dataclasses

import numpy as np
import pytest
import torch

import oracle
import paged_attention_fp8_gb300 as pa
from common import oracle_on
from gpu_common import assert_close, run_gpu
from paged_attention_fp8_gb300.workloads import make_batch, new_tokens, raw_numpy

pytestmark = pytest.mark.gpu


def as_16_token_pages(b):
    """The same batch with every page of P = 16 m tokens split into m pages."""
    m = b.page_size // 16
    pool = b.k_cache.shape[0]
    kc = b.k_cache.reshape(pool * m, 16, *b.k_cache.shape[2:])
    vc = b.v_cache.reshape(pool * m, 16, *b.v_cache.shape[2:])
    indptr, indices, last = [0], [], []
    for i, kv in enumerate(b.kv_lens):
        pages = b.kv_indices[b.kv_indptr[i]:b.kv_indptr[i + 1]].tolist()
        n16 = (kv + 15) // 16
        sub = [p * m + s for p in pages for s in range(m)][:n16]
        indices += sub
        indptr.append(indptr[-1] + n16)
        last.append(kv - (n16 - 1) * 16 if n16 else 0)
    return dataclasses.replace(b, k_cache=kc, v_cache=vc, page_size=16, num_pages=pool * m,
                               kv_indptr=torch.tensor(indptr, dtype=torch.int32),
                               kv_indices=torch.tensor(indices, dtype=torch.int32),
                               last_page_len=torch.tensor(last, dtype=torch.int32))


def _run(b, dev, **kw):
    from gpu_common import DeviceBatch
    db = DeviceBatch(b, dev, **kw)
    db.run()
    return db.result()


@pytest.mark.parametrize("P", [32, 64, 128])
@pytest.mark.parametrize("kv,q", [("e4m3fn", "bf16"), ("bf16", "bf16"), ("e5m2", "f16")])
def test_decode_page_sizes(cuda_device, P, kv, q):
    b = make_batch([1, 15, 33, 300, 2049], num_qo_heads=16, num_kv_heads=4, q_dtype=q, kv_dtype=kv, page_size=P,
                   seed=91 + P, pool_pages=4200 // P)
    o, lse = _run(b, cuda_device, num_ctas=11)
    ro, rl = oracle_on(b)
    assert_close(o, lse, ro, rl, f"decode page_size {P} {q}/{kv}")
    o16, l16 = _run(as_16_token_pages(b), cuda_device, num_ctas=11)
    assert np.array_equal(o, o16) and np.array_equal(lse, l16)


@pytest.mark.parametrize("P", [32, 64])
@pytest.mark.parametrize("q,kv", [("bf16", "e4m3fn"), ("e4m3fn", "e4m3fn"), ("bf16", "bf16")])
def test_prefill_page_sizes(cuda_device, P, q, kv):
    b = make_batch([300, 129, 77], [200, 129, 50], num_qo_heads=16, num_kv_heads=4, q_dtype=q, kv_dtype=kv,
                   page_size=P, seed=97 + P, pool_pages=1200 // P)
    o, lse = _run(b, cuda_device, num_ctas=7)
    ro, rl = oracle_on(b)
    assert_close(o, lse, ro, rl, f"prefill page_size {P} {q}/{kv}")
    o16, l16 = _run(as_16_token_pages(b), cuda_device, num_ctas=7)
    assert np.array_equal(o, o16) and np.array_equal(lse, l16)


def test_out_of_range_page_with_large_pages_is_reported(cuda_device):
    b = make_batch([100, 70], num_qo_heads=8, num_kv_heads=2, page_size=32, seed=101, pool_pages=8)
    b.kv_indices = b.kv_indices.clone()
    b.kv_indices[1] = 2 ** 30  # would overflow if multiplied before the check
    from gpu_common import DeviceBatch
    db = DeviceBatch(b, cuda_device, num_ctas=3)
    db.run()
    with pytest.raises(pa.Pafp8Error) as ei:
        db.plan.device_status(db.ws)
    assert ei.value.status == 7  # PAFP8_ERR_BOUNDS


@pytest.mark.parametrize("P", [32, 64])
def test_append_page_sizes(cuda_device, P):
    base = make_batch([40, 129, 300], [40, 1, 77], num_qo_heads=8, num_kv_heads=4, page_size=P, seed=103 + P,
                      pool_pages=800 // P)
    a = new_tokens(base, src_dtype="bf16", seed=8)
    dev = cuda_device
    kc, vc = base.k_cache.to(dev), base.v_cache.to(dev)
    pa.pafp8_append_kv(a.k_new.to(dev), a.v_new.to(dev), a.batch_indices.to(dev), a.positions.to(dev),
                       base.kv_indptr.to(dev), base.kv_indices.to(dev), kc, vc, k_scale=base.k_scale,
                       v_scale=base.v_scale)
    torch.cuda.synchronize()
    rk, rv, skipped = oracle.append_kv(
        fmt="e4m3fn", k_new=oracle.as_f32(raw_numpy(a.k_new), "bf16"), v_new=oracle.as_f32(raw_numpy(a.v_new), "bf16"),
        batch_indices=a.batch_indices.numpy(), positions=a.positions.numpy(), kv_indptr=base.kv_indptr.numpy(),
        kv_indices=base.kv_indices.numpy(), k_cache=raw_numpy(base.k_cache), v_cache=raw_numpy(base.v_cache),
        k_scale=base.k_scale, v_scale=base.v_scale)
    assert skipped == 0
    assert np.array_equal(raw_numpy(kc), rk) and np.array_equal(raw_numpy(vc), rv)
