"""Prefill parity: ragged causal prefill on the tcgen05 path against the fp64
CPU oracle, element by element, plus page-indexing invariance and the named
prefill workloads (scaled-down in full, full size on sampled rows)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import paged_attention_fp8_gb300 as pa
from common import oracle_on
from gpu_common import assert_close, run_gpu
from paged_attention_fp8_gb300.workloads import make_batch, workload

pytestmark = pytest.mark.gpu


def test_single_small_request(cuda_device):
    b = make_batch([40], [40], num_qo_heads=8, num_kv_heads=2, seed=3)
    o, lse = run_gpu(b, cuda_device, num_ctas=4)
    ro, rl = oracle_on(b)
    assert_close(o, lse, ro, rl, "single square prefill")


@pytest.mark.parametrize("kv,qo", [
    ([5, 200], [5, 40]), ([129, 128, 127], [129, 1, 100]), ([300, 700], [300, 33]),
    ([1, 2, 3, 16, 17], [1, 1, 3, 16, 9])])
def test_ragged_prefix_and_tails(cuda_device, kv, qo):
    b = make_batch(kv, qo, num_qo_heads=8, num_kv_heads=2, seed=sum(kv))
    o, lse = run_gpu(b, cuda_device, num_ctas=7)
    ro, rl = oracle_on(b)
    assert_close(o, lse, ro, rl, f"ragged prefill {kv}/{qo}")


@pytest.mark.parametrize("hq,hkv", [(8, 8), (16, 2), (32, 8), (16, 1), (24, 8), (6, 2), (10, 2)])
def test_group_shapes(cuda_device, hq, hkv):
    b = make_batch([150, 290], [150, 70], num_qo_heads=hq, num_kv_heads=hkv, seed=hq + hkv)
    o, lse = run_gpu(b, cuda_device, num_ctas=9)
    ro, rl = oracle_on(b)
    assert_close(o, lse, ro, rl, f"prefill Hq {hq} Hkv {hkv}")


@pytest.mark.parametrize("q_dtype,kv_dtype,o_dtype", [
    ("bf16", "e4m3fn", "bf16"), ("f16", "e4m3fn", "f16"), ("bf16", "e5m2", "f16"),
    ("f16", "e5m2", "bf16"), ("e4m3fn", "e4m3fn", "bf16"), ("e4m3fn", "e5m2", "f16"),
    ("e5m2", "e4m3fn", "bf16")])
def test_dtype_combinations(cuda_device, q_dtype, kv_dtype, o_dtype):
    b = make_batch([260, 77], [200, 77], num_qo_heads=16, num_kv_heads=4, q_dtype=q_dtype,
                   kv_dtype=kv_dtype, o_dtype=o_dtype, seed=11)
    o, lse = run_gpu(b, cuda_device, num_ctas=11)
    ro, rl = oracle_on(b)
    assert_close(o, lse, ro, rl, f"prefill {q_dtype}/{kv_dtype}/{o_dtype}")


def test_large_bf16_query_range(cuda_device):
    b = make_batch([100], [60], num_qo_heads=8, num_kv_heads=2, seed=19, sm_scale=1e-6)
    b.q = (b.q.float() * 1e5).to(torch.bfloat16)
    o, lse = run_gpu(b, cuda_device, num_ctas=3)
    ro, rl = oracle_on(b)
    assert_close(o, lse, ro, rl, "prefill large query")


def test_page_permutation_is_bitwise_invariant(cuda_device):
    b = make_batch([333, 90], [120, 90], num_qo_heads=8, num_kv_heads=2, seed=23, pool_pages=40)
    o1, l1 = run_gpu(b, cuda_device, num_ctas=5)
    g = torch.Generator().manual_seed(5)
    perm = torch.randperm(b.num_pages, generator=g)
    k2 = torch.empty_like(b.k_cache.view(torch.uint8))
    v2 = torch.empty_like(k2)
    k2[perm] = b.k_cache.view(torch.uint8)
    v2[perm] = b.v_cache.view(torch.uint8)
    b.k_cache, b.v_cache = k2.view(b.k_cache.dtype), v2.view(b.v_cache.dtype)
    b.kv_indices = perm[b.kv_indices.long()].to(torch.int32)
    o2, l2 = run_gpu(b, cuda_device, num_ctas=5)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_qo_len_one_matches_decode(cuda_device):
    """One new token per request is decode; the two paths agree within the
    parity tolerance of each against the oracle."""
    kv = [37, 300, 1000]
    bp = make_batch(kv, [1, 1, 1], num_qo_heads=32, num_kv_heads=8, seed=29)
    op, lp = run_gpu(bp, cuda_device, num_ctas=6)
    ro, rl = oracle_on(bp)
    assert_close(op, lp, ro, rl, "prefill qo=1")
    bd = make_batch(kv, num_qo_heads=32, num_kv_heads=8, seed=29)
    od, ld = run_gpu(bd, cuda_device)
    assert_close(od, ld, ro, rl, "decode of the same rows")


def test_ragged_workload_scaled_down_all_outputs(cuda_device):
    """The ragged prefill workload's shape mix at 1/8 length, every output."""
    b = workload(4, scale_down=8)
    o, lse = run_gpu(b, cuda_device)
    ro, rl = oracle_on(b)
    assert_close(o, lse, ro, rl, "ragged prefill / 8")


def _sample_rows(b, n, seed):
    g = np.random.default_rng(seed)
    rows = g.integers(0, b.nnz_qo, n)
    heads = g.integers(0, b.num_qo_heads, n)
    # always include each request's first and last new row
    firsts = b.qo_indptr[:-1].numpy()
    lasts = b.qo_indptr[1:].numpy() - 1
    rows = np.concatenate([rows, firsts, lasts])
    heads = np.concatenate([heads, np.zeros_like(firsts), np.full_like(lasts, b.num_qo_heads - 1)])
    return rows, heads


def test_ragged_workload_full_size_sampled(cuda_device):
    b = workload(4)
    o, lse = run_gpu(b, cuda_device)
    rows, heads = _sample_rows(b, 160, 4)
    ro, rl = oracle_on(b, rows=rows, heads=heads)
    assert_close(o[rows, heads], lse[rows, heads], ro, rl, "ragged prefill full")
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse))


def test_fp8_workload_full_size_sampled(cuda_device):
    b = workload(5)
    o, lse = run_gpu(b, cuda_device)
    rows, heads = _sample_rows(b, 160, 5)
    ro, rl = oracle_on(b, rows=rows, heads=heads)
    assert_close(o[rows, heads], lse[rows, heads], ro, rl, "fp8 prefill full")
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse))


def test_fp8_output_refused(cuda_device):
    b = workload(5, scale_down=64)
    with pytest.raises(pa.Pafp8Error) as ei:
        pa.Plan(
            mode="prefill", num_qo_heads=32, num_kv_heads=8, num_pages=b.num_pages,
            kv_indptr=b.kv_indptr, last_page_len=b.last_page_len, qo_indptr=b.qo_indptr,
            q_dtype="e4m3fn", kv_dtype="e4m3fn", o_dtype="e4m3fn")
    assert ei.value.status == 1 and "float8_e4m3fn" in str(ei.value)


@pytest.mark.parametrize("dt", ["f16", "bf16"])
@pytest.mark.parametrize("kv,qo", [([260, 77], [200, 77]), ([129, 128, 127, 1000], [129, 1, 100, 333])])
def test_2byte_cache_of_the_query_dtype(cuda_device, dt, kv, qo):
    """A 16-bit cache of the query's dtype: K tiles come in by TMA as they
    are, V is transposed in shared memory; ragged rows, partial tiles."""
    b = make_batch(kv, qo, num_qo_heads=16, num_kv_heads=4, q_dtype=dt, kv_dtype=dt, o_dtype=dt,
                   seed=29 + len(kv))
    o, lse = run_gpu(b, cuda_device, num_ctas=11)
    ro, rl = oracle_on(b)
    assert_close(o, lse, ro, rl, f"prefill {dt} cache {kv}/{qo}")


@pytest.mark.parametrize("kv_dtype", ["e4m3fn", "e5m2"])
def test_fp8_cache_equals_its_f16_dequantization_bitwise(cuda_device, kv_dtype):
    """With an f16 query, the fp8 path dequantizes into the same f16 K and
    V^T tiles the 2-byte path builds from the widened cache, so both give
    bit-identical o and lse."""
    import dataclasses
    b = make_batch([260, 77, 1000], [200, 77, 150], num_qo_heads=16, num_kv_heads=4, q_dtype="f16",
                   kv_dtype=kv_dtype, o_dtype="f16", seed=31)
    o1, l1 = run_gpu(b, cuda_device, num_ctas=11)
    b16 = dataclasses.replace(b, kv_dtype="f16", k_cache=b.k_cache.to(torch.float16),
                              v_cache=b.v_cache.to(torch.float16))
    o2, l2 = run_gpu(b16, cuda_device, num_ctas=11)
    assert np.array_equal(o1, o2)
    assert np.array_equal(l1, l2)


@pytest.mark.parametrize("q_dtype", ["bf16", "e4m3fn"])
def test_output_only_16_byte_aligned(cuda_device, q_dtype):
    """o at 16 bytes past a 32-byte boundary (the interface asks for 16): the
    rows that are not written by bulk tensor stores take 16-byte stores, and
    the result is bitwise the same as with an aligned buffer."""
    from gpu_common import DeviceBatch
    b = make_batch([300, 150], [300, 90], num_qo_heads=8, num_kv_heads=2, q_dtype=q_dtype, seed=29)
    db = DeviceBatch(b, cuda_device, num_ctas=5)
    db.run()
    o1, l1 = db.result()
    big = torch.full((db.o.numel() + 8,), float("nan"), dtype=db.o.dtype, device=cuda_device)
    db.o = big[8:].view(db.o.shape)
    assert db.o.data_ptr() % 32 == 16
    db.run()
    o2, l2 = db.result()
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
    ro, rl = oracle_on(b)
    assert_close(o2, l2, ro, rl, f"prefill {q_dtype}, o 16-byte aligned")
