"""KV append parity: new tokens quantized into the paged fp8 cache on the GPU
against the CPU oracle, byte for byte over the whole cache (the rows written
and every row that must stay untouched), plus skipped tokens, special
values and an append followed by decode."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import paged_attention_fp8_gb300 as pa
from common import oracle_on
from gpu_common import assert_close, run_gpu
from paged_attention_fp8_gb300.workloads import (TORCH_DTYPES, append_workload, make_batch, new_tokens,
                                                 raw_numpy)

pytestmark = pytest.mark.gpu


def _oracle_src(t: torch.Tensor, src_dtype: str) -> np.ndarray:
    return oracle.as_f32(raw_numpy(t) if src_dtype != "f32" else t.numpy(), src_dtype)


def device_append(a, dev, *, kv_indices=None, status=True):
    b = a.base
    kc = b.k_cache.to(dev)
    vc = b.v_cache.to(dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev) if status else None
    pa.pafp8_append_kv(a.k_new.to(dev), a.v_new.to(dev), a.batch_indices.to(dev), a.positions.to(dev),
                       b.kv_indptr.to(dev), (b.kv_indices if kv_indices is None else kv_indices).to(dev),
                       kc, vc, k_scale=b.k_scale, v_scale=b.v_scale, status=st)
    torch.cuda.synchronize()
    return raw_numpy(kc), raw_numpy(vc), (int(st.item()) if status else None)


def oracle_append(a, *, kv_indices=None):
    b = a.base
    return oracle.append_kv(fmt=b.kv_dtype, k_new=_oracle_src(a.k_new, a.src_dtype),
                            v_new=_oracle_src(a.v_new, a.src_dtype), batch_indices=a.batch_indices.numpy(),
                            positions=a.positions.numpy(), kv_indptr=b.kv_indptr.numpy(),
                            kv_indices=(b.kv_indices if kv_indices is None else kv_indices).numpy(),
                            k_cache=raw_numpy(b.k_cache), v_cache=raw_numpy(b.v_cache),
                            k_scale=b.k_scale, v_scale=b.v_scale)


@pytest.mark.parametrize("src", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("fmt", ["e4m3fn", "e5m2"])
def test_append_bitwise_against_the_oracle(cuda_device, src, fmt):
    base = make_batch([40, 129, 300, 17], [40, 1, 77, 17], num_qo_heads=8, num_kv_heads=2, kv_dtype=fmt,
                      seed=31, pool_pages=50)
    a = new_tokens(base, src_dtype=src, seed=5, std=2.0)
    gk, gv, st = device_append(a, cuda_device)
    rk, rv, skipped = oracle_append(a)
    assert skipped == 0 and st == 0
    assert np.array_equal(gk, rk) and np.array_equal(gv, rv)


@pytest.mark.parametrize("fmt", ["e4m3fn", "e5m2"])
def test_special_values_and_ties(cuda_device, fmt):
    """+-0, +-inf, NaN, saturating magnitudes, subnormal-range values and exact
    midpoints between neighbouring codes (scale 1/4: fl32(1/scale) = 4 is
    exact, so y = 4x lands on the midpoint)."""
    base = make_batch([64], [64], num_qo_heads=4, num_kv_heads=1, kv_dtype=fmt, seed=37)
    base.k_scale = base.v_scale = 0.25
    table = oracle.fp8_table(fmt)
    fin = np.sort(np.unique(table[np.isfinite(table) & (table >= 0)]))
    mids = (fin[:-1] + fin[1:]) / 2
    vals = np.concatenate([[0.0, -0.0, np.inf, -np.inf, np.nan, 1e30, -1e30, 3e-45], mids, -mids,
                           fin * 1.0000001, -fin * 0.9999999]).astype(np.float32) / 4
    n = 64 * 128
    x = np.resize(vals, n).reshape(64, 1, 128).astype(np.float32)
    a = new_tokens(base, src_dtype="f32", seed=1)
    a.k_new = torch.from_numpy(x.copy())
    a.v_new = torch.from_numpy(-x.copy())
    gk, gv, _ = device_append(a, cuda_device)
    rk, rv, _ = oracle_append(a)
    for g, r in ((gk, rk), (gv, rv)):
        nan_r = np.isnan(table[r])
        assert np.array_equal(np.isnan(table[g]), nan_r)
        assert np.array_equal(g[~nan_r], r[~nan_r])


def test_out_of_range_tokens_are_skipped_and_reported(cuda_device):
    base = make_batch([50, 20], [10, 20], num_qo_heads=4, num_kv_heads=2, seed=41, pool_pages=12)
    a = new_tokens(base, src_dtype="bf16", seed=2)
    bi, ps = a.batch_indices.clone(), a.positions.clone()
    bi[0], ps[1], ps[2], bi[3] = 2, 64, -1, -1   # no request 2; past the pages; negative; negative
    a.batch_indices, a.positions = bi, ps
    kvi = base.kv_indices.clone()
    kvi[-1] = base.num_pages + 3                  # request 1's last page id out of the pool
    gk, gv, st = device_append(a, cuda_device, kv_indices=kvi)
    rk, rv, skipped = oracle_append(a, kv_indices=kvi)
    assert skipped == 4 + int((a.batch_indices == 1).logical_and(a.positions >= 16).sum())
    assert st == 1
    assert np.array_equal(gk, rk) and np.array_equal(gv, rv)
    # without a status word the same tokens are written
    gk2, gv2, _ = device_append(a, cuda_device, kv_indices=kvi, status=False)
    assert np.array_equal(gk2, rk) and np.array_equal(gv2, rv)


def test_append_then_decode(cuda_device):
    """One decode step's new tokens written by the GPU, then attended: the
    result matches the oracle's attention over the oracle-written cache."""
    base = make_batch([33, 300, 1000], num_qo_heads=16, num_kv_heads=4, seed=43, pool_pages=100)
    a = new_tokens(base, src_dtype="bf16", seed=3)
    gk, gv, _ = device_append(a, cuda_device)
    rk, rv, _ = oracle_append(a)
    assert np.array_equal(gk, rk) and np.array_equal(gv, rv)
    base.k_cache = torch.from_numpy(gk).view(TORCH_DTYPES[base.kv_dtype])
    base.v_cache = torch.from_numpy(gv).view(TORCH_DTYPES[base.kv_dtype])
    o, lse = run_gpu(base, cuda_device, num_ctas=6)
    ro, rl = oracle_on(base)
    assert_close(o, lse, ro, rl, "decode after append")


@pytest.mark.parametrize("index", [8, 9])
def test_named_append_workloads_full_size(cuda_device, index):
    a = append_workload(index)
    gk, gv, st = device_append(a, cuda_device)
    rk, rv, skipped = oracle_append(a)
    assert skipped == 0 and st == 0
    assert np.array_equal(gk, rk) and np.array_equal(gv, rv)
