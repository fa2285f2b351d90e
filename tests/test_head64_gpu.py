"""head_dim 64 (the other head size the equivalence tests of "fp8 KV cache in
the in-tree prefill kernel" cover) against the oracle.  Decode: every cache
dtype, fp8 queries, split and unsplit rows, partial pages, both layouts,
large pages and per-head scales.  Prefill: every query/cache/output dtype
pairing, ragged causal rows with partial tiles, group shapes, large pages,
per-head scales, one new token per request against decode.  Both: the fp8
cache against its f16 widening bit for bit.  And the append at head_dim
64."""
from __future__ import annotations

import dataclasses

import numpy as np
import pytest
import torch

import oracle
import paged_attention_fp8_gb300 as pa
from common import oracle_on
from gpu_common import DeviceBatch, assert_close, run_gpu
from paged_attention_fp8_gb300.workloads import make_batch, new_tokens, raw_numpy, with_layout

pytestmark = pytest.mark.gpu

LENS = [1, 15, 16, 17, 100, 555, 2100]


@pytest.mark.parametrize("q,kv", [("bf16", "e4m3fn"), ("f16", "e5m2"), ("e4m3fn", "e4m3fn"),
                                  ("e5m2", "e5m2"), ("bf16", "bf16"), ("f16", "f16"), ("f16", "bf16")])
@pytest.mark.parametrize("hq,hkv", [(8, 2), (32, 8), (8, 8), (16, 2)])
def test_decode_head64(cuda_device, q, kv, hq, hkv):
    b = make_batch(LENS, num_qo_heads=hq, num_kv_heads=hkv, head_dim=64, q_dtype=q, kv_dtype=kv,
                   seed=107 + hq + hkv, pool_pages=300)
    for ctas in (152, 5):
        o, lse = run_gpu(b, cuda_device, num_ctas=ctas)
        ro, rl = oracle_on(b)
        assert_close(o, lse, ro, rl, f"decode head_dim 64 {q}/{kv} {hq}/{hkv} ctas {ctas}")


@pytest.mark.parametrize("kv", ["e4m3fn", "e5m2"])
def test_head64_fp8_cache_equals_its_f16_widening_bitwise(cuda_device, kv):
    b = make_batch(LENS, num_qo_heads=16, num_kv_heads=4, head_dim=64, q_dtype="f16", kv_dtype=kv, seed=109,
                   pool_pages=300)
    o1, l1 = run_gpu(b, cuda_device, num_ctas=20)
    b16 = dataclasses.replace(b, kv_dtype="f16", k_cache=b.k_cache.to(torch.float16),
                              v_cache=b.v_cache.to(torch.float16))
    o2, l2 = run_gpu(b16, cuda_device, num_ctas=20)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


@pytest.mark.parametrize("variant", ["hnd", "page32", "head_scales"])
def test_head64_variants(cuda_device, variant):
    b = make_batch(LENS, num_qo_heads=16, num_kv_heads=4, head_dim=64, q_dtype="bf16", kv_dtype="e4m3fn",
                   seed=113, pool_pages=300, page_size=32 if variant == "page32" else 16)
    if variant == "hnd":
        b = with_layout(b, "HND")
    if variant == "head_scales":
        db = DeviceBatch(b, cuda_device, num_ctas=20)
        rng = np.random.default_rng(4)
        ks = (rng.uniform(0.5, 2, 4) * b.k_scale).astype(np.float32)
        vs = (rng.uniform(0.5, 2, 4) * b.v_scale).astype(np.float32)
        db.plan.run_head_scales(db.q, db.k, db.v, db.kv_indices, db.o, db.lse, db.ws,
                                k_scales=torch.from_numpy(ks).to(cuda_device), v_scales=torch.from_numpy(vs).to(cuda_device))
        o, lse = db.result()
        ro, rl = oracle_on(b, k_scale=ks, v_scale=vs)
    else:
        o, lse = run_gpu(b, cuda_device, num_ctas=20)
        ro, rl = oracle_on(b)
    assert_close(o, lse, ro, rl, f"decode head_dim 64 {variant}")


def test_append_head64(cuda_device):
    base = make_batch([40, 129, 300], [40, 1, 77], num_qo_heads=8, num_kv_heads=4, head_dim=64, seed=127,
                      pool_pages=40)
    a = new_tokens(base, src_dtype="bf16", seed=9)
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


# ---------------------------------------------------------------- prefill

PKV, PQO = [1, 17, 129, 300, 700], [1, 9, 128, 33, 700]


@pytest.mark.parametrize("q,kv,o", [("bf16", "e4m3fn", "bf16"), ("f16", "e5m2", "f16"),
                                    ("bf16", "e5m2", "f16"), ("e4m3fn", "e4m3fn", "bf16"),
                                    ("e5m2", "e4m3fn", "f16"), ("e4m3fn", "e5m2", "bf16"),
                                    ("bf16", "bf16", "bf16"), ("f16", "f16", "f16")])
def test_prefill_head64_dtypes(cuda_device, q, kv, o):
    b = make_batch(PKV, PQO, num_qo_heads=16, num_kv_heads=4, head_dim=64, q_dtype=q, kv_dtype=kv,
                   o_dtype=o, seed=131, pool_pages=120)
    for ctas in (152, 7):
        oo, lse = run_gpu(b, cuda_device, num_ctas=ctas)
        ro, rl = oracle_on(b)
        assert_close(oo, lse, ro, rl, f"prefill head_dim 64 {q}/{kv}/{o} ctas {ctas}")


@pytest.mark.parametrize("hq,hkv", [(8, 8), (16, 2), (32, 8), (16, 1), (6, 2)])
def test_prefill_head64_groups(cuda_device, hq, hkv):
    b = make_batch([150, 290, 64], [150, 70, 64], num_qo_heads=hq, num_kv_heads=hkv, head_dim=64,
                   seed=137 + hq + hkv, pool_pages=60)
    oo, lse = run_gpu(b, cuda_device, num_ctas=9)
    ro, rl = oracle_on(b)
    assert_close(oo, lse, ro, rl, f"prefill head_dim 64 Hq {hq} Hkv {hkv}")


@pytest.mark.parametrize("q,kv", [("bf16", "e4m3fn"), ("e4m3fn", "e4m3fn"), ("bf16", "bf16")])
def test_prefill_head64_page32(cuda_device, q, kv):
    b = make_batch([300, 129, 77], [200, 129, 50], num_qo_heads=16, num_kv_heads=4, head_dim=64, q_dtype=q,
                   kv_dtype=kv, page_size=32, seed=139, pool_pages=40)
    oo, lse = run_gpu(b, cuda_device, num_ctas=7)
    ro, rl = oracle_on(b)
    assert_close(oo, lse, ro, rl, f"prefill head_dim 64 page_size 32 {q}/{kv}")


@pytest.mark.parametrize("kv", ["e4m3fn", "e5m2"])
def test_prefill_head64_fp8_cache_equals_its_f16_widening_bitwise(cuda_device, kv):
    b = make_batch([260, 77, 1000], [200, 77, 150], num_qo_heads=16, num_kv_heads=4, head_dim=64,
                   q_dtype="f16", kv_dtype=kv, o_dtype="f16", seed=149, pool_pages=120)
    o1, l1 = run_gpu(b, cuda_device, num_ctas=11)
    b16 = dataclasses.replace(b, kv_dtype="f16", k_cache=b.k_cache.to(torch.float16),
                              v_cache=b.v_cache.to(torch.float16))
    o2, l2 = run_gpu(b16, cuda_device, num_ctas=11)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


@pytest.mark.parametrize("q", ["bf16", "e4m3fn"])
def test_prefill_head64_head_scales(cuda_device, q):
    b = make_batch([300, 129], [200, 129], num_qo_heads=16, num_kv_heads=4, head_dim=64, q_dtype=q,
                   kv_dtype="e4m3fn", seed=151, pool_pages=40)
    db = DeviceBatch(b, cuda_device, num_ctas=5)
    rng = np.random.default_rng(6)
    qs = (rng.uniform(0.5, 2, 16) * b.q_scale).astype(np.float32) if q == "e4m3fn" else None
    ks = (rng.uniform(0.5, 2, 4) * b.k_scale).astype(np.float32)
    vs = (rng.uniform(0.5, 2, 4) * b.v_scale).astype(np.float32)
    t = lambda a: None if a is None else torch.from_numpy(a).to(cuda_device)
    db.plan.run_head_scales(db.q, db.k, db.v, db.kv_indices, db.o, db.lse, db.ws, q_scales=t(qs),
                            k_scales=t(ks), v_scales=t(vs))
    o, lse = db.result()
    ro, rl = oracle_on(b, q_scale=qs if qs is not None else b.q_scale, k_scale=ks, v_scale=vs)
    assert_close(o, lse, ro, rl, f"prefill head_dim 64 per-head scales {q}")


def test_prefill_head64_qo_len_one_matches_decode(cuda_device):
    kv = [37, 300, 1000]
    bp = make_batch(kv, [1, 1, 1], num_qo_heads=32, num_kv_heads=8, head_dim=64, seed=157, pool_pages=100)
    op, lp = run_gpu(bp, cuda_device, num_ctas=6)
    ro, rl = oracle_on(bp)
    assert_close(op, lp, ro, rl, "prefill head_dim 64 qo=1")
    bd = make_batch(kv, num_qo_heads=32, num_kv_heads=8, head_dim=64, seed=157, pool_pages=100)
    od, ld = run_gpu(bd, cuda_device)
    assert_close(od, ld, ro, rl, "decode head_dim 64 of the same rows")
