"""Decode parity: the CUDA path against the fp64 CPU oracle, element by
element, on seeded inputs (tolerance in gpu_common), plus the bit-exact page
indexing checks and the named workloads at full size."""
from __future__ import annotations

import dataclasses

import numpy as np
import pytest
import torch

from common import oracle_on
from gpu_common import DeviceBatch, assert_close, run_gpu
from paged_attention_fp8_gb300.workloads import make_batch, workload

pytestmark = pytest.mark.gpu


def test_tiny_named_workload_all_outputs(cuda_device):
    b = workload(1)
    o, lse = run_gpu(b, cuda_device)
    ro, rl = oracle_on(b)
    assert_close(o, lse, ro, rl, "tiny decode")


@pytest.mark.parametrize("plan_kw", [
    dict(num_ctas=1), dict(num_ctas=3), dict(num_ctas=1000), dict(fixed_split_pages=1),
    dict(fixed_split_pages=3), dict(disable_split_kv=True), dict(disable_split_kv=True, num_ctas=2)])
def test_tiny_workload_every_plan_mode(cuda_device, plan_kw):
    b = workload(1)
    o, lse = run_gpu(b, cuda_device, **plan_kw)
    ro, rl = oracle_on(b)
    assert_close(o, lse, ro, rl, f"tiny decode {plan_kw}")


RAGGED = [1, 2, 15, 16, 17, 31, 33, 100, 255, 256, 257, 1000]


@pytest.mark.parametrize("hq,hkv", [(8, 8), (8, 1), (16, 2), (24, 4), (64, 8), (24, 12), (6, 3), (5, 5)])
def test_group_and_head_block_shapes(cuda_device, hq, hkv):
    b = make_batch(RAGGED, num_qo_heads=hq, num_kv_heads=hkv, seed=hq * 31 + hkv,
                   pool_pages=sum((L + 15) // 16 for L in RAGGED) + 7)
    o, lse = run_gpu(b, cuda_device, num_ctas=20)
    ro, rl = oracle_on(b)
    assert_close(o, lse, ro, rl, f"Hq {hq} Hkv {hkv}")


@pytest.mark.parametrize("q_dtype,kv_dtype,o_dtype", [
    ("bf16", "e4m3fn", "bf16"), ("f16", "e4m3fn", "f16"), ("bf16", "e5m2", "f16"),
    ("f16", "e5m2", "bf16"), ("e4m3fn", "e4m3fn", "bf16"), ("e5m2", "e4m3fn", "f16"),
    ("e4m3fn", "e5m2", "bf16")])
def test_dtype_combinations(cuda_device, q_dtype, kv_dtype, o_dtype):
    b = make_batch(RAGGED, num_qo_heads=16, num_kv_heads=4, q_dtype=q_dtype, kv_dtype=kv_dtype,
                   o_dtype=o_dtype, seed=5, pool_pages=140)
    o, lse = run_gpu(b, cuda_device, num_ctas=16)
    ro, rl = oracle_on(b)
    assert_close(o, lse, ro, rl, f"{q_dtype}/{kv_dtype}/{o_dtype}")


def test_outliers_and_scales(cuda_device):
    """Heavy-tailed K/V (1% at x20) on e5m2 with small per-tensor scales, and
    a non-default sm_scale."""
    b = make_batch([700, 1300, 9], num_qo_heads=16, num_kv_heads=2, q_dtype="f16", kv_dtype="e5m2",
                   o_dtype="f16", kv_std=0.5, outlier_frac=0.01, seed=9, sm_scale=0.05)
    o, lse = run_gpu(b, cuda_device, num_ctas=7)
    ro, rl = oracle_on(b)
    assert_close(o, lse, ro, rl, "outliers")


def test_large_bf16_query_range(cuda_device):
    """A bf16 query beyond the f16 range is brought into range by an exact
    power-of-two scaling inside the kernel."""
    b = make_batch([64, 200], num_qo_heads=8, num_kv_heads=2, seed=13, sm_scale=1e-6)
    b.q = (b.q.float() * 1e5).to(torch.bfloat16)
    o, lse = run_gpu(b, cuda_device, num_ctas=4)
    ro, rl = oracle_on(b)
    assert_close(o, lse, ro, rl, "large query")


def test_empty_requests(cuda_device):
    b = make_batch([0, 40, 0, 1, 0], num_qo_heads=8, num_kv_heads=2, seed=17, pool_pages=6)
    for kw in (dict(num_ctas=2), dict(disable_split_kv=True), dict(fixed_split_pages=1)):
        o, lse = run_gpu(b, cuda_device, **kw)
        ro, rl = oracle_on(b)
        assert_close(o, lse, ro, rl, f"empty requests {kw}")
        assert np.all(o[0] == 0) and np.all(np.isneginf(lse[0]))


def test_all_requests_empty(cuda_device):
    b = make_batch([0, 0], num_qo_heads=4, num_kv_heads=4, seed=1, pool_pages=1)
    o, lse = run_gpu(b, cuda_device)
    assert np.all(o == 0) and np.all(np.isneginf(lse))


def test_page_permutation_is_bitwise_invariant(cuda_device):
    """Moving every page of the pool and relabelling kv_indices to match must
    not change a single output bit (page-table indexing is exact)."""
    b = workload(1)
    o1, l1 = run_gpu(b, cuda_device, num_ctas=5)
    g = torch.Generator().manual_seed(99)
    perm = torch.randperm(b.num_pages, generator=g)
    k2 = torch.empty_like(b.k_cache.view(torch.uint8))
    v2 = torch.empty_like(k2)
    k2[perm] = b.k_cache.view(torch.uint8)
    v2[perm] = b.v_cache.view(torch.uint8)
    b.k_cache, b.v_cache = k2.view(b.k_cache.dtype), v2.view(b.v_cache.dtype)
    b.kv_indices = perm[b.kv_indices.long()].to(torch.int32)
    o2, l2 = run_gpu(b, cuda_device, num_ctas=5)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_stray_bytes_do_not_leak(cuda_device):
    """Slots past a request's last token and pages no request owns hold NaN
    codes: the result must not change (they are masked, never mixed in)."""
    b = workload(1)
    o1, l1 = run_gpu(b, cuda_device)
    owned = torch.zeros(b.num_pages, 16, dtype=torch.bool)
    for r in range(b.batch):
        pages = b.kv_indices[b.kv_indptr[r]:b.kv_indptr[r + 1]].long()
        for t in range(b.kv_lens[r]):
            owned[pages[t // 16], t % 16] = True
    for name in ("k_cache", "v_cache"):
        raw = getattr(b, name).view(torch.uint8).clone()
        raw[~owned] = 0x7F  # e4m3fn NaN
        setattr(b, name, raw.view(torch.float8_e4m3fn))
    o2, l2 = run_gpu(b, cuda_device)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_out_of_range_page_is_reported_not_read(cuda_device):
    b = workload(1)
    b.kv_indices = b.kv_indices.clone()
    b.kv_indices[3] = b.num_pages + 5
    db = DeviceBatch(b, cuda_device)
    db.run()
    import paged_attention_fp8_gb300 as pa
    with pytest.raises(pa.Pafp8Error) as ei:
        db.plan.device_status(db.ws)
    assert ei.value.status == 7


def test_stages_compose(cuda_device):
    """Stage 1 (attention) then stage 2 (merge) equals the whole run, bit for bit."""
    b = make_batch([900, 37, 2500], num_qo_heads=32, num_kv_heads=8, seed=21)
    db = DeviceBatch(b, cuda_device, num_ctas=40)
    db.run()
    o1, l1 = db.result()
    db.o.zero_()
    db.lse.zero_()
    db.run(stage=1)
    db.run(stage=2)
    o2, l2 = db.result()
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_serving_workload_full_size(cuda_device):
    """64 requests, kv U[512,4096], GQA 32/8, e4m3fn, in the benchmark's launch
    configuration (balanced plan over every SM); every output checked."""
    b = workload(2)
    o, lse = run_gpu(b, cuda_device)
    ro, rl = oracle_on(b)
    assert_close(o, lse, ro, rl, "serving decode")


def test_long_context_workload_sampled(cuda_device):
    """8 x 32768 tokens, GQA 64/8, e5m2 with outliers, f16: split-KV plus
    merge.  Sampled (row, head) outputs against the oracle, all outputs finite."""
    b = workload(3)
    o, lse = run_gpu(b, cuda_device)
    g = np.random.default_rng(3)
    rows = g.integers(0, b.batch, 96)
    heads = g.integers(0, b.num_qo_heads, 96)
    ro, rl = oracle_on(b, rows=rows, heads=heads)
    assert_close(o[rows, heads], lse[rows, heads], ro, rl, "long-context decode")
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse))


def test_merge_many_partials_and_repeat_runs(cuda_device):
    """One-page splits give up to 256 partial states per (request, KV head),
    combined by the merge kernel; running the same plan again gives
    bit-identical results."""
    b = make_batch([4096, 1, 700, 0, 33], num_qo_heads=32, num_kv_heads=8, seed=41)
    db = DeviceBatch(b, cuda_device, fixed_split_pages=1)
    db.run()
    o1, l1 = db.result()
    ro, rl = oracle_on(b)
    assert_close(o1, l1, ro, rl, "one-page splits")
    for _ in range(2):
        db.o.zero_()
        db.lse.zero_()
        db.run()
        o2, l2 = db.result()
        assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_balanced_plan_on_few_ctas_repeats_bitwise(cuda_device):
    b = workload(1)
    db = DeviceBatch(b, cuda_device, num_ctas=3)
    db.run()
    o1, l1 = db.result()
    db.run()
    o2, l2 = db.result()
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


@pytest.mark.parametrize("q_dtype,kv_dtype,o_dtype", [
    ("f16", "f16", "f16"), ("bf16", "f16", "bf16"), ("bf16", "bf16", "bf16"), ("f16", "bf16", "f16")])
def test_2byte_cache(cuda_device, q_dtype, kv_dtype, o_dtype):
    """A 16-bit cache through the same decode kernel (ragged lengths, splits,
    every partial-page case), against the oracle."""
    b = make_batch(RAGGED, num_qo_heads=16, num_kv_heads=4, q_dtype=q_dtype, kv_dtype=kv_dtype,
                   o_dtype=o_dtype, seed=17, pool_pages=140)
    o, lse = run_gpu(b, cuda_device, num_ctas=16)
    ro, rl = oracle_on(b)
    assert_close(o, lse, ro, rl, f"{q_dtype} q / {kv_dtype} cache")


@pytest.mark.parametrize("kv_dtype", ["e4m3fn", "e5m2"])
@pytest.mark.parametrize("q_dtype", ["f16", "bf16"])
def test_fp8_cache_equals_its_f16_dequantization_bitwise(cuda_device, kv_dtype, q_dtype):
    """fp8 codes widen to f16 exactly, and the 2-byte path feeds the tensor
    cores the same operand words in the same order, so an fp8 cache and its
    f16 copy (same scales) give bit-identical o and lse, split or not."""
    b = make_batch(RAGGED, num_qo_heads=16, num_kv_heads=4, q_dtype=q_dtype, kv_dtype=kv_dtype, seed=23,
                   pool_pages=140)
    o1, l1 = run_gpu(b, cuda_device, num_ctas=16)
    b16 = dataclasses.replace(b, kv_dtype="f16", k_cache=b.k_cache.to(torch.float16),
                              v_cache=b.v_cache.to(torch.float16))
    o2, l2 = run_gpu(b16, cuda_device, num_ctas=16)
    assert np.array_equal(o1, o2)
    assert np.array_equal(l1, l2)


def test_2byte_cache_serving_size_sampled(cuda_device):
    """The serving workload's shape with a bf16 cache (600 MB of KV), sampled
    outputs against the oracle."""
    b = workload(6)
    o, lse = run_gpu(b, cuda_device)
    g = np.random.default_rng(6)
    rows = g.integers(0, b.batch, 64)
    heads = g.integers(0, b.num_qo_heads, 64)
    ro, rl = oracle_on(b, rows=rows, heads=heads)
    assert_close(o[rows, heads], lse[rows, heads], ro, rl, "serving decode, bf16 cache")


def test_serving_workload_repeats_bitwise_with_run_time_chunks(cuda_device):
    """The serving batch's plan hands part of its pages out at run time from
    a counter in the workspace (which the last CTA resets); whichever CTA takes
    a chunk, its partial state is the same, so repeated runs (and a run after
    the stage-by-stage path) are bit-identical."""
    b = workload(2)
    db = DeviceBatch(b, cuda_device)
    assert int(db.plan.metadata()[22]) > 0  # the plan has run-time chunks
    db.run()
    o1, l1 = db.result()
    for stage_by_stage in (False, True, False):
        db.o.zero_()
        db.lse.zero_()
        if stage_by_stage:
            db.run(stage=1)
            db.run(stage=2)
        else:
            db.run()
        o2, l2 = db.result()
        assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_more_ctas_than_sms_takes_the_merge_kernel(cuda_device):
    """With more CTAs than SMs the CTAs cannot all be resident, so the decode
    kernel does not merge itself (no grid barrier); the merge kernel does."""
    b = make_batch([3000, 1700, 900, 4096, 37], num_qo_heads=32, num_kv_heads=8, seed=45)
    sms = torch.cuda.get_device_properties(cuda_device).multi_processor_count
    for ctas in (sms, 3 * sms):
        o, lse = run_gpu(b, cuda_device, num_ctas=ctas)
        ro, rl = oracle_on(b)
        assert_close(o, lse, ro, rl, f"{ctas} CTAs")


def test_many_uploads_back_to_back(cuda_device):
    """Plan uploads go through a small page-locked staging ring; more plans
    than ring slots, uploaded back to back before any run, each keep their own
    metadata."""
    batches = [make_batch([17 + 150 * i, 900, 37 * i + 1], num_qo_heads=16, num_kv_heads=4, seed=60 + i)
               for i in range(7)]
    dbs = [DeviceBatch(bt, cuda_device, num_ctas=10 + 3 * i) for i, bt in enumerate(batches)]
    for db in dbs:
        db.run()
    for db, bt in zip(dbs, batches):
        o, lse = db.result()
        ro, rl = oracle_on(bt)
        assert_close(o, lse, ro, rl, "upload ring")
