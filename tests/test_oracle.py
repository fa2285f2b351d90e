"""Pins for the CPU oracle: checks against what the pages and the mathematics
fix, never against the oracle itself.  No GPU needed.

Each test is chosen so that a plausible mistake in the oracle fails it: a
wrong fp8 bias or special-code set (tables), a wrong gather index or cache
layout (brute force, dense re-layout, permutation), a wrong GQA mapping, a
shifted causal diagonal, a dropped or misplaced scale, a wrong LSE base or a
wrong merge weight.
"""
from __future__ import annotations

import math
import os

import numpy as np
import pytest
import torch

import brute
import oracle
from common import oracle_on
from paged_attention_fp8_gb300.workloads import TORCH_DTYPES, make_batch, raw_numpy, workload

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _spot_values():
    rows = []
    with open(os.path.join(GOLDEN, "fp8_spot_values.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            fmt, code, val = line.split()
            v = float(val) if val in ("nan", "inf", "-inf") else float.fromhex(val)
            rows.append((fmt, int(code, 16), v))
    return rows


def _page_number(key):
    with open(os.path.join(GOLDEN, "page_measurements.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line and line.split()[0] == key:
                return float(line.split()[1])
    raise KeyError(key)


# ---------------------------------------------------------------- fp8 tables

@pytest.mark.parametrize("fmt,code,value", _spot_values())
def test_fp8_spot_values(fmt, code, value):
    got = oracle.fp8_table(fmt)[code]
    if math.isnan(value):
        assert math.isnan(got)
    else:
        assert got == value and math.copysign(1.0, got) == math.copysign(1.0, value)


@pytest.mark.parametrize("fmt", ["e4m3fn", "e5m2"])
def test_fp8_table_matches_torch_cast(fmt):
    """All 256 codes against torch's float8 dtypes, an independent decoder."""
    ours = oracle.fp8_table(fmt)
    ref = torch.arange(256, dtype=torch.uint8).view(TORCH_DTYPES[fmt]).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    fin = ~np.isnan(ref)
    assert np.array_equal(ours[fin], ref[fin])


@pytest.mark.parametrize("fmt,n_nan,n_inf", [("e4m3fn", 2, 0), ("e5m2", 6, 2)])
def test_fp8_special_codes(fmt, n_nan, n_inf):
    t = oracle.fp8_table(fmt)
    assert int(np.isnan(t).sum()) == n_nan
    assert int(np.isinf(t).sum()) == n_inf
    fin = t[np.isfinite(t)]
    assert fin.max() == {"e4m3fn": 448.0, "e5m2": 57344.0}[fmt]


@pytest.mark.parametrize("fmt", ["e4m3fn", "e5m2"])
@pytest.mark.parametrize("wide", ["f16", "bf16"])
def test_fp8_values_exact_in_16bit(fmt, wide):
    """Every finite fp8 value is exactly a 16-bit float of either kind, so a
    kernel that widens fp8 to f16/bf16 before its matrix products loses
    nothing; GPU-vs-oracle differences are then accumulation order only."""
    t = oracle.fp8_table(fmt)
    fin = t[np.isfinite(t)]
    back = torch.tensor(fin, dtype=torch.float64).to(TORCH_DTYPES[wide]).to(torch.float64).numpy()
    assert np.array_equal(back, fin)


@pytest.mark.parametrize("dt", ["f16", "bf16"])
def test_16bit_decode_matches_torch_all_codes(dt):
    codes = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle.decode(dt, codes)
    ref = torch.from_numpy(codes.view(np.int16).copy()).view(TORCH_DTYPES[dt]).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    fin = ~np.isnan(ref)
    assert np.array_equal(ours[fin], ref[fin])


# ------------------------------------------------------------ brute force

TINY_CASES = [
    # kv_lens, qo_lens, Hq, Hkv, D, P, q_dtype, kv_dtype
    ([5, 1, 3], None, 4, 2, 8, 4, "bf16", "e4m3fn"),
    ([7, 9], None, 6, 3, 8, 4, "f16", "e5m2"),
    ([6, 4], [6, 2], 4, 1, 8, 4, "bf16", "e4m3fn"),
    ([10, 5], [3, 5], 2, 2, 4, 3, "e4m3fn", "e4m3fn"),
    ([9], [4], 8, 2, 8, 2, "e5m2", "e4m3fn"),
    ([33], None, 4, 4, 16, 16, "bf16", "e4m3fn"),
]


@pytest.mark.parametrize("case", TINY_CASES)
def test_oracle_matches_brute_force(case):
    kv, qo, hq, hkv, d, p, qd, kd = case
    b = make_batch(kv, qo, num_qo_heads=hq, num_kv_heads=hkv, head_dim=d, page_size=p,
                   q_dtype=qd, kv_dtype=kd, seed=7, pool_pages=sum((x + p - 1) // p for x in kv) + 3)
    o, lse = oracle_on(b)
    bo, blse = brute.attention(b)
    assert np.max(np.abs(o - bo)) < 1e-12
    assert np.max(np.abs(lse - blse)) < 1e-12


def test_oracle_matches_brute_force_on_tiny_named_workload():
    """The 4-request GQA-4 decode workload, whole."""
    b = workload(1)
    o, lse = oracle_on(b)
    bo, blse = brute.attention(b)
    assert np.max(np.abs(o - bo)) < 1e-12
    assert np.max(np.abs(lse - blse)) < 1e-12


# ----------------------------------------------------------- page table

def test_page_permutation_invariance():
    """Relabel the pool (move every page and rewrite kv_indices to match):
    the result must not change at all."""
    b = make_batch([37, 64, 100, 129], num_qo_heads=8, num_kv_heads=2, seed=3, pool_pages=64)
    o1, l1 = oracle_on(b)
    g = torch.Generator().manual_seed(11)
    perm = torch.randperm(b.num_pages, generator=g)  # new position of old page i
    k2 = torch.empty_like(b.k_cache.view(torch.uint8))
    v2 = torch.empty_like(k2)
    k2[perm] = b.k_cache.view(torch.uint8)
    v2[perm] = b.v_cache.view(torch.uint8)
    idx2 = perm[b.kv_indices.long()].to(torch.int32)
    o2, l2 = oracle_on(b, k_cache=k2.view(b.k_cache.dtype), v_cache=v2.view(b.v_cache.dtype),
                       kv_indices=idx2)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_gather_equals_dense_relayout():
    """The paged result equals attention over the same rows laid out densely
    (K_dense[t] = cache[kv_indices[t // P], t % P]), bit for bit."""
    b = make_batch([23, 50], [5, 50], num_qo_heads=4, num_kv_heads=2, head_dim=16,
                   page_size=8, seed=5, pool_pages=20)
    o, lse = oracle_on(b)
    kt = oracle.decode(b.kv_dtype, raw_numpy(b.k_cache)) * b.k_scale
    vt = oracle.decode(b.kv_dtype, raw_numpy(b.v_cache)) * b.v_scale
    qt = oracle.decode(b.q_dtype, raw_numpy(b.q)) * b.q_scale
    P = b.page_size
    for r in range(b.batch):
        pages = b.kv_indices[b.kv_indptr[r]:b.kv_indptr[r + 1]].tolist()
        L, qo = b.kv_lens[r], b.qo_lens[r]
        K = np.stack([kt[pages[t // P], t % P] for t in range(L)])
        V = np.stack([vt[pages[t // P], t % P] for t in range(L)])
        for i in range(qo):
            row = int(b.qo_indptr[r]) + i
            n_keys = i + L - qo + 1  # bottom-right causal: keys 0 .. i + L - qo
            do, dl = oracle.dense_attention_row(qt[row], K[:n_keys], V[:n_keys], b.num_kv_heads,
                                                b.sm_scale)
            assert np.array_equal(do, o[row]) and np.array_equal(dl, lse[row])


# ------------------------------------------------------ closed-form cases

def test_single_token_returns_v_times_scale():
    b = make_batch([1, 1, 1], num_qo_heads=4, num_kv_heads=2, seed=9, pool_pages=8)
    o, lse = oracle_on(b)
    vt = oracle.fp8_table(b.kv_dtype)
    kt = oracle.fp8_table(b.kv_dtype)
    g = b.num_qo_heads // b.num_kv_heads
    for r in range(3):
        page = int(b.kv_indices[r])
        for h in range(b.num_qo_heads):
            vrow = raw_numpy(b.v_cache)[page, 0, h // g]
            assert np.array_equal(o[r, h], vt[vrow] * b.v_scale)
            krow = kt[raw_numpy(b.k_cache)[page, 0, h // g]] * b.k_scale
            qrow = b.q[r, h].double().numpy()
            s0 = b.sm_scale * float(np.dot(qrow, krow))
            assert abs(lse[r, h] - s0) <= 1e-12 * max(1.0, abs(s0))


def test_constant_v_gives_constant_output():
    b = make_batch([40, 17], [9, 17], num_qo_heads=4, num_kv_heads=2, head_dim=16, seed=13,
                   pool_pages=12)
    code = 0x3A  # e4m3fn 1.25
    v = torch.full_like(b.v_cache.view(torch.uint8), code).view(b.v_cache.dtype)
    o, _ = oracle_on(b, v_cache=v)
    c = oracle.fp8_table("e4m3fn")[code] * b.v_scale
    assert np.max(np.abs(o - c)) <= 1e-14 * abs(c)


def test_empty_kv_gives_zero_and_minus_inf():
    b = make_batch([0, 5], num_qo_heads=2, num_kv_heads=1, head_dim=8, page_size=4, seed=1,
                   pool_pages=3)
    o, lse = oracle_on(b)
    assert np.all(o[0] == 0) and np.all(np.isneginf(lse[0]))
    assert np.all(np.isfinite(lse[1]))


def test_gqa_equals_repeated_mha():
    """Hq = g * Hkv with KV heads shared by contiguous query-head groups
    equals plain multi-head attention on K/V with each head repeated g times
    (head h reads KV head h // g, not h % Hkv)."""
    g = 3
    b = make_batch([20, 33], num_qo_heads=2 * g, num_kv_heads=2, head_dim=16, page_size=4,
                   seed=17, pool_pages=16)
    o, lse = oracle_on(b)
    k_rep = b.k_cache.view(torch.uint8).repeat_interleave(g, dim=2).view(b.k_cache.dtype)
    v_rep = b.v_cache.view(torch.uint8).repeat_interleave(g, dim=2).view(b.v_cache.dtype)
    mha = make_batch([20, 33], num_qo_heads=2 * g, num_kv_heads=2 * g, head_dim=16, page_size=4,
                     seed=17, pool_pages=16)
    o2, l2 = oracle_on(mha, q=b.q, k_cache=k_rep, v_cache=v_rep, kv_indices=b.kv_indices,
                       k_scale=b.k_scale, v_scale=b.v_scale)
    assert np.array_equal(o, o2) and np.array_equal(lse, l2)
    # The two KV heads hold different data, so a wrong group mapping shows.
    assert not np.allclose(o[:, 0], o[:, g])


def test_causal_square_is_lower_triangular_and_qo1_is_decode():
    b = make_batch([12], [12], num_qo_heads=2, num_kv_heads=1, head_dim=8, page_size=4,
                   seed=19, pool_pages=4)
    o, lse = oracle_on(b)
    o_full, _ = oracle_on(b, causal=False)
    # Row 0 sees only key 0: output is V row 0 exactly (rows differ beyond).
    vt = oracle.fp8_table(b.kv_dtype)
    page0 = int(b.kv_indices[0])
    assert np.array_equal(o[0, 0], vt[raw_numpy(b.v_cache)[page0, 0, 0]] * b.v_scale)
    # The last row sees every key: it equals the unmasked result.
    assert np.array_equal(o[-1], o_full[-1])
    assert not np.allclose(o[5], o_full[5])
    # qo_len = 1 under the causal rule admits every key: identical to decode.
    d = make_batch([12], num_qo_heads=2, num_kv_heads=1, head_dim=8, page_size=4, seed=19,
                   pool_pages=4)
    od, ld = oracle_on(d)
    op, lp = oracle_on(d, causal=True)
    assert np.array_equal(od, op) and np.array_equal(ld, lp)


# ------------------------------------------------------------- scale folds

def test_scale_folds():
    """k_scale folds into sm_scale and v_scale is linear on the output, the
    two folds named in the test plan of "fp8 KV cache in the in-tree prefill
    kernel"; lse does not depend on v_scale."""
    b = make_batch([29, 64], [3, 1], num_qo_heads=4, num_kv_heads=2, head_dim=16, seed=23,
                   pool_pages=10)
    s = 0.37
    o1, l1 = oracle_on(b, k_scale=s, sm_scale=0.25)
    o2, l2 = oracle_on(b, k_scale=1.0, sm_scale=0.25 * s)
    assert np.max(np.abs(o1 - o2)) < 1e-12 and np.max(np.abs(l1 - l2)) < 1e-12
    o3, l3 = oracle_on(b, v_scale=s)
    o4, l4 = oracle_on(b, v_scale=1.0)
    assert np.max(np.abs(o3 - s * o4)) < 1e-12 * max(1.0, np.abs(o4).max())
    assert np.array_equal(l3, l4)
    # The fold matters: dropping k_scale changes the result.
    o5, _ = oracle_on(b, k_scale=1.0, sm_scale=0.25)
    assert np.max(np.abs(o5 - o1)) > 1e-3


def test_fp8_query_scale_folds_like_k_scale():
    b = make_batch([30], [4], num_qo_heads=4, num_kv_heads=2, head_dim=16, seed=29,
                   q_dtype="e4m3fn", pool_pages=4)
    o1, l1 = oracle_on(b, q_scale=0.5, k_scale=0.2, sm_scale=0.3)
    o2, l2 = oracle_on(b, q_scale=1.0, k_scale=1.0, sm_scale=0.3 * 0.5 * 0.2)
    assert np.max(np.abs(o1 - o2)) < 1e-12 and np.max(np.abs(l1 - l2)) < 1e-12


# ------------------------------------------------------------------- merge

def test_split_and_merge_equals_unsplit():
    """Attention over disjoint key subsets, combined by their LSE, equals
    attention over the union (decode: split a request's pages into chunks,
    each chunk a request of its own with the same query row)."""
    P = 4
    b = make_batch([45], num_qo_heads=4, num_kv_heads=2, head_dim=16, page_size=P, seed=31,
                   pool_pages=14)
    o, lse = oracle_on(b)
    pages = b.kv_indices.tolist()  # 12 pages, last holds 1 token
    cuts = [0, 3, 4, 9, 12]
    parts_o, parts_l = [], []
    for a, c in zip(cuts[:-1], cuts[1:]):
        last = int(b.last_page_len[0]) if c == len(pages) else P
        o_c, l_c = oracle_on(b, kv_indptr=torch.tensor([0, c - a], dtype=torch.int32),
                             kv_indices=torch.tensor(pages[a:c], dtype=torch.int32),
                             last_page_len=torch.tensor([last], dtype=torch.int32))
        parts_o.append(o_c[0])
        parts_l.append(l_c[0])
    for h in range(b.num_qo_heads):
        mo, ml = oracle.merge_states(np.stack([p[h] for p in parts_o]),
                                     np.array([p[h] for p in parts_l]))
        assert np.max(np.abs(mo - o[0, h])) < 1e-12
        assert abs(ml - lse[0, h]) < 1e-12
    # An empty partial state (lse = -inf) is ignored.
    mo, ml = oracle.merge_states(np.stack([parts_o[0][0], np.zeros(16)]),
                                 np.array([parts_l[0][0], -np.inf]))
    assert np.array_equal(mo, parts_o[0][0]) and ml == parts_l[0][0]


# ----------------------------------------------------- mixed 2-byte decode

def test_mixed_2byte_decode_agrees_with_bf16_bf16():
    """fp16 query with a bf16 cache vs bf16/bf16 decode: the page reports
    that the two agree to 0.0024.  In fp64 the only difference is the
    query's rounding (f16 vs bf16), so the oracle's gap must stay within the
    page's measured figure."""
    g = torch.Generator().manual_seed(37)
    B, Hq, Hkv, D, P = 8, 8, 2, 128, 16
    kv = [int(x) for x in torch.randint(64, 512, (B,), generator=g)]
    base = make_batch(kv, num_qo_heads=Hq, num_kv_heads=Hkv, head_dim=D, page_size=P, seed=41)
    qf = torch.randn(B, Hq, D, generator=g)
    kf = torch.randn(base.num_pages, P, Hkv, D, generator=g)
    vf = torch.randn(base.num_pages, P, Hkv, D, generator=g)
    kb, vb = kf.to(torch.bfloat16), vf.to(torch.bfloat16)
    kw = dict(k_cache=kb, v_cache=vb, kv_dtype="bf16", k_scale=1.0, v_scale=1.0)
    o_mixed, _ = oracle_on(base, q=qf.to(torch.float16), q_dtype="f16", **kw)
    o_bf, _ = oracle_on(base, q=qf.to(torch.bfloat16), q_dtype="bf16", **kw)
    gap = float(np.max(np.abs(o_mixed - o_bf)))
    assert 0 < gap <= _page_number("mixed_2byte_decode_max_abs_diff")


@pytest.mark.parametrize("mode", ["decode", "prefill"])
def test_hnd_layout_reads_the_same_rows(mode):
    """The head-major cache is the token-major one with (slot, head) swapped
    by numpy; the oracle's HND gather gives the same result bit for bit, and
    a gather that mixed slot and head (a wrong stride) would not."""
    from paged_attention_fp8_gb300.workloads import with_layout
    qo = None if mode == "decode" else [20, 5, 33]
    b = make_batch([20, 70, 33], qo, num_qo_heads=8, num_kv_heads=4, seed=61, pool_pages=12)
    o1, l1 = oracle_on(b)
    h = with_layout(b, "HND")
    assert h.k_cache.shape == (b.num_pages, 4, 16, 128)
    o2, l2 = oracle_on(h)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
    # the HND bytes read as NHD are a different cache, and give a different result
    o3, _ = oracle_on(b, k_cache=h.k_cache.view(b.k_cache.shape), v_cache=h.v_cache.view(b.v_cache.shape))
    assert not np.allclose(o1, o3)


@pytest.mark.parametrize("q_dtype", ["bf16", "e4m3fn"])
def test_per_head_scales_reduce_to_per_tensor_scales_head_by_head(q_dtype):
    """Per-head scale tensors: equal entries give the per-tensor result bit for
    bit, and with distinct entries every query head's output is the
    per-tensor result computed with that head's own scales (its KV head's k
    and v scales), so a scale applied to the wrong head fails."""
    mode_qo = [40, 9, 64]
    b = make_batch([40, 100, 64], mode_qo, num_qo_heads=8, num_kv_heads=2, q_dtype=q_dtype, seed=67,
                   pool_pages=16)
    hq, hkv = 8, 2
    same = oracle_on(b, q_scale=np.full(hq, b.q_scale), k_scale=np.full(hkv, b.k_scale),
                     v_scale=np.full(hkv, b.v_scale))
    ref = oracle_on(b)
    assert np.array_equal(same[0], ref[0]) and np.array_equal(same[1], ref[1])
    rng = np.random.default_rng(3)
    qs = rng.uniform(0.5, 2.0, hq) * b.q_scale if q_dtype == "e4m3fn" else np.ones(hq)
    ks = rng.uniform(0.5, 2.0, hkv) * b.k_scale
    vs = rng.uniform(0.5, 2.0, hkv) * b.v_scale
    o, lse = oracle_on(b, q_scale=qs, k_scale=ks, v_scale=vs)
    for h in range(hq):
        hk = h // (hq // hkv)
        oh, lh = oracle_on(b, q_scale=qs[h], k_scale=ks[hk], v_scale=vs[hk])
        assert np.allclose(o[:, h], oh[:, h], rtol=1e-12, atol=1e-15)
        assert np.allclose(lse[:, h], lh[:, h], rtol=1e-12, atol=1e-12)
    assert not np.allclose(o, ref[0])


@pytest.mark.parametrize("P", [32, 64])
def test_large_pages_read_as_16_token_pages(P):
    """A page of 16 m tokens is m consecutive 16-token pages: the oracle reads
    both descriptions of the same bytes to the same result bit for bit."""
    import dataclasses
    b = make_batch([1, 15, 33, 300], [1, 15, 20, 64], num_qo_heads=8, num_kv_heads=2, page_size=P, seed=71,
                   pool_pages=800 // P)
    m = P // 16
    pool = b.k_cache.shape[0]
    indptr, indices, last = [0], [], []
    for i, kv in enumerate(b.kv_lens):
        pages = b.kv_indices[b.kv_indptr[i]:b.kv_indptr[i + 1]].tolist()
        n16 = (kv + 15) // 16
        indices += [p * m + s for p in pages for s in range(m)][:n16]
        indptr.append(indptr[-1] + n16)
        last.append(kv - (n16 - 1) * 16 if n16 else 0)
    b16 = dataclasses.replace(b, k_cache=b.k_cache.reshape(pool * m, 16, 2, 128),
                              v_cache=b.v_cache.reshape(pool * m, 16, 2, 128), page_size=16,
                              num_pages=pool * m, kv_indptr=torch.tensor(indptr, dtype=torch.int32),
                              kv_indices=torch.tensor(indices, dtype=torch.int32),
                              last_page_len=torch.tensor(last, dtype=torch.int32))
    o1, l1 = oracle_on(b)
    o2, l2 = oracle_on(b16)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
