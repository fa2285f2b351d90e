"""Host-side checks of libpafp8 (no GPU): the library loads and exports every
entry point its header declares, the plan's partition words equal the
independently restated rule bit for bit, the partition covers every page
exactly once, and every refused dtype or shape combination returns a status
and a sentence instead of running."""
from __future__ import annotations

import ctypes
import os
import re

import numpy as np
import pytest
import torch

import paged_attention_fp8_gb300 as pa
from oracle import plan as plan_rule
from paged_attention_fp8_gb300 import build as pbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built_library():
    pbuild.build()
    return pa.lib()


def header_symbols():
    text = open(os.path.join(ROOT, "include", "pafp8.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pafp8_[a-z0-9_]+)\s*\(", text)))


def test_exports_every_declared_symbol():
    syms = header_symbols()
    assert "pafp8_run" in syms and "pafp8_plan_create" in syms
    L = ctypes.CDLL(pa.LIB_PATH)
    for s in syms:
        assert hasattr(L, s), f"{s} declared in include/pafp8.h but not exported"
    assert set(pa.EXPORTS) == set(syms)
    assert pa.pafp8_abi_version() == 1


# ------------------------------------------------------------------- plans

def _decode_plan(kv_lens, *, hq=32, hkv=8, num_ctas=152, page_size=16, **kw):
    P = page_size
    npages = [(L + P - 1) // P for L in kv_lens]
    indptr = np.concatenate([[0], np.cumsum(npages)]).astype(np.int32)
    last = np.array([(L - (n - 1) * P) if n else 0 for L, n in zip(kv_lens, npages)], dtype=np.int32)
    plan = pa.Plan(mode="decode", num_qo_heads=hq, num_kv_heads=hkv, num_pages=max(1, int(indptr[-1])),
                   kv_indptr=indptr, last_page_len=last, q_dtype="bf16", kv_dtype="e4m3fn",
                   num_ctas=num_ctas, page_size=P, **kw)
    ref = plan_rule.decode_metadata(indptr, last, num_qo_heads=hq, num_kv_heads=hkv,
                                    num_ctas=num_ctas, page_size=P,
                                    fixed_split_pages=kw.get("fixed_split_pages", 0),
                                    disable_split_kv=kw.get("disable_split_kv", False))
    return plan, np.array(ref, dtype=np.int32), [(L + 15) // 16 for L in kv_lens]


PLAN_CASES = [
    dict(kv_lens=[37, 64, 100, 129], hq=8, hkv=2, num_ctas=152),
    dict(kv_lens=[37, 64, 100, 129], hq=8, hkv=2, num_ctas=3),
    dict(kv_lens=[0, 5, 0, 300, 17], hq=8, hkv=8, num_ctas=7),
    dict(kv_lens=[32768] * 8, hq=64, hkv=8, num_ctas=152),
    dict(kv_lens=list(range(512, 4097, 57))[:64], hq=32, hkv=8, num_ctas=152),
    dict(kv_lens=[1000, 17, 4096], hq=32, hkv=8, num_ctas=152, fixed_split_pages=16),
    dict(kv_lens=[1000, 17, 4096], hq=32, hkv=8, num_ctas=2, disable_split_kv=True),
    dict(kv_lens=[100] * 5, hq=24, hkv=12, num_ctas=9),  # 12 KV heads -> blocks of 6
    dict(kv_lens=[0, 0], hq=4, hkv=4, num_ctas=152),
    dict(kv_lens=[], hq=4, hkv=4, num_ctas=152),
    dict(kv_lens=[37, 64, 100, 129, 3000], hq=8, hkv=2, num_ctas=11, page_size=32),
    dict(kv_lens=[1, 1000, 17, 4096], hq=32, hkv=8, num_ctas=152, page_size=64),
    dict(kv_lens=[129, 300], hq=8, hkv=8, num_ctas=5, page_size=128, fixed_split_pages=3),
]


@pytest.mark.parametrize("case", PLAN_CASES)
def test_plan_metadata_bit_exact(case):
    plan, ref, _ = _decode_plan(**case)
    got = plan.metadata()
    assert got.dtype == np.int32
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("case", PLAN_CASES)
def test_plan_partition_covers_every_page_once(case):
    plan, _, npages = _decode_plan(**case)
    m = plan.metadata()
    nhb = m[3]
    G, nseg = m[6], m[7]
    cta = m[m[12]:m[12] + G + 1]
    segs = m[m[13]:m[13] + 4 * nseg].reshape(-1, 4)
    chunks = m[m[23]:m[23] + 4 * m[22]].reshape(-1, 4)  # handed out at run time
    cover = {}
    for r, a, e, _ in np.concatenate([segs, chunks]):
        for p in range(a, e):
            key = (int(r), p)
            assert key not in cover
            cover[key] = 1
    want = {(b * nhb + hb, p) for b, n in enumerate(npages) for hb in range(nhb) for p in range(n)}
    assert set(cover) == want
    assert cta[0] == 0 and cta[-1] == nseg and np.all(np.diff(cta) >= 1)
    if not case.get("fixed_split_pages") and not case.get("disable_split_kv") and G > 0:
        loads = [int((segs[cta[i]:cta[i + 1], 2] - segs[cta[i]:cta[i + 1], 1]).sum()) for i in range(G)]
        assert max(loads) - min(loads) <= 1  # static shares balanced to within one page
        T = sum(n for n in npages for _ in range(nhb))
        R = len(npages) * nhb
        run_time = int((chunks[:, 2] - chunks[:, 1]).sum()) if len(chunks) else 0
        assert run_time == (sum(n // 16 for n in npages) * nhb if T >= 16 * G and 4 * R >= G else 0)
        assert all(e - a <= max(4, -(-run_time // G)) for _, a, e, _ in chunks)
        for r, a, e, _ in chunks:  # a row's chunks are its last pages
            assert e <= npages[int(r) // nhb] and a >= npages[int(r) // nhb] - npages[int(r) // nhb] // 16


def test_workspace_grows_with_partials():
    p1, _, _ = _decode_plan([4096] * 4, num_ctas=1)
    p2, _, _ = _decode_plan([4096] * 4, num_ctas=152)
    assert p2.workspace_bytes > p1.workspace_bytes > 0


# ---------------------------------------------------------------- refusals

def _desc(**over):
    d = dict(mode=0, batch=1, num_qo_heads=8, num_kv_heads=2, head_dim=128, page_size=16, num_pages=4,
             q_dtype=pa.BF16, kv_dtype=pa.E4M3FN, o_dtype=0, sm_scale=0.0, fixed_split_pages=0,
             disable_split_kv=0, num_ctas=4)
    d.update(over)
    return pa.plan_desc(**d)


def _create(**over):
    return pa.pafp8_plan_create(_desc(**over), np.array([0, 2], np.int32), np.array([5], np.int32))


@pytest.mark.parametrize("kv,words", [
    (pa.INT8, ["int8", "integer"]), (pa.UINT8, ["uint8", "integer"]), (pa.F32, ["float32"]),
    (99, ["unknown"])])
def test_plan_refuses_kv_dtype(kv, words):
    with pytest.raises(pa.Pafp8Error) as ei:
        _create(kv_dtype=kv)
    assert ei.value.status == 1
    for w in words:
        assert w in str(ei.value)


@pytest.mark.parametrize("kv", [pa.F16, pa.BF16])
@pytest.mark.parametrize("q", [pa.F16, pa.BF16])
def test_decode_plan_takes_2byte_cache_with_2byte_query(kv, q):
    # decode is exempt from the rule that the cache matches the query
    plan = _create(kv_dtype=kv, q_dtype=q)
    pa.pafp8_plan_destroy(plan)


@pytest.mark.parametrize("kv", [pa.F16, pa.BF16])
def test_decode_plan_refuses_fp8_query_with_2byte_cache(kv):
    with pytest.raises(pa.Pafp8Error) as ei:
        _create(kv_dtype=kv, q_dtype=pa.E4M3FN)
    assert ei.value.status == 1 and "fp8 query" in str(ei.value)


@pytest.mark.parametrize("q,kv", [(pa.F16, pa.BF16), (pa.BF16, pa.F16)])
def test_prefill_plan_refuses_2byte_cache_of_another_dtype(q, kv):
    with pytest.raises(pa.Pafp8Error) as ei:
        pa.pafp8_plan_create(_desc(mode=1, q_dtype=q, kv_dtype=kv), np.array([0, 2], np.int32),
                             np.array([5], np.int32), np.array([0, 3], np.int32))
    assert ei.value.status == 1 and "own dtype" in str(ei.value)


@pytest.mark.parametrize("kv", [pa.F16, pa.BF16])
def test_prefill_plan_takes_2byte_cache_of_the_query_dtype(kv):
    plan = pa.pafp8_plan_create(_desc(mode=1, q_dtype=kv, kv_dtype=kv), np.array([0, 2], np.int32),
                                np.array([5], np.int32), np.array([0, 3], np.int32))
    pa.pafp8_plan_destroy(plan)


@pytest.mark.parametrize("q", [pa.F32, pa.INT8, pa.UINT8, 42])
def test_plan_refuses_q_dtype(q):
    with pytest.raises(pa.Pafp8Error) as ei:
        _create(q_dtype=q)
    assert ei.value.status == 1


@pytest.mark.parametrize("o,word", [(pa.E4M3FN, "float8_e4m3fn"), (pa.E5M2, "float8_e5m2"),
                                    (pa.F32, "float32"), (pa.INT8, "int8")])
def test_plan_refuses_o_dtype(o, word):
    with pytest.raises(pa.Pafp8Error) as ei:
        _create(o_dtype=o)
    assert ei.value.status == 1 and word in str(ei.value)


@pytest.mark.parametrize("over,status", [
    (dict(num_qo_heads=6, num_kv_heads=4), 2), (dict(head_dim=96), 8), (dict(head_dim=32), 8), (dict(page_size=24), 8),
    (dict(page_size=0), 8),
    (dict(num_qo_heads=32, num_kv_heads=2), 8), (dict(mode=5), 3), (dict(num_ctas=-1), 3),
    (dict(fixed_split_pages=-2), 3), (dict(sm_scale=float("nan")), 3), (dict(kv_layout=2), 3)])
def test_plan_refuses_shapes_and_args(over, status):
    with pytest.raises(pa.Pafp8Error) as ei:
        _create(**over)
    assert ei.value.status == status and len(str(ei.value)) > 20


@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("d", [64, 128])
def test_plan_accepts_both_head_sizes_in_both_modes(mode, d):
    qo = np.array([0, 3], np.int32) if mode == 1 else None
    h = pa.pafp8_plan_create(_desc(mode=mode, head_dim=d), np.array([0, 2], np.int32), np.array([5], np.int32), qo)
    pa.pafp8_plan_destroy(h)


@pytest.mark.parametrize("layout", [0, 1])
@pytest.mark.parametrize("P", [32, 48, 256])
def test_plan_accepts_large_pages_in_both_layouts(layout, P):
    h = pa.pafp8_plan_create(_desc(page_size=P, kv_layout=layout), np.array([0, 2], np.int32),
                             np.array([5], np.int32))
    pa.pafp8_plan_destroy(h)


def test_plan_refuses_bad_page_table():
    with pytest.raises(pa.Pafp8Error, match="last_page_len"):
        pa.pafp8_plan_create(_desc(), np.array([0, 2], np.int32), np.array([17], np.int32))
    with pytest.raises(pa.Pafp8Error, match="last_page_len"):
        pa.pafp8_plan_create(_desc(), np.array([0, 2], np.int32), np.array([0], np.int32))
    with pytest.raises(pa.Pafp8Error, match="decreases"):
        pa.pafp8_plan_create(_desc(batch=2), np.array([0, 2, 1], np.int32), np.array([3, 3], np.int32))


def test_default_o_dtype():
    """o_data_type defaults to a 2-byte query's dtype and to bf16 for an fp8 query."""
    import paged_attention_fp8_gb300 as m
    for q, want in [(pa.F16, "float16"), (pa.BF16, "bfloat16"), (pa.E4M3FN, "bfloat16")]:
        h = _create(q_dtype=q)
        try:
            # A run with a mismatched o dtype names the planned one.
            other = pa.BF16 if want == "float16" else pa.F16
            st = m.lib().pafp8_run(h, q, 16, pa.E4M3FN, 16, pa.E4M3FN, 16, 16, 1.0, 1.0, 1.0, other,
                                   16, None, 256, 1 << 20, None)
            assert st == 1 and want in pa.pafp8_last_error()
        finally:
            pa.pafp8_plan_destroy(h)


@pytest.mark.parametrize("k,v,q,o,qs,status,word", [
    (pa.E4M3FN, pa.E5M2, pa.BF16, pa.BF16, 1.0, 1, "v_cache has float8_e5m2"),
    (pa.F16, pa.BF16, pa.BF16, pa.BF16, 1.0, 1, "k_cache has dtype float16 but v_cache has bfloat16"),
    (pa.INT8, pa.INT8, pa.BF16, pa.BF16, 1.0, 1, "integer"),
    (pa.E5M2, pa.E5M2, pa.BF16, pa.BF16, 1.0, 1, "plan was made for float8_e4m3fn"),
    (pa.E4M3FN, pa.E4M3FN, pa.F16, pa.BF16, 1.0, 1, "plan was made for bfloat16"),
    (pa.E4M3FN, pa.E4M3FN, pa.BF16, pa.E4M3FN, 1.0, 1, "refused"),
    (pa.E4M3FN, pa.E4M3FN, pa.BF16, pa.BF16, 0.5, 3, "silently ignored"),
])
def test_run_refuses_before_touching_memory(k, v, q, o, qs, status, word):
    """The run-time dtype checks come before any device access, so fake
    (never dereferenced) pointers suffice here."""
    h = _create()
    try:
        st = pa.lib().pafp8_run(h, q, 16, k, 16, v, 16, 16, qs, 1.0, 1.0, o, 16, None, 256, 1 << 20, None)
        assert st == status
        assert word in pa.pafp8_last_error()
    finally:
        pa.pafp8_plan_destroy(h)


def test_run_refuses_workspace_not_uploaded():
    h = _create()
    try:
        st = pa.lib().pafp8_run(h, pa.BF16, 16, pa.E4M3FN, 16, pa.E4M3FN, 16, 16, 1.0, 1.0, 1.0, pa.BF16,
                                16, None, 256, 1 << 20, None)
        assert st == 4 and "uploaded" in pa.pafp8_last_error()
    finally:
        pa.pafp8_plan_destroy(h)


def test_run_refuses_bad_scales():
    h = _create()
    try:
        for ks in (0.0, -1.0, float("inf"), float("nan")):
            st = pa.lib().pafp8_run(h, pa.BF16, 16, pa.E4M3FN, 16, pa.E4M3FN, 16, 16, 1.0, ks, 1.0,
                                    pa.BF16, 16, None, 256, 1 << 20, None)
            assert st == 3 and "scales" in pa.pafp8_last_error()
    finally:
        pa.pafp8_plan_destroy(h)


def test_run_host_refuses_a_small_workspace():
    """pafp8_run_host checks its workspace (the plan's bytes, then staging for
    q, kv_indices, o and lse) before any device work."""
    h = _create()
    try:
        need = pa.lib().pafp8_host_workspace_bytes(h, pa.BF16)
        assert need > pa.pafp8_workspace_bytes(h)
        assert pa.lib().pafp8_host_workspace_bytes(h, pa.E4M3FN) < need  # 1-byte q staging
        st = pa.lib().pafp8_run_host(h, pa.BF16, 16, pa.E4M3FN, 16, pa.E4M3FN, 16, 16, 1.0, 1.0, 1.0,
                                     pa.BF16, 16, None, 256, need - 1, None)
        assert st == 4 and "host-buffer step" in pa.pafp8_last_error()
    finally:
        pa.pafp8_plan_destroy(h)


# ------------------------------------------------------------ prefill plans

def _prefill_plan(kv_lens, qo_lens, *, hq=32, hkv=8, num_ctas=152, page_size=16, head_dim=128, kv_dtype="e4m3fn"):
    P = page_size
    npages = [(L + P - 1) // P for L in kv_lens]
    indptr = np.concatenate([[0], np.cumsum(npages)]).astype(np.int32)
    last = np.array([(L - (n - 1) * P) if n else 0 for L, n in zip(kv_lens, npages)], dtype=np.int32)
    qo_indptr = np.concatenate([[0], np.cumsum(qo_lens)]).astype(np.int32)
    plan = pa.Plan(mode="prefill", num_qo_heads=hq, num_kv_heads=hkv, num_pages=max(1, int(indptr[-1])),
                   kv_indptr=indptr, last_page_len=last, qo_indptr=qo_indptr, q_dtype="bf16",
                   kv_dtype=kv_dtype, num_ctas=num_ctas, page_size=P, head_dim=head_dim)
    ref = plan_rule.prefill_metadata(indptr, last, qo_indptr, num_qo_heads=hq, num_kv_heads=hkv,
                                     num_ctas=num_ctas, page_size=P, head_dim=head_dim, kv_dtype=kv_dtype)
    return plan, np.array(ref, dtype=np.int32)


PREFILL_CASES = [
    dict(kv_lens=[40], qo_lens=[40], hq=8, hkv=2),
    dict(kv_lens=[5, 200, 1000, 3000], qo_lens=[5, 40, 1000, 17], hq=32, hkv=8, num_ctas=7),
    dict(kv_lens=[129, 128, 127, 0], qo_lens=[129, 1, 100, 0], hq=16, hkv=1),
    dict(kv_lens=[300, 700], qo_lens=[300, 33], hq=24, hkv=8, num_ctas=2),
    dict(kv_lens=[2048] * 8, qo_lens=[2048] * 8, hq=32, hkv=8),
    dict(kv_lens=[100, 90], qo_lens=[60, 90], hq=6, hkv=2, num_ctas=1000),
    dict(kv_lens=[5, 200, 1000, 3000], qo_lens=[5, 40, 1000, 17], hq=32, hkv=8, num_ctas=7, page_size=64),
    dict(kv_lens=[5, 200, 1000, 3000], qo_lens=[5, 40, 1000, 17], hq=32, hkv=8, num_ctas=7, head_dim=64),
    # a 2-byte cache at head_dim 128 runs on CTA pairs (items of four tiles' tokens, even CTA counts)
    dict(kv_lens=[5, 200, 1000, 3000], qo_lens=[5, 40, 1000, 17], hq=32, hkv=8, num_ctas=7, kv_dtype="bf16"),
    dict(kv_lens=[129, 128, 127, 0], qo_lens=[129, 1, 100, 0], hq=16, hkv=1, num_ctas=1, kv_dtype="bf16"),
    dict(kv_lens=[2048] * 8, qo_lens=[2048] * 8, hq=32, hkv=8, kv_dtype="bf16"),
    dict(kv_lens=[300, 700], qo_lens=[300, 33], hq=24, hkv=8, num_ctas=5, head_dim=64, kv_dtype="bf16"),
]


def _pairs(case):
    return case.get("head_dim", 128) == 128 and case.get("kv_dtype", "e4m3fn") in ("f16", "bf16")


@pytest.mark.parametrize("case", PREFILL_CASES)
def test_prefill_plan_metadata_bit_exact(case):
    plan, ref = _prefill_plan(**case)
    assert np.array_equal(plan.metadata(), ref)


@pytest.mark.parametrize("case", PREFILL_CASES)
def test_prefill_tiles_cover_every_row_head_once(case):
    plan, _ = _prefill_plan(**case)
    m = plan.metadata()
    hq, hkv = case.get("hq", 32), case.get("hkv", 8)
    g = hq // hkv
    tq = int(m[20])
    tiles = m[m[19]:m[19] + 8 * int(m[18])].reshape(-1, 8)
    qo_ptr = np.concatenate([[0], np.cumsum(case["qo_lens"])])
    seen = set()
    for b, hk, t0, nkv, qo0, qo_len, kv_len, page0 in tiles:
        qo, kv = case["qo_lens"][b], case["kv_lens"][b]
        # the record repeats the request's own fields
        assert (qo0, qo_len, kv_len) == (qo_ptr[b], qo, kv)
        assert page0 == m[m[10] + b]
        span = (4 if _pairs(case) else 2) * tq  # two query tiles (of TQ tokens per CTA of a pair)
        for tok in range(t0, min(t0 + span, qo)):
            for h in range(hk * g, hk * g + g):
                assert (b, tok, h) not in seen
                seen.add((b, tok, h))
            # every key the token may see lies in the tile's KV tiles
            assert tok + kv - qo < nkv * 128
    want = {(b, t, h) for b, qo in enumerate(case["qo_lens"]) for t in range(qo) for h in range(hq)}
    assert seen == want
    assert list(tiles[:, 3]) == sorted(tiles[:, 3], reverse=True)
    if _pairs(case):
        assert m[6] % 2 == 0 and (m[6] > 0 or len(tiles) == 0)


@pytest.mark.parametrize("qo,kv,word", [([50], [40], "qo_len"), ([3, 2], [2, 5], "qo_len")])
def test_prefill_refuses_more_rows_than_keys(qo, kv, word):
    with pytest.raises(pa.Pafp8Error, match=word):
        _prefill_plan(kv, qo, hq=8, hkv=2)


def test_prefill_refusals():
    indptr = np.array([0, 2], np.int32)
    last = np.array([5], np.int32)
    with pytest.raises(pa.Pafp8Error, match="qo_indptr"):
        pa.Plan(mode="prefill", num_qo_heads=8, num_kv_heads=2, num_pages=4, kv_indptr=indptr,
                last_page_len=last, q_dtype="bf16", kv_dtype="e4m3fn", num_ctas=4)
    with pytest.raises(pa.Pafp8Error) as ei:
        pa.Plan(mode="prefill", num_qo_heads=64, num_kv_heads=2, num_pages=4, kv_indptr=indptr,
                last_page_len=last, qo_indptr=np.array([0, 3], np.int32), q_dtype="bf16",
                kv_dtype="e4m3fn", num_ctas=4)
    assert ei.value.status == 8 and "prefill" in str(ei.value)
    with pytest.raises(pa.Pafp8Error) as ei:
        pa.Plan(mode="prefill", num_qo_heads=8, num_kv_heads=2, num_pages=4, kv_indptr=indptr,
                last_page_len=last, qo_indptr=np.array([0, 3], np.int32), q_dtype="e4m3fn",
                kv_dtype="e4m3fn", o_dtype="e5m2", num_ctas=4)
    assert ei.value.status == 1


def _append_raw(**over):
    """pafp8_append_kv with plausible arguments (fake, aligned device
    addresses: every refusal below happens before any of them is used)."""
    a = dict(src=pa.BF16, k_new=0x10000, v_new=0x20000, nnz=4, hkv=2, d=128, bi=0x30000, pos=0x40000, batch=2,
             indptr=0x50000, indices=0x60000, kv=pa.E4M3FN, layout=0, k_cache=0x70000, v_cache=0x80000,
             num_pages=8, page_size=16, ks=0.5, vs=0.25, status=None)
    a.update(over)
    return pa.lib().pafp8_append_kv(a["src"], a["k_new"], a["v_new"], a["nnz"], a["hkv"], a["d"], a["bi"],
                                    a["pos"], a["batch"], a["indptr"], a["indices"], a["kv"], a["layout"],
                                    a["k_cache"], a["v_cache"], a["num_pages"], a["page_size"], a["ks"],
                                    a["vs"], a["status"], None)


@pytest.mark.parametrize("over,status,word", [
    (dict(src=pa.E4M3FN), 1, "append takes"), (dict(src=pa.INT8), 1, "int8"),
    (dict(kv=pa.BF16), 8, "bfloat16"), (dict(kv=pa.F16), 8, "float16"), (dict(kv=pa.UINT8), 1, "uint8"),
    (dict(kv=pa.F32), 1, "float32"), (dict(d=96), 8, "head_dim"), (dict(page_size=24), 8, "page_size"),
    (dict(hkv=0), 2, "num_kv_heads"), (dict(nnz=-1), 2, "negative"), (dict(ks=0.0), 3, "scales"),
    (dict(vs=float("inf")), 3, "scales"), (dict(layout=3), 3, "kv_layout"), (dict(k_new=None), 3, "non-NULL"),
    (dict(indices=None), 3, "non-NULL"), (dict(k_cache=0x70008), 3, "16-byte"), (dict(pos=0x40002), 3, "4-byte")])
def test_append_refuses_before_touching_memory(over, status, word):
    st = _append_raw(**over)
    assert st == status and word in pa.pafp8_last_error(), (st, pa.pafp8_last_error())


def test_append_of_nothing_is_a_no_op():
    assert _append_raw(nnz=0, k_new=None, v_new=None, k_cache=None, v_cache=None) == 0


@pytest.mark.parametrize("q,qs,ks,vs,word", [
    (pa.BF16, None, None, 64, "k_scales and v_scales"), (pa.BF16, None, 64, None, "k_scales and v_scales"),
    (pa.BF16, 64, 64, 64, "silently ignored"), (pa.E4M3FN, 66, 64, 64, "4-byte"),
    (pa.E4M3FN, None, 64, 62, "4-byte")])
def test_run_head_scales_refuses_before_touching_memory(q, qs, ks, vs, word):
    h = _create(q_dtype=q)
    try:
        st = pa.lib().pafp8_run_head_scales(h, q, 16, pa.E4M3FN, 16, pa.E4M3FN, 16, 16, qs, ks, vs, pa.BF16, 16,
                                            None, 256, 1 << 20, None)
        assert st == 3 and word in pa.pafp8_last_error(), pa.pafp8_last_error()
    finally:
        pa.pafp8_plan_destroy(h)


@pytest.mark.parametrize("case", PLAN_CASES)
def test_partial_slots_are_consecutive_per_merge_row(case):
    """The merge reads a split row's partial states at slots mptr[e] ..
    mptr[e+1]-1 without an index list: the slot list must be 0, 1, 2, ...
    and every partial segment's slot must lie in its own row's range, in page
    order."""
    plan, _, _ = _decode_plan(**case)
    m = plan.metadata()
    nseg, nparts, nmerge = int(m[7]), int(m[8]), int(m[9])
    segs = np.concatenate([m[m[13]:m[13] + 4 * nseg].reshape(-1, 4), m[m[23]:m[23] + 4 * m[22]].reshape(-1, 4)])
    mptr = m[m[14]:m[14] + nmerge + 1]
    mrow = m[m[15]:m[15] + nmerge]
    mslot = m[m[16]:m[16] + nparts]
    assert np.array_equal(mslot, np.arange(nparts))
    for e in range(nmerge):
        mine = sorted((int(p0), int(sl)) for r, p0, p1, sl in segs if r == mrow[e] and sl >= 0)
        assert [sl for _, sl in mine] == list(range(mptr[e], mptr[e + 1]))


# ---------------------------------------------------------------- POD refusals

def _pod_plans(pre=None, dec=None):
    hp = pa.pafp8_plan_create(_desc(mode=1, **(pre or {})), np.array([0, 2], np.int32),
                              np.array([5], np.int32), np.array([0, 5], np.int32))
    hd = _create(**(dec or {}))
    return hp, hd


def _pod_call(hp, hd, *, ws_p=1 << 20, ws_d=1 << 24, q=pa.BF16, swap=False):
    pre = pa.pod_phase(hp, 256, 16, 512, 1024, ws_p, 4096)
    dec = pa.pod_phase(hd, 256, 16, 512, 1024, ws_d, 4096)
    if swap:
        pre, dec = dec, pre
    return pa.lib().pafp8_run_pod(ctypes.byref(pre), ctypes.byref(dec), q, pa.E4M3FN, 16, pa.E4M3FN, 16,
                                  1.0, 1.0, 1.0, pa.BF16, None)


@pytest.mark.parametrize("case,status,word", [
    ("swap", 3, "decode plan"),
    ("pages", 2, "different caches"),
    ("heads", 2, "different caches"),
    ("overlap", 4, "overlap"),
    ("qdtype", 1, "plan was made for"),
])
def test_run_pod_refuses_before_any_launch(case, status, word):
    """Every refusal comes back before a CUDA call (none can succeed here:
    this host has no GPU, so reaching one would give ERR_CUDA instead)."""
    pre, dec = {}, {}
    if case == "pages":
        dec = dict(num_pages=8)
    if case == "heads":
        pre = dict(num_qo_heads=16, num_kv_heads=4)
    hp, hd = _pod_plans(pre, dec)
    try:
        kw = {}
        if case == "swap":
            kw["swap"] = True
        if case == "overlap":
            kw["ws_d"] = (1 << 20) + 2048
        if case == "qdtype":
            kw["q"] = pa.F16
        st = _pod_call(hp, hd, **kw)
        assert st == status and word in pa.pafp8_last_error(), pa.pafp8_last_error()
    finally:
        pa.pafp8_plan_destroy(hp)
        pa.pafp8_plan_destroy(hd)


def test_run_pod_refuses_missing_phase():
    st = pa.lib().pafp8_run_pod(None, None, pa.BF16, pa.E4M3FN, 16, pa.E4M3FN, 16, 1.0, 1.0, 1.0, pa.BF16,
                                None)
    assert st == 3 and "both phases" in pa.pafp8_last_error()


def test_run_pod_binding_passes_both_phases():
    """The Python wrapper marshals both phases: a cache mismatch between the
    two plans comes back as the C library's refusal (no GPU is touched)."""
    import torch
    hp, hd = _pod_plans(None, dict(num_pages=8))
    try:
        q = torch.zeros(5, 8, 128, dtype=torch.bfloat16)
        qd = torch.zeros(1, 8, 128, dtype=torch.bfloat16)
        kc = torch.zeros(8, 16, 2, 128, dtype=torch.uint8)
        idx = torch.zeros(2, dtype=torch.int32)
        o, od = torch.zeros_like(q), torch.zeros_like(qd)
        lse, lsed = torch.zeros(5, 8), torch.zeros(1, 8)
        wp, wd = torch.zeros(64, dtype=torch.uint8), torch.zeros(64, dtype=torch.uint8)
        with pytest.raises(pa.Pafp8Error) as ei:
            pa.pafp8_run_pod(hp, q, idx, o, lse, wp, hd, qd, idx, od, lsed, wd, kc, kc, k_dtype=pa.E4M3FN,
                             v_dtype=pa.E4M3FN, stream=0)
        assert ei.value.status == 2 and "different caches" in str(ei.value)
    finally:
        pa.pafp8_plan_destroy(hp)
        pa.pafp8_plan_destroy(hd)


@pytest.mark.parametrize("seed", range(6))
def test_random_plans_match_the_restated_rule(seed):
    """Seeded random batches (request counts, lengths with empty and one-token
    requests, head shapes, page sizes, CTA counts and split modes): the
    library's decode and prefill metadata equal the restated rule word for word."""
    g = np.random.default_rng(100 + seed)
    for _ in range(12):
        B = int(g.choice([1, 2, 5, 33, 200]))
        hkv = int(g.choice([1, 2, 4, 8, 12]))
        hq = hkv * int(g.choice([1, 2, 4, 8]))
        P = int(g.choice([16, 32, 64]))
        kv = [int(x) for x in g.choice([0, 1, 15, 16, 17, 129, 1000, 5000], size=B)]
        ctas = int(g.choice([1, 3, 37, 152, 400]))
        kw = [{}, {"fixed_split_pages": int(g.integers(1, 40))}, {"disable_split_kv": True}][int(g.integers(0, 3))]
        plan, ref, _ = _decode_plan(kv, hq=hq, hkv=hkv, num_ctas=ctas, page_size=P, **kw)
        assert np.array_equal(plan.metadata(), ref), (B, hq, hkv, P, ctas, kw)
        if hq // hkv <= 16:
            qo = [int(g.integers(0, L + 1)) for L in kv]
            plan, ref = _prefill_plan(kv, qo, hq=hq, hkv=hkv, num_ctas=ctas, page_size=P)
            assert np.array_equal(plan.metadata(), ref), (B, hq, hkv, P, ctas, "prefill")


def test_dtype_codes_of_torch_dtypes_names_and_codes():
    import torch
    pairs = [(torch.float16, pa.F16), (torch.bfloat16, pa.BF16), (torch.float8_e4m3fn, pa.E4M3FN),
             (torch.float8_e5m2, pa.E5M2), (torch.float32, pa.F32), (torch.int8, pa.INT8),
             (torch.uint8, pa.UINT8)]
    for _ in range(2):  # the second round is served from the cache
        for dt, code in pairs:
            assert pa.dtype_code(dt) == code
    assert pa.dtype_code("bf16") == pa.BF16 and pa.dtype_code("float8_e5m2") == pa.E5M2
    assert pa.dtype_code(pa.E4M3FN) == pa.E4M3FN
    with pytest.raises(ValueError):
        pa.dtype_code(torch.float64)


def test_plan_takes_torch_and_numpy_page_tables_alike():
    """CPU int32 tensors (passed by pointer), int64 or strided tensors and
    numpy arrays give the same plan."""
    import torch
    kv = [37, 0, 700, 16, 4096]
    npg = [(L + 15) // 16 for L in kv]
    ind = np.concatenate([[0], np.cumsum(npg)]).astype(np.int32)
    last = np.array([(L - (k - 1) * 16) if k else 0 for L, k in zip(kv, npg)], dtype=np.int32)
    qo = np.array([0, 10, 10, 300, 316, 1000], dtype=np.int32)
    for mode in ("decode", "prefill"):
        ref = None
        for conv in (np.asarray, torch.from_numpy, lambda a: torch.from_numpy(a).long(),
                     lambda a: torch.from_numpy(np.repeat(a, 2))[::2]):
            p = pa.Plan(mode=mode, num_qo_heads=32, num_kv_heads=8, num_pages=int(ind[-1]), kv_indptr=conv(ind),
                        last_page_len=conv(last), qo_indptr=conv(qo) if mode == "prefill" else None,
                        q_dtype="bf16", kv_dtype="e4m3fn", num_ctas=37)
            got = p.metadata()
            if ref is None:
                ref = got
            assert np.array_equal(got, ref)
