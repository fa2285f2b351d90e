"""Pins for the oracle's cache writer (new tokens quantized into the paged
fp8 cache).  No GPU needed.

What pins it, so that a plausible mistake fails a test: every finite code
round-trips (a wrong bias, mantissa width or subnormal rule); exact midpoints
between neighbouring codes go to the even code and their float32 neighbours
to the nearer code (truncation, ties away from zero); saturation at the
largest finite value and the special inputs; torch's own float32 -> fp8 cast,
an independent library routine, on in-range values; the multiply by
fl32(1/scale) (a dropped or inverted scale); and brute force over a tiny
page table for the scatter (a wrong page, slot or row offset, or writing
tokens that must be skipped).
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle

FMTS = {"e4m3fn": (torch.float8_e4m3fn, 448.0, 0x7E), "e5m2": (torch.float8_e5m2, 57344.0, 0x7B)}


@pytest.mark.parametrize("fmt", sorted(FMTS))
def test_every_finite_code_round_trips(fmt):
    table = oracle.fp8_table(fmt)
    for c in range(256):
        if np.isfinite(table[c]):
            assert oracle.encode_fp8(fmt, table[c]) == c, (fmt, hex(c), table[c])


@pytest.mark.parametrize("fmt", sorted(FMTS))
def test_midpoints_go_to_the_even_code(fmt):
    table = oracle.fp8_table(fmt)
    _, mx, _ = FMTS[fmt]
    for sign in (0x00, 0x80):
        for c in range(0x00, 0x7F):
            lo, hi = table[sign | c], table[sign | (c + 1)]
            if not (np.isfinite(lo) and np.isfinite(hi)) or abs(hi) > mx:
                continue
            mid = np.float32((lo + hi) / 2)
            assert float(mid) == (lo + hi) / 2  # the midpoint is exact in fp32
            even = sign | c if c % 2 == 0 else sign | (c + 1)
            assert oracle.encode_fp8(fmt, mid) == even, (fmt, hex(sign | c), float(mid))
            below = np.nextafter(mid, np.float32(lo), dtype=np.float32)
            above = np.nextafter(mid, np.float32(hi), dtype=np.float32)
            assert oracle.encode_fp8(fmt, below) == sign | c
            assert oracle.encode_fp8(fmt, above) == sign | (c + 1)


@pytest.mark.parametrize("fmt", sorted(FMTS))
def test_saturation_and_special_inputs(fmt):
    _, mx, mxc = FMTS[fmt]
    for v in (mx, mx * 1.01, mx * 4, 1e30, np.inf):
        assert oracle.encode_fp8(fmt, v) == mxc
        assert oracle.encode_fp8(fmt, -v) == 0x80 | mxc
    assert oracle.encode_fp8(fmt, 0.0) == 0x00
    assert oracle.encode_fp8(fmt, -0.0) == 0x80
    assert np.isnan(oracle.fp8_table(fmt)[oracle.encode_fp8(fmt, np.nan)])
    tiny = float(np.float32(1e-30))  # far below half the smallest subnormal
    assert oracle.encode_fp8(fmt, tiny) == 0x00 and oracle.encode_fp8(fmt, -tiny) == 0x80


@pytest.mark.parametrize("fmt", sorted(FMTS))
def test_agrees_with_torch_cast_in_range(fmt):
    td, mx, _ = FMTS[fmt]
    rng = np.random.default_rng(7)
    x = (rng.standard_normal(100000) * np.exp2(rng.uniform(-24, 17, 100000))).astype(np.float32)
    x = x[np.abs(x) <= mx]
    ref = torch.from_numpy(x).to(td).view(torch.uint8).numpy()
    assert np.array_equal(oracle.quantize(fmt, x, 1.0), ref)


@pytest.mark.parametrize("fmt", sorted(FMTS))
def test_scale_is_a_multiply_by_its_fp32_reciprocal(fmt):
    td, mx, _ = FMTS[fmt]
    rng = np.random.default_rng(8)
    x = rng.standard_normal(20000).astype(np.float32) * 3
    for scale in (np.float32(3.0 / 448), np.float32(0.37), np.float32(7.5)):
        inv = np.float32(1) / scale
        y = (x * inv).astype(np.float32)
        keep = np.abs(y) <= mx
        ref = torch.from_numpy(y[keep]).to(td).view(torch.uint8).numpy()
        assert np.array_equal(oracle.quantize(fmt, x, float(scale))[keep], ref)
        # and the dequantized value is within half a spacing (times scale) of x
        back = oracle.decode(fmt, oracle.quantize(fmt, x[keep], float(scale))) * float(scale)
        rel = np.abs(back - x[keep]) / np.maximum(np.abs(x[keep]), 1e-30)
        small = np.abs(x[keep]) * float(inv) >= (2.0 ** -6 if fmt == "e4m3fn" else 2.0 ** -14)
        mbits = 3 if fmt == "e4m3fn" else 2
        assert rel[small].max() <= 2.0 ** -(mbits + 1) * (1 + 1e-6)


def test_scatter_matches_brute_force_on_a_tiny_table():
    rng = np.random.default_rng(9)
    page_size, hkv, d, num_pages = 16, 2, 128, 9
    kv_indptr = np.array([0, 3, 3, 5], dtype=np.int32)          # request 1 has no pages
    kv_indices = np.array([4, 0, 7, 2, 8], dtype=np.int32)
    # tokens: (request, position); the last four must be skipped
    toks = [(0, 0), (0, 17), (0, 47), (2, 5), (2, 31), (0, 48), (1, 0), (3, 0), (2, -1)]
    nnz = len(toks)
    bi = np.array([t[0] for t in toks], dtype=np.int32)
    ps = np.array([t[1] for t in toks], dtype=np.int32)
    k_new = rng.standard_normal((nnz, hkv, d)).astype(np.float32)
    v_new = rng.standard_normal((nnz, hkv, d)).astype(np.float32) * 5
    k0 = rng.integers(0, 256, (num_pages, page_size, hkv, d), dtype=np.uint8)
    v0 = rng.integers(0, 256, (num_pages, page_size, hkv, d), dtype=np.uint8)
    kc, vc, skipped = oracle.append_kv(fmt="e4m3fn", k_new=k_new, v_new=v_new, batch_indices=bi, positions=ps,
                                       kv_indptr=kv_indptr, kv_indices=kv_indices, k_cache=k0, v_cache=v0,
                                       k_scale=0.01, v_scale=0.05)
    assert skipped == 4
    ek, ev = k0.copy(), v0.copy()
    for i, (b, p) in enumerate(toks[:5]):
        page = kv_indices[kv_indptr[b] + p // page_size]
        for h in range(hkv):
            for j in range(d):
                ek[page, p % page_size, h, j] = oracle.encode_fp8("e4m3fn", np.float32(k_new[i, h, j]) *
                                                                  (np.float32(1) / np.float32(0.01)))
                ev[page, p % page_size, h, j] = oracle.encode_fp8("e4m3fn", np.float32(v_new[i, h, j]) *
                                                                  (np.float32(1) / np.float32(0.05)))
    assert np.array_equal(kc, ek) and np.array_equal(vc, ev)


def test_hnd_scatter_is_the_transposed_nhd_scatter():
    rng = np.random.default_rng(10)
    kv_indptr = np.array([0, 2, 5], dtype=np.int32)
    kv_indices = np.array([3, 0, 6, 1, 5], dtype=np.int32)
    bi = np.array([0, 0, 1, 1, 1], dtype=np.int32)
    ps = np.array([3, 20, 0, 37, 47], dtype=np.int32)
    k_new = rng.standard_normal((5, 4, 128)).astype(np.float32)
    v_new = rng.standard_normal((5, 4, 128)).astype(np.float32)
    k0 = rng.integers(0, 256, (8, 16, 4, 128), dtype=np.uint8)
    v0 = rng.integers(0, 256, (8, 16, 4, 128), dtype=np.uint8)
    common = dict(fmt="e5m2", k_new=k_new, v_new=v_new, batch_indices=bi, positions=ps, kv_indptr=kv_indptr,
                  kv_indices=kv_indices, k_scale=0.02, v_scale=0.03)
    kn, vn, sn = oracle.append_kv(k_cache=k0, v_cache=v0, **common)
    kh, vh, sh = oracle.append_kv(k_cache=k0.transpose(0, 2, 1, 3), v_cache=v0.transpose(0, 2, 1, 3),
                                  kv_layout="HND", **common)
    assert sn == sh == 0
    assert np.array_equal(kh, kn.transpose(0, 2, 1, 3)) and np.array_equal(vh, vn.transpose(0, 2, 1, 3))
