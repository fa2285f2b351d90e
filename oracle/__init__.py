"""CPU oracle for paged attention over an fp8 KV cache.

TEST INFRASTRUCTURE ONLY.  The tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference leg may import this package; the product
library (``paged_attention_fp8_gb300``) never does, and the two share no code.

The arithmetic lives in ``oracle.c`` (plain C, fp64).  This module only builds
it with gcc (once, next to the source), loads it with ctypes, and marshals
numpy arrays.  Quantized inputs are passed as raw codes: ``uint8`` arrays for
fp8 elements, ``uint16`` arrays for f16/bf16 elements; the C code decodes them
from the format definitions.

Dtype names: ``"f16"``, ``"bf16"``, ``"e4m3fn"``, ``"e5m2"``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_SO = os.path.join(_HERE, "liboracle.so")

DTYPE_CODES = {"f16": 1, "bf16": 2, "e4m3fn": 3, "e5m2": 4}
_ELEM_NP = {"f16": np.uint16, "bf16": np.uint16, "e4m3fn": np.uint8, "e5m2": np.uint8}

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``liboracle.so`` (with OpenMP when gcc has it)."""
    if not force and os.path.exists(_SO) and os.path.getmtime(_SO) >= os.path.getmtime(_SRC):
        return _SO
    tmp = _SO + ".tmp.%d" % os.getpid()
    base = ["gcc", "-O2", "-fPIC", "-shared", "-std=c11", "-o", tmp, _SRC, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        build()
        lib = ctypes.CDLL(_SO)
        i64, i32, dbl, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_double, ctypes.c_void_p
        lib.orc_decode_array.argtypes = [i32, vp, i64, vp]
        lib.orc_decode_array.restype = i32
        lib.orc_num_threads.argtypes = []
        lib.orc_num_threads.restype = i32
        lib.orc_set_num_threads.argtypes = [i32]
        lib.orc_set_num_threads.restype = i32
        lib.orc_paged_attention.argtypes = (
            [i64] * 6 + [vp] * 4 + [i32, vp, dbl, i32, vp, vp, dbl, dbl, dbl, i32, i32, vp, vp, vp, i64, vp, vp,
                                     vp, vp])
        lib.orc_paged_attention.restype = i32
        lib.orc_dense_attention_row.argtypes = [i64, i64, i64, vp, i64, vp, vp, dbl, vp, vp]
        lib.orc_dense_attention_row.restype = i32
        lib.orc_merge_states.argtypes = [i64, i64, vp, vp, vp, vp]
        lib.orc_merge_states.restype = None
        lib.orc_encode_fp8.argtypes = [i32, ctypes.c_float]
        lib.orc_encode_fp8.restype = ctypes.c_uint8
        lib.orc_quantize_array.argtypes = [i32, vp, i64, ctypes.c_float, vp]
        lib.orc_quantize_array.restype = i32
        lib.orc_append_kv.argtypes = [i32, vp, vp, i64, i32, i32, vp, vp, i32, vp, vp, i32, i32, i32,
                                      ctypes.c_float, ctypes.c_float, vp, vp]
        lib.orc_append_kv.restype = i64
        _lib = lib
        return lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _raw(a, dtype: str) -> np.ndarray:
    a = np.ascontiguousarray(a)
    want = _ELEM_NP[dtype]
    if a.dtype != want:
        if a.dtype.itemsize != np.dtype(want).itemsize:
            raise TypeError(f"raw {dtype} codes must be {np.dtype(want).name}, got {a.dtype}")
        a = a.view(want)
    return a


def num_threads() -> int:
    """Threads the oracle's OpenMP loop uses (1 when built without OpenMP)."""
    return int(_load().orc_num_threads())


def set_num_threads(n: int) -> int:
    """Threads for later oracle calls (every host core by default); returns
    the count in effect (1 when built without OpenMP)."""
    return int(_load().orc_set_num_threads(int(n)))


def decode(dtype: str, raw) -> np.ndarray:
    """Decode raw element codes of ``dtype`` to fp64 (same shape)."""
    raw = _raw(raw, dtype)
    out = np.empty(raw.shape, dtype=np.float64)
    rc = _load().orc_decode_array(DTYPE_CODES[dtype], _ptr(raw), raw.size, _ptr(out))
    if rc != 0:
        raise ValueError(f"oracle decode failed ({rc})")
    return out


def fp8_table(fmt: str) -> np.ndarray:
    """The 256 values of an fp8 format, indexed by code."""
    return decode(fmt, np.arange(256, dtype=np.uint8))


def as_f32(src, src_dtype: str) -> np.ndarray:
    """New-token rows as fp32: raw f16/bf16 codes decoded (exact), or fp32."""
    if src_dtype == "f32":
        return np.ascontiguousarray(src, dtype=np.float32)
    return decode(src_dtype, src).astype(np.float32)


def encode_fp8(fmt: str, y: float) -> int:
    """Code of the fp32 value ``y`` in ``fmt`` (nearest, ties to even,
    saturating; NaN -> 0x7F)."""
    return int(_load().orc_encode_fp8(DTYPE_CODES[fmt], float(np.float32(y))))


def quantize(fmt: str, x, scale: float) -> np.ndarray:
    """fp8 codes of fl32(x * fl32(1/scale)) for fp32 ``x`` (same shape)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint8)
    rc = _load().orc_quantize_array(DTYPE_CODES[fmt], _ptr(x), x.size, float(scale), _ptr(out))
    if rc != 0:
        raise ValueError(f"oracle quantize failed ({rc})")
    return out


def append_kv(*, fmt, k_new, v_new, batch_indices, positions, kv_indptr, kv_indices, k_cache,
              v_cache, k_scale, v_scale, kv_layout="NHD"):
    """Write new tokens (fp32 rows [nnz, hkv, d]) into copies of the fp8 caches
    (uint8 codes [num_pages, page_size, hkv, d], or [num_pages, hkv,
    page_size, d] for kv_layout "HND").  Returns (k_cache, v_cache, tokens
    not written)."""
    k_new = np.ascontiguousarray(k_new, dtype=np.float32)
    v_new = np.ascontiguousarray(v_new, dtype=np.float32)
    kc = np.array(k_cache, dtype=np.uint8, copy=True, order="C")
    vc = np.array(v_cache, dtype=np.uint8, copy=True, order="C")
    bi = np.ascontiguousarray(batch_indices, dtype=np.int32)
    ps = np.ascontiguousarray(positions, dtype=np.int32)
    ip = np.ascontiguousarray(kv_indptr, dtype=np.int32)
    ix = np.ascontiguousarray(kv_indices, dtype=np.int32)
    nnz, hkv, d = k_new.shape
    hnd = {"NHD": 0, "HND": 1}[kv_layout]
    page_size = kc.shape[2] if hnd else kc.shape[1]
    skipped = _load().orc_append_kv(DTYPE_CODES[fmt], _ptr(k_new), _ptr(v_new), nnz, hkv, d, _ptr(bi),
                                    _ptr(ps), len(ip) - 1, _ptr(ip), _ptr(ix), kc.shape[0], page_size, hnd,
                                    float(k_scale), float(v_scale), _ptr(kc), _ptr(vc))
    if skipped < 0:
        raise ValueError("oracle append failed")
    return kc, vc, int(skipped)


def paged_attention(*, q, q_dtype, k_cache, v_cache, kv_dtype, qo_indptr, kv_indptr,
                    kv_indices, last_page_len, num_qo_heads, num_kv_heads,
                    q_scale=1.0, k_scale=1.0, v_scale=1.0, sm_scale=None,
                    causal=True, rows=None, heads=None, kv_layout="NHD"):
    """fp64 attention of q against the paged cache; see ``oracle.c``.

    q: raw codes [nnz_qo, Hq, D]; k_cache/v_cache: raw codes
    [num_pages, P, Hkv, D] (kv_layout "NHD") or [num_pages, Hkv, P, D]
    ("HND"); index arrays int32.  ``q_scale``, ``k_scale`` and ``v_scale``
    are floats (per tensor) or arrays of one scale per query head (q) or per
    KV head (k, v).  ``rows``/``heads`` (equal
    length) select which (query row, head) outputs to compute; None = all.
    Returns (o, lse): o [n, D] fp64 and lse [n] fp64 in selection order
    (all: n = nnz_qo * Hq, row-major over (row, head)).
    """
    lib = _load()
    scales = {}
    for name, val, n_heads in (("q", q_scale, num_qo_heads), ("k", k_scale, num_kv_heads),
                               ("v", v_scale, num_kv_heads)):
        if np.ndim(val) == 0:
            scales[name] = (float(val), None)
        else:
            arr = np.ascontiguousarray(val, dtype=np.float64)
            if arr.shape != (n_heads,):
                raise ValueError(f"oracle: {name}_scale has shape {arr.shape}, expected ({n_heads},)")
            scales[name] = (1.0, arr)
    q = _raw(q, q_dtype)
    k_cache = _raw(k_cache, kv_dtype)
    v_cache = _raw(v_cache, kv_dtype)
    hnd = {"NHD": 0, "HND": 1}[kv_layout]
    if hnd:
        num_pages, hkv, page_size, head_dim = k_cache.shape
    else:
        num_pages, page_size, hkv, head_dim = k_cache.shape
    if hkv != num_kv_heads or q.shape[-1] != head_dim or q.shape[-2] != num_qo_heads:
        raise ValueError("oracle: shape mismatch between q, cache and head counts")
    qo_indptr = np.ascontiguousarray(qo_indptr, dtype=np.int32)
    kv_indptr = np.ascontiguousarray(kv_indptr, dtype=np.int32)
    kv_indices = np.ascontiguousarray(kv_indices, dtype=np.int32)
    last_page_len = np.ascontiguousarray(last_page_len, dtype=np.int32)
    batch = len(kv_indptr) - 1
    if sm_scale is None:
        sm_scale = 1.0 / np.sqrt(head_dim)
    if rows is None:
        n = int(qo_indptr[-1]) * num_qo_heads
        sel_r = sel_h = None
    else:
        sel_r = np.ascontiguousarray(rows, dtype=np.int64)
        sel_h = np.ascontiguousarray(heads, dtype=np.int32)
        n = len(sel_r)
    o = np.empty((n, head_dim), dtype=np.float64)
    lse = np.empty((n,), dtype=np.float64)
    rc = lib.orc_paged_attention(
        batch, num_qo_heads, num_kv_heads, head_dim, page_size, num_pages,
        _ptr(qo_indptr), _ptr(kv_indptr), _ptr(kv_indices), _ptr(last_page_len),
        DTYPE_CODES[q_dtype], _ptr(q), scales["q"][0],
        DTYPE_CODES[kv_dtype], _ptr(k_cache), _ptr(v_cache),
        scales["k"][0], scales["v"][0], float(sm_scale), int(bool(causal)), hnd,
        *[None if scales[x][1] is None else _ptr(scales[x][1]) for x in ("q", "k", "v")],
        n, None if sel_r is None else _ptr(sel_r), None if sel_h is None else _ptr(sel_h),
        _ptr(o), _ptr(lse))
    if rc != 0:
        raise ValueError(f"oracle rejected its arguments (code {rc})")
    return o, lse


def dense_attention_row(q, k, v, num_kv_heads, sm_scale):
    """Attention of one query row q [Hq, D] (fp64) over dense fp64 K/V rows
    [n, Hkv, D]; no paging.  Returns (o [Hq, D], lse [Hq])."""
    q = np.ascontiguousarray(q, dtype=np.float64)
    k = np.ascontiguousarray(k, dtype=np.float64)
    v = np.ascontiguousarray(v, dtype=np.float64)
    hq, d = q.shape
    o = np.empty((hq, d), dtype=np.float64)
    lse = np.empty((hq,), dtype=np.float64)
    rc = _load().orc_dense_attention_row(hq, num_kv_heads, d, _ptr(q), k.shape[0], _ptr(k),
                                         _ptr(v), float(sm_scale), _ptr(o), _ptr(lse))
    if rc != 0:
        raise ValueError(f"oracle rejected its arguments (code {rc})")
    return o, lse


def merge_states(o_parts, lse_parts):
    """Combine partial states [n, D] / [n] of one (row, head) by their lse."""
    o_parts = np.ascontiguousarray(o_parts, dtype=np.float64)
    lse_parts = np.ascontiguousarray(lse_parts, dtype=np.float64)
    n, d = o_parts.shape
    o = np.empty((d,), dtype=np.float64)
    lse = np.empty((1,), dtype=np.float64)
    _load().orc_merge_states(n, d, _ptr(o_parts), _ptr(lse_parts), _ptr(o), _ptr(lse))
    return o, float(lse[0])
