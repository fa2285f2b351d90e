"""paged_attention_fp8_gb300 -- Python binding of libpafp8.

Paged attention of a bf16/f16 (or fp8) query against a KV cache stored in
fp8 (e4m3fn/e5m2) with per-tensor scales, on GB300 (sm_103a).  Every step of
the computation runs in the CUDA library ``libpafp8.so``; this module only
marshals arguments through its C ABI (``include/pafp8.h``) with ctypes.  The
functions carry the C names.  There is no fallback: if the library is not
built, every call raises.

Typical use::

    plan = Plan(mode="decode", num_qo_heads=32, num_kv_heads=8, num_pages=...,
                kv_indptr=..., last_page_len=..., q_dtype=torch.bfloat16,
                kv_dtype=torch.float8_e4m3fn)
    ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device="cuda")
    plan.upload(ws)
    plan.run(q, k_cache, v_cache, kv_indices, o, lse, ws, k_scale=..., v_scale=...)
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpafp8.so")

# dtype codes of include/pafp8.h
DTYPE_DEFAULT, F16, BF16, E4M3FN, E5M2, F32, INT8, UINT8 = range(8)
MODE_DECODE, MODE_PREFILL = 0, 1
LAYOUT_NHD, LAYOUT_HND = 0, 1
_LAYOUTS = {"NHD": LAYOUT_NHD, "HND": LAYOUT_HND}
STATUS = {0: "OK", 1: "ERR_DTYPE", 2: "ERR_SHAPE", 3: "ERR_ARG", 4: "ERR_WORKSPACE", 5: "ERR_CUDA",
          6: "ERR_TIMEOUT", 7: "ERR_BOUNDS", 8: "ERR_UNSUPPORTED"}
_NAME_CODES = {"default": DTYPE_DEFAULT, "f16": F16, "float16": F16, "bf16": BF16, "bfloat16": BF16,
               "e4m3fn": E4M3FN, "float8_e4m3fn": E4M3FN, "e5m2": E5M2, "float8_e5m2": E5M2,
               "f32": F32, "float32": F32, "int8": INT8, "uint8": UINT8}

# Every entry point include/pafp8.h declares.
EXPORTS = ("pafp8_abi_version", "pafp8_last_error", "pafp8_plan_create", "pafp8_plan_destroy",
           "pafp8_workspace_bytes", "pafp8_plan_metadata", "pafp8_plan_upload", "pafp8_run",
           "pafp8_run_stage", "pafp8_device_status", "pafp8_run_decode_noalloc", "pafp8_append_kv",
           "pafp8_run_head_scales", "pafp8_run_pod", "pafp8_host_workspace_bytes", "pafp8_run_host")


class Pafp8Error(RuntimeError):
    """A non-OK status from libpafp8, with its sentence."""

    def __init__(self, status: int, message: str):
        self.status = status
        self.status_name = STATUS.get(status, str(status))
        super().__init__(f"{self.status_name}: {message}")


class plan_desc(ctypes.Structure):
    _fields_ = [("mode", ctypes.c_int32), ("batch", ctypes.c_int32),
                ("num_qo_heads", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("page_size", ctypes.c_int32),
                ("num_pages", ctypes.c_int32), ("q_dtype", ctypes.c_int32),
                ("kv_dtype", ctypes.c_int32), ("o_dtype", ctypes.c_int32),
                ("sm_scale", ctypes.c_float), ("fixed_split_pages", ctypes.c_int32),
                ("disable_split_kv", ctypes.c_int32), ("num_ctas", ctypes.c_int32),
                ("kv_layout", ctypes.c_int32)]


class pod_phase(ctypes.Structure):
    _fields_ = [("plan", ctypes.c_void_p), ("q", ctypes.c_void_p), ("kv_indices", ctypes.c_void_p),
                ("o", ctypes.c_void_p), ("lse", ctypes.c_void_p), ("workspace", ctypes.c_void_p),
                ("workspace_bytes", ctypes.c_size_t)]


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded libpafp8.so; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"libpafp8.so is not built ({LIB_PATH} missing); run "
                           "paged_attention_fp8_gb300.build.build() first")
    L = ctypes.CDLL(LIB_PATH)
    vp, i32, sz, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t, ctypes.c_float
    L.pafp8_abi_version.argtypes, L.pafp8_abi_version.restype = [], i32
    L.pafp8_last_error.argtypes, L.pafp8_last_error.restype = [], ctypes.c_char_p
    L.pafp8_plan_create.argtypes = [ctypes.POINTER(plan_desc), vp, vp, vp, ctypes.POINTER(vp)]
    L.pafp8_plan_create.restype = i32
    L.pafp8_plan_destroy.argtypes, L.pafp8_plan_destroy.restype = [vp], None
    L.pafp8_workspace_bytes.argtypes, L.pafp8_workspace_bytes.restype = [vp], sz
    L.pafp8_plan_metadata.argtypes = [vp, ctypes.POINTER(ctypes.POINTER(ctypes.c_int32)),
                                      ctypes.POINTER(sz)]
    L.pafp8_plan_metadata.restype = i32
    L.pafp8_plan_upload.argtypes, L.pafp8_plan_upload.restype = [vp, vp, sz, vp], i32
    L.pafp8_run.argtypes = [vp, i32, vp, i32, vp, i32, vp, vp, f32, f32, f32, i32, vp, vp, vp, sz, vp]
    L.pafp8_run.restype = i32
    L.pafp8_run_stage.argtypes = [vp, i32, i32, vp, i32, vp, i32, vp, vp, f32, f32, f32, i32, vp, vp,
                                  vp, sz, vp]
    L.pafp8_run_stage.restype = i32
    L.pafp8_host_workspace_bytes.argtypes, L.pafp8_host_workspace_bytes.restype = [vp, i32], sz
    L.pafp8_run_host.argtypes = [vp, i32, vp, i32, vp, i32, vp, vp, f32, f32, f32, i32, vp, vp, vp, sz, vp]
    L.pafp8_run_host.restype = i32
    L.pafp8_device_status.argtypes, L.pafp8_device_status.restype = [vp, vp, vp], i32
    L.pafp8_run_decode_noalloc.argtypes = [vp, i32, vp, i32, vp, i32, vp, vp, f32, f32, f32, i32, vp,
                                           vp, vp]
    L.pafp8_run_decode_noalloc.restype = i32
    L.pafp8_append_kv.argtypes = [i32, vp, vp, ctypes.c_int64, i32, i32, vp, vp, i32, vp, vp, i32, i32, vp,
                                  vp, i32, i32, f32, f32, vp, vp]
    L.pafp8_append_kv.restype = i32
    L.pafp8_run_head_scales.argtypes = [vp, i32, vp, i32, vp, i32, vp, vp, vp, vp, vp, i32, vp, vp, vp, sz, vp]
    L.pafp8_run_head_scales.restype = i32
    L.pafp8_run_pod.argtypes = [ctypes.POINTER(pod_phase), ctypes.POINTER(pod_phase), i32, i32, vp, i32, vp,
                                f32, f32, f32, i32, vp]
    L.pafp8_run_pod.restype = i32
    _lib = L
    return L


_OBJ_CODES = {}  # dtype objects seen before -> code (the run calls pass torch dtypes)


def dtype_code(x) -> int:
    """int32 dtype code for a torch dtype, a name or a code."""
    if isinstance(x, int):
        return x
    if isinstance(x, str):
        return _NAME_CODES[x]
    code = _OBJ_CODES.get(x)
    if code is not None:
        return code
    name = str(x).replace("torch.", "")
    if name not in _NAME_CODES:
        raise ValueError(f"no libpafp8 dtype code for {x}")
    _OBJ_CODES[x] = _NAME_CODES[name]
    return _NAME_CODES[name]


def _check(status: int) -> None:
    if status != 0:
        raise Pafp8Error(status, pafp8_last_error())


def _i32_host(a):
    """A host int32 array: a contiguous CPU int32 tensor as it is (its
    data_ptr is passed), anything else as a contiguous numpy int32 array."""
    if a is None:
        return None
    if hasattr(a, "cpu"):
        if a.device.type == "cpu" and str(a.dtype) == "torch.int32" and a.is_contiguous():
            return a
        a = a.cpu().numpy()
    return np.ascontiguousarray(a, dtype=np.int32)


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, np.ndarray):
        return t.ctypes.data
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return getattr(stream, "cuda_stream", stream)


# ---- the C entry points, same names --------------------------------------

def pafp8_abi_version() -> int:
    return int(lib().pafp8_abi_version())


def pafp8_last_error() -> str:
    return lib().pafp8_last_error().decode()


def pafp8_plan_create(desc: plan_desc, kv_indptr, last_page_len, qo_indptr=None) -> int:
    kv_indptr, last_page_len, qo_indptr = _i32_host(kv_indptr), _i32_host(last_page_len), _i32_host(qo_indptr)
    out = ctypes.c_void_p()
    _check(lib().pafp8_plan_create(ctypes.byref(desc), _ptr(kv_indptr), _ptr(last_page_len),
                                   _ptr(qo_indptr), ctypes.byref(out)))
    return out.value


def pafp8_plan_destroy(handle: int) -> None:
    lib().pafp8_plan_destroy(handle)


def pafp8_workspace_bytes(handle: int) -> int:
    return int(lib().pafp8_workspace_bytes(handle))


def pafp8_plan_metadata(handle: int) -> np.ndarray:
    words = ctypes.POINTER(ctypes.c_int32)()
    n = ctypes.c_size_t()
    _check(lib().pafp8_plan_metadata(handle, ctypes.byref(words), ctypes.byref(n)))
    return np.ctypeslib.as_array(words, shape=(n.value,)).copy()


def pafp8_plan_upload(handle: int, workspace, stream=None) -> None:
    _check(lib().pafp8_plan_upload(handle, _ptr(workspace), workspace.numel() * workspace.element_size(),
                                   _stream(stream)))


def pafp8_run(handle: int, q, k_cache, v_cache, kv_indices, o, lse, workspace, *, q_scale=1.0,
              k_scale=1.0, v_scale=1.0, q_dtype=None, k_dtype=None, v_dtype=None, o_dtype=None,
              stream=None) -> None:
    """Dtype codes default to the tensors' own dtypes."""
    _check(lib().pafp8_run(
        handle, dtype_code(q_dtype if q_dtype is not None else q.dtype), _ptr(q),
        dtype_code(k_dtype if k_dtype is not None else k_cache.dtype), _ptr(k_cache),
        dtype_code(v_dtype if v_dtype is not None else v_cache.dtype), _ptr(v_cache),
        _ptr(kv_indices), float(q_scale), float(k_scale), float(v_scale),
        dtype_code(o_dtype if o_dtype is not None else o.dtype), _ptr(o), _ptr(lse),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))


def pafp8_host_workspace_bytes(handle: int, q_dtype) -> int:
    return int(lib().pafp8_host_workspace_bytes(handle, dtype_code(q_dtype)))


def pafp8_run_host(handle: int, q_h, k_cache, v_cache, kv_indices_h, o_h, lse_h, workspace, *, q_scale=1.0,
                   k_scale=1.0, v_scale=1.0, q_dtype=None, k_dtype=None, v_dtype=None, o_dtype=None,
                   stream=None) -> None:
    """One step from and to host memory (q_h, kv_indices_h, o_h, lse_h: CPU
    tensors, preferably pinned); dtype codes default to the tensors' own."""
    _check(lib().pafp8_run_host(
        handle, dtype_code(q_dtype if q_dtype is not None else q_h.dtype), _ptr(q_h),
        dtype_code(k_dtype if k_dtype is not None else k_cache.dtype), _ptr(k_cache),
        dtype_code(v_dtype if v_dtype is not None else v_cache.dtype), _ptr(v_cache),
        _ptr(kv_indices_h), float(q_scale), float(k_scale), float(v_scale),
        dtype_code(o_dtype if o_dtype is not None else o_h.dtype), _ptr(o_h), _ptr(lse_h),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))


def pafp8_run_stage(handle: int, stage: int, q, k_cache, v_cache, kv_indices, o, lse, workspace, *,
                    q_scale=1.0, k_scale=1.0, v_scale=1.0, q_dtype=None, k_dtype=None, v_dtype=None,
                    o_dtype=None, stream=None) -> None:
    """pafp8_run limited to stage 1 (attention kernel) or 2 (merge); 0 = all."""
    _check(lib().pafp8_run_stage(
        handle, int(stage), dtype_code(q_dtype if q_dtype is not None else q.dtype), _ptr(q),
        dtype_code(k_dtype if k_dtype is not None else k_cache.dtype), _ptr(k_cache),
        dtype_code(v_dtype if v_dtype is not None else v_cache.dtype), _ptr(v_cache),
        _ptr(kv_indices), float(q_scale), float(k_scale), float(v_scale),
        dtype_code(o_dtype if o_dtype is not None else o.dtype), _ptr(o), _ptr(lse),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))


def pafp8_run_head_scales(handle: int, q, k_cache, v_cache, kv_indices, o, lse, workspace, *, q_scales=None,
                          k_scales, v_scales, q_dtype=None, k_dtype=None, v_dtype=None, o_dtype=None,
                          stream=None) -> None:
    """pafp8_run with per-head scale tensors (device float32: q_scales [Hq] or
    None, k_scales and v_scales [Hkv])."""
    _check(lib().pafp8_run_head_scales(
        handle, dtype_code(q_dtype if q_dtype is not None else q.dtype), _ptr(q),
        dtype_code(k_dtype if k_dtype is not None else k_cache.dtype), _ptr(k_cache),
        dtype_code(v_dtype if v_dtype is not None else v_cache.dtype), _ptr(v_cache),
        _ptr(kv_indices), _ptr(q_scales), _ptr(k_scales), _ptr(v_scales),
        dtype_code(o_dtype if o_dtype is not None else o.dtype), _ptr(o), _ptr(lse),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))


def pafp8_device_status(handle: int, workspace, stream=None) -> None:
    _check(lib().pafp8_device_status(handle, _ptr(workspace), _stream(stream)))


def pafp8_run_decode_noalloc(handle: int, q, k_cache, v_cache, kv_indices, o, lse, *, q_scale=1.0,
                             k_scale=1.0, v_scale=1.0, q_dtype=None, k_dtype=None, v_dtype=None,
                             o_dtype=None, stream=None) -> None:
    """Decode with the library's built-in scratch instead of a workspace, for
    callers that may not allocate device memory (see include/pafp8.h)."""
    _check(lib().pafp8_run_decode_noalloc(
        handle, dtype_code(q_dtype if q_dtype is not None else q.dtype), _ptr(q),
        dtype_code(k_dtype if k_dtype is not None else k_cache.dtype), _ptr(k_cache),
        dtype_code(v_dtype if v_dtype is not None else v_cache.dtype), _ptr(v_cache),
        _ptr(kv_indices), float(q_scale), float(k_scale), float(v_scale),
        dtype_code(o_dtype if o_dtype is not None else o.dtype), _ptr(o), _ptr(lse), _stream(stream)))


def _phase(handle, q, kv_indices, o, lse, workspace) -> pod_phase:
    return pod_phase(handle, _ptr(q), _ptr(kv_indices), _ptr(o), _ptr(lse), _ptr(workspace),
                     workspace.numel() * workspace.element_size())


def pafp8_run_pod(prefill_handle: int, prefill_q, prefill_kv_indices, prefill_o, prefill_lse, prefill_workspace,
                  decode_handle: int, decode_q, decode_kv_indices, decode_o, decode_lse, decode_workspace,
                  k_cache, v_cache, *, q_scale=1.0, k_scale=1.0, v_scale=1.0, q_dtype=None, k_dtype=None,
                  v_dtype=None, o_dtype=None, stream=None) -> None:
    """A prefill plan's phase and a decode plan's phase over one cache in one
    call, side by side on the SMs their plans' num_ctas give (see
    include/pafp8.h).  Dtype codes default to the prefill tensors' dtypes."""
    pre = _phase(prefill_handle, prefill_q, prefill_kv_indices, prefill_o, prefill_lse, prefill_workspace)
    dec = _phase(decode_handle, decode_q, decode_kv_indices, decode_o, decode_lse, decode_workspace)
    _check(lib().pafp8_run_pod(
        ctypes.byref(pre), ctypes.byref(dec), dtype_code(q_dtype if q_dtype is not None else prefill_q.dtype),
        dtype_code(k_dtype if k_dtype is not None else k_cache.dtype), _ptr(k_cache),
        dtype_code(v_dtype if v_dtype is not None else v_cache.dtype), _ptr(v_cache),
        float(q_scale), float(k_scale), float(v_scale),
        dtype_code(o_dtype if o_dtype is not None else prefill_o.dtype), _stream(stream)))


def pafp8_append_kv(k_new, v_new, batch_indices, positions, kv_indptr, kv_indices, k_cache, v_cache, *,
                    k_scale=1.0, v_scale=1.0, status=None, src_dtype=None, kv_dtype=None,
                    kv_layout="NHD", num_pages=None, stream=None) -> None:
    """Quantize new tokens k_new/v_new [nnz, Hkv, D] into the paged fp8 cache
    (see include/pafp8.h).  Index arrays are device int32; dtype codes,
    head counts and sizes default to what the tensors say."""
    nnz, hkv, d = k_new.shape
    layout = _LAYOUTS[kv_layout] if isinstance(kv_layout, str) else int(kv_layout)
    page_size = int(k_cache.shape[2] if layout == LAYOUT_HND else k_cache.shape[1])
    _check(lib().pafp8_append_kv(
        dtype_code(src_dtype if src_dtype is not None else k_new.dtype), _ptr(k_new), _ptr(v_new), int(nnz),
        int(hkv), int(d), _ptr(batch_indices), _ptr(positions), int(kv_indptr.numel() - 1), _ptr(kv_indptr),
        _ptr(kv_indices), dtype_code(kv_dtype if kv_dtype is not None else k_cache.dtype), layout,
        _ptr(k_cache), _ptr(v_cache), int(num_pages if num_pages is not None else k_cache.shape[0]),
        page_size, float(k_scale), float(v_scale), _ptr(status), _stream(stream)))


# ---- convenience owner of a plan ---------------------------------------

class Plan:
    """Owns one pafp8_plan.  Shapes served: head_dim 128 or 64,
    page_size a multiple of 16 in either layout."""

    def __init__(self, *, mode: str, num_qo_heads: int, num_kv_heads: int, num_pages: int,
                 kv_indptr, last_page_len, qo_indptr=None, q_dtype, kv_dtype, o_dtype=None,
                 head_dim: int = 128, page_size: int = 16, sm_scale: float = 0.0,
                 fixed_split_pages: int = 0, disable_split_kv: bool = False, num_ctas: int = 0,
                 kv_layout: str = "NHD"):
        kv_indptr_h = _i32_host(kv_indptr)
        self.desc = plan_desc(
            mode=MODE_DECODE if mode == "decode" else MODE_PREFILL, batch=len(kv_indptr_h) - 1,
            num_qo_heads=num_qo_heads, num_kv_heads=num_kv_heads, head_dim=head_dim,
            page_size=page_size, num_pages=num_pages, q_dtype=dtype_code(q_dtype),
            kv_dtype=dtype_code(kv_dtype),
            o_dtype=DTYPE_DEFAULT if o_dtype is None else dtype_code(o_dtype),
            sm_scale=float(sm_scale), fixed_split_pages=int(fixed_split_pages),
            disable_split_kv=int(bool(disable_split_kv)), num_ctas=int(num_ctas),
            kv_layout=_LAYOUTS[kv_layout] if isinstance(kv_layout, str) else int(kv_layout))
        self.handle = None
        self.handle = pafp8_plan_create(self.desc, kv_indptr_h, last_page_len, qo_indptr)

    def __del__(self):
        if getattr(self, "handle", None):
            pafp8_plan_destroy(self.handle)
            self.handle = None

    @property
    def workspace_bytes(self) -> int:
        return pafp8_workspace_bytes(self.handle)

    def metadata(self) -> np.ndarray:
        return pafp8_plan_metadata(self.handle)

    def upload(self, workspace, stream=None) -> None:
        pafp8_plan_upload(self.handle, workspace, stream)

    def run(self, q, k_cache, v_cache, kv_indices, o, lse, workspace, **kw) -> None:
        pafp8_run(self.handle, q, k_cache, v_cache, kv_indices, o, lse, workspace, **kw)

    def host_workspace_bytes(self, q_dtype) -> int:
        return pafp8_host_workspace_bytes(self.handle, q_dtype)

    def run_host(self, q_h, k_cache, v_cache, kv_indices_h, o_h, lse_h, workspace, **kw) -> None:
        pafp8_run_host(self.handle, q_h, k_cache, v_cache, kv_indices_h, o_h, lse_h, workspace, **kw)

    def run_head_scales(self, q, k_cache, v_cache, kv_indices, o, lse, workspace, **kw) -> None:
        pafp8_run_head_scales(self.handle, q, k_cache, v_cache, kv_indices, o, lse, workspace, **kw)

    def run_stage(self, stage, q, k_cache, v_cache, kv_indices, o, lse, workspace, **kw) -> None:
        pafp8_run_stage(self.handle, stage, q, k_cache, v_cache, kv_indices, o, lse, workspace, **kw)

    def device_status(self, workspace, stream=None) -> None:
        pafp8_device_status(self.handle, workspace, stream)
