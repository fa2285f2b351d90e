"""Seeded synthetic inputs for paged attention over an fp8 KV cache.

This module only *draws* inputs: request lengths, a shuffled page pool, query
values and K/V values quantized to fp8 with per-tensor scales.  It holds none
of the attention arithmetic; both the CUDA library's tests/benchmark and the
CPU oracle consume the tensors it returns.

Recipe (every draw from one CPU ``torch.Generator`` seeded per workload, in
this order): request lengths -> page permutation -> q -> K -> V -> outlier
masks -> filler bytes for cache slots no request owns.

* Values are N(0, std) in fp32.  Outliers (long-context workload) multiply a
  Bernoulli(frac) subset by ``outlier_mult``.
* fp8 quantization is per tensor: scale = amax(|x|) / fp8_max (448 for
  e4m3fn, 57344 for e5m2); code = round-to-nearest-even(clamp(x / scale)).
  An fp8 query gets its own q_scale the same way.  A 2-byte query is a
  round-to-nearest cast of the fp32 draw, with q_scale = 1.
* Pages are a random permutation of a pool (``pool_pages`` >= pages needed);
  every cache byte no request owns (unused pages, slots past a request's
  last token) holds a random code, so a stray read shows up in the result.
* Layout: ``k_cache``/``v_cache`` are ``[num_pages, page_size, Hkv, D]``
  (token-major within a page); ``q`` is ``[nnz_qo, Hq, D]``.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional, Sequence

import numpy as np
import torch

TORCH_DTYPES = {
    "f16": torch.float16,
    "bf16": torch.bfloat16,
    "e4m3fn": torch.float8_e4m3fn,
    "e5m2": torch.float8_e5m2,
}
FP8_MAX = {"e4m3fn": 448.0, "e5m2": 57344.0}


@dataclasses.dataclass
class PagedBatch:
    """One batch of paged-attention inputs (all host tensors)."""

    name: str
    mode: str  # "decode" (one query row per request) or "prefill" (causal, ragged)
    num_qo_heads: int
    num_kv_heads: int
    head_dim: int
    page_size: int
    num_pages: int
    q_dtype: str
    kv_dtype: str
    o_dtype: str
    q: torch.Tensor  # [nnz_qo, Hq, D], torch dtype of q_dtype
    k_cache: torch.Tensor  # [num_pages, P, Hkv, D], torch fp8 dtype
    v_cache: torch.Tensor
    qo_indptr: torch.Tensor  # int32 [B+1]
    kv_indptr: torch.Tensor  # int32 [B+1]
    kv_indices: torch.Tensor  # int32 [nnz_pages]
    last_page_len: torch.Tensor  # int32 [B]
    qo_lens: List[int]
    kv_lens: List[int]
    q_scale: float
    k_scale: float
    v_scale: float
    sm_scale: float
    kv_layout: str = "NHD"  # "HND": caches are [num_pages, Hkv, P, D]

    @property
    def batch(self) -> int:
        return len(self.kv_lens)

    @property
    def causal(self) -> bool:
        return self.mode == "prefill"

    @property
    def nnz_qo(self) -> int:
        return int(self.qo_indptr[-1])

    def kv_bytes(self) -> int:
        """Bytes of K and V the requests own (1 byte per fp8 element, 2 for a
        2-byte cache)."""
        esz = 1 if self.kv_dtype in FP8_MAX else 2
        return 2 * sum(self.kv_lens) * self.num_kv_heads * self.head_dim * esz

    def causal_flops(self) -> int:
        """4*D*Hq per admitted (query row, key) pair, causal pairs only."""
        pairs = 0
        for qo, kv in zip(self.qo_lens, self.kv_lens):
            if self.mode == "prefill":
                prefix = kv - qo
                pairs += qo * prefix + qo * (qo + 1) // 2
            else:
                pairs += qo * kv
        return 4 * self.head_dim * self.num_qo_heads * pairs


def raw_numpy(t: torch.Tensor) -> np.ndarray:
    """Raw element codes of a host tensor: uint8 for 1-byte, uint16 for 2-byte."""
    t = t.contiguous().cpu()
    if t.element_size() == 1:
        return t.view(torch.uint8).numpy()
    if t.element_size() == 2:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def _quantize(x: torch.Tensor, fmt: str):
    amax = float(x.abs().max()) if x.numel() else 0.0
    scale = amax / FP8_MAX[fmt] if amax > 0 else 1.0
    y = (x / scale).clamp_(-FP8_MAX[fmt], FP8_MAX[fmt])
    return y.to(TORCH_DTYPES[fmt]), scale


def make_batch(kv_lens: Sequence[int], qo_lens: Optional[Sequence[int]] = None, *,
               num_qo_heads: int, num_kv_heads: int, head_dim: int = 128,
               page_size: int = 16, q_dtype: str = "bf16", kv_dtype: str = "e4m3fn",
               o_dtype: Optional[str] = None, seed: int = 0, pool_pages: Optional[int] = None,
               q_std: float = 1.0, kv_std: float = 1.0, outlier_frac: float = 0.0,
               outlier_mult: float = 20.0, name: str = "custom",
               gen: Optional[torch.Generator] = None, sm_scale: Optional[float] = None) -> PagedBatch:
    """Draw one batch.  ``qo_lens`` None means decode (one query row per
    request, no mask); otherwise causal prefill with qo_lens[b] <= kv_lens[b].
    ``gen`` continues an existing generator (so lengths drawn by the caller
    come first in the draw order); otherwise one is seeded with ``seed``."""
    if gen is None:
        gen = torch.Generator().manual_seed(seed)
    kv_lens = [int(x) for x in kv_lens]
    mode = "decode" if qo_lens is None else "prefill"
    qo_lens = [1] * len(kv_lens) if qo_lens is None else [int(x) for x in qo_lens]
    B, P, Hq, Hkv, D = len(kv_lens), page_size, num_qo_heads, num_kv_heads, head_dim
    if o_dtype is None:
        o_dtype = q_dtype if q_dtype in ("f16", "bf16") else "bf16"

    npages = [(L + P - 1) // P for L in kv_lens]
    need = sum(npages)
    pool = need if pool_pages is None else int(pool_pages)
    if pool < need:
        raise ValueError("page pool smaller than the pages the requests need")
    pool = max(pool, 1)

    perm = torch.randperm(pool, generator=gen)[:need].to(torch.int32)
    kv_indptr = torch.zeros(B + 1, dtype=torch.int32)
    kv_indptr[1:] = torch.tensor(np.cumsum(npages), dtype=torch.int32)
    qo_indptr = torch.zeros(B + 1, dtype=torch.int32)
    qo_indptr[1:] = torch.tensor(np.cumsum(qo_lens), dtype=torch.int32)
    last_page_len = torch.tensor([(L - (n - 1) * P) if n > 0 else 0 for L, n in zip(kv_lens, npages)],
                                 dtype=torch.int32)

    nnz_qo = sum(qo_lens)
    total_kv = sum(kv_lens)
    qf = torch.randn(nnz_qo, Hq, D, generator=gen) * q_std
    kf = torch.randn(total_kv, Hkv, D, generator=gen) * kv_std
    vf = torch.randn(total_kv, Hkv, D, generator=gen) * kv_std
    if outlier_frac > 0:
        mk = torch.rand(kf.shape, generator=gen) < outlier_frac
        kf[mk] *= outlier_mult
        del mk
        mv = torch.rand(vf.shape, generator=gen) < outlier_frac
        vf[mv] *= outlier_mult
        del mv

    if q_dtype in FP8_MAX:
        q, q_scale = _quantize(qf, q_dtype)
    else:
        q, q_scale = qf.to(TORCH_DTYPES[q_dtype]), 1.0
    del qf
    if kv_dtype in FP8_MAX:
        kq, k_scale = _quantize(kf, kv_dtype)
        del kf
        vq, v_scale = _quantize(vf, kv_dtype)
        del vf
    else:  # a 2-byte cache holds the values themselves (decode only)
        kq, k_scale = kf.to(TORCH_DTYPES[kv_dtype]), 1.0
        vq, v_scale = vf.to(TORCH_DTYPES[kv_dtype]), 1.0
        del kf, vf

    # Pool filled with random codes first; the requests' tokens overwrite
    # their own slots.
    esz = 1 if kv_dtype in FP8_MAX else 2
    shape = (pool, P, Hkv, D * esz)
    k_cache = torch.randint(0, 256, shape, generator=gen, dtype=torch.uint8)
    v_cache = torch.randint(0, 256, shape, generator=gen, dtype=torch.uint8)
    if total_kv:
        rows = torch.empty(total_kv, dtype=torch.int64)
        pos = 0
        for b, L in enumerate(kv_lens):
            t = torch.arange(L, dtype=torch.int64)
            pages = perm[kv_indptr[b]:kv_indptr[b + 1]].to(torch.int64)
            rows[pos:pos + L] = pages[t // P] * P + t % P
            pos += L
        k_cache.view(pool * P, Hkv, D * esz).index_copy_(0, rows, kq.view(torch.uint8))
        v_cache.view(pool * P, Hkv, D * esz).index_copy_(0, rows, vq.view(torch.uint8))
    k_cache = k_cache.view(TORCH_DTYPES[kv_dtype])
    v_cache = v_cache.view(TORCH_DTYPES[kv_dtype])

    return PagedBatch(
        name=name, mode=mode, num_qo_heads=Hq, num_kv_heads=Hkv, head_dim=D, page_size=P,
        num_pages=pool, q_dtype=q_dtype, kv_dtype=kv_dtype, o_dtype=o_dtype, q=q,
        k_cache=k_cache, v_cache=v_cache, qo_indptr=qo_indptr, kv_indptr=kv_indptr,
        kv_indices=perm, last_page_len=last_page_len, qo_lens=qo_lens, kv_lens=kv_lens,
        q_scale=float(q_scale), k_scale=float(k_scale), v_scale=float(v_scale),
        sm_scale=float(sm_scale) if sm_scale is not None else 1.0 / math.sqrt(D))


def with_layout(batch: PagedBatch, layout: str) -> PagedBatch:
    """The same batch with its caches stored in ``layout`` ("NHD" or "HND");
    every value is unchanged, only the order of the (slot, head) rows."""
    if layout == batch.kv_layout:
        return batch

    def perm(c):
        return c.view(torch.uint8).permute(0, 2, 1, 3).contiguous().view(c.dtype)
    return dataclasses.replace(batch, k_cache=perm(batch.k_cache), v_cache=perm(batch.v_cache), kv_layout=layout)


WORKLOADS = {
    1: "tiny batch decode (B=4, kv {37,64,100,129}, Hq 8/Hkv 2, e4m3fn KV, bf16 q/o)",
    2: "serving batch decode (B=64, kv U[512,4096], Hq 32/Hkv 8, e4m3fn KV, bf16 q/o)",
    3: "long-context decode (B=8, kv 32768, Hq 64/Hkv 8, e5m2 KV with 1% x20 outliers, f16 q/o)",
    4: "ragged causal prefill (B=16, qo U[128,1024], prefix U[0,2048], Hq 32/Hkv 8, e4m3fn KV, bf16 q/o)",
    5: "fp8 x fp8 causal prefill (B=8, qo=kv=2048, Hq 32/Hkv 8, e4m3fn q/KV, bf16 o)",
    6: "serving batch decode with a 2-byte cache (B=64, kv U[512,4096], Hq 32/Hkv 8, bf16 q/KV/o)",
    7: "ragged causal prefill with a 2-byte cache (B=16, qo U[128,1024], prefix U[0,2048], Hq 32/Hkv 8, bf16 q/KV/o)",
}


def workload(index: int, *, scale_down: int = 1) -> PagedBatch:
    """The named workloads, seed 1000 + index.  ``scale_down`` > 1
    divides every length (keeping at least one token) for quick runs of the
    same shape mix; it changes the draws, so use it only where the full size
    is not required."""
    gen = torch.Generator().manual_seed(1000 + index)
    sd = max(1, int(scale_down))

    def shrink(xs):
        return [max(1, int(x) // sd) for x in xs]

    if index == 1:
        return make_batch(shrink([37, 64, 100, 129]), num_qo_heads=8, num_kv_heads=2,
                          q_dtype="bf16", kv_dtype="e4m3fn", o_dtype="bf16",
                          pool_pages=64, gen=gen, name="tiny_decode")
    if index == 2:
        kv = torch.randint(512, 4097, (64,), generator=gen).tolist()
        return make_batch(shrink(kv), num_qo_heads=32, num_kv_heads=8, q_dtype="bf16",
                          kv_dtype="e4m3fn", o_dtype="bf16", gen=gen, name="serving_decode")
    if index == 3:
        return make_batch(shrink([32768] * 8), num_qo_heads=64, num_kv_heads=8, q_dtype="f16",
                          kv_dtype="e5m2", o_dtype="f16", kv_std=0.5, outlier_frac=0.01,
                          outlier_mult=20.0, gen=gen, name="long_decode")
    if index == 4:
        qo = torch.randint(128, 1025, (16,), generator=gen).tolist()
        prefix = torch.randint(0, 2049, (16,), generator=gen).tolist()
        qo = shrink(qo)
        prefix = [p // sd for p in prefix]
        kv = [a + b for a, b in zip(qo, prefix)]
        return make_batch(kv, qo, num_qo_heads=32, num_kv_heads=8, q_dtype="bf16",
                          kv_dtype="e4m3fn", o_dtype="bf16", gen=gen, name="ragged_prefill")
    if index == 5:
        L = shrink([2048] * 8)
        return make_batch(L, L, num_qo_heads=32, num_kv_heads=8, q_dtype="e4m3fn",
                          kv_dtype="e4m3fn", o_dtype="bf16", gen=gen, name="fp8_prefill")
    if index == 6:
        kv = torch.randint(512, 4097, (64,), generator=gen).tolist()
        return make_batch(shrink(kv), num_qo_heads=32, num_kv_heads=8, q_dtype="bf16",
                          kv_dtype="bf16", o_dtype="bf16", gen=gen, name="serving_decode_bf16_cache")
    if index == 7:
        qo = torch.randint(128, 1025, (16,), generator=gen).tolist()
        prefix = torch.randint(0, 2049, (16,), generator=gen).tolist()
        qo = shrink(qo)
        prefix = [p // sd for p in prefix]
        kv = [a + b for a, b in zip(qo, prefix)]
        return make_batch(kv, qo, num_qo_heads=32, num_kv_heads=8, q_dtype="bf16",
                          kv_dtype="bf16", o_dtype="bf16", gen=gen, name="ragged_prefill_bf16_cache")
    raise ValueError(f"unknown workload {index}")


@dataclasses.dataclass
class AppendBatch:
    """New tokens to be written into the paged cache of ``base``: one row of
    K and of V per (token, KV head), at the given (request, position)."""
    base: PagedBatch
    src_dtype: str                 # "f16", "bf16" or "f32"
    k_new: torch.Tensor            # [nnz, Hkv, D] of src_dtype
    v_new: torch.Tensor
    batch_indices: torch.Tensor    # int32 [nnz]
    positions: torch.Tensor        # int32 [nnz]

    @property
    def nnz(self) -> int:
        return int(self.batch_indices.numel())


SRC_DTYPES = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}


def new_tokens(base: PagedBatch, *, src_dtype: str = "bf16", seed: int = 0, std: float = 1.0) -> AppendBatch:
    """The last qo_len positions of every request of ``base`` (a prefill's new
    tokens, or one token per request for a decode batch), drawn N(0, std) in
    fp32 from a generator seeded with ``seed`` (K, then V) and cast to
    ``src_dtype`` (round to nearest)."""
    gen = torch.Generator().manual_seed(seed)
    b_idx, pos = [], []
    for b, (qo, kv) in enumerate(zip(base.qo_lens, base.kv_lens)):
        b_idx.extend([b] * qo)
        pos.extend(range(kv - qo, kv))
    nnz = len(b_idx)
    shape = (nnz, base.num_kv_heads, base.head_dim)
    kf = torch.randn(shape, generator=gen) * std
    vf = torch.randn(shape, generator=gen) * std
    dt = SRC_DTYPES[src_dtype]
    return AppendBatch(base=base, src_dtype=src_dtype, k_new=kf.to(dt), v_new=vf.to(dt),
                       batch_indices=torch.tensor(b_idx, dtype=torch.int32),
                       positions=torch.tensor(pos, dtype=torch.int32))


APPEND_WORKLOADS = {
    8: "KV append of the ragged prefill's new tokens (workload 4: 16 requests, qo U[128,1024], "
       "Hkv 8, bf16 rows -> e4m3fn cache)",
    9: "KV append of one decode step (workload 2: 64 requests, one token each, Hkv 8, "
       "bf16 rows -> e4m3fn cache)",
}


def append_workload(index: int, *, scale_down: int = 1) -> AppendBatch:
    """The named append workloads: new tokens (seed 1000 + index) for the cache
    of workload 4 (index 8) or workload 2 (index 9)."""
    if index == 8:
        return new_tokens(workload(4, scale_down=scale_down), src_dtype="bf16", seed=1008)
    if index == 9:
        return new_tokens(workload(2, scale_down=scale_down), src_dtype="bf16", seed=1009)
    raise ValueError(f"unknown append workload {index}")


@dataclasses.dataclass
class PodBatch:
    """A prefill batch and a decode batch over one page pool: ``prefill`` and
    ``decode`` share the same ``k_cache``/``v_cache`` tensors, ``num_pages``
    and per-tensor scales; the decode requests own pages of the pool that no
    prefill request owns."""
    prefill: PagedBatch
    decode: PagedBatch


POD_WORKLOADS = {
    10: "prefill and decode in one call over one page pool: the ragged causal prefill of workload 4 "
        "(16 requests) and the serving decode of workload 2 (64 requests), e4m3fn KV, bf16 q/o",
}


def pod_batch(prefill: PagedBatch, decode: PagedBatch) -> PodBatch:
    """Join two batches' pools (prefill pages first) into one; the decode
    requests' page indices move past the prefill pool and both phases use the
    prefill batch's per-tensor scales, q_scale included (one call takes one set
    of scales; the decode batch's fp8 codes are kept, so its values scale with
    them)."""
    if (prefill.kv_dtype, prefill.num_kv_heads, prefill.head_dim, prefill.page_size, prefill.kv_layout) != (
            decode.kv_dtype, decode.num_kv_heads, decode.head_dim, decode.page_size, decode.kv_layout):
        raise ValueError("the two batches' caches differ in dtype or shape")
    k = torch.cat([prefill.k_cache.view(torch.uint8), decode.k_cache.view(torch.uint8)]).view(prefill.k_cache.dtype)
    v = torch.cat([prefill.v_cache.view(torch.uint8), decode.v_cache.view(torch.uint8)]).view(prefill.v_cache.dtype)
    pool = prefill.num_pages + decode.num_pages
    pre = dataclasses.replace(prefill, k_cache=k, v_cache=v, num_pages=pool)
    dec = dataclasses.replace(decode, k_cache=k, v_cache=v, num_pages=pool,
                              kv_indices=decode.kv_indices + prefill.num_pages,
                              q_scale=prefill.q_scale, k_scale=prefill.k_scale, v_scale=prefill.v_scale)
    return PodBatch(prefill=pre, decode=dec)


def pod_workload(index: int, *, scale_down: int = 1) -> PodBatch:
    """The named POD workloads (index 10: workloads 4 and 2 over one pool)."""
    if index == 10:
        return pod_batch(workload(4, scale_down=scale_down), workload(2, scale_down=scale_down))
    raise ValueError(f"unknown POD workload {index}")
