// append.cu -- quantize new K/V tokens into the paged fp8 cache.  sm_103a.
//
// The cache every other kernel reads holds fp8 codes whose values times the
// per-tensor scale are the keys and values ("fp8 KV cache in the in-tree
// prefill kernel", What changed: KV stays fp8 in HBM and is dequantized on
// load).  Writing a new token is the inverse: code = fp8(RNE, saturating)(
// fp32(x) * fp32(1/scale)).
//
// One thread per 16 elements of one (token, KV head) row, K and V both:
// 16-byte loads of the source (two for a 2-byte type, four for fp32), issued
// for K and V before the page-table lookups they do not depend on, the
// product with fp32(1/scale) rounded once in fp32 (__fmul_rn), pairs packed by
// cvt.rn.satfinite.{e4m3x2,e5m2x2}.f32 (round to nearest even, magnitudes
// above the largest finite value saturate to it, NaN stays NaN), one 16-byte
// store of the 16 codes.  head_dim / 16 consecutive threads cover a row (8
// for head_dim 128, 4 for 64), so a warp reads consecutive rows and writes
// rows of one page slot (consecutive in the NHD layout [page][slot][head][d],
// a page-slot stride apart in the HND layout [page][head][slot][d]).  The
// page comes from the request's CSR page table; a token whose request,
// position or page lies outside the table or the pool is skipped and
// reported in *status.  The work is a pure stream of reads and writes,
// bounded by HBM bandwidth.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "../../include/pafp8.h"
#include "internal.h"

namespace pafp8 {
namespace {

constexpr int kThreads = 256;

// Raw source words of 16 elements: 8 words for a 2-byte type, 16 for fp32.
template <int SRC>
struct Raw16 {
    static constexpr int kWords = SRC == PAFP8_F32 ? 16 : 8;
    uint32_t w[kWords];
};

template <int SRC>
__device__ __forceinline__ void load_raw(const void* base, size_t off, Raw16<SRC>& r) {
    const uint4* s = reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(base) +
                                                    off * (SRC == PAFP8_F32 ? 4 : 2));
#pragma unroll
    for (int i = 0; i < Raw16<SRC>::kWords / 4; ++i) {
        const uint4 v = __ldcs(s + i);
        r.w[4 * i] = v.x;
        r.w[4 * i + 1] = v.y;
        r.w[4 * i + 2] = v.z;
        r.w[4 * i + 3] = v.w;
    }
}

// Element i of the 16 as fp32 (exact: f16 and bf16 are subsets of fp32).
template <int SRC>
__device__ __forceinline__ float elem(const Raw16<SRC>& r, int i) {
    if constexpr (SRC == PAFP8_F32) {
        return __uint_as_float(r.w[i]);
    } else if constexpr (SRC == PAFP8_BF16) {
        return __uint_as_float((i & 1) ? (r.w[i >> 1] & 0xFFFF0000u) : (r.w[i >> 1] << 16));
    } else {
        return __half2float(__ushort_as_half((unsigned short)((i & 1) ? (r.w[i >> 1] >> 16) : (r.w[i >> 1] & 0xFFFFu))));
    }
}

// Codes of (lo, hi): lo in the low byte.
template <int KV>
__device__ __forceinline__ uint32_t cvt_pair(float lo, float hi) {
    unsigned short d;
    if constexpr (KV == PAFP8_E4M3FN)
        asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(d) : "f"(hi), "f"(lo));
    else
        asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(d) : "f"(hi), "f"(lo));
    return d;
}

template <int KV, int SRC>
__device__ __forceinline__ uint4 quantize16(const Raw16<SRC>& r, float inv) {
    uint32_t w[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint32_t a = cvt_pair<KV>(__fmul_rn(elem(r, 4 * k), inv), __fmul_rn(elem(r, 4 * k + 1), inv));
        const uint32_t b = cvt_pair<KV>(__fmul_rn(elem(r, 4 * k + 2), inv), __fmul_rn(elem(r, 4 * k + 3), inv));
        w[k] = a | (b << 16);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

template <int SRC, int KV, int DH>
__global__ void __launch_bounds__(kThreads) append_kernel(const AppendParams p) {
    constexpr int CPR = DH / 16;  // threads per (token, KV head) row
    const long long total = p.nnz * (long long)p.num_kv_heads * CPR;
    for (long long t = (long long)blockIdx.x * kThreads + threadIdx.x; t < total;
         t += (long long)gridDim.x * kThreads) {
        const long long row = t / CPR;  // (token, KV head)
        const int c = (int)(t - row * CPR);
        const long long tok = row / p.num_kv_heads;
        const int h = (int)(row - tok * p.num_kv_heads);
        // The source rows do not depend on the page: their loads go first and
        // overlap the page-table lookups.
        const size_t src = (size_t)row * DH + 16 * c;
        Raw16<SRC> rk, rv;
        load_raw<SRC>(p.k_new, src, rk);
        load_raw<SRC>(p.v_new, src, rv);
        const int b = __ldg(p.batch_indices + tok);
        const int pos = __ldg(p.positions + tok);
        int page = -1;
        if (b >= 0 && b < p.batch && pos >= 0) {
            const int e0 = __ldg(p.kv_indptr + b), e1 = __ldg(p.kv_indptr + b + 1);
            const long long e = (long long)e0 + pos / p.page_size;
            if (e0 >= 0 && e < e1) {
                const int pg = __ldg(p.kv_indices + e);
                if (pg >= 0 && pg < p.num_pages) page = pg;
            }
        }
        if (page < 0) {
            if (c == 0 && p.status != nullptr) atomicOr(p.status, kStatusBounds);
            continue;
        }
        const size_t slot = (size_t)(pos % p.page_size);
        const size_t dst = (p.hnd ? ((size_t)page * p.num_kv_heads + h) * p.page_size + slot
                                  : ((size_t)page * p.page_size + slot) * p.num_kv_heads + h) *
                               DH +
                           16 * c;
        *reinterpret_cast<uint4*>(static_cast<uint8_t*>(p.k_cache) + dst) = quantize16<KV>(rk, p.k_inv);
        *reinterpret_cast<uint4*>(static_cast<uint8_t*>(p.v_cache) + dst) = quantize16<KV>(rv, p.v_inv);
    }
}

template <int SRC, int KV, int DH>
cudaError_t launch_t(const AppendParams& p, cudaStream_t stream) {
    const long long total = p.nnz * (long long)p.num_kv_heads * (DH / 16);
    const long long blocks = (total + kThreads - 1) / kThreads;
    const int grid = (int)(blocks < 65535 ? blocks : 65535);
    append_kernel<SRC, KV, DH><<<grid, kThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

template <int SRC, int KV>
cudaError_t launch_kv(const AppendParams& p, cudaStream_t stream) {
    return p.head_dim == 64 ? launch_t<SRC, KV, 64>(p, stream) : launch_t<SRC, KV, 128>(p, stream);
}

template <int SRC>
cudaError_t launch_src(const AppendParams& p, cudaStream_t stream) {
    return p.kv_dtype == PAFP8_E4M3FN ? launch_kv<SRC, PAFP8_E4M3FN>(p, stream)
                                      : launch_kv<SRC, PAFP8_E5M2>(p, stream);
}

}  // namespace

cudaError_t launch_append(const AppendParams& p, cudaStream_t stream) {
    if (p.nnz == 0) return cudaSuccess;
    switch (p.src_dtype) {
        case PAFP8_F16:
            return launch_src<PAFP8_F16>(p, stream);
        case PAFP8_BF16:
            return launch_src<PAFP8_BF16>(p, stream);
        case PAFP8_F32:
            return launch_src<PAFP8_F32>(p, stream);
        default:
            return cudaErrorInvalidValue;
    }
}

}  // namespace pafp8
