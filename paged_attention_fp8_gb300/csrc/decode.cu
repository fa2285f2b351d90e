// decode.cu -- paged decode attention over an fp8 KV cache, and the split-KV
// merge.  sm_103a.
//
// What it computes: for every request b and query head h (KV head
// h / group), o = v_scale * softmax_j(sm_scale * q_scale * k_scale * q.k_j) V_j
// over the request's kv_len cached tokens, with lse = ln sum_j exp(logit_j).
// The KV bytes stay fp8 in HBM and are dequantized on load ("fp8 KV cache in
// the in-tree prefill kernel", Kernel note and Architecture / design notes);
// k_scale (with q_scale) folds into the softmax scale and v_scale multiplies
// the output once, the two folds of that page's Test plan.
//
// Design (one persistent CTA per SM):
//  * Warp `HPC` is the producer.  It walks the CTA's segments (row, page
//    range) from the plan, prefetches 32 page indices per warp-wide load, and
//    for each page issues one TMA box per tensor covering the block's KV
//    heads (or one per head), 16 tokens x 128 bytes per head, 128B-swizzled,
//    head-major in shared memory, into a ring of stages guarded by
//    full/empty mbarriers.  Every wait is bounded; on expiry the kernel sets a
//    status bit and returns after its copies in flight have landed.
//  * Warps 0..HPC-1 are consumers, one per KV head of the block.  Each
//    consumer keeps the whole GQA group (up to 8 query heads) of its KV head,
//    so every KV byte is read from HBM once.  Per 16-token page:
//      S^T[16 tok x 8 heads] = K[16 x 128] . Q^T   (m16n8k16, f16 in, f32 acc)
//    with fp8 -> f16 conversion in registers (exact for e4m3fn and e5m2), an
//    online softmax in the log2 domain (column max by warp shuffles), P
//    transposed in registers with movmatrix, then
//      O^T[128 x 8] += V^T[128 x 16 tok] . P^T.
//    The head dimension is permuted consistently between K and Q (thread t
//    owns dims 32t..32t+31 of every row) and between V and O (thread g owns
//    dims 16g..16g+15), so every shared-memory read is one conflict-free
//    16-byte load.
//  * A 2-byte cache (f16 or bf16, which the pages exempt from the rule that
//    the cache matches the query in decode) runs through the same kernel:
//    each 128-element row arrives as two 128-byte halves, every thread loads
//    the same dims of the same tokens as in the fp8 case, and the MMA operand
//    words it assembles are exactly the converted words the fp8 path feeds
//    the tensor cores.  So an fp8 cache and its f16 dequantization give
//    bit-identical results.  A bf16 cache runs bf16 MMAs with P rounded to
//    bf16; an f16 query enters them as two bf16 words whose sum is exact.
//  * A segment covering its whole request writes o and lse; a partial one
//    writes (O/l, lse in log2 units) to the workspace, and a separate merge
//    kernel (one block per split row and query head, launched as a
//    programmatic dependent) combines them by their log-sum-exp.  Folding
//    the merge into this kernel made the warps that merged stall their
//    CTA's page ring.  A request with no KV writes o = 0, lse = -inf.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <mutex>

#include "../../include/pafp8.h"
#include "internal.h"
#include "ptx.cuh"

namespace pafp8 {
namespace {

using namespace ptx;


constexpr int P = kPageSize;
constexpr int kStageBudget = 192 * 1024;    // shared memory for the page ring
constexpr int kChunkSlots = 2;              // chunk-id queue depth
__host__ __device__ constexpr bool is_2byte_kv(int kt) { return kt == PAFP8_F16 || kt == PAFP8_BF16; }
// One KV head of one page in shared memory: 16 token rows of dh bytes (fp8:
// 128 B with the 128-byte swizzle, or 64 B with the 64-byte swizzle), or of
// 2 dh bytes (2-byte cache: two swizzled 128-B halves per row for dh 128,
// one 128-B row for dh 64).
__host__ __device__ constexpr int tile_bytes(int kt, int dh) { return P * dh * (is_2byte_kv(kt) ? 2 : 1); }
__device__ __forceinline__ void flag(uint32_t* status, uint32_t bit) { atomicOr(status, bit); }

template <bool kBF16>
__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    if (kBF16)
        mma_16816_bf16(c, a0, a1, a2, a3, b0, b1);
    else
        mma_16816(c, a0, a1, a2, a3, b0, b1);
}

// Q fragment for the QK product: B operand (K = head dim, N = 8 query heads).
// Lane (g, t) holds head g of the group, dims (DH/4)t .. (DH/4)t + DH/4 - 1, as
// DH/8 f16x2 words; word j = dims (DH/4)t+2j, (DH/4)t+2j+1.  Returns the
// power-of-two factor the logits must be multiplied by (a bf16 query is
// brought into f16 range by an exact power-of-two scaling when its magnitude
// needs it).
template <bool kBF16, int DH>
__device__ __forceinline__ float load_q(uint32_t (&qf)[16], uint32_t (&qlo)[16], const void* q, int q_dtype,
                                        size_t head_off, bool active, int t) {
    constexpr int QW = DH / 8;   // words per lane
    constexpr int Q4 = QW / 4;   // 16-byte loads of a 2-byte query
    float factor = 1.0f;
    if (kBF16) {
        // bf16 MMAs (bf16 cache): a bf16 query as is; an f16 query as the sum
        // of two bf16 words, its bf16 rounding (qf) and the exact remainder
        // (qlo: an f16 has 11 significant bits, so the remainder needs at most
        // 4 of bf16's 8), so the QK product loses nothing.
        uint4 w[Q4] = {};
        if (active) {
            const uint4* src = reinterpret_cast<const uint4*>(
                static_cast<const uint16_t*>(q) + head_off + (DH / 4) * t);
#pragma unroll
            for (int i = 0; i < Q4; ++i) w[i] = __ldg(src + i);
        }
        const uint32_t* ws = reinterpret_cast<const uint32_t*>(w);
#pragma unroll
        for (int j = 0; j < QW; ++j) {
            if (q_dtype == PAFP8_BF16) {
                qf[j] = ws[j];
            } else {
                const __half2 h = *reinterpret_cast<const __half2*>(&ws[j]);
                const float2 f = __half22float2(h);
                const float hx = __bfloat162float(__float2bfloat16_rn(f.x));
                const float hy = __bfloat162float(__float2bfloat16_rn(f.y));
                qf[j] = pack_bf162(hx, hy);
                qlo[j] = pack_bf162(f.x - hx, f.y - hy);
            }
        }
    } else if (q_dtype == PAFP8_F16 || q_dtype == PAFP8_BF16) {
        uint4 w[Q4] = {};
        if (active) {
            const uint4* src = reinterpret_cast<const uint4*>(
                static_cast<const uint16_t*>(q) + head_off + (DH / 4) * t);
#pragma unroll
            for (int i = 0; i < Q4; ++i) w[i] = __ldg(src + i);
        }
        const uint32_t* ws = reinterpret_cast<const uint32_t*>(w);
        if (q_dtype == PAFP8_F16) {
#pragma unroll
            for (int j = 0; j < QW; ++j) qf[j] = ws[j];
        } else {
            // Largest |q| over the warp decides the power-of-two shift.
            uint32_t mx = 0;
#pragma unroll
            for (int j = 0; j < QW; ++j) {
                mx = max(mx, (ws[j] & 0x7FFFu) << 16);
                mx = max(mx, ws[j] & 0x7FFF0000u);
            }
            mx = __reduce_max_sync(0xFFFFFFFFu, mx);
            const int e = (int)((mx >> 23) & 0xFF) - 127;
            const int shift = e > 14 ? e - 14 : 0;
            const float down = __int_as_float((127 - shift) << 23);
            factor = __int_as_float((127 + shift) << 23);
#pragma unroll
            for (int j = 0; j < QW; ++j) {
                const float lo = __uint_as_float(ws[j] << 16) * down;
                const float hi = __uint_as_float(ws[j] & 0xFFFF0000u) * down;
                qf[j] = pack_half2(lo, hi);
            }
        }
    } else {
        // fp8 query: DH/4 bytes per lane, DH/64 16-byte loads.
        uint4 w[DH / 64] = {};
        if (active) {
            const uint4* src = reinterpret_cast<const uint4*>(
                static_cast<const uint8_t*>(q) + head_off + (DH / 4) * t);
#pragma unroll
            for (int i = 0; i < DH / 64; ++i) w[i] = __ldg(src + i);
        }
        const uint32_t* ws = reinterpret_cast<const uint32_t*>(w);
#pragma unroll
        for (int j = 0; j < QW / 2; ++j) {
            if (q_dtype == PAFP8_E4M3FN) {
                qf[2 * j] = fp8x2_lo<PAFP8_E4M3FN>(ws[j]);
                qf[2 * j + 1] = fp8x2_hi<PAFP8_E4M3FN>(ws[j]);
            } else {
                qf[2 * j] = fp8x2_lo<PAFP8_E5M2>(ws[j]);
                qf[2 * j + 1] = fp8x2_hi<PAFP8_E5M2>(ws[j]);
            }
        }
    }
    return factor;
}

// Combine the partial states of each split (request, KV-head block) row.
// The plan numbers a row's partial states consecutively (slots mptr[e] ..
// mptr[e+1] - 1, in page order), so no slot list is read.
// One warp per (merge entry, query head of the block), kMergeWarps per block;
// lane l holds dims (D/32) l .. (D/32) l + D/32 - 1.  The warp loads the
// row's slots in batches of kMergeBatch (every lane the batch's lse values
// and its own dims of the O vectors, all loads of a batch in flight
// together), keeps a running max m of the log2-domain lse_c and the rescaled
// sums of 2^lse_c and 2^lse_c O_c, and writes
// o = v_scale * sum(2^lse_c O_c) / sum(2^lse_c), lse = ln(sum) + m.
// Launched as a programmatic dependent of the decode kernel: the row's
// metadata (written by the host) is read before griddepcontrol.wait, which
// returns once the decode grid has completed and its writes are visible.
constexpr int kMergeBatch = 8;
constexpr int kMergeWarps = 4;  // query heads per merge block

// kMergeBatch lse values and O vectors (DPL floats) of partial states, all
// loads issued in one instruction block (L2, bypassing L1), so the batch's
// latencies overlap.
template <int DPL>
__device__ __forceinline__ void load_batch(const float* const (&lp)[kMergeBatch], const float* const (&op)[kMergeBatch],
                                           float (&l)[kMergeBatch], float (&o)[kMergeBatch][DPL]);
template <>
__device__ __forceinline__ void load_batch<4>(const float* const (&lp)[kMergeBatch], const float* const (&op)[kMergeBatch],
                                              float (&l)[kMergeBatch], float (&o)[kMergeBatch][4]) {
    asm volatile(
        "ld.global.cg.f32 %0, [%40];\n ld.global.cg.f32 %1, [%41];\n ld.global.cg.f32 %2, [%42];\n"
        " ld.global.cg.f32 %3, [%43];\n ld.global.cg.f32 %4, [%44];\n ld.global.cg.f32 %5, [%45];\n"
        " ld.global.cg.f32 %6, [%46];\n ld.global.cg.f32 %7, [%47];\n"
        " ld.global.cg.v4.f32 {%8, %9, %10, %11}, [%48];\n ld.global.cg.v4.f32 {%12, %13, %14, %15}, [%49];\n"
        " ld.global.cg.v4.f32 {%16, %17, %18, %19}, [%50];\n ld.global.cg.v4.f32 {%20, %21, %22, %23}, [%51];\n"
        " ld.global.cg.v4.f32 {%24, %25, %26, %27}, [%52];\n ld.global.cg.v4.f32 {%28, %29, %30, %31}, [%53];\n"
        " ld.global.cg.v4.f32 {%32, %33, %34, %35}, [%54];\n ld.global.cg.v4.f32 {%36, %37, %38, %39}, [%55];\n"
        : "=f"(l[0]), "=f"(l[1]), "=f"(l[2]), "=f"(l[3]), "=f"(l[4]), "=f"(l[5]), "=f"(l[6]), "=f"(l[7]),
          "=f"(o[0][0]), "=f"(o[0][1]), "=f"(o[0][2]), "=f"(o[0][3]), "=f"(o[1][0]), "=f"(o[1][1]), "=f"(o[1][2]),
          "=f"(o[1][3]), "=f"(o[2][0]), "=f"(o[2][1]), "=f"(o[2][2]), "=f"(o[2][3]), "=f"(o[3][0]), "=f"(o[3][1]),
          "=f"(o[3][2]), "=f"(o[3][3]), "=f"(o[4][0]), "=f"(o[4][1]), "=f"(o[4][2]), "=f"(o[4][3]), "=f"(o[5][0]),
          "=f"(o[5][1]), "=f"(o[5][2]), "=f"(o[5][3]), "=f"(o[6][0]), "=f"(o[6][1]), "=f"(o[6][2]), "=f"(o[6][3]),
          "=f"(o[7][0]), "=f"(o[7][1]), "=f"(o[7][2]), "=f"(o[7][3])
        : "l"(lp[0]), "l"(lp[1]), "l"(lp[2]), "l"(lp[3]), "l"(lp[4]), "l"(lp[5]), "l"(lp[6]), "l"(lp[7]),
          "l"(op[0]), "l"(op[1]), "l"(op[2]), "l"(op[3]), "l"(op[4]), "l"(op[5]), "l"(op[6]), "l"(op[7])
        : "memory");
    // Every result is live here, so no use of one can be scheduled before
    // the last load of the batch has been issued.
    asm volatile("" ::"f"(l[0]), "f"(l[1]), "f"(l[2]), "f"(l[3]), "f"(l[4]), "f"(l[5]), "f"(l[6]), "f"(l[7]),
                 "f"(o[0][0]), "f"(o[0][1]), "f"(o[0][2]), "f"(o[0][3]), "f"(o[1][0]), "f"(o[1][1]), "f"(o[1][2]),
                 "f"(o[1][3]), "f"(o[2][0]), "f"(o[2][1]), "f"(o[2][2]), "f"(o[2][3]), "f"(o[3][0]), "f"(o[3][1]),
                 "f"(o[3][2]), "f"(o[3][3]), "f"(o[4][0]), "f"(o[4][1]), "f"(o[4][2]), "f"(o[4][3]), "f"(o[5][0]),
                 "f"(o[5][1]), "f"(o[5][2]), "f"(o[5][3]), "f"(o[6][0]), "f"(o[6][1]), "f"(o[6][2]), "f"(o[6][3]),
                 "f"(o[7][0]), "f"(o[7][1]), "f"(o[7][2]), "f"(o[7][3]));
}
template <>
__device__ __forceinline__ void load_batch<2>(const float* const (&lp)[kMergeBatch], const float* const (&op)[kMergeBatch],
                                              float (&l)[kMergeBatch], float (&o)[kMergeBatch][2]) {
    asm volatile(
        "ld.global.cg.f32 %0, [%24];\n ld.global.cg.f32 %1, [%25];\n ld.global.cg.f32 %2, [%26];\n"
        " ld.global.cg.f32 %3, [%27];\n ld.global.cg.f32 %4, [%28];\n ld.global.cg.f32 %5, [%29];\n"
        " ld.global.cg.f32 %6, [%30];\n ld.global.cg.f32 %7, [%31];\n"
        " ld.global.cg.v2.f32 {%8, %9}, [%32];\n ld.global.cg.v2.f32 {%10, %11}, [%33];\n"
        " ld.global.cg.v2.f32 {%12, %13}, [%34];\n ld.global.cg.v2.f32 {%14, %15}, [%35];\n"
        " ld.global.cg.v2.f32 {%16, %17}, [%36];\n ld.global.cg.v2.f32 {%18, %19}, [%37];\n"
        " ld.global.cg.v2.f32 {%20, %21}, [%38];\n ld.global.cg.v2.f32 {%22, %23}, [%39];\n"
        : "=f"(l[0]), "=f"(l[1]), "=f"(l[2]), "=f"(l[3]), "=f"(l[4]), "=f"(l[5]), "=f"(l[6]), "=f"(l[7]),
          "=f"(o[0][0]), "=f"(o[0][1]), "=f"(o[1][0]), "=f"(o[1][1]), "=f"(o[2][0]), "=f"(o[2][1]), "=f"(o[3][0]),
          "=f"(o[3][1]), "=f"(o[4][0]), "=f"(o[4][1]), "=f"(o[5][0]), "=f"(o[5][1]), "=f"(o[6][0]), "=f"(o[6][1]),
          "=f"(o[7][0]), "=f"(o[7][1])
        : "l"(lp[0]), "l"(lp[1]), "l"(lp[2]), "l"(lp[3]), "l"(lp[4]), "l"(lp[5]), "l"(lp[6]), "l"(lp[7]),
          "l"(op[0]), "l"(op[1]), "l"(op[2]), "l"(op[3]), "l"(op[4]), "l"(op[5]), "l"(op[6]), "l"(op[7])
        : "memory");
    asm volatile("" ::"f"(l[0]), "f"(l[1]), "f"(l[2]), "f"(l[3]), "f"(l[4]), "f"(l[5]), "f"(l[6]), "f"(l[7]),
                 "f"(o[0][0]), "f"(o[0][1]), "f"(o[1][0]), "f"(o[1][1]), "f"(o[2][0]), "f"(o[2][1]), "f"(o[3][0]),
                 "f"(o[3][1]), "f"(o[4][0]), "f"(o[4][1]), "f"(o[5][0]), "f"(o[5][1]), "f"(o[6][0]), "f"(o[6][1]),
                 "f"(o[7][0]), "f"(o[7][1]));
}

template <int DPL>
__device__ __forceinline__ void merge_head(const DecodeParams& p, int hpb, int hh, int s0, int s1, size_t oh,
                                           float vscale) {
    const int lane = threadIdx.x & 31;
    float m = -INFINITY, sum = 0.f, acc[DPL];
#pragma unroll
    for (int i = 0; i < DPL; ++i) acc[i] = 0.f;
    for (int s = s0; s < s1; s += kMergeBatch) {
        float l[kMergeBatch], o[kMergeBatch][DPL];
        const float* lp[kMergeBatch];
        const float* op[kMergeBatch];
#pragma unroll
        for (int k = 0; k < kMergeBatch; ++k) {
            const size_t idx = (size_t)(s + k < s1 ? s + k : s) * hpb + hh;  // a row's slots are consecutive
            lp[k] = p.part_lse + idx;
            op[k] = p.part_o + idx * p.head_dim + DPL * lane;
        }
        load_batch<DPL>(lp, op, l, o);  // every load of the batch in flight together
        // Slot s (k = 0) exists, so m is finite from here on; padding slots
        // (lse -inf) get weight 0.
#pragma unroll
        for (int k = 0; k < kMergeBatch; ++k) {
            const float lk = s + k < s1 ? l[k] : -INFINITY;
            const float mn = fmaxf(m, lk);
            const float a = ex2(m - mn), wt = ex2(lk - mn);
            sum = sum * a + wt;
#pragma unroll
            for (int i = 0; i < DPL; ++i) acc[i] = acc[i] * a + wt * o[k][i];
            m = mn;
        }
    }
    const float inv = vscale / sum;
    uint32_t wd[DPL / 2];
#pragma unroll
    for (int i = 0; i < DPL / 2; ++i) wd[i] = pack_out2(acc[2 * i] * inv, acc[2 * i + 1] * inv, p.o_dtype);
    uint16_t* dst = static_cast<uint16_t*>(p.o) + oh * p.head_dim + DPL * lane;
    if constexpr (DPL == 4)
        *reinterpret_cast<uint2*>(dst) = make_uint2(wd[0], wd[DPL > 2 ? 1 : 0]);
    else
        *reinterpret_cast<uint32_t*>(dst) = wd[0];
    if (lane == 0 && p.lse != nullptr) p.lse[oh] = (m + __log2f(sum)) * 0.69314718055994531f;
}

// One (merge entry, query head) pair's metadata: its slots, output row and
// v_scale.  The metadata is the host's, so it may be read before the
// partial states are complete.
struct MergePair {
    int hh, s0, s1;
    size_t oh;
    float vscale;
};

__device__ __forceinline__ MergePair merge_pair_args(const DecodeParams& p, int hpc, int group, int e, int hh) {
    const int* meta = p.meta;
    const int nhb = meta[kMetaHeadBlocks];
    const int* mptr = meta + meta[kMetaOffMergePtr];
    const int* mrow = meta + meta[kMetaOffMergeRow];
    const int hpb = hpc * group;
    const int row = mrow[e];
    const int b = row / nhb, hb = row - b * nhb;
    const int head = hb * hpb + hh;  // query head: (hb * hpc + hh / group) * group + hh % group
    MergePair a;
    a.hh = hh;
    a.s0 = mptr[e];
    a.s1 = mptr[e + 1];
    a.oh = (size_t)b * p.num_qo_heads + head;
    a.vscale = p.v_scales != nullptr ? __ldg(p.v_scales + head / group) : p.v_scale;
    return a;
}

__device__ __forceinline__ void merge_pair(const DecodeParams& p, int hpb, const MergePair& a) {
    if (p.head_dim == 64)
        merge_head<2>(p, hpb, a.hh, a.s0, a.s1, a.oh, a.vscale);
    else
        merge_head<4>(p, hpb, a.hh, a.s0, a.s1, a.oh, a.vscale);
}

template <int KT, int DH, bool kDiag, bool kSlots>
__global__ void __launch_bounds__(32 * 9, 1)
    decode_kernel(const __grid_constant__ DecodeParams p, const __grid_constant__ CUtensorMap tmk,
                  const __grid_constant__ CUtensorMap tmv, int hpc, int group, int stages,
                  int heads_per_box) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;      // 128B swizzle wants 1024-B alignment
    constexpr bool k2 = is_2byte_kv(KT), kBF = KT == PAFP8_BF16;
    constexpr uint32_t kTileBytes = (uint32_t)tile_bytes(KT, DH);
    constexpr int NA = DH / 16;    // PV accumulators (MMAs) per lane; also QK k-steps
    const uint32_t stage_bytes = 2u * hpc * kTileBytes;  // K heads then V heads
    const uint32_t bar_full = base + stages * stage_bytes;
    const uint32_t bar_empty = bar_full + 8u * stages;
    // Queue of chunk ids (run-time work) from the producer to the consumers:
    // kChunkSlots slots with full / empty barriers.
    const uint32_t cq_full = bar_empty + 8u * stages;
    const uint32_t cq_empty = cq_full + 8u * kChunkSlots;
    const uint32_t cq_id = cq_empty + 8u * kChunkSlots;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int* meta = p.meta;
    const int nhb = meta[kMetaHeadBlocks];
    const int* req_page = meta + meta[kMetaOffReqPage];
    const int* req_kv = meta + meta[kMetaOffReqKvLen];
    const int* cta_seg = meta + meta[kMetaOffCtaSeg];
    const int* segs = meta + meta[kMetaOffSeg];
    const int seg_begin = cta_seg[blockIdx.x], seg_end = cta_seg[blockIdx.x + 1];
    const int n_chunks = meta[kMetaNumChunks];
    const int* chunk_rec = meta + meta[kMetaOffChunk];

    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(bar_full + 8u * s, 1);
            mbar_init(bar_empty + 8u * s, 32u * hpc);
        }
        for (int s = 0; s < kChunkSlots; ++s) {
            mbar_init(cq_full + 8u * s, 1);
            mbar_init(cq_empty + 8u * s, (uint32_t)hpc);
        }

        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    __syncthreads();
    // Let the merge grid (launched as a programmatic dependent) start now
    // rather than when the last CTA of this grid exits: its small blocks fit
    // beside this CTA, read their metadata and wait in griddepcontrol.wait,
    // which still returns only once this grid has completed and its writes
    // are visible.  A no-op when no merge follows.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if (warp == hpc) {
        // ---------------------------------------------------------- producer
        if (lane == 0) {
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmk)) : "memory");
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmv)) : "memory");
        }
        int stage = 0;
        uint32_t phase = 0;
        long long issued = 0;
        bool ok = true;
        int si = seg_begin, cq = 0;
        uint32_t cqphase = 0;
        uint32_t* const ctr = p.status + kChunkCounterWord;
        for (;;) {
            // This CTA's own segments, then chunks taken from the counter
            // until none is left; each chunk id goes to the consumers first.
            const int* rec;
            if (si < seg_end) {
                rec = segs + 4 * si++;
            } else {
                if (n_chunks == 0) break;
                int c = -1;
                if (lane == 0) {
                    c = (int)atomicAdd(ctr, 1u);
                    if (c >= n_chunks) c = -1;
                    ok = pipe_wait<kDiag>(cq_empty + 8u * cq, cqphase ^ 1u, p.wait_cycles);
                    if (ok) {
                        sts32(cq_id + 4u * cq, (uint32_t)c);
                        mbar_arrive(cq_full + 8u * cq);
                    }
                }
                ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
                c = __shfl_sync(0xFFFFFFFFu, c, 0);
                if (++cq == kChunkSlots) {
                    cq = 0;
                    cqphase ^= 1u;
                }
                if (!ok || c < 0) break;
                rec = chunk_rec + 4 * c;
            }
            const int row = rec[0], p0 = rec[1], p1 = rec[2];
            const int b = row / nhb, hb = row - b * nhb;
            const int* idx = p.kv_indices + req_page[b];
            for (int pb = p0; pb < p1 && ok; pb += 32) {
                const int n = min(32, p1 - pb);
                // Pool pages and token slots of 16-token sub-pages (a page of
                // 16 * m tokens is m of them); an id outside the pool reads page
                // 0 instead.
                // (kSlots: pages of 16 m tokens, m > 1; the 16-token path keeps
                // its lookup free of the division by m.)
                bool bad = false;
                SubPageAt sp{0, 0};
                if constexpr (kSlots) {
                    if (lane < n) sp = sub_page(idx, pb + lane, p.page_mult, p.num_pages, bad);
                } else if (lane < n) {
                    const int pg = __ldg(idx + pb + lane);
                    bad = pg < 0 || pg >= p.num_pages;
                    sp.page = bad ? 0 : pg;
                }
                if (__any_sync(0xFFFFFFFFu, bad) && lane == 0) flag(p.status, kStatusBounds);
                for (int j = 0; j < n; ++j) {
                    SubPageAt at;
                    at.page = __shfl_sync(0xFFFFFFFFu, sp.page, j);
                    at.slot = kSlots ? __shfl_sync(0xFFFFFFFFu, sp.slot, j) : 0;
                    if (lane == 0) {
                        if (!pipe_wait<kDiag>(bar_empty + 8u * stage, phase ^ 1u, p.wait_cycles)) {
                            ok = false;
                        } else {
                            const uint32_t fb = bar_full + 8u * stage;
                            mbar_arrive_expect_tx(fb, stage_bytes);
                            const uint32_t sk = base + stage * stage_bytes;
                            const uint32_t sv = sk + hpc * kTileBytes;
                            if (k2) {
                                // (d % 64, d / 64, token, head, page) or, per head,
                                // (d % 64, d / 64, head, token, page)
                                if (heads_per_box == hpc) {
                                    tma_load_5d(sk, &tmk, fb, 0, 0, at.slot, hb * hpc, at.page);
                                    tma_load_5d(sv, &tmv, fb, 0, 0, at.slot, hb * hpc, at.page);
                                } else {
                                    for (int h = 0; h < hpc; ++h) {
                                        tma_load_5d(sk + h * kTileBytes, &tmk, fb, 0, 0, hb * hpc + h, at.slot,
                                                    at.page);
                                        tma_load_5d(sv + h * kTileBytes, &tmv, fb, 0, 0, hb * hpc + h, at.slot,
                                                    at.page);
                                    }
                                }
                            } else if (heads_per_box == hpc) {
                                // one box = every head of the block: (d, token, head, page)
                                tma_load_4d(sk, &tmk, fb, 0, at.slot, hb * hpc, at.page);
                                tma_load_4d(sv, &tmv, fb, 0, at.slot, hb * hpc, at.page);
                            } else {
                                // one box per head: (d, head, token, page)
                                for (int h = 0; h < hpc; ++h) {
                                    tma_load_4d(sk + h * kTileBytes, &tmk, fb, 0, hb * hpc + h, at.slot, at.page);
                                    tma_load_4d(sv + h * kTileBytes, &tmv, fb, 0, hb * hpc + h, at.slot, at.page);
                                }
                            }
                            ++issued;
                        }
                    }
                    ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
                    if (!ok) break;
                    if (++stage == stages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok) break;
        }
        if (lane == 0) {
            if (n_chunks > 0) {
                // The last CTA done taking chunks resets the counters for the
                // next launch (every CTA's last take comes before its count).
                uint32_t* const done = p.status + kChunkDoneWord;
                __threadfence();
                if (atomicAdd(done, 1u) == gridDim.x - 1) {
                    atomicExch(ctr, 0u);
                    atomicExch(done, 0u);
                }
            }
            if (!ok) flag(p.status, kStatusTimeout);
            // Let every copy this CTA issued land before it may exit.
            for (int s = 0; s < stages && s < issued; ++s) {
                const long long times = (issued - 1 - s) / stages + 1;
                if (!mbar_wait(bar_full + 8u * s, (uint32_t)((times - 1) & 1))) {
                    flag(p.status, kStatusTimeout);
                    break;
                }
            }
        }
    } else {

    // -------------------------------------------------------------- consumers
    const int g = lane >> 2, t = lane & 3;
    const int Hq = p.num_qo_heads;
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    int si = seg_begin, cq = 0;
    uint32_t cqphase = 0;
    for (;;) {
        const int* rec;
        if (si < seg_end) {
            rec = segs + 4 * si++;
        } else {
            // The next chunk the producer took (id -1: none left).
            if (n_chunks == 0) break;
            ok = __all_sync(0xFFFFFFFFu, pipe_wait<kDiag>(cq_full + 8u * cq, cqphase, p.wait_cycles));
            if (!ok) break;
            uint32_t c;
            asm volatile("ld.shared.u32 %0, [%1];" : "=r"(c) : "r"(cq_id + 4u * cq) : "memory");
            __syncwarp();
            if (lane == 0) mbar_arrive(cq_empty + 8u * cq);
            if (++cq == kChunkSlots) {
                cq = 0;
                cqphase ^= 1u;
            }
            if ((int)c < 0) break;
            rec = chunk_rec + 4 * (int)c;
        }
        const int row = rec[0], p0 = rec[1], p1 = rec[2];
        const int slot = rec[3];
        const int b = row / nhb, hb = row - b * nhb;
        const int kvh = hb * hpc + warp;
        const int kv_len = req_kv[b];

        if (p0 == p1) {  // a request with no KV: o = 0, lse = -inf
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int n = 2 * t + hh;
                if (n >= group) continue;
                const size_t oh = (size_t)b * Hq + (size_t)kvh * group + n;
                uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.o) + oh * DH + (DH / 8) * g);
#pragma unroll
                for (int i = 0; i < DH / 64; ++i) dst[i] = make_uint4(0, 0, 0, 0);
                if (g == 0 && p.lse != nullptr) p.lse[oh] = -INFINITY;
            }
            continue;
        }

        uint32_t qf[16], qlo[16];
        const size_t q_head_off = ((size_t)b * Hq + (size_t)kvh * group + g) * DH;
        const float qfactor = load_q<kBF, DH>(qf, qlo, p.q, p.q_dtype, q_head_off, g < group, t);
        const bool split_q = kBF && p.q_dtype == PAFP8_F16;
        // log2 softmax scale of heads 2t and 2t+1 (this lane's S columns).
        // Per-query-head scales exist only for an fp8 query, which a 2-byte
        // cache never has: there one scale serves both columns.
        float sc0 = p.sm_scale_log2 * qfactor, sc1 = sc0;
        if (p.k_scales != nullptr) {
            const float ks = __ldg(p.k_scales + kvh);
            if constexpr (k2) {
                sc0 = fold_scale_log2(p.sm_scale, 1.0f, ks) * qfactor;
            } else {
                const int h0 = kvh * group + min(2 * t, group - 1), h1 = kvh * group + min(2 * t + 1, group - 1);
                const float q0 = p.q_scales != nullptr ? __ldg(p.q_scales + h0) : 1.0f;
                const float q1 = p.q_scales != nullptr ? __ldg(p.q_scales + h1) : 1.0f;
                sc0 = fold_scale_log2(p.sm_scale, q0, ks) * qfactor;
                sc1 = fold_scale_log2(p.sm_scale, q1, ks) * qfactor;
            }
        }
        if constexpr (k2) sc1 = sc0;

        float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
        float acc[NA][4];
#pragma unroll
        for (int i = 0; i < NA; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;

        for (int pg = p0; pg < p1; ++pg) {
            // mma.sync and movmatrix below are warp-collective: the warp
            // leaves together if any lane's wait gave up.
            if (!__all_sync(0xFFFFFFFFu, pipe_wait<kDiag>(bar_full + 8u * stage, phase, p.wait_cycles))) {
                ok = false;
                break;
            }
            const uint32_t kt = base + stage * stage_bytes + warp * kTileBytes;
            const uint32_t vt = kt + hpc * kTileBytes;
            // fp8 cache: K rows g and g+8, 16-byte chunks 2t and 2t+1 (swizzled by
            // row & 7 = g), converted pairwise right before each MMA; V rows 2t,
            // 2t+1, 2t+8, 2t+9, chunk g.  2-byte cache: the same dims of the same
            // tokens as 16-bit words (K: dims 32t .. 32t+31 of tokens g and g+8,
            // word w = dims 32t+2w, 32t+2w+1; V: dims 16g .. 16g+15 of the four
            // tokens, word w = dims 16g+2w, 16g+2w+1), so the operand words match
            // the fp8 path's converted words exactly.
            // Head dim 64 takes the same fragments at half the width: K dims
            // 16t .. 16t+15 (one chunk), V dims 8g .. 8g+7, from 64-B fp8 rows
            // under the 64-byte swizzle (16-byte chunk c of row r at c ^ ((r >> 1)
            // & 3)) or from 128-B rows of a 2-byte cache.
            uint4 k0, k1, k2w, k3, v0, v1, v2, v3;
            uint32_t kw0[16], kw8[16], vw[4][8];
            if constexpr (k2 && DH == 64) {
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    const int c = 2 * t + i;
                    const uint4 x = lds128(kt + g * 128 + ((c ^ g) << 4));
                    const uint4 y = lds128(kt + (g + 8) * 128 + ((c ^ g) << 4));
                    kw0[4 * i] = x.x, kw0[4 * i + 1] = x.y, kw0[4 * i + 2] = x.z, kw0[4 * i + 3] = x.w;
                    kw8[4 * i] = y.x, kw8[4 * i + 1] = y.y, kw8[4 * i + 2] = y.z, kw8[4 * i + 3] = y.w;
                }
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    const int tok = 2 * t + (r & 1) + 8 * (r >> 1);
                    const uint4 x = lds128(vt + tok * 128 + ((g ^ (tok & 7)) << 4));
                    vw[r][0] = x.x, vw[r][1] = x.y, vw[r][2] = x.z, vw[r][3] = x.w;
                }
            } else if constexpr (DH == 64) {
                const int sw = (g >> 1) & 3;  // rows g and g+8 share it
                k0 = lds128(kt + g * 64 + ((t ^ sw) << 4));
                k2w = lds128(kt + (g + 8) * 64 + ((t ^ sw) << 4));
                k1 = k3 = make_uint4(0, 0, 0, 0);
                auto vrow = [&](int tok) {
                    const uint2 x = lds64(vt + tok * 64 + ((((g >> 1) ^ ((tok >> 1) & 3))) << 4) + (g & 1) * 8);
                    return make_uint4(x.x, x.y, 0u, 0u);
                };
                v0 = vrow(2 * t);
                v1 = vrow(2 * t + 1);
                v2 = vrow(2 * t + 8);
                v3 = vrow(2 * t + 9);
            } else if constexpr (k2) {
                // A token row is two swizzled 128-B rows (dims 0-63, 64-127):
                // row index 2 * token + half.
                const int rk = (t >> 1) + 2 * g;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int c = 4 * (t & 1) + i;
                    const uint4 x = lds128(kt + rk * 128 + ((c ^ (rk & 7)) << 4));
                    const uint4 y = lds128(kt + (rk + 16) * 128 + ((c ^ (rk & 7)) << 4));
                    kw0[4 * i] = x.x, kw0[4 * i + 1] = x.y, kw0[4 * i + 2] = x.z, kw0[4 * i + 3] = x.w;
                    kw8[4 * i] = y.x, kw8[4 * i + 1] = y.y, kw8[4 * i + 2] = y.z, kw8[4 * i + 3] = y.w;
                }
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    const int rv = (g >> 2) + 2 * (2 * t + (r & 1) + 8 * (r >> 1));
#pragma unroll
                    for (int i = 0; i < 2; ++i) {
                        const int c = 2 * (g & 3) + i;
                        const uint4 x = lds128(vt + rv * 128 + ((c ^ (rv & 7)) << 4));
                        vw[r][4 * i] = x.x, vw[r][4 * i + 1] = x.y, vw[r][4 * i + 2] = x.z, vw[r][4 * i + 3] = x.w;
                    }
                }
            } else {
                k0 = lds128(kt + g * 128 + (((2 * t) ^ g) << 4));
                k1 = lds128(kt + g * 128 + (((2 * t + 1) ^ g) << 4));
                k2w = lds128(kt + (g + 8) * 128 + (((2 * t) ^ g) << 4));
                k3 = lds128(kt + (g + 8) * 128 + (((2 * t + 1) ^ g) << 4));
                v0 = lds128(vt + (2 * t) * 128 + ((g ^ (2 * t)) << 4));
                v1 = lds128(vt + (2 * t + 1) * 128 + ((g ^ (2 * t + 1)) << 4));
                v2 = lds128(vt + (2 * t + 8) * 128 + ((g ^ (2 * t)) << 4));
                v3 = lds128(vt + (2 * t + 9) * 128 + ((g ^ (2 * t + 1)) << 4));
            }
            mbar_arrive(bar_empty + 8u * stage);
            if (++stage == stages) {
                stage = 0;
                phase ^= 1u;
            }

            const int valid = kv_len - pg * P;  // tokens of this page that exist (>= 1)
            if (valid < P) {
                if constexpr (k2) {
#pragma unroll
                    for (int r = 0; r < 4; ++r)
                        if (2 * t + (r & 1) + 8 * (r >> 1) >= valid) {
#pragma unroll
                            for (int w = 0; w < 8; ++w) vw[r][w] = 0u;
                        }
                } else {
                    const uint4 z = make_uint4(0, 0, 0, 0);
                    if (2 * t >= valid) v0 = z;
                    if (2 * t + 1 >= valid) v1 = z;
                    if (2 * t + 8 >= valid) v2 = z;
                    if (2 * t + 9 >= valid) v3 = z;
                }
            }

            // S^T = K . Q^T over 8 k-steps, two accumulators for ILP.
            float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
            if constexpr (k2) {
#pragma unroll
                for (int s = 0; s < NA; ++s) {
                    if (s & 1)
                        mma16816<kBF>(sb, kw0[2 * s], kw8[2 * s], kw0[2 * s + 1], kw8[2 * s + 1], qf[2 * s],
                                      qf[2 * s + 1]);
                    else
                        mma16816<kBF>(sa, kw0[2 * s], kw8[2 * s], kw0[2 * s + 1], kw8[2 * s + 1], qf[2 * s],
                                      qf[2 * s + 1]);
                }
                if (kBF && split_q) {
#pragma unroll
                    for (int s = 0; s < NA; ++s) {
                        if (s & 1)
                            mma16816<kBF>(sb, kw0[2 * s], kw8[2 * s], kw0[2 * s + 1], kw8[2 * s + 1], qlo[2 * s],
                                          qlo[2 * s + 1]);
                        else
                            mma16816<kBF>(sa, kw0[2 * s], kw8[2 * s], kw0[2 * s + 1], kw8[2 * s + 1], qlo[2 * s],
                                          qlo[2 * s + 1]);
                    }
                }
            } else {
                const uint32_t kr0[8] = {k0.x, k0.y, k0.z, k0.w, k1.x, k1.y, k1.z, k1.w};
                const uint32_t kr8[8] = {k2w.x, k2w.y, k2w.z, k2w.w, k3.x, k3.y, k3.z, k3.w};
#pragma unroll
                for (int s = 0; s < NA; ++s) {
                    const uint32_t a0 = fp8x2_lo<KT>(kr0[s]), a1 = fp8x2_lo<KT>(kr8[s]);
                    const uint32_t a2 = fp8x2_hi<KT>(kr0[s]), a3 = fp8x2_hi<KT>(kr8[s]);
                    if (s & 1)
                        mma_16816(sb, a0, a1, a2, a3, qf[2 * s], qf[2 * s + 1]);
                    else
                        mma_16816(sa, a0, a1, a2, a3, qf[2 * s], qf[2 * s + 1]);
                }
            }
            // (tok g | tok g+8) x (head 2t | head 2t+1), log2 units.
            float x0 = (sa[0] + sb[0]) * sc0, x1 = (sa[1] + sb[1]) * sc1;
            float x2 = (sa[2] + sb[2]) * sc0, x3 = (sa[3] + sb[3]) * sc1;
            if (g >= valid) x0 = x1 = -INFINITY;
            if (g + 8 >= valid) x2 = x3 = -INFINITY;
            float mx0 = fmaxf(x0, x2), mx1 = fmaxf(x1, x3);
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xFFFFFFFFu, mx0, off));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xFFFFFFFFu, mx1, off));
            }
            const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
            const float al0 = ex2(m0 - mn0), al1 = ex2(m1 - mn1);
            const float e0 = ex2(x0 - mn0), e1 = ex2(x1 - mn1);
            const float e2 = ex2(x2 - mn0), e3 = ex2(x3 - mn1);
            l0 = l0 * al0 + e0 + e2;
            l1 = l1 * al1 + e1 + e3;
            m0 = mn0;
            m1 = mn1;
#pragma unroll
            for (int i = 0; i < NA; ++i) {
                acc[i][0] *= al0;
                acc[i][1] *= al1;
                acc[i][2] *= al0;
                acc[i][3] *= al1;
            }
            // P^T as the B operand: transpose the two 8x8 (token x head) blocks.
            const uint32_t pb0 = movmatrix_t(kBF ? pack_bf162(e0, e1) : pack_half2(e0, e1));
            const uint32_t pb1 = movmatrix_t(kBF ? pack_bf162(e2, e3) : pack_half2(e2, e3));

            // O^T += V^T . P^T: MMA 2j takes dims 16g+4j (rows g) and 16g+4j+1
            // (rows g+8), MMA 2j+1 the next two; the k columns are the tokens
            // (2t, 2t+1 | 2t+8, 2t+9), each operand word one dim of two tokens.
            if constexpr (k2) {
#pragma unroll
                for (int w = 0; w < NA; ++w)
                    mma16816<kBF>(acc[w], prmt(vw[0][w], vw[1][w], 0x5410u), prmt(vw[0][w], vw[1][w], 0x7632u),
                                  prmt(vw[2][w], vw[3][w], 0x5410u), prmt(vw[2][w], vw[3][w], 0x7632u), pb0, pb1);
            } else {
                const uint32_t va[4] = {v0.x, v0.y, v0.z, v0.w}, vb[4] = {v1.x, v1.y, v1.z, v1.w};
                const uint32_t vc[4] = {v2.x, v2.y, v2.z, v2.w}, vd[4] = {v3.x, v3.y, v3.z, v3.w};
#pragma unroll
                for (int j = 0; j < NA / 2; ++j) {
                    const uint32_t ab_lo = prmt(va[j], vb[j], 0x5140u), ab_hi = prmt(va[j], vb[j], 0x7362u);
                    const uint32_t cd_lo = prmt(vc[j], vd[j], 0x5140u), cd_hi = prmt(vc[j], vd[j], 0x7362u);
                    mma_16816(acc[2 * j], fp8x2_lo<KT>(ab_lo), fp8x2_hi<KT>(ab_lo), fp8x2_lo<KT>(cd_lo),
                              fp8x2_hi<KT>(cd_lo), pb0, pb1);
                    mma_16816(acc[2 * j + 1], fp8x2_lo<KT>(ab_hi), fp8x2_hi<KT>(ab_hi), fp8x2_lo<KT>(cd_hi),
                              fp8x2_hi<KT>(cd_hi), pb0, pb1);
                }
            }
        }
        if (!ok) break;

        // ------------------------------------------------------- epilogue
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            l0 += __shfl_xor_sync(0xFFFFFFFFu, l0, off);
            l1 += __shfl_xor_sync(0xFFFFFFFFu, l1, off);
        }
        // This lane holds dims 16g .. 16g+15 of heads 2t and 2t+1 of the group.
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const int n = 2 * t + hh;
            if (n >= group) continue;
            const float l = hh ? l1 : l0, m = hh ? m1 : m0;
            const float inv = 1.0f / l;
            float vals[2 * NA];  // dims (DH/8)g .. (DH/8)g + DH/8 - 1
#pragma unroll
            for (int i = 0; i < NA; ++i) {
                vals[2 * i] = acc[i][hh] * inv;
                vals[2 * i + 1] = acc[i][2 + hh] * inv;
            }
            const int head = kvh * group + n;
            if (slot < 0) {
                const float vs = p.v_scales != nullptr ? __ldg(p.v_scales + kvh) : p.v_scale;
                uint32_t w[NA];
#pragma unroll
                for (int i = 0; i < NA; ++i) w[i] = pack_out2(vals[2 * i] * vs, vals[2 * i + 1] * vs, p.o_dtype);
                uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.o) +
                                                      ((size_t)b * Hq + head) * DH + (DH / 8) * g);
#pragma unroll
                for (int i = 0; i < NA / 4; ++i) dst[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
                if (g == 0 && p.lse != nullptr)
                    p.lse[(size_t)b * Hq + head] = (m + __log2f(l)) * 0.69314718055994531f;
            } else {
                const int hpb = hpc * group;
                float4* dst = reinterpret_cast<float4*>(
                    p.part_o + ((size_t)slot * hpb + warp * group + n) * DH + (DH / 8) * g);
#pragma unroll
                for (int i = 0; i < NA / 2; ++i)
                    dst[i] = make_float4(vals[4 * i], vals[4 * i + 1], vals[4 * i + 2], vals[4 * i + 3]);
                if (g == 0) p.part_lse[(size_t)slot * hpb + warp * group + n] = m + __log2f(l);
            }
        }
    }
    if (!ok && lane == 0) flag(p.status, kStatusTimeout);
    }  // consumers
}

__global__ void __launch_bounds__(32 * kMergeWarps)
    merge_kernel(const __grid_constant__ DecodeParams p, int hpc, int group) {
    // The metadata (written by the host) is read before the wait.
    const int hpb = hpc * group;
    const int bpr = (hpb + kMergeWarps - 1) / kMergeWarps;  // blocks per merge row
    const int e = blockIdx.x / bpr;
    const int hh = (blockIdx.x - e * bpr) * kMergeWarps + (threadIdx.x >> 5);
    MergePair a{};
    if (hh < hpb) a = merge_pair_args(p, hpc, group, e, hh);
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (hh >= hpb) return;
    merge_pair(p, hpb, a);
}

}  // namespace

// Built-in scratch for callers that cannot allocate device memory (see
// pafp8_run_decode_noalloc).  It stands in for the caller's workspace: the
// plan's metadata, the split-KV partial states and the status word.  Every
// GPU that loads the library holds these bytes until the process exits, and
// every call shares them.
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of g_noalloc_scratch on the current device.  The symbol's
// host-side name is only a stand-in, so the address is looked up once per
// device (with that device current) and cached.
cudaError_t noalloc_scratch(void** ptr) {
    static std::mutex mu;
    static void* addr[kMaxDevices] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (addr[dev] == nullptr) {
        void* a = nullptr;
        e = cudaGetSymbolAddress(&a, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        addr[dev] = a;
    }
    *ptr = addr[dev];
    return cudaSuccess;
}

template <int KT, int DH>
cudaError_t launch_decode_t(const DecodeParams& p, const CUtensorMap& tmap_k, const CUtensorMap& tmap_v,
                            int num_ctas, int hpc, int group, int heads_per_box, cudaStream_t stream) {
    const int stage_bytes = 2 * hpc * tile_bytes(KT, DH);
    int stages = kStageBudget / stage_bytes;
    if (stages > 8) stages = 8;
    if (stages < 2) stages = 2;
    const size_t smem = 1024 + (size_t)stages * stage_bytes + 16 * (size_t)stages + 20 * kChunkSlots;
    const dim3 grid(num_ctas), block(32 * (hpc + 1));
    // The diagnostic instantiation runs only under a shortened wait bound.
    const bool diag = p.wait_cycles < kWaitCyclesDefault;
    // Pages of 16 tokens and of 16 m tokens have an instantiation each; the
    // diagnostic one takes any page size.
    auto kern = diag ? decode_kernel<KT, DH, true, true>
                     : (p.page_mult != 1 ? decode_kernel<KT, DH, false, true> : decode_kernel<KT, DH, false, false>);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<grid, block, smem, stream>>>(p, tmap_k, tmap_v, hpc, group, stages, heads_per_box);
    return cudaGetLastError();
}

template <int KT>
cudaError_t launch_decode_kt(const DecodeParams& p, const CUtensorMap& tmap_k, const CUtensorMap& tmap_v,
                             int num_ctas, int hpc, int group, int heads_per_box, cudaStream_t stream) {
    if (p.head_dim == 64)
        return launch_decode_t<KT, 64>(p, tmap_k, tmap_v, num_ctas, hpc, group, heads_per_box, stream);
    return launch_decode_t<KT, 128>(p, tmap_k, tmap_v, num_ctas, hpc, group, heads_per_box, stream);
}

cudaError_t launch_decode(const DecodeParams& p, const CUtensorMap& tmap_k, const CUtensorMap& tmap_v,
                          int num_ctas, int hpc, int group, int heads_per_box, cudaStream_t stream) {
    switch (p.kv_dtype) {
        case PAFP8_E4M3FN:
            return launch_decode_kt<PAFP8_E4M3FN>(p, tmap_k, tmap_v, num_ctas, hpc, group, heads_per_box, stream);
        case PAFP8_E5M2:
            return launch_decode_kt<PAFP8_E5M2>(p, tmap_k, tmap_v, num_ctas, hpc, group, heads_per_box, stream);
        case PAFP8_F16:
            return launch_decode_kt<PAFP8_F16>(p, tmap_k, tmap_v, num_ctas, hpc, group, heads_per_box, stream);
        case PAFP8_BF16:
            return launch_decode_kt<PAFP8_BF16>(p, tmap_k, tmap_v, num_ctas, hpc, group, heads_per_box, stream);
        default:
            return cudaErrorInvalidValue;
    }
}

cudaError_t launch_merge(const DecodeParams& p, int num_merge, int hpc, int group, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(num_merge * ((hpc * group + kMergeWarps - 1) / kMergeWarps));
    cfg.blockDim = dim3(32 * kMergeWarps);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, merge_kernel, p, hpc, group);
}

}  // namespace pafp8
