// ptx.cuh -- inline-PTX building blocks shared by the sm_103a kernels:
// mbarriers with bounded waits, TMA tile loads, fp8 -> f16 register
// conversion, warp-level MMA, and the tcgen05 (tensor memory) instructions.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "../../include/pafp8.h"
#include "internal.h"

namespace pafp8 {
namespace ptx {

// Bound of every wait, in SM clock cycles (~1 s at 2 GHz).  The diagnostic
// instantiations of the kernels (PAFP8_WAIT_CYCLES set) bound their pipeline
// waits by the shorter value the host passes instead; a CTA's final waits for
// its own copies and MMAs in flight always take this one, since those
// complete whatever the other roles did.
constexpr long long kWaitCycles = kWaitCyclesDefault;

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

// ---------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_init_fence() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Non-blocking test of the phase of `parity`.
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Poll without suspending; false after `limit` cycles.  Used by the kernels'
// diagnostic instantiations (a shortened bound): try_wait may suspend the
// thread until the phase completes, which would outlast a short bound.
__device__ __forceinline__ bool mbar_poll(uint32_t bar, uint32_t parity, long long limit) {
    const long long t0 = clock64();
    while (!mbar_test_wait(bar, parity))
        if (clock64() - t0 > limit) return false;
    return true;
}

// Wait for the phase of `parity` to complete; false after ~kWaitCycles.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity))
        if (clock64() - t0 > kWaitCycles) return false;
    return true;
}

// A pipeline wait: mbar_wait, or in a diagnostic instantiation (kDiag) a
// poll bounded by `limit`.  The production instantiations compile to exactly
// mbar_wait: the kernels are sensitive to every instruction of their waits.
template <bool kDiag>
__device__ __forceinline__ bool pipe_wait(uint32_t bar, uint32_t parity, long long limit) {
    if constexpr (kDiag) return mbar_poll(bar, parity, limit);
    return mbar_wait(bar, parity);
}

// Generic-proxy shared-memory writes become visible to the async proxy
// (TMA, tensor core) after this fence.
__device__ __forceinline__ void fence_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// --------------------------------------------------------------------- TMA

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int c0, int c1, int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int c0, int c1, int c2, int c3) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void tma_load_5d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int c0, int c1, int c2, int c3, int c4) {
    asm volatile(
        "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4), "r"(bar)
        : "memory");
}

// Bulk tensor store shared -> global (one box), tracked by this thread's bulk
// groups: commit closes a group; wait_group.read 0 returns once every group's
// shared-memory reads are done, wait_group 0 once its writes are complete.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, uint32_t src, int c0, int c1, int c2) {
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];"
                 ::"l"(reinterpret_cast<uint64_t>(map)), "r"(src), "r"(c0), "r"(c1), "r"(c2)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read_all() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Eight words to global memory in one 32-byte access (address 32-byte aligned).
__device__ __forceinline__ void stg256(void* addr, const uint32_t* w) {
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(addr), "r"(w[0]), "r"(w[1]),
                 "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
                 : "memory");
}

// ------------------------------------------------------------ shared memory

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

__device__ __forceinline__ uint2 lds64(uint32_t addr) {
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ void sts32(uint32_t addr, uint32_t a) {
    asm volatile("st.shared.b32 [%0], %1;" ::"r"(addr), "r"(a) : "memory");
}

__device__ __forceinline__ void sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
                 : "memory");
}

// ------------------------------------------------------- fp8 -> f16 (exact)

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t r;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
    return r;
}

// Two fp8 codes (bytes 0,1 or 2,3 of w) -> f16x2 with the same values.
// e4m3fn uses the hardware conversion; an e5m2 code is the high byte of the
// f16 of equal value (same exponent width and bias, two mantissa bits).
template <int KT>
__device__ __forceinline__ uint32_t fp8x2_lo(uint32_t w);
template <int KT>
__device__ __forceinline__ uint32_t fp8x2_hi(uint32_t w);

template <>
__device__ __forceinline__ uint32_t fp8x2_lo<PAFP8_E4M3FN>(uint32_t w) {
    uint32_t r;
    asm("{\n .reg .b16 l, h;\n mov.b32 {l, h}, %1;\n cvt.rn.f16x2.e4m3x2 %0, l;\n}\n"
        : "=r"(r)
        : "r"(w));
    return r;
}
template <>
__device__ __forceinline__ uint32_t fp8x2_hi<PAFP8_E4M3FN>(uint32_t w) {
    uint32_t r;
    asm("{\n .reg .b16 l, h;\n mov.b32 {l, h}, %1;\n cvt.rn.f16x2.e4m3x2 %0, h;\n}\n"
        : "=r"(r)
        : "r"(w));
    return r;
}
template <>
__device__ __forceinline__ uint32_t fp8x2_lo<PAFP8_E5M2>(uint32_t w) {
    return prmt(w, 0u, 0x1404u);
}
template <>
__device__ __forceinline__ uint32_t fp8x2_hi<PAFP8_E5M2>(uint32_t w) {
    return prmt(w, 0u, 0x3424u);
}

// ------------------------------------------------------------- arithmetic

__device__ __forceinline__ float ex2(float x) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

// Three-input maximum (one instruction on sm_100 and later).
__device__ __forceinline__ float max3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// Packed pairs of fp32 (sm_100 and later): one instruction for two lanes of
// work.  A pair is held as .b64 with element 0 in the low word.
struct f32x2 {
    uint64_t v;
};
__device__ __forceinline__ f32x2 make_f32x2(float lo, float hi) {
    f32x2 r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r.v) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void split_f32x2(f32x2 a, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(a.v));
}
__device__ __forceinline__ f32x2 fma2(f32x2 a, f32x2 b, f32x2 c) {
    f32x2 r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r.v) : "l"(a.v), "l"(b.v), "l"(c.v));
    return r;
}
__device__ __forceinline__ f32x2 add2(f32x2 a, f32x2 b) {
    f32x2 r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r.v) : "l"(a.v), "l"(b.v));
    return r;
}
__device__ __forceinline__ f32x2 mul2(f32x2 a, f32x2 b) {
    f32x2 r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r.v) : "l"(a.v), "l"(b.v));
    return r;
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ uint32_t pack_out2(float lo, float hi, int o_dtype) {
    if (o_dtype == PAFP8_BF16) {
        __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&h);
    }
    return pack_half2(lo, hi);
}

// ------------------------------------------------------ warp-level MMA (decode)

__device__ __forceinline__ void mma_16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7},"
        " {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// The same MMA with bf16 A and B (both operands must share the type).
__device__ __forceinline__ void mma_16816_bf16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                               uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7},"
        " {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf162(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
    uint32_t r;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(r) : "r"(x));
    return r;
}

// ------------------------------------------------------------- tcgen05

// Shared-memory matrix descriptor, K-major, 128-byte swizzle: rows of 128
// bytes, 8-row atoms 1024 bytes apart (stride byte offset), descriptor
// version 1, layout type 2 (SWIZZLE_128B).  The leading byte offset is unused
// for this layout and set to 1 (16 bytes).
__device__ __forceinline__ uint64_t sw128_kmajor_desc(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)1 << 16;            // leading byte offset (unused), 16 B
    d |= (uint64_t)(1024 >> 4) << 32;  // stride byte offset: 8 rows x 128 B
    d |= (uint64_t)1 << 46;            // descriptor version
    d |= (uint64_t)2 << 61;            // SWIZZLE_128B
    return d;
}

// The same for 64-byte rows under the 64-byte swizzle (an fp8 row of 64
// elements): 8-row atoms of 512 bytes, layout type 4 (SWIZZLE_64B).
__device__ __forceinline__ uint64_t sw64_kmajor_desc(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)1 << 16;            // leading byte offset (unused), 16 B
    d |= (uint64_t)(512 >> 4) << 32;   // stride byte offset: 8 rows x 64 B
    d |= (uint64_t)1 << 46;            // descriptor version
    d |= (uint64_t)4 << 61;            // SWIZZLE_64B
    return d;
}

// An MN-major operand under the 128-byte swizzle: 128-byte rows of 64 2-byte
// elements along M or N, one row per K index, 8-row atoms 1024 bytes apart
// along K (stride byte offset); `lbo` bytes between the 64-element column
// blocks along M or N (leading byte offset).  This is the layout a TMA box of
// [K rows][64 elements] lands in, so a tile stored K-index-major (keys x dims)
// serves as the B operand of O = P V without a transpose.
__device__ __forceinline__ uint64_t sw128_mnmajor_desc(uint32_t saddr, uint32_t lbo) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;  // leading byte offset: next 64 columns
    d |= (uint64_t)(1024 >> 4) << 32;              // stride byte offset: next 8 K rows
    d |= (uint64_t)1 << 46;                        // descriptor version
    d |= (uint64_t)2 << 61;                        // SWIZZLE_128B
    return d;
}

// Instruction descriptor: f32 accumulator, K-major A and B, M x N.
// a_fmt/b_fmt: kind::f16 -> 0 f16, 1 bf16; kind::f8f6f4 -> 0 e4m3, 1 e5m2.
__host__ __device__ constexpr uint32_t make_idesc(int a_fmt, int b_fmt, int m, int n) {
    return (1u << 4) | ((uint32_t)a_fmt << 7) | ((uint32_t)b_fmt << 10) |
           ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}
// The same with an MN-major B operand (bit 16: B transposed).
__host__ __device__ constexpr uint32_t make_idesc_bmn(int a_fmt, int b_fmt, int m, int n) {
    return make_idesc(a_fmt, b_fmt, m, n) | (1u << 16);
}

// One product's K steps from a single asm statement: the descriptors'
// start offsets (16-byte units) are immediate operands, the first MMA
// accumulates into D when `accum` is nonzero and the others always, so an MMA
// costs two 64-bit adds besides itself (instead of also widening a register
// offset and setting its own predicate).  kind::f16 A and B in shared memory
// with K = 8 x 16 over two 128-byte halves (ha, hb: bytes between a
// descriptor's first and second half), kind::f16 with K = 4 x 16 in one half,
// kind::f8f6f4 with K = 4 x 32 or 2 x 32, and kind::f16 with A in TMEM (8
// columns per K step of 16 2-byte elements) and an MN-major B.
#define PAFP8_K8_SS_BODY(CG)                                                                          \
    "{\n .reg .pred p, t;\n .reg .b64 da, db;\n setp.ne.b32 p, %4, 0;\n setp.eq.b32 t, %4, %4;\n"     \
    " tcgen05.mma.cta_group::" CG ".kind::f16 [%0], %1, %2, %3, p;\n"                                \
    " add.s64 da, %1, 2;\n add.s64 db, %2, 2;\n tcgen05.mma.cta_group::" CG ".kind::f16 [%0], da, db, %3, t;\n" \
    " add.s64 da, %1, 4;\n add.s64 db, %2, 4;\n tcgen05.mma.cta_group::" CG ".kind::f16 [%0], da, db, %3, t;\n" \
    " add.s64 da, %1, 6;\n add.s64 db, %2, 6;\n tcgen05.mma.cta_group::" CG ".kind::f16 [%0], da, db, %3, t;\n" \
    " add.s64 da, %1, %5;\n add.s64 db, %2, %6;\n tcgen05.mma.cta_group::" CG ".kind::f16 [%0], da, db, %3, t;\n" \
    " add.s64 da, %1, %7;\n add.s64 db, %2, %8;\n tcgen05.mma.cta_group::" CG ".kind::f16 [%0], da, db, %3, t;\n" \
    " add.s64 da, %1, %9;\n add.s64 db, %2, %10;\n tcgen05.mma.cta_group::" CG ".kind::f16 [%0], da, db, %3, t;\n" \
    " add.s64 da, %1, %11;\n add.s64 db, %2, %12;\n tcgen05.mma.cta_group::" CG ".kind::f16 [%0], da, db, %3, t;\n}\n"
#define PAFP8_K8_SS_ARGS(HA, HB)                                                                       \
    "r"(d_tmem), "l"(a), "l"(b), "r"(idesc), "r"(accum), "n"((HA) >> 4), "n"((HB) >> 4), "n"(((HA) >> 4) + 2), \
        "n"(((HB) >> 4) + 2), "n"(((HA) >> 4) + 4), "n"(((HB) >> 4) + 4), "n"(((HA) >> 4) + 6), "n"(((HB) >> 4) + 6)
// The MN-major B (sw128_mnmajor_desc) of kind::f16 with A in TMEM: a K step
// of 16 is 16 rows of 128 bytes, 2048 bytes on.
#define PAFP8_K8_TS_MN_BODY(CG)                                                                       \
    "{\n .reg .pred p, t;\n .reg .b64 db;\n .reg .b32 ta;\n setp.ne.b32 p, %4, 0;\n setp.eq.b32 t, %4, %4;\n" \
    " tcgen05.mma.cta_group::" CG ".kind::f16 [%0], [%1], %2, %3, p;\n"                              \
    " add.u32 ta, %1, 8;\n add.s64 db, %2, 128;\n tcgen05.mma.cta_group::" CG ".kind::f16 [%0], [ta], db, %3, t;\n" \
    " add.u32 ta, %1, 16;\n add.s64 db, %2, 256;\n tcgen05.mma.cta_group::" CG ".kind::f16 [%0], [ta], db, %3, t;\n" \
    " add.u32 ta, %1, 24;\n add.s64 db, %2, 384;\n tcgen05.mma.cta_group::" CG ".kind::f16 [%0], [ta], db, %3, t;\n" \
    " add.u32 ta, %1, 32;\n add.s64 db, %2, 512;\n tcgen05.mma.cta_group::" CG ".kind::f16 [%0], [ta], db, %3, t;\n" \
    " add.u32 ta, %1, 40;\n add.s64 db, %2, 640;\n tcgen05.mma.cta_group::" CG ".kind::f16 [%0], [ta], db, %3, t;\n" \
    " add.u32 ta, %1, 48;\n add.s64 db, %2, 768;\n tcgen05.mma.cta_group::" CG ".kind::f16 [%0], [ta], db, %3, t;\n" \
    " add.u32 ta, %1, 56;\n add.s64 db, %2, 896;\n tcgen05.mma.cta_group::" CG ".kind::f16 [%0], [ta], db, %3, t;\n}\n"

template <uint32_t HA, uint32_t HB>
__device__ __forceinline__ void tc_mma_f16_ss_k8(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                                 uint32_t accum) {
    asm volatile(PAFP8_K8_SS_BODY("1")::PAFP8_K8_SS_ARGS(HA, HB) : "memory");
}
template <uint32_t HA, uint32_t HB>
__device__ __forceinline__ void tc_mma_pair_f16_ss_k8(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                                      uint32_t accum) {
    asm volatile(PAFP8_K8_SS_BODY("2")::PAFP8_K8_SS_ARGS(HA, HB) : "memory");
}
__device__ __forceinline__ void tc_mma_f16_ts_mn_k8(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                                    uint32_t accum) {
    asm volatile(PAFP8_K8_TS_MN_BODY("1")::"r"(d_tmem), "r"(a_tmem), "l"(b), "r"(idesc), "r"(accum) : "memory");
}
__device__ __forceinline__ void tc_mma_pair_f16_ts_mn_k8(uint32_t d_tmem, uint32_t a_tmem, uint64_t b,
                                                         uint32_t idesc, uint32_t accum) {
    asm volatile(PAFP8_K8_TS_MN_BODY("2")::"r"(d_tmem), "r"(a_tmem), "l"(b), "r"(idesc), "r"(accum) : "memory");
}
__device__ __forceinline__ void tc_mma_f16_ss_k4(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                                 uint32_t accum) {
    asm volatile(
        "{\n .reg .pred p, t;\n .reg .b64 da, db;\n setp.ne.b32 p, %4, 0;\n setp.eq.b32 t, %4, %4;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n"
        " add.s64 da, %1, 2;\n add.s64 db, %2, 2;\n tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %3, t;\n"
        " add.s64 da, %1, 4;\n add.s64 db, %2, 4;\n tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %3, t;\n"
        " add.s64 da, %1, 6;\n add.s64 db, %2, 6;\n tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %3, t;\n}\n"
        ::"r"(d_tmem), "l"(a), "l"(b), "r"(idesc), "r"(accum)
        : "memory");
}
__device__ __forceinline__ void tc_mma_f8_ss_k4(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                                uint32_t accum) {
    asm volatile(
        "{\n .reg .pred p, t;\n .reg .b64 da, db;\n setp.ne.b32 p, %4, 0;\n setp.eq.b32 t, %4, %4;\n"
        " tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n"
        " add.s64 da, %1, 2;\n add.s64 db, %2, 2;\n tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], da, db, %3, t;\n"
        " add.s64 da, %1, 4;\n add.s64 db, %2, 4;\n tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], da, db, %3, t;\n"
        " add.s64 da, %1, 6;\n add.s64 db, %2, 6;\n tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], da, db, %3, t;\n}\n"
        ::"r"(d_tmem), "l"(a), "l"(b), "r"(idesc), "r"(accum)
        : "memory");
}
__device__ __forceinline__ void tc_mma_f8_ss_k2(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                                uint32_t accum) {
    asm volatile(
        "{\n .reg .pred p, t;\n .reg .b64 da, db;\n setp.ne.b32 p, %4, 0;\n setp.eq.b32 t, %4, %4;\n"
        " tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n"
        " add.s64 da, %1, 2;\n add.s64 db, %2, 2;\n tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], da, db, %3, t;\n}\n"
        ::"r"(d_tmem), "l"(a), "l"(b), "r"(idesc), "r"(accum)
        : "memory");
}
#undef PAFP8_K8_SS_BODY
#undef PAFP8_K8_SS_ARGS
#undef PAFP8_K8_TS_MN_BODY

// Arrive (count 1) on `bar` when every tcgen05 operation this thread issued
// before has completed.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Warp-wide: allocate `ncols` TMEM columns, address written to smem `dst`.
__device__ __forceinline__ void tc_alloc(uint32_t dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tc_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

// ------------------------------------------------- CTA pairs (2-SM MMA)
// A cluster of two CTAs on two SMs runs one MMA stream: the leader (rank 0)
// issues tcgen05.mma.cta_group::2 with M = 256, each CTA holding its 128 rows
// of A (and of D in its TMEM) and half of B's N rows at the same shared-memory
// offset.  Every tcgen05 MMA, commit, alloc and dealloc of such a kernel uses
// .cta_group::2.

// Every thread of both CTAs.
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// The shared::cluster address of `addr` (a shared::cta offset) in CTA `rank`.
__device__ __forceinline__ uint32_t map_shared(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}
// Arrive on an mbarrier of either CTA of the cluster (shared::cluster address).
// The release is at CTA scope: what an arrival in these kernels orders is the
// arriving CTA's own shared memory and TMEM against the tensor cores' reads of
// them (already ordered by fence.proxy.async and the tcgen05 fences before the
// arrive), never data that the other CTA's threads load.  A cluster-scope
// release made the arriving thread wait about half a microsecond per arrive.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cbar) {
    asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cbar) : "memory");
}
// One arrival for the whole warp (all 32 lanes call it): the warp barrier
// orders every lane's earlier work before lane 0's arrive.  Cross-SM arrives
// are transactions between SMs, so a warp sends one instead of 32.
__device__ __forceinline__ void warp_arrive_cluster(uint32_t cbar) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive_cluster(cbar);
}
__device__ __forceinline__ void warp_arrive(uint32_t bar) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
}
// try_wait acquiring at cluster scope (for arrivals from the peer CTA).
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ bool mbar_test_wait_cluster(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.test_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
// Warp-wide in each CTA of the pair: allocate `ncols` TMEM columns (the same
// address in both), written to smem `dst`; then give up further allocation.
__device__ __forceinline__ void tc_alloc_pair(uint32_t dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst), "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tc_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
// Arrive (count 1) on the mbarrier at offset `bar` in each CTA of `mask` when
// every pair MMA this thread issued before has completed.
__device__ __forceinline__ void tc_commit_pair(uint32_t bar, uint16_t mask) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(bar),
        "h"(mask)
        : "memory");
}
// TMA loads into this CTA's shared memory whose completion (bytes) is counted
// on the mbarrier `cbar` (a shared::cluster address, here the leader's).
__device__ __forceinline__ void tma_load_3d_pair(uint32_t dst, const CUtensorMap* map, uint32_t cbar, int c0, int c1,
                                                 int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(cbar)
        : "memory");
}
__device__ __forceinline__ void tma_load_5d_pair(uint32_t dst, const CUtensorMap* map, uint32_t cbar, int c0, int c1,
                                                 int c2, int c3, int c4) {
    asm volatile(
        "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2"
        " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4), "r"(cbar)
        : "memory");
}

// 32 lanes x 32 consecutive 32-bit columns: thread i gets lane (base + i).
__device__ __forceinline__ void tc_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11,"
        " %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29,"
        " %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]),
          "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]),
          "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
}

__device__ __forceinline__ void tc_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10,"
        " %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}

__device__ __forceinline__ void tc_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10,"
        " %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28,"
        " %29, %30, %31, %32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]),
        "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]),
        "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]),
        "r"(r[30]), "r"(r[31])
        : "memory");
}

__device__ __forceinline__ void tc_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tc_wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

}  // namespace ptx
}  // namespace pafp8
