// prefill.cuh -- ragged causal prefill attention over a paged fp8 KV cache on
// the tcgen05 tensor cores (sm_103a).  Included by one translation unit per
// head size (prefill_d128.cu, prefill_d64.cu), which compile in parallel.
//
// What it computes: for request b with qo_len new query rows and kv_len keys,
// query row i (0-based among the new rows) of head h attends to keys
// j <= i + kv_len - qo_len (bottom-right aligned causal mask) of KV head
// h / group: o = v_scale * softmax(sm_scale * q_scale * k_scale * q.k) V,
// lse = ln sum exp(logits).  KV stays fp8 in HBM and is dequantized on load
// ("fp8 KV cache in the in-tree prefill kernel", Kernel note: KV is widened
// into a 2-byte shared-memory tile in the global -> shared path); with an fp8
// query the QK product runs natively in fp8 ("Enable Hopper FA3 FP8 attention
// in decode.py", review note on q_scale folding into sm_scale for FP8 BMM1).
//
// Work item: one KV head of one request and two query tiles A and B of 128
// rows each, packed as (token, head-of-group) pairs -- 128/group consecutive
// new tokens times the group's query heads per tile, B right after A -- so a
// dequantized K/V tile serves 256 query rows.  KV tiles are 128 keys (8
// pages).  Persistent CTAs take items from a longest-first list built by the
// plan, dealt in snake order (item_at).
//
// Roles (512 threads, four warpgroups; registers are moved by setmaxnreg from
// the dequant warpgroup (64) and the producer/MMA warpgroup (64) to the two
// softmax warpgroups (192), which hold a whole S row without spilling):
//   warps 0-3   dequant: raw fp8 K -> f16 K tile (2-byte query path); raw fp8
//               V -> f16 V tile (both paths; a 2-byte V tile is copied), in
//               the layout a 2-byte tile lands in ([64-dim half][key][128 B]),
//               zero beyond the request's keys;
//   warps 4-7   softmax of tile A, warps 8-11 softmax of tile B: thread r owns
//               TMEM lane r = query row r of its tile.  Reads S, masks, keeps
//               the running max and sum, writes P (f16) over the first half of
//               S in TMEM, rescales O in TMEM only when the max rises by more
//               than 2^8, and in the epilogue normalizes O and stores o, lse.
//               With a bf16 query on an fp8 cache each thread brings its Q
//               row into f16 range by an exact power of two and converts it in
//               place, for the next item as soon as its last pass of the
//               current one is done (before that item's epilogue);
//   warp 12     TMA producer: both Q tiles, K and V pages (one box per page);
//   warp 13     MMA issuer and TMEM owner (warps 14-15 idle).  Per KV tile j:
//                 S_A = Q_A K_j^T, S_B = Q_B K_j^T    (kind::f16 or kind::f8f6f4)
//                 O_A += P_A V_j,  O_B += P_B V_j      (kind::f16, A = P from TMEM)
//               issued as ... PV_A(j), QK_A(j+1), PV_B(j), QK_B(j+1) ... so
//               each tile's softmax overlaps the other tile's tensor work.
// TMEM columns: S_A/P_A 0-127, S_B/P_B 128-255, O_A 256-383, O_B 384-511.
// O_X is released by its softmax warps after each epilogue they run; the
// MMA warp waits for that release only before the first O_X write of the
// next item in which tile X has rows (so an empty tile B never advances the
// barrier ahead of the wait).
// The tensor pipe runs one CTA's MMAs in order, so an MMA writing S_X after
// O_X += P_X V has been issued cannot overtake it, and s_full(X, j) implies
// that the previous O update of X is complete.  Q and K in shared memory are
// K-major operands with the 128-byte swizzle (64-byte for the 64-byte fp8 rows
// of head_dim 64); V is the MN-major B operand of P V (dims along 128-byte
// rows, one row per key), so no role transposes it.  All waits are bounded; on
// expiry the kernel records a status bit and winds down.
//
// Pages of 16 m tokens (m > 1) are read as m sub-pages of 16: the TMA box of
// sub-page j is at token slot 16 j of its page, which covers both layouts.
// That path (kSlots) is its own instantiation so that the 16-token path keeps
// a producer loop without the division by m.
#pragma once
#include "../../include/pafp8.h"
#include "internal.h"
#include "ptx.cuh"

namespace pafp8 {
namespace {

using namespace ptx;

constexpr int kThreads = 512;  // four warpgroups; warps 14-15 only lend registers
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kHalfTile = kTileKeys * 128;  // 16 KB: 128 rows x 128 B
__device__ __forceinline__ uint32_t col_s(int x) { return 128u * (uint32_t)x; }  // S_X / P_X

// Sizes that depend on the head size DH (128 or 64).  A 2-byte row of DH
// elements is DH / 64 rows of 128 B ("halves", each under the 128-byte
// swizzle); an fp8 row is DH bytes (128-byte swizzle for 128, 64-byte for 64).
template <int DH>
struct Dims {
    static constexpr int NH = DH / 64;                       // 128-B halves of a 2-byte row
    static constexpr uint32_t kRawTile = kTileKeys * DH;      // fp8 K or V tile (128 keys)
    static constexpr uint32_t kRawPage = kPageSize * DH;      // fp8 page box (16 tokens)
    static constexpr uint32_t kF16Tile = NH * kHalfTile;      // 2-byte K or V tile (128 keys) or Q tile
};
template <int DH>
__device__ __forceinline__ uint32_t col_o(int x) { return 256u + (uint32_t)DH * (uint32_t)x; }  // O_X

template <bool kF8, bool k2, int DH>
struct Layout {
    using Dm = Dims<DH>;
    // The 2-byte-query path spends its shared memory on two f16 K tiles (the
    // dequant of K_{j+1} may start while QK_B(j) still reads K_j) and keeps a
    // single raw fp8 stage per tensor; the fp8 path multiplies raw K directly.
    // A 2-byte cache (k2) brings K straight into the 16-bit K tiles and only
    // copies V (zeroing the keys past the request's end), so it has no raw K
    // stage and a 2-byte raw V stage.
    static constexpr int NKR = kF8 ? 4 : (k2 ? 0 : 1);  // raw K stages
    static constexpr int NVR = kF8 ? 2 : 1;             // raw V stages
    static constexpr uint32_t kRawV = k2 ? Dm::kF16Tile : Dm::kRawTile;
    static constexpr int NK16 = kF8 ? 0 : 2;   // f16 K stages
    static constexpr int NV16 = 2;             // f16 V stages
    static constexpr uint32_t kQTile = kF8 ? kTileRows * DH : Dm::kF16Tile;
    static constexpr uint32_t q = 0;                     // Q_A, then Q_B
    static constexpr uint32_t kr = 2 * kQTile;
    static constexpr uint32_t vr = kr + NKR * Dm::kRawTile;
    static constexpr uint32_t k16 = vr + NVR * kRawV;
    static constexpr uint32_t v16 = k16 + NK16 * Dm::kF16Tile;
    // fp8 query: a 16 KB staging half per query tile for the output's bulk
    // tensor stores (64 dims of 128 rows, 128-byte rows swizzled).
    static constexpr uint32_t ostage = v16 + NV16 * Dm::kF16Tile;
    static constexpr uint32_t bars = ostage + (kF8 ? 2 * kHalfTile : 0);
    // barrier indices (8 bytes each)
    static constexpr int bQFull = 0, bQReady = 1, bQEmpty = 2;
    static constexpr int bKrFull = 3, bKrEmpty = bKrFull + NKR;
    static constexpr int bVrFull = bKrEmpty + NKR, bVrEmpty = bVrFull + NVR;
    static constexpr int bK16Full = bVrEmpty + NVR, bK16Empty = bK16Full + NK16;
    static constexpr int bV16Full = bK16Empty + NK16, bV16Empty = bV16Full + NV16;
    static constexpr int bSFull = bV16Empty + NV16;  // [2]
    static constexpr int bPFull = bSFull + 2;        // [2]
    static constexpr int bOFull = bPFull + 2;        // [2]
    static constexpr int bOEmpty = bOFull + 2;       // [2]
    static constexpr int bStageFree = bOEmpty + 2;    // [2]
    static constexpr int bStageReady = bStageFree + 2;  // [2]
    static constexpr int bDrain = bStageReady + 2;
    static constexpr int nBars = bDrain + 1;
    static constexpr uint32_t tmem_slot = bars + 8 * nBars;
    static constexpr uint32_t abort_flag = tmem_slot + 4;
    static constexpr uint32_t bytes = abort_flag + 4;
};
static_assert(1024 + Layout<false, false, 128>::bytes <= 232448, "shared memory budget (2-byte query)");
static_assert(1024 + Layout<true, false, 128>::bytes <= 232448, "shared memory budget (fp8 query)");
static_assert(1024 + Layout<false, true, 128>::bytes <= 232448, "shared memory budget (2-byte cache)");
static_assert(1024 + Layout<false, false, 64>::bytes <= 232448, "shared memory budget (2-byte query, D 64)");
static_assert(1024 + Layout<true, false, 64>::bytes <= 232448, "shared memory budget (fp8 query, D 64)");
static_assert(1024 + Layout<false, true, 64>::bytes <= 232448, "shared memory budget (2-byte cache, D 64)");
// Swizzled tiles start on 1024-byte boundaries (the 128-byte swizzle's atom).
static_assert(Layout<true, false, 64>::kr % 1024 == 0 && Layout<true, false, 64>::v16 % 1024 == 0 &&
                  Layout<false, false, 64>::v16 % 1024 == 0 && Layout<false, true, 64>::v16 % 1024 == 0,
              "1024-byte alignment of the D 64 tiles");

struct Ring {
    int idx = 0;
    uint32_t phase = 0;
    __device__ __forceinline__ void next(int n) {
        if (++idx == n) {
            idx = 0;
            phase ^= 1u;
        }
    }
};

struct Item {
    int b, hk, t0, nkv;          // nkv: KV tiles of the item (tile B's, or A's if B is empty)
    int qo0, qo_len, kv_len, page0;  // the request's first query row, rows, keys, first page entry
};

// One plan record per item, with the request fields the kernel needs, so an
// item start costs one round of independent loads.
__device__ __forceinline__ Item load_item(const int* items, int t) {
    const int* r = items + 8 * t;
    return Item{__ldg(r), __ldg(r + 1), __ldg(r + 2), __ldg(r + 3), __ldg(r + 4), __ldg(r + 5), __ldg(r + 6), __ldg(r + 7)};
}

// KV tiles that query tile `x` (0 = A, 1 = B) of an item needs: its last
// token's causal limit, capped by the request's own key tiles; 0 if the tile
// has no rows.
__device__ __forceinline__ int tile_nkv(int t0, int x, int TQ, int qo_len, int kv_len) {
    const int first = t0 + x * TQ;
    if (first >= qo_len) return 0;
    const int last = min(first + TQ, qo_len) - 1;
    const int lim = last + kv_len - qo_len;
    return min((kv_len + kTileKeys - 1) / kTileKeys, lim / kTileKeys + 1);
}

// The item that persistent worker i of G takes in round r.  Items are sorted
// longest first; even rounds deal them to workers 0 .. G-1, odd rounds back
// from G-1 to 0 (a snake), so each worker's total evens out while the items
// in flight at any time are the same neighbours as in plain round robin.  A
// worker stops at its first round whose item is past the list (no later
// round has one for it).
__device__ __forceinline__ int item_at(int r, int i, int G) { return r * G + ((r & 1) ? G - 1 - i : i); }

__device__ __forceinline__ void set_abort(uint32_t flag_addr, uint32_t* status) {
    asm volatile("st.shared.u32 [%0], 1;" ::"r"(flag_addr) : "memory");
    atomicOr(status, kStatusTimeout);
}

__device__ __forceinline__ bool aborted(uint32_t flag_addr) {
    uint32_t v;
    asm volatile("ld.volatile.shared.u32 %0, [%1];" : "=r"(v) : "r"(flag_addr) : "memory");
    return v != 0;
}

// Bounded wait that also gives up once another role has aborted.  A
// diagnostic instantiation (kDiag) polls with the host's shortened bound.
template <bool kDiag>
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity, uint32_t flag_addr,
                                              uint32_t* status, long long limit) {
    if constexpr (kDiag) {
        if (mbar_poll(bar, parity, limit)) return true;
        set_abort(flag_addr, status);
        return false;
    }
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (aborted(flag_addr)) return false;
        if (clock64() - t0 > kWaitCycles) {
            set_abort(flag_addr, status);
            return false;
        }
    }
    return true;
}

template <bool kF8, int KT, bool kDiag, int DH, bool kSlots>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ PrefillParams p, const __grid_constant__ CUtensorMap tmq,
                   const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                   const __grid_constant__ CUtensorMap tmo) {
    constexpr bool k2 = KT == PAFP8_F16 || KT == PAFP8_BF16;  // 2-byte cache, same dtype as q
    constexpr bool kBF = KT == PAFP8_BF16;                    // bf16 MMA operands
    // A bf16 query on an fp8 cache is brought into f16 range (per row, by the
    // softmax warps) before the QK MMAs; every other path multiplies Q as loaded.
    const bool fit_q = !kF8 && !k2 && p.q_dtype == PAFP8_BF16;
    using L = Layout<kF8, k2, DH>;
    using Dm = Dims<DH>;
    constexpr int NH = Dm::NH;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t base = (smem_addr(smem_raw) + 1023u) & ~1023u;
    auto bar = [&](int i) -> uint32_t { return base + L::bars + 8u * (uint32_t)i; };
    const uint32_t flag_addr = base + L::abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int* meta = p.meta;
    const int n_items = meta[kMetaNumTiles];
    const int* items = meta + meta[kMetaOffTile];
    const int g = p.group, TQ = p.tile_tokens;

    if (threadIdx.x == 0) {
        mbar_init(bar(L::bQFull), 1);
        mbar_init(bar(L::bQReady), 256);
        mbar_init(bar(L::bQEmpty), 1);
        for (int i = 0; i < L::NKR; ++i) {
            mbar_init(bar(L::bKrFull + i), 1);
            mbar_init(bar(L::bKrEmpty + i), kF8 ? 1 : 128);
        }
        for (int i = 0; i < L::NVR; ++i) {
            mbar_init(bar(L::bVrFull + i), 1);
            mbar_init(bar(L::bVrEmpty + i), 128);
        }
        for (int i = 0; i < L::NK16; ++i) {
            mbar_init(bar(L::bK16Full + i), k2 ? 1 : 128);  // TMA, or the dequant warps
            mbar_init(bar(L::bK16Empty + i), 1);
        }
        for (int i = 0; i < L::NV16; ++i) {
            mbar_init(bar(L::bV16Full + i), 128);
            mbar_init(bar(L::bV16Empty + i), 1);
        }
        for (int x = 0; x < 2; ++x) {
            mbar_init(bar(L::bSFull + x), 1);
            mbar_init(bar(L::bPFull + x), 128);
            mbar_init(bar(L::bOFull + x), 1);
            mbar_init(bar(L::bOEmpty + x), 128);
            mbar_init(bar(L::bStageFree + x), 1);
            mbar_init(bar(L::bStageReady + x), 128);
        }
        mbar_init(bar(L::bDrain), 1);
        asm volatile("st.shared.u32 [%0], 0;" ::"r"(flag_addr) : "memory");
        mbar_init_fence();
    }
    if (warp == 13) tc_alloc(base + L::tmem_slot, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    uint32_t tmem;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(tmem) : "r"(base + L::tmem_slot) : "memory");
    // Registers per thread: launched at 128; each warpgroup's branch below
    // starts by resizing: softmax 192, dequant 64, producer/MMA 64
    // (4 x 32 x (64 + 2 x 192 + 64) = 65,536, what the block launched with).

    if (warp >= 12) {
      asm volatile("setmaxnreg.dec.sync.aligned.u32 64;" ::: "memory");
      if (warp == 12) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            prefetch_tmap(&tmq);
            prefetch_tmap(&tmk);
            prefetch_tmap(&tmv);
        }
        Ring kr, vr;  // kr: raw K ring, or the 16-bit K ring for a 2-byte cache
        uint32_t qphase = 0;
        long long issued_k = 0, issued_v = 0, issued_q = 0;
        constexpr int nkr = k2 ? L::NK16 : L::NKR;
        constexpr int bkf = k2 ? L::bK16Full : L::bKrFull, bke = k2 ? L::bK16Empty : L::bKrEmpty;
        bool ok = true;
        for (int rnd = 0, t = blockIdx.x; t < n_items && ok; t = item_at(++rnd, blockIdx.x, gridDim.x)) {
            const Item it = load_item(items, t);
            const int q0 = it.qo0 + it.t0;
            if (lane == 0) {
                ok = wait_or_abort<kDiag>(bar(L::bQEmpty), qphase ^ 1u, flag_addr, p.status, p.wait_cycles);
                if (ok) {
                    const uint32_t qb = bar(L::bQFull);
                    if (kF8) {
                        mbar_arrive_expect_tx(qb, (uint32_t)(2 * DH * g * TQ));
                        tma_load_3d(base + L::q, &tmq, qb, 0, it.hk * g, q0);
                        tma_load_3d(base + L::q + L::kQTile, &tmq, qb, 0, it.hk * g, q0 + TQ);
                    } else {
                        mbar_arrive_expect_tx(qb, (uint32_t)(4 * DH * g * TQ));
                        for (int x = 0; x < 2; ++x) {
                            const uint32_t dst = base + L::q + x * L::kQTile;
                            for (int h = 0; h < NH; ++h)
                                tma_load_3d(dst + h * kHalfTile, &tmq, qb, 64 * h, it.hk * g, q0 + x * TQ);
                        }
                    }
                    ++issued_q;
                }
            }
            ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
            qphase ^= 1u;
            const int kv_len = it.kv_len;
            // 16-token sub-pages of the request (a page of 16 * m tokens is m
            // of them).  The page entries of the next KV tile are loaded one
            // tile ahead and checked only when used, so the load's latency
            // stays hidden.
            const int m = p.page_mult;
            const int npages = (kv_len + kPageSize - 1) / kPageSize;
            const int* idx = p.kv_indices + it.page0;
            int page_next = 0;
            {
                const int np0 = min(kTileKeys / kPageSize, npages);
                if (lane < np0) page_next = __ldg(idx + (m == 1 ? lane : lane / m));
            }
            for (int j = 0; j < it.nkv && ok; ++j) {
                const int pg0 = j * (kTileKeys / kPageSize);
                const int np = min(kTileKeys / kPageSize, npages - pg0);
                int page = page_next;
                if (j + 1 < it.nkv) {
                    const int pg1 = pg0 + kTileKeys / kPageSize;
                    const int np1 = min(kTileKeys / kPageSize, npages - pg1);
                    page_next = lane < np1 ? __ldg(idx + (m == 1 ? pg1 + lane : (pg1 + lane) / m)) : 0;
                }
                const bool bad = lane < np && (page < 0 || page >= p.num_pages);
                if (bad) page = 0;
                else if (kSlots) page = page * m + (pg0 + lane) % m;
                if (__any_sync(0xFFFFFFFFu, bad) && lane == 0) atomicOr(p.status, kStatusBounds);
                // Lane i < np holds the id of the tile's sub-page i (page * m + j
                // with kSlots; sub-page j of a page is the box at token slot 16 j
                // of that page) and issues its copies through load(slot, page).
                auto for_page = [&](auto&& load) {
                    if constexpr (kSlots) {
                        const int pg = page / m;
                        load((page - pg * m) * kPageSize, pg);
                    } else {
                        load(0, page);
                    }
                };
                // A 2-byte cache has two boxes per page (the 64-dim halves): lane
                // 8 h + i issues half h of page i, so 16 lanes share them.
                const int hpage = __shfl_sync(0xFFFFFFFFu, page, lane & 7);
                auto for_half_page = [&](auto&& load) {
                    if constexpr (kSlots) {
                        const int pg = hpage / m;
                        load((hpage - pg * m) * kPageSize, pg);
                    } else {
                        load(0, hpage);
                    }
                };
                const bool half_lane = (lane & 7) < np && (lane >> 3) < NH;
                // Lane 0 waits for the stage and posts the byte count; then lane
                // i issues page i's box, or lane 8 h + i half h of it for a
                // 2-byte cache (a thread needs about 100 cycles per TMA box, so
                // the pages go out from several lanes at once).
                if (lane == 0) {
                    ok = wait_or_abort<kDiag>(bar(bke + kr.idx), kr.phase ^ 1u, flag_addr, p.status, p.wait_cycles);
                    if (ok) mbar_arrive_expect_tx(bar(bkf + kr.idx), (uint32_t)np * kPageSize * DH * (k2 ? 2 : 1));
                }
                ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
                if (!ok) break;
                if (k2) {
                    if (half_lane) {
                        // Each page as one box per 64-dim half into the halves of
                        // the 16-bit K tile: [half][key][128 B].
                        const uint32_t dst = base + L::k16 + kr.idx * Dm::kF16Tile;
                        const int h = lane >> 3, i = lane & 7;
                        for_half_page([&](int slot, int pg) {
                            tma_load_5d(dst + h * kHalfTile + i * 2048u, &tmk, bar(bkf + kr.idx), 0, h, slot, it.hk, pg);
                        });
                    }
                } else if (lane < np) {
                    const uint32_t dst = base + L::kr + kr.idx * Dm::kRawTile;
                    for_page([&](int slot, int pg) {
                        tma_load_4d(dst + lane * Dm::kRawPage, &tmk, bar(bkf + kr.idx), 0, it.hk, slot, pg);
                    });
                }
                ++issued_k;
                kr.next(nkr);
                if (lane == 0) {
                    ok = wait_or_abort<kDiag>(bar(L::bVrEmpty + vr.idx), vr.phase ^ 1u, flag_addr, p.status, p.wait_cycles);
                    if (ok) mbar_arrive_expect_tx(bar(L::bVrFull + vr.idx), (uint32_t)np * kPageSize * DH * (k2 ? 2 : 1));
                }
                ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
                if (!ok) break;
                if (k2) {
                    if (half_lane) {
                        const uint32_t dst = base + L::vr + vr.idx * L::kRawV;
                        const int h = lane >> 3, i = lane & 7;
                        for_half_page([&](int slot, int pg) {
                            tma_load_5d(dst + h * kHalfTile + i * 2048u, &tmv, bar(L::bVrFull + vr.idx), 0, h, slot, it.hk,
                                        pg);
                        });
                    }
                } else if (lane < np) {
                    const uint32_t dst = base + L::vr + vr.idx * L::kRawV;
                    for_page([&](int slot, int pg) {
                        tma_load_4d(dst + lane * Dm::kRawPage, &tmv, bar(L::bVrFull + vr.idx), 0, it.hk, slot, pg);
                    });
                }
                ++issued_v;
                vr.next(L::NVR);
            }
        }
        if (lane == 0) {
            // Let every copy issued by this CTA land before it may exit.
            if (issued_q > 0) mbar_wait(bar(L::bQFull), (uint32_t)((issued_q - 1) & 1));
            for (int s = 0; s < nkr && s < issued_k; ++s)
                mbar_wait(bar(bkf + s), (uint32_t)(((issued_k - 1 - s) / nkr) & 1));
            for (int s = 0; s < L::NVR && s < issued_v; ++s)
                mbar_wait(bar(L::bVrFull + s), (uint32_t)(((issued_v - 1 - s) / L::NVR) & 1));
        }
      } else if (warp == 13) {
        // ------------------------------------------------------------- MMA
        if (lane == 0) {
            const uint32_t idesc_qk =
                kF8 ? make_idesc(p.q_dtype == PAFP8_E5M2 ? 1 : 0, KT == PAFP8_E5M2 ? 1 : 0, 128, 128)
                    : make_idesc(kBF ? 1 : 0, kBF ? 1 : 0, 128, 128);
            const uint32_t idesc_pv = make_idesc_bmn(kBF ? 1 : 0, kBF ? 1 : 0, 128, DH);
            const int nk = kF8 ? L::NKR : L::NK16;
            const int kfull = kF8 ? L::bKrFull : L::bK16Full;
            const int kempty = kF8 ? L::bKrEmpty : L::bK16Empty;
            Ring kring, v16;
            uint32_t qphase = 0;
            uint32_t pphase[2] = {0, 0};
            int nonempty[2] = {0, 0};  // earlier items in which tile A / B had rows
            long long issued_any = 0;
            bool ok = true;
            // S_X = Q_X K^T for the K tile at the head of kring.
            auto qk = [&](int x) {
                const uint32_t dS = tmem + col_s(x);
                const uint32_t qa = base + L::q + x * L::kQTile;
                // The K steps' descriptor offsets are immediates inside one asm
                // statement (tc_mma_*_k*): start addresses are 16-byte units.
                if (kF8) {
                    // fp8 rows of DH bytes: 128- or 64-byte swizzle, 32 B per K step
                    const uint64_t dq = DH == 128 ? sw128_kmajor_desc(qa) : sw64_kmajor_desc(qa);
                    const uint32_t ka = base + L::kr + kring.idx * Dm::kRawTile;
                    const uint64_t dk = DH == 128 ? sw128_kmajor_desc(ka) : sw64_kmajor_desc(ka);
                    if constexpr (DH == 128) tc_mma_f8_ss_k4(dS, dq, dk, idesc_qk, 0u);
                    else tc_mma_f8_ss_k2(dS, dq, dk, idesc_qk, 0u);
                } else {
                    // 2-byte rows of DH elements: DH / 64 halves of 128 B, 32 B per K step
                    const uint64_t dq = sw128_kmajor_desc(qa);
                    const uint64_t dk = sw128_kmajor_desc(base + L::k16 + kring.idx * Dm::kF16Tile);
                    if constexpr (DH == 128) tc_mma_f16_ss_k8<kHalfTile, kHalfTile>(dS, dq, dk, idesc_qk, 0u);
                    else tc_mma_f16_ss_k4(dS, dq, dk, idesc_qk, 0u);
                }
                tc_commit(bar(L::bSFull + x));
                ++issued_any;
            };
            // O_X (+)= P_X V for the V tile at the head of the v16 ring.
            auto pv = [&](int x, bool accumulate) -> bool {
                // The first O_X write of an item waits for the epilogue of the
                // previous item that used O_X.
                if (!accumulate && nonempty[x] > 0 &&
                    !wait_or_abort<kDiag>(bar(L::bOEmpty + x), (uint32_t)((nonempty[x] - 1) & 1), flag_addr,
                                   p.status, p.wait_cycles))
                    return false;
                if (!wait_or_abort<kDiag>(bar(L::bPFull + x), pphase[x], flag_addr, p.status, p.wait_cycles)) return false;
                pphase[x] ^= 1u;
                tc_fence_after();
                // V [64-dim half][key][128 B] as the MN-major B operand: K = 128
                // keys in 8 steps of 16 rows, the dim halves kHalfTile apart.
                const uint64_t dv = sw128_mnmajor_desc(base + L::v16 + v16.idx * Dm::kF16Tile, kHalfTile);
                tc_mma_f16_ts_mn_k8(tmem + col_o<DH>(x), tmem + col_s(x), dv, idesc_pv, accumulate ? 1u : 0u);
                ++issued_any;
                return true;
            };
            for (int rnd = 0, t = blockIdx.x; t < n_items && ok; t = item_at(++rnd, blockIdx.x, gridDim.x)) {
                const Item it = load_item(items, t);
                const int qo_len = it.qo_len;
                const int kv_len = it.kv_len;
                const int nA = tile_nkv(it.t0, 0, TQ, qo_len, kv_len);
                const int nB = tile_nkv(it.t0, 1, TQ, qo_len, kv_len);
                const int n = it.nkv;
                ok = wait_or_abort<kDiag>(bar(fit_q ? L::bQReady : L::bQFull), qphase, flag_addr, p.status, p.wait_cycles);
                qphase ^= 1u;
                if (!ok) break;
                tc_fence_after();
                // K tile 0 for both query tiles.
                ok = wait_or_abort<kDiag>(bar(kfull + kring.idx), kring.phase, flag_addr, p.status, p.wait_cycles);
                if (!ok) break;
                tc_fence_after();
                if (nA > 0) qk(0);
                if (nB > 0) qk(1);
                tc_commit(bar(kempty + kring.idx));
                kring.next(nk);
                if (n == 1) tc_commit(bar(L::bQEmpty));
                for (int j = 0; j < n && ok; ++j) {
                    ok = wait_or_abort<kDiag>(bar(L::bV16Full + v16.idx), v16.phase, flag_addr, p.status, p.wait_cycles);
                    if (!ok) break;
                    tc_fence_after();
                    if (j < nA) {
                        if (!(ok = pv(0, j > 0))) break;
                        if (j == nA - 1) tc_commit(bar(L::bOFull + 0));
                    }
                    const bool more = j + 1 < n;
                    if (more) {
                        ok = wait_or_abort<kDiag>(bar(kfull + kring.idx), kring.phase, flag_addr, p.status, p.wait_cycles);
                        if (!ok) break;
                        tc_fence_after();
                        if (j + 1 < nA) qk(0);
                    }
                    if (j < nB) {
                        if (!(ok = pv(1, j > 0))) break;
                        if (j == nB - 1) tc_commit(bar(L::bOFull + 1));
                    }
                    tc_commit(bar(L::bV16Empty + v16.idx));
                    v16.next(L::NV16);
                    if (more) {
                        if (j + 1 < nB) qk(1);
                        tc_commit(bar(kempty + kring.idx));
                        kring.next(nk);
                        if (j + 1 == n - 1) tc_commit(bar(L::bQEmpty));
                    }
                }
                nonempty[0] += nA > 0;
                nonempty[1] += nB > 0;
            }
            // Drain: every MMA issued above completes before TMEM is freed.
            if (issued_any > 0) {
                tc_commit(bar(L::bDrain));
                mbar_wait(bar(L::bDrain), 0);
            }
        }
        __syncwarp();
      }
    } else if (warp < 4) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 64;" ::: "memory");
        // ---------------------------------------------------------- dequant
        const int wd = warp, q8 = lane >> 3, e = lane & 7;
        Ring kr, vr, k16, v16;
        bool ok = true;
        // A raw fp8 K or V tile [key][DH bytes] -> f16 [64-dim half][key][128 B]
        // under the 128-byte swizzle (the layout a 2-byte tile lands in), keys
        // `valid` and beyond zeroed.  K serves as the K-major B operand of Q K^T,
        // V as the MN-major B operand of P V.
        auto widen = [&](uint32_t src, uint32_t dst, int valid) {
            if constexpr (k2) {
                return;  // a 2-byte cache has no fp8 tile
            } else if constexpr (DH == 128) {
#pragma unroll 2
                for (int i = 0; i < 8; ++i) {
                    const int combo = wd * 8 + i;
                    const int row = (combo >> 1) * 8 + e;
                    const int c = (combo & 1) * 4 + q8;
                    uint4 w = lds128(src + row * 128 + ((c ^ e) << 4));
                    if (row >= valid) w = make_uint4(0u, 0u, 0u, 0u);
                    const uint32_t hb = dst + (c >> 2) * kHalfTile + row * 128;
                    sts128(hb + (((2 * q8) ^ e) << 4), fp8x2_lo<KT>(w.x), fp8x2_hi<KT>(w.x), fp8x2_lo<KT>(w.y),
                           fp8x2_hi<KT>(w.y));
                    sts128(hb + (((2 * q8 + 1) ^ e) << 4), fp8x2_lo<KT>(w.z), fp8x2_hi<KT>(w.z), fp8x2_lo<KT>(w.w),
                           fp8x2_hi<KT>(w.w));
                }
            } else {
                // 64-B fp8 rows under the 64-byte swizzle (16-byte chunk c of
                // row r at c ^ ((r >> 1) & 3)) -> one 128-B f16 half.
#pragma unroll 2
                for (int i = 0; i < 4; ++i) {
                    const int row = (wd * 4 + i) * 8 + e, c = q8;
                    uint4 w = lds128(src + row * 64 + ((c ^ ((row >> 1) & 3)) << 4));
                    if (row >= valid) w = make_uint4(0u, 0u, 0u, 0u);
                    const uint32_t hb = dst + row * 128;
                    sts128(hb + (((2 * c) ^ e) << 4), fp8x2_lo<KT>(w.x), fp8x2_hi<KT>(w.x), fp8x2_lo<KT>(w.y),
                           fp8x2_hi<KT>(w.y));
                    sts128(hb + (((2 * c + 1) ^ e) << 4), fp8x2_lo<KT>(w.z), fp8x2_hi<KT>(w.z), fp8x2_lo<KT>(w.w),
                           fp8x2_hi<KT>(w.w));
                }
            }
        };
        for (int rnd = 0, t = blockIdx.x; t < n_items && ok; t = item_at(++rnd, blockIdx.x, gridDim.x)) {
            const Item it = load_item(items, t);
            const int kv_len = it.kv_len;
            for (int j = 0; j < it.nkv && ok; ++j) {
                const int valid = min(kTileKeys, kv_len - j * kTileKeys);
                if constexpr (!kF8 && !k2) {
                    ok = wait_or_abort<kDiag>(bar(L::bKrFull + kr.idx), kr.phase, flag_addr, p.status, p.wait_cycles) &&
                         wait_or_abort<kDiag>(bar(L::bK16Empty + k16.idx), k16.phase ^ 1u, flag_addr, p.status, p.wait_cycles);
                    if (!ok) break;
                    widen(base + L::kr + kr.idx * Dm::kRawTile, base + L::k16 + k16.idx * Dm::kF16Tile, kTileKeys);
                    fence_async_smem();
                    mbar_arrive(bar(L::bK16Full + k16.idx));
                    mbar_arrive(bar(L::bKrEmpty + kr.idx));
                    kr.next(L::NKR);
                    k16.next(L::NK16);
                }
                ok = wait_or_abort<kDiag>(bar(L::bVrFull + vr.idx), vr.phase, flag_addr, p.status, p.wait_cycles) &&
                     wait_or_abort<kDiag>(bar(L::bV16Empty + v16.idx), v16.phase ^ 1u, flag_addr, p.status, p.wait_cycles);
                if (!ok) break;
                const uint32_t src = base + L::vr + vr.idx * L::kRawV;
                const uint32_t dst = base + L::v16 + v16.idx * Dm::kF16Tile;
                if constexpr (k2) {
                    // A 2-byte V tile is already in the layout the MMA reads: copied
                    // 16 bytes per thread and step (consecutive threads, consecutive
                    // chunks), keys past the request's end zeroed.
#pragma unroll 2
                    for (int i = 0; i < 8 * NH; ++i) {
                        const int q = i * 128 + (int)threadIdx.x;
                        const uint32_t off = (uint32_t)q * 16u;  // [half][key][128 B]
                        const int row = (q >> 3) & (kTileKeys - 1);
                        uint4 w = lds128(src + off);
                        if (row >= valid) w = make_uint4(0u, 0u, 0u, 0u);
                        sts128(dst + off, w.x, w.y, w.z, w.w);
                    }
                } else {
                    widen(src, dst, valid);
                }
                fence_async_smem();
                mbar_arrive(bar(L::bV16Full + v16.idx));
                mbar_arrive(bar(L::bVrEmpty + vr.idx));
                vr.next(L::NVR);
                v16.next(L::NV16);
            }
        }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 192;" ::: "memory");
        // ---------------------------------------------------------- softmax
        const int x = warp < 8 ? 0 : 1;        // query tile A or B
        const int r = threadIdx.x - 128 * (1 + x);  // row of the tile = TMEM lane
        const uint32_t lane_base = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
        const uint32_t tS = lane_base + col_s(x), tO = lane_base + col_o<DH>(x);
        uint32_t qphase = 0, sphase = 0, ophase = 0;
        uint32_t stage_round = 0;  // staging rounds of this tile so far (fp8 query)
        const bool issuer = (threadIdx.x & 127) == 0;
        const bool o_32b = (reinterpret_cast<uintptr_t>(p.o) & 31u) == 0;  // rows are 256 B apart
        bool ok = true;
        // Range fit of this thread's Q row (bf16 query on an fp8 cache): wait
        // for the item's Q tiles, scale the row into f16 range by an exact power
        // of two, convert it in place and return the power (it multiplies the
        // logit scale).  Both warpgroups arrive on q_ready for every item.
        auto fit_row = [&]() -> float {
            float up = 1.f;
            ok = __all_sync(0xFFFFFFFFu, wait_or_abort<kDiag>(bar(L::bQFull), qphase, flag_addr, p.status, p.wait_cycles));
            qphase ^= 1u;
            if (!ok) return up;
            if (r < TQ * g) {
                const uint32_t qrow = base + L::q + x * L::kQTile + r * 128;
                uint32_t mx = 0;
#pragma unroll
                for (int c = 0; c < 8 * NH; ++c) {
                    const uint4 w = lds128(qrow + (c >> 3) * kHalfTile + (((c & 7) ^ (r & 7)) << 4));
                    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        mx = max(mx, (ws[k] & 0x7FFFu) << 16);
                        mx = max(mx, ws[k] & 0x7FFF0000u);
                    }
                }
                const int ex = (int)((mx >> 23) & 0xFF) - 127;
                const int shift = ex > 14 ? ex - 14 : 0;
                const float down = __int_as_float((127 - shift) << 23);
                up = __int_as_float((127 + shift) << 23);
#pragma unroll 4
                for (int c = 0; c < 8 * NH; ++c) {
                    const uint32_t a = qrow + (c >> 3) * kHalfTile + (((c & 7) ^ (r & 7)) << 4);
                    const uint4 w = lds128(a);
                    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
                    uint32_t o4[4];
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        o4[k] = pack_half2(__uint_as_float(ws[k] << 16) * down,
                                           __uint_as_float(ws[k] & 0xFFFF0000u) * down);
                    sts128(a, o4[0], o4[1], o4[2], o4[3]);
                }
                fence_async_smem();
            }
            mbar_arrive(bar(L::bQReady));
            return up;
        };
        // The next item's Q is fitted right after this item's last softmax pass
        // and before its epilogue, so the next item's first QK does not wait
        // for the epilogues.
        float up_next = 1.f;
        if (fit_q && (int)blockIdx.x < n_items) up_next = fit_row();
        Item it_next = (int)blockIdx.x < n_items ? load_item(items, blockIdx.x) : Item{};
        for (int rnd = 0, t = blockIdx.x; t < n_items && ok; t = item_at(++rnd, blockIdx.x, gridDim.x)) {
            const Item it = it_next;
            const int qo0 = it.qo0;
            const int qo_len = it.qo_len;
            const int kv_len = it.kv_len;
            const int t0 = it.t0 + x * TQ;
            const int nX = tile_nkv(it.t0, x, TQ, qo_len, kv_len);
            const int tok = r / g, hh = r - tok * g;
            const bool valid_row = (tok < TQ) && (t0 + tok < qo_len);
            const int limit = valid_row ? t0 + tok + kv_len - qo_len : -1;
            float scale = p.sm_scale_log2 * up_next;
            float vsc = p.v_scale;
            if (p.k_scales != nullptr) {  // per-head scale tensors
                const int qh = it.hk * g + min(hh, g - 1);
                scale = fold_scale_log2(p.sm_scale, p.q_scales != nullptr ? __ldg(p.q_scales + qh) : 1.0f,
                                        __ldg(p.k_scales + it.hk)) *
                        up_next;
                vsc = __ldg(p.v_scales + it.hk);
            }
            float m = -INFINITY, l = 0.f;  // m in scaled (log2) units
            for (int j = 0; j < nX && ok; ++j) {
                ok = __all_sync(0xFFFFFFFFu, wait_or_abort<kDiag>(bar(L::bSFull + x), sphase, flag_addr, p.status, p.wait_cycles));
                sphase ^= 1u;
                if (!ok) break;
                tc_fence_after();
                const int key0 = j * kTileKeys;
                const bool need_mask = key0 + kTileKeys - 1 > limit;
                // The whole S row (128 columns) in registers, one wait.
                uint32_t v[128];
#pragma unroll
                for (int c = 0; c < 4; ++c) tc_ld32(tS + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(v + 32 * c));
                tc_wait_ld();
                // row max of the raw logits (scale > 0); masked logits -> -inf.
                // Eight independent partial maxima keep the chain short.
                if (need_mask) {
                    const int lim = limit - key0;
#pragma unroll
                    for (int i = 0; i < 128; ++i)
                        if (i > lim) v[i] = __float_as_uint(-INFINITY);
                }
                // Four independent three-input maxima keep the chain short.
                float pm[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) pm[k] = __uint_as_float(v[k]);
#pragma unroll
                for (int i = 4; i < 128; i += 2)
                    pm[(i >> 1) & 3] = max3(pm[(i >> 1) & 3], __uint_as_float(v[i]), __uint_as_float(v[i + 1]));
                const float mx = fmaxf(max3(pm[0], pm[1], pm[2]), pm[3]);
                const float m_new = fmaxf(m, mx * scale);
                float m_use = m;
                bool rescale = false;
                if (j == 0) {
                    m_use = m_new;
                } else if (m_new > m + 8.0f) {
                    m_use = m_new;
                    rescale = true;
                }
                if (m_use == -INFINITY) m_use = 0.f;  // row with no admissible key so far
                // tcgen05.ld/st are warp-collective: the whole warp rescales
                // when any of its rows must (alpha = 1 for the others).
                if (__any_sync(0xFFFFFFFFu, rescale)) {
                    // O_X += P V of the previous KV tile has completed (in-order
                    // tensor pipe, S of this tile was written after it).
                    const float alpha = rescale ? ex2(m - m_use) : 1.f;
                    const f32x2 alpha2 = make_f32x2(alpha, alpha);
                    l *= alpha;
#pragma unroll 1
                    for (int c = 0; c < DH / 32; ++c) {
                        uint32_t v[32];
                        tc_ld32(tO + 32 * c, v);
                        tc_wait_ld();
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            float a, b;
                            split_f32x2(mul2(make_f32x2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1])),
                                             alpha2),
                                        a, b);
                            v[2 * i] = __float_as_uint(a);
                            v[2 * i + 1] = __float_as_uint(b);
                        }
                        tc_st32(tO + 32 * c, v);
                    }
                    tc_wait_st();
                }
                // P = exp2(s * scale - m) (masked logits are -inf: P = 0), row
                // sum, P -> TMEM as f16 over the first half of S.  Pairs of
                // columns go through the packed fp32 pipe.
                const f32x2 scale2 = make_f32x2(scale, scale), negm2 = make_f32x2(-m_use, -m_use);
                // P overwrites the S values it consumed: P of columns 2i, 2i+1
                // goes to v[i], which held column i (already used).  Two
                // independent packed partial sums keep the chain short.
                f32x2 ps[2] = {make_f32x2(0.f, 0.f), make_f32x2(0.f, 0.f)};
#pragma unroll
                for (int i = 0; i < 64; ++i) {
                    float a, b;
                    split_f32x2(fma2(make_f32x2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1])), scale2,
                                     negm2),
                                a, b);
                    const float e0 = ex2(a), e1 = ex2(b);
                    const f32x2 e = make_f32x2(e0, e1);
                    ps[i & 1] = add2(ps[i & 1], e);
                    v[i] = kBF ? pack_bf162(e0, e1) : pack_half2(e0, e1);
                }
                {
                    float a, b, c, d;
                    split_f32x2(ps[0], a, b);
                    split_f32x2(ps[1], c, d);
                    l += (a + b) + (c + d);
                }
                tc_st32(tS, *reinterpret_cast<uint32_t(*)[32]>(v));
                tc_st32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(v + 32));
                tc_wait_st();
                tc_fence_before();
                mbar_arrive(bar(L::bPFull + x));
                m = m_use;
            }
            if (!ok) break;
            // The next item's record, loaded here so that its latency passes
            // during the epilogue rather than before the next item's first pass.
            {
                const int tn = item_at(rnd + 1, blockIdx.x, gridDim.x);
                if (tn < n_items) it_next = load_item(items, tn);
            }
            if (fit_q && item_at(rnd + 1, blockIdx.x, gridDim.x) < n_items) {
                up_next = fit_row();
                if (!ok) break;
            }
            if (nX == 0) continue;  // tile B past the request's last row
            // epilogue: the tile's last O update must have completed.
            ok = __all_sync(0xFFFFFFFFu, wait_or_abort<kDiag>(bar(L::bOFull + x), ophase, flag_addr, p.status, p.wait_cycles));
            ophase ^= 1u;
            if (!ok) break;
            tc_fence_after();
            const float inv = valid_row && l > 0.f ? vsc / l : 0.f;
            const size_t orow = (size_t)(qo0 + t0 + tok) * p.num_qo_heads + (size_t)it.hk * g + hh;
            if (kF8 && t0 + TQ <= qo_len) {
                // A full tile: two rounds of 64 dims through this tile's staging
                // half, each written out by one bulk tensor store (asynchronous;
                // the next round waits until the store has read the staging).
                const uint32_t stg = base + L::ostage + (uint32_t)x * kHalfTile;
                bool sok = true;
#pragma unroll 1
                for (int h = 0; h < NH && sok; ++h, ++stage_round) {
                    uint32_t v[64];
                    tc_ld32(tO + 64 * h, *reinterpret_cast<uint32_t(*)[32]>(v));
                    tc_ld32(tO + 64 * h + 32, *reinterpret_cast<uint32_t(*)[32]>(v + 32));
                    tc_wait_ld();
                    if (h == NH - 1) {
                        // O_X is read: release it to the next item's first PV.
                        tc_fence_before();
                        mbar_arrive(bar(L::bOEmpty + x));
                    }
                    uint32_t w[32];
                    const f32x2 inv2 = make_f32x2(inv, inv);
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        float a0, a1;
                        split_f32x2(mul2(make_f32x2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1])), inv2),
                                    a0, a1);
                        w[i] = pack_out2(a0, a1, p.o_dtype);
                    }
                    if (issuer) {
                        bulk_wait_read_all();
                        mbar_arrive(bar(L::bStageFree + x));
                    }
                    sok = __all_sync(0xFFFFFFFFu, wait_or_abort<kDiag>(bar(L::bStageFree + x), stage_round & 1u, flag_addr,
                                                                p.status, p.wait_cycles));
                    if (!sok) break;
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        sts128(stg + r * 128 + ((c ^ (r & 7)) << 4), w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
                    fence_async_smem();
                    mbar_arrive(bar(L::bStageReady + x));
                    if (issuer) {
                        sok = wait_or_abort<kDiag>(bar(L::bStageReady + x), stage_round & 1u, flag_addr, p.status, p.wait_cycles);
                        if (sok) {
                            tma_store_3d(&tmo, stg, 64 * h, it.hk * g, qo0 + t0);
                            bulk_commit();
                        }
                    }
                    sok = __all_sync(0xFFFFFFFFu, sok);
                }
                ok = sok;
                if (!ok) break;
                if (valid_row && p.lse != nullptr) p.lse[orow] = (m + __log2f(l)) * 0.69314718055994531f;
                continue;
            }
#pragma unroll 1
            for (int c = 0; c < DH / 32; ++c) {
                uint32_t v[32];
                tc_ld32(tO + 32 * c, v);
                tc_wait_ld();
                if (valid_row) {
                    uint32_t w[16];
                    const f32x2 inv2 = make_f32x2(inv, inv);
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        float a, b;
                        split_f32x2(mul2(make_f32x2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1])), inv2),
                                    a, b);
                        w[i] = pack_out2(a, b, p.o_dtype);
                    }
                    uint16_t* dst = static_cast<uint16_t*>(p.o) + orow * DH + 32 * c;
                    if (o_32b) {
                        // 32-byte stores: every access fills whole sectors.
                        stg256(dst, w);
                        stg256(dst + 16, w + 8);
                    } else {
                        uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
                        for (int i = 0; i < 4; ++i) d4[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
                    }
                }
            }
            if (valid_row && p.lse != nullptr) p.lse[orow] = (m + __log2f(l)) * 0.69314718055994531f;
            tc_fence_before();
            mbar_arrive(bar(L::bOEmpty + x));
        }
    }

    if (kF8 && (warp == 4 || warp == 8) && lane == 0) bulk_wait_all();  // this thread's output stores
    tc_fence_before();
    __syncthreads();
    if (warp == 13) {
        tc_fence_after();
        tc_dealloc(tmem, kTmemCols);
    }
}

template <bool kF8, int KT, bool kDiag, int DH, bool kSlots>
cudaError_t launch_t(const PrefillParams& p, const CUtensorMap& tq, const CUtensorMap& tk,
                     const CUtensorMap& tv, const CUtensorMap& to, int num_ctas, cudaStream_t stream) {
    const size_t smem = 1024 + Layout<kF8, KT == PAFP8_F16 || KT == PAFP8_BF16, DH>::bytes;
    cudaError_t e = cudaFuncSetAttribute(prefill_kernel<kF8, KT, kDiag, DH, kSlots>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    prefill_kernel<kF8, KT, kDiag, DH, kSlots><<<num_ctas, kThreads, smem, stream>>>(p, tq, tk, tv, to);
    return cudaGetLastError();
}

// The diagnostic instantiation runs only under a shortened wait bound (and
// takes any page size); pages of 16 tokens and of 16 m tokens have one each.
template <bool kF8, int KT, int DH>
cudaError_t launch_one(const PrefillParams& p, const CUtensorMap& tq, const CUtensorMap& tk,
                       const CUtensorMap& tv, const CUtensorMap& to, int num_ctas, cudaStream_t stream) {
    if (p.wait_cycles < kWaitCyclesDefault)
        return launch_t<kF8, KT, true, DH, true>(p, tq, tk, tv, to, num_ctas, stream);
    return p.page_mult != 1 ? launch_t<kF8, KT, false, DH, true>(p, tq, tk, tv, to, num_ctas, stream)
                            : launch_t<kF8, KT, false, DH, false>(p, tq, tk, tv, to, num_ctas, stream);
}

// Dispatch on the query and cache dtypes for head size DH.
template <int DH>
cudaError_t launch_prefill_head(const PrefillParams& p, const CUtensorMap& tmap_q, const CUtensorMap& tmap_k,
                                const CUtensorMap& tmap_v, const CUtensorMap& tmap_o, int num_ctas,
                                cudaStream_t stream) {
    const bool f8 = p.q_dtype == PAFP8_E4M3FN || p.q_dtype == PAFP8_E5M2;
    if (f8)
        return p.kv_dtype == PAFP8_E4M3FN
                   ? launch_one<true, PAFP8_E4M3FN, DH>(p, tmap_q, tmap_k, tmap_v, tmap_o, num_ctas, stream)
                   : launch_one<true, PAFP8_E5M2, DH>(p, tmap_q, tmap_k, tmap_v, tmap_o, num_ctas, stream);
    switch (p.kv_dtype) {
        case PAFP8_E4M3FN: return launch_one<false, PAFP8_E4M3FN, DH>(p, tmap_q, tmap_k, tmap_v, tmap_o, num_ctas, stream);
        case PAFP8_E5M2: return launch_one<false, PAFP8_E5M2, DH>(p, tmap_q, tmap_k, tmap_v, tmap_o, num_ctas, stream);
        case PAFP8_F16: return launch_one<false, PAFP8_F16, DH>(p, tmap_q, tmap_k, tmap_v, tmap_o, num_ctas, stream);
        case PAFP8_BF16: return launch_one<false, PAFP8_BF16, DH>(p, tmap_q, tmap_k, tmap_v, tmap_o, num_ctas, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace
}  // namespace pafp8
