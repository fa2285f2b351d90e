// prefill_pair.cuh -- the ragged causal prefill of prefill.cuh at head_dim 128
// over a 2-byte (f16 or bf16) cache, run by CTA pairs (clusters of two CTAs
// on two SMs) with 2-SM MMAs.
//
// What it computes is prefill.cuh's: for query row i of request b (0-based
// among its qo_len new rows) and head h, o = v_scale * softmax(sm_scale *
// k_scale * q.k) V over the keys j <= i + kv_len - qo_len of KV head
// h / group (bottom-right causal mask), lse = ln sum exp(logits).  The query
// and the cache have the same 2-byte dtype, which the MMAs take as loaded.
//
// Why pairs here: with a 2-byte cache a single CTA spends its producer on the
// TMA issue of 32 half-page boxes per tile.  A pair issues
// tcgen05.mma.cta_group::2 with M = 256 from the leader CTA: each CTA holds
// its 128 rows of the query tile (and of S, P and O in its TMEM) and half of
// the other operand's N columns at the same shared-memory offset -- keys
// 64 r .. 64 r + 63 of each K tile (QK: N = keys), dims 64 r .. 64 r + 63 of
// each V tile (PV: N = dims).  So each CTA loads half of every K and V tile.
// V is the MN-major B operand of P V exactly as its page boxes land
// ([key][64 dims of 128 B]), so nothing transforms it.  (With an fp8 cache
// the single-CTA kernel stays faster: there the serial per-tile chain QK ->
// softmax -> P hand-off -> PV bounds it, and a pair lengthens the hand-offs,
// which cross SMs.)
//
// Work item: (request, KV head, two query tiles A and B of 2 TQ tokens each);
// CTA r of the pair owns tokens [t0 + 2 TQ x + TQ r, + TQ) of tile x, i.e.
// 128 packed (token, head) rows per tile, as one CTA of prefill.cuh.
//
// Roles per CTA (512 threads; registers moved by setmaxnreg as in prefill.cuh):
//   warps 0-3   V release: zero the keys past the request's end in a request's
//               last V tile, then mark the tile ready for the leader;
//   warps 4-7   softmax of tile A, warps 8-11 of tile B (prefill.cuh's);
//   warp 12     TMA producer: this CTA's Q rows, its K pages, its V dim half;
//   warp 13     in the leader: MMA issuer (warps 14-15 and the peer's 13-15
//               idle; warp 13 of each CTA allocates the pair's TMEM).
// Synchronization across the pair: barriers that the leader's MMA thread
// waits on live in the leader and count arrivals from both CTAs (one arrive
// per warp, and TMA loads of both CTAs whose bytes complete on the leader's
// barrier); barriers that the MMAs release are signalled in both CTAs by
// multicast commits.  All waits are bounded; on expiry a CTA records a status
// bit and winds down.
#pragma once
#include "prefill.cuh"

namespace pafp8 {
namespace {

constexpr int kPairKeys = kTileKeys / 2;       // K rows each CTA holds (QK: N / 2)
constexpr uint32_t kHalf64 = kPairKeys * 128;  // 8 KB: 64 rows x 128 B

struct PairLayout {
    // Q: two tiles of [dim half][128 rows][128 B]; 16-bit K: [dim half][64
    // keys][128 B] (this CTA's keys); V: [128 keys][128 B] (this CTA's 64
    // dims), four stages, each held from its copy to the P V MMAs' commit.
    static constexpr int NK16 = 2, NVR = 4;
    static constexpr uint32_t kQTile = 2 * kHalfTile;  // 32 KB
    static constexpr uint32_t kK16 = 2 * kHalf64;      // 16 KB
    static constexpr uint32_t kRawV = kTileKeys * 128;  // 16 KB
    static constexpr uint32_t q = 0;
    static constexpr uint32_t k16 = 2 * kQTile;
    static constexpr uint32_t vr = k16 + NK16 * kK16;
    // Output staging: per query tile a [64-dim half][128 rows][128 B] copy of
    // this CTA's O rows (the Q tile's swizzled layout), written out by two
    // bulk tensor stores.
    static constexpr uint32_t ostage = vr + NVR * kRawV;
    static constexpr uint32_t kStage = 2 * kHalfTile;  // 32 KB
    static constexpr uint32_t bars = ostage + 2 * kStage;
    static constexpr int bQFull = 0, bQEmpty = 1;
    static constexpr int bK16Full = 2, bK16Empty = bK16Full + NK16;
    static constexpr int bVrFull = bK16Empty + NK16, bVrEmpty = bVrFull + NVR;
    static constexpr int bVReady = bVrEmpty + NVR;   // [NVR], in the leader
    static constexpr int bSFull = bVReady + NVR;     // [2]
    static constexpr int bPFull = bSFull + 2;        // [2]
    static constexpr int bOFull = bPFull + 2;        // [2]
    static constexpr int bOEmpty = bOFull + 2;       // [2]
    static constexpr int bStageFree = bOEmpty + 2;     // [2]
    static constexpr int bStageReady = bStageFree + 2;  // [2]
    static constexpr int bDrain = bStageReady + 2;
    static constexpr int nBars = bDrain + 1;
    static constexpr uint32_t tmem_slot = bars + 8 * nBars;
    static constexpr uint32_t abort_flag = tmem_slot + 4;
    static constexpr uint32_t bytes = abort_flag + 4;
};
static_assert(1024 + PairLayout::bytes <= 232448, "shared memory budget (pair)");
static_assert(PairLayout::k16 % 1024 == 0 && PairLayout::vr % 1024 == 0 && PairLayout::ostage % 1024 == 0,
              "1024-byte alignment of the pair tiles");

// wait_or_abort with acquire at cluster scope, for barriers that the peer CTA
// arrives on.
template <bool kDiag>
__device__ __forceinline__ bool wait_or_abort_cl(uint32_t bar, uint32_t parity, uint32_t flag_addr, uint32_t* status,
                                                 long long limit) {
    if constexpr (kDiag) {
        const long long t0 = clock64();
        while (!mbar_test_wait_cluster(bar, parity))
            if (clock64() - t0 > limit) {
                set_abort(flag_addr, status);
                return false;
            }
        return true;
    }
    if (mbar_try_wait_cluster(bar, parity)) return true;
    const long long t0 = clock64();
    while (!mbar_try_wait_cluster(bar, parity)) {
        if (aborted(flag_addr)) return false;
        if (clock64() - t0 > kWaitCycles) {
            set_abort(flag_addr, status);
            return false;
        }
    }
    return true;
}

template <int KT, bool kDiag, bool kSlots>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_pair_kernel(const __grid_constant__ PrefillParams p, const __grid_constant__ CUtensorMap tmq,
                        const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                        const __grid_constant__ CUtensorMap tmo) {
    static_assert(KT == PAFP8_F16 || KT == PAFP8_BF16, "a 2-byte cache");
    constexpr bool kBF = KT == PAFP8_BF16;  // bf16 MMA operands
    constexpr int DH = 128;
    using L = PairLayout;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t base = (smem_addr(smem_raw) + 1023u) & ~1023u;
    auto bar = [&](int i) -> uint32_t { return base + L::bars + 8u * (uint32_t)i; };
    const uint32_t flag_addr = base + L::abort_flag;
    // Clusters are (2, 1, 1) over a 1-D grid, so %cluster_ctarank is blockIdx.x & 1
    // (read from blockIdx, the compiler need not keep it live).  0: the leader,
    // which issues the MMAs.
    const uint32_t rank = blockIdx.x & 1u;
    const bool leader = rank == 0;
    // Barrier i of the leader, as a shared::cluster address.
    auto lbar = [&](int i) -> uint32_t { return map_shared(bar(i), 0); };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int* meta = p.meta;
    const int n_items = meta[kMetaNumTiles];
    const int* items = meta + meta[kMetaOffTile];
    const int g = p.group, TQ = p.tile_tokens, TQ2 = 2 * TQ;
    const int pair_id = blockIdx.x >> 1, n_pairs = gridDim.x >> 1;

    if (threadIdx.x == 0) {
        // Arrivals from threads are counted per warp (one arrive per warp).
        mbar_init(bar(L::bQFull), 1);
        mbar_init(bar(L::bQEmpty), 1);
        for (int i = 0; i < L::NK16; ++i) {
            mbar_init(bar(L::bK16Full + i), 1);
            mbar_init(bar(L::bK16Empty + i), 1);
        }
        for (int i = 0; i < L::NVR; ++i) {
            mbar_init(bar(L::bVrFull + i), 1);
            mbar_init(bar(L::bVrEmpty + i), 1);  // the P V MMAs' commit
            mbar_init(bar(L::bVReady + i), 8);   // both CTAs' V-release warps
        }
        for (int x = 0; x < 2; ++x) {
            mbar_init(bar(L::bSFull + x), 1);
            mbar_init(bar(L::bPFull + x), 8);   // both CTAs' softmax warps of tile x
            mbar_init(bar(L::bOFull + x), 1);
            mbar_init(bar(L::bOEmpty + x), 8);
            mbar_init(bar(L::bStageFree + x), 1);
            mbar_init(bar(L::bStageReady + x), 128);
        }
        mbar_init(bar(L::bDrain), 1);
        asm volatile("st.shared.u32 [%0], 0;" ::"r"(flag_addr) : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 13) tc_alloc_pair(base + L::tmem_slot, kTmemCols);
    __syncwarp();
    tc_fence_before();
    cluster_sync_all();
    tc_fence_after();
    uint32_t tmem;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(tmem) : "r"(base + L::tmem_slot) : "memory");

    if (warp >= 12) {
      asm volatile("setmaxnreg.dec.sync.aligned.u32 64;" ::: "memory");
      if (warp == 12) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            prefetch_tmap(&tmq);
            prefetch_tmap(&tmk);
            prefetch_tmap(&tmv);
        }
        Ring kr, vr;
        uint32_t qphase = 0;
        long long issued_k = 0, issued_v = 0, issued_q = 0;
        bool ok = true;
        for (int rnd = 0, t = pair_id; t < n_items && ok; t = item_at(++rnd, pair_id, n_pairs)) {
            const Item it = load_item(items, t);
            // Q: this CTA's rows of tiles A and B (tokens t0 + 2 TQ x + TQ r),
            // one box per 64-dim half, lane 2 x + h; the bytes of both CTAs
            // complete on the leader's barrier.
            if (lane == 0) {
                ok = wait_or_abort<kDiag>(bar(L::bQEmpty), qphase ^ 1u, flag_addr, p.status, p.wait_cycles);
                if (ok && leader) mbar_arrive_expect_tx(bar(L::bQFull), (uint32_t)(2 * 4 * DH * g * TQ));
            }
            ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
            qphase ^= 1u;
            if (!ok) break;
            if (lane < 4) {
                const int x = lane >> 1, h = lane & 1;
                tma_load_3d_pair(base + L::q + x * L::kQTile + h * kHalfTile, &tmq, lbar(L::bQFull), 64 * h,
                                 it.hk * g, it.qo0 + it.t0 + x * TQ2 + (int)rank * TQ);
            }
            ++issued_q;
            const int kv_len = it.kv_len;
            // 16-token sub-pages of the request; the entries of the next KV
            // tile are loaded one tile ahead and checked only when used.
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
                // TMA coordinates (token slot, page) of sub-page id v (page * m + j
                // with kSlots: sub-page j of a page is the box at slot 16 j).
                auto at = [&](int v, int& slot, int& pg) {
                    if constexpr (kSlots) {
                        pg = v / m;
                        slot = (v - pg * m) * kPageSize;
                    } else {
                        pg = v;
                        slot = 0;
                    }
                };
                // K: this CTA's keys 64 r .. 64 r + 63, i.e. pages 4 r .. 4 r + 3 of
                // the tile, lane 4 h + i issuing dim half h of page i; the bytes of
                // both CTAs complete on the leader's barrier.
                const int myk = max(0, min(4, np - 4 * (int)rank));
                if (lane == 0) {
                    ok = wait_or_abort<kDiag>(bar(L::bK16Empty + kr.idx), kr.phase ^ 1u, flag_addr, p.status,
                                              p.wait_cycles);
                    if (ok && leader)
                        mbar_arrive_expect_tx(bar(L::bK16Full + kr.idx), (uint32_t)np * kPageSize * DH * 2);
                }
                ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
                if (!ok) break;
                {
                    const int i = lane & 3, h = (lane >> 2) & 1;
                    const int v = __shfl_sync(0xFFFFFFFFu, page, min(4 * (int)rank + i, 7));
                    if (lane < 8 && i < myk) {
                        int slot, pg;
                        at(v, slot, pg);
                        tma_load_5d_pair(base + L::k16 + kr.idx * L::kK16 + h * kHalf64 + i * 2048u, &tmk,
                                         lbar(L::bK16Full + kr.idx), 0, h, slot, it.hk, pg);
                    }
                }
                ++issued_k;
                kr.next(L::NK16);
                // V: this CTA's dim half of every page, lane i issuing page i.
                if (lane == 0) {
                    ok = wait_or_abort<kDiag>(bar(L::bVrEmpty + vr.idx), vr.phase ^ 1u, flag_addr, p.status,
                                              p.wait_cycles);
                    if (ok) mbar_arrive_expect_tx(bar(L::bVrFull + vr.idx), (uint32_t)np * kPageSize * 64 * 2);
                }
                ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
                if (!ok) break;
                if (lane < np) {
                    int slot, pg;
                    at(page, slot, pg);
                    tma_load_5d(base + L::vr + vr.idx * L::kRawV + lane * 2048u, &tmv, bar(L::bVrFull + vr.idx), 0,
                                (int)rank, slot, it.hk, pg);
                }
                ++issued_v;
                vr.next(L::NVR);
            }
        }
        if (lane == 0) {
            // Let every copy land before the pair may exit: this CTA's V
            // copies on its own barriers; the leader also waits for the pair's
            // Q and K barriers, which count the other CTA's copies too.
            if (leader) {
                if (issued_q > 0) mbar_wait(bar(L::bQFull), (uint32_t)((issued_q - 1) & 1));
                for (int s = 0; s < L::NK16 && s < issued_k; ++s)
                    mbar_wait(bar(L::bK16Full + s), (uint32_t)(((issued_k - 1 - s) / L::NK16) & 1));
            }
            for (int s = 0; s < L::NVR && s < issued_v; ++s)
                mbar_wait(bar(L::bVrFull + s), (uint32_t)(((issued_v - 1 - s) / L::NVR) & 1));
        }
      } else if (warp == 13 && leader) {
        // ------------------------------------------------------ MMA (leader)
        // Per KV tile j, as prefill.cuh: ... PV_A(j), QK_A(j+1), PV_B(j),
        // QK_B(j+1) ..., each MMA covering both CTAs' rows (M = 256), each
        // commit arriving in both CTAs.
        if (lane == 0) {
            const uint32_t idesc_qk = make_idesc(kBF ? 1 : 0, kBF ? 1 : 0, 256, 128);
            const uint32_t idesc_pv = make_idesc_bmn(kBF ? 1 : 0, kBF ? 1 : 0, 256, DH);
            constexpr uint16_t kBoth = 3;  // commit multicast to both CTAs of the pair
            Ring kring, vring;
            uint32_t qphase = 0;
            uint32_t pphase[2] = {0, 0};
            int nonempty[2] = {0, 0};  // earlier items in which tile A / B had rows
            long long issued_any = 0;
            bool ok = true;
            // S_X = Q_X K^T: A = Q [dim half][128 rows][128 B] of each CTA, B = K
            // [dim half][64 keys][128 B] of each CTA (N = 128 keys).
            auto qk = [&](int x) {
                const uint64_t dq = sw128_kmajor_desc(base + L::q + x * L::kQTile);
                const uint64_t dk = sw128_kmajor_desc(base + L::k16 + kring.idx * L::kK16);
                tc_mma_pair_f16_ss_k8<kHalfTile, kHalf64>(tmem + col_s(x), dq, dk, idesc_qk, 0u);
                tc_commit_pair(bar(L::bSFull + x), kBoth);
                ++issued_any;
            };
            // O_X (+)= P_X V: A = P_X from each CTA's TMEM, B = V [key][64 dims
            // of 128 B] of each CTA, MN-major (N = 128 dims, 64 per CTA).
            auto pv = [&](int x, bool accumulate) -> bool {
                // The first O_X write of an item waits for the epilogue of the
                // previous item that used O_X.
                if (!accumulate && nonempty[x] > 0 &&
                    !wait_or_abort_cl<kDiag>(bar(L::bOEmpty + x), (uint32_t)((nonempty[x] - 1) & 1), flag_addr,
                                             p.status, p.wait_cycles))
                    return false;
                if (!wait_or_abort_cl<kDiag>(bar(L::bPFull + x), pphase[x], flag_addr, p.status, p.wait_cycles))
                    return false;
                pphase[x] ^= 1u;
                tc_fence_after();
                // (one 64-column block per CTA: the leading byte offset is unused)
                const uint64_t dv = sw128_mnmajor_desc(base + L::vr + vring.idx * L::kRawV, 16u);
                tc_mma_pair_f16_ts_mn_k8(tmem + col_o<DH>(x), tmem + col_s(x), dv, idesc_pv, accumulate ? 1u : 0u);
                ++issued_any;
                return true;
            };
            for (int rnd = 0, t = pair_id; t < n_items && ok; t = item_at(++rnd, pair_id, n_pairs)) {
                const Item it = load_item(items, t);
                const int nA = tile_nkv(it.t0, 0, TQ2, it.qo_len, it.kv_len);
                const int nB = tile_nkv(it.t0, 1, TQ2, it.qo_len, it.kv_len);
                const int n = it.nkv;
                ok = wait_or_abort_cl<kDiag>(bar(L::bQFull), qphase, flag_addr, p.status, p.wait_cycles);
                qphase ^= 1u;
                if (!ok) break;
                tc_fence_after();
                // K tile 0 for both query tiles.
                ok = wait_or_abort_cl<kDiag>(bar(L::bK16Full + kring.idx), kring.phase, flag_addr, p.status,
                                             p.wait_cycles);
                if (!ok) break;
                tc_fence_after();
                if (nA > 0) qk(0);
                if (nB > 0) qk(1);
                tc_commit_pair(bar(L::bK16Empty + kring.idx), kBoth);
                kring.next(L::NK16);
                if (n == 1) tc_commit_pair(bar(L::bQEmpty), kBoth);
                for (int j = 0; j < n && ok; ++j) {
                    ok = wait_or_abort_cl<kDiag>(bar(L::bVReady + vring.idx), vring.phase, flag_addr, p.status,
                                                 p.wait_cycles);
                    if (!ok) break;
                    tc_fence_after();
                    if (j < nA) {
                        if (!(ok = pv(0, j > 0))) break;
                        if (j == nA - 1) tc_commit_pair(bar(L::bOFull + 0), kBoth);
                    }
                    const bool more = j + 1 < n;
                    if (more) {
                        ok = wait_or_abort_cl<kDiag>(bar(L::bK16Full + kring.idx), kring.phase, flag_addr, p.status,
                                                     p.wait_cycles);
                        if (!ok) break;
                        tc_fence_after();
                        if (j + 1 < nA) qk(0);
                    }
                    if (j < nB) {
                        if (!(ok = pv(1, j > 0))) break;
                        if (j == nB - 1) tc_commit_pair(bar(L::bOFull + 1), kBoth);
                    }
                    tc_commit_pair(bar(L::bVrEmpty + vring.idx), kBoth);
                    vring.next(L::NVR);
                    if (more) {
                        if (j + 1 < nB) qk(1);
                        tc_commit_pair(bar(L::bK16Empty + kring.idx), kBoth);
                        kring.next(L::NK16);
                        if (j + 1 == n - 1) tc_commit_pair(bar(L::bQEmpty), kBoth);
                    }
                }
                nonempty[0] += nA > 0;
                nonempty[1] += nB > 0;
            }
            // Drain: every MMA issued above completes before TMEM is freed.
            if (issued_any > 0) {
                tc_commit_pair(bar(L::bDrain), 1);
                mbar_wait(bar(L::bDrain), 0);
            }
        }
        __syncwarp();
      }
    } else if (warp < 4) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 64;" ::: "memory");
        // ------------------------------------------------------- V release
        // Each V tile is read by the P V MMAs as it landed.  In a request's last
        // tile the keys past its end (the tail of its last page, and rows no
        // page of this tile filled) are zeroed first -- thread t takes key row
        // t -- so that P = 0 there never meets a stray non-finite value.  Both
        // CTAs arrive on the leader's barrier.
        Ring vr;
        bool ok = true;
        for (int rnd = 0, t = pair_id; t < n_items && ok; t = item_at(++rnd, pair_id, n_pairs)) {
            const Item it = load_item(items, t);
            for (int j = 0; j < it.nkv && ok; ++j) {
                const int valid = min(kTileKeys, it.kv_len - j * kTileKeys);
                ok = wait_or_abort<kDiag>(bar(L::bVrFull + vr.idx), vr.phase, flag_addr, p.status, p.wait_cycles);
                if (!ok) break;
                if (valid < kTileKeys) {
                    if ((int)threadIdx.x >= valid) {
                        const uint32_t row = base + L::vr + vr.idx * L::kRawV + threadIdx.x * 128u;
#pragma unroll
                        for (int c = 0; c < 8; ++c) sts128(row + 16u * c, 0u, 0u, 0u, 0u);
                    }
                    fence_async_smem();
                }
                warp_arrive_cluster(lbar(L::bVReady + vr.idx));
                vr.next(L::NVR);
            }
        }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 192;" ::: "memory");
        // ---------------------------------------------------------- softmax
        // prefill.cuh's softmax on this CTA's 128 rows of query tile x (its
        // TMEM lanes hold them); P and the release of O go to the leader's
        // barriers, one arrive per warp.
        const int x = warp < 8 ? 0 : 1;
        const int r = threadIdx.x - 128 * (1 + x);
        const uint32_t lane_base = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
        const uint32_t tS = lane_base + col_s(x), tO = lane_base + col_o<DH>(x);
        uint32_t sphase = 0, ophase = 0;
        uint32_t stage_round = 0;  // staged epilogues of this tile so far
        const bool issuer = r == 0;
        const bool o_32b = (reinterpret_cast<uintptr_t>(p.o) & 31u) == 0;  // rows are 256 B apart
        bool ok = true;
        Item it_next = pair_id < n_items ? load_item(items, pair_id) : Item{};
        for (int rnd = 0, t = pair_id; t < n_items && ok; t = item_at(++rnd, pair_id, n_pairs)) {
            const Item it = it_next;
            const int qo0 = it.qo0;
            const int qo_len = it.qo_len;
            const int kv_len = it.kv_len;
            const int t0 = it.t0 + x * TQ2 + (int)rank * TQ;         // this CTA's first token of tile x
            const int nX = tile_nkv(it.t0, x, TQ2, qo_len, kv_len);  // the pair's KV tiles for tile x
            const int tok = r / g, hh = r - tok * g;
            const bool valid_row = (tok < TQ) && (t0 + tok < qo_len);
            const int limit = valid_row ? t0 + tok + kv_len - qo_len : -1;
            float scale = p.sm_scale_log2;
            float vsc = p.v_scale;
            if (p.k_scales != nullptr) {  // per-head scale tensors
                const int qh = it.hk * g + min(hh, g - 1);
                scale = fold_scale_log2(p.sm_scale, p.q_scales != nullptr ? __ldg(p.q_scales + qh) : 1.0f,
                                        __ldg(p.k_scales + it.hk));
                vsc = __ldg(p.v_scales + it.hk);
            }
            float m = -INFINITY, l = 0.f;  // m in scaled (log2) units
            for (int j = 0; j < nX && ok; ++j) {
                ok = __all_sync(0xFFFFFFFFu,
                                wait_or_abort<kDiag>(bar(L::bSFull + x), sphase, flag_addr, p.status, p.wait_cycles));
                sphase ^= 1u;
                if (!ok) break;
                tc_fence_after();
                const int key0 = j * kTileKeys;
                const bool need_mask = key0 + kTileKeys - 1 > limit;
                uint32_t v[128];
#pragma unroll
                for (int c = 0; c < 4; ++c) tc_ld32(tS + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(v + 32 * c));
                tc_wait_ld();
                if (need_mask) {
                    const int lim = limit - key0;
#pragma unroll
                    for (int i = 0; i < 128; ++i)
                        if (i > lim) v[i] = __float_as_uint(-INFINITY);
                }
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
                if (__any_sync(0xFFFFFFFFu, rescale)) {
                    // O_X += P_X V of the previous KV tile has completed (in-order
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
                            split_f32x2(mul2(make_f32x2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1])), alpha2),
                                        a, b);
                            v[2 * i] = __float_as_uint(a);
                            v[2 * i + 1] = __float_as_uint(b);
                        }
                        tc_st32(tO + 32 * c, v);
                    }
                    tc_wait_st();
                }
                // P = exp2(s * scale - m) over the first half of S in TMEM.
                const f32x2 scale2 = make_f32x2(scale, scale), negm2 = make_f32x2(-m_use, -m_use);
                f32x2 ps[2] = {make_f32x2(0.f, 0.f), make_f32x2(0.f, 0.f)};
#pragma unroll
                for (int i = 0; i < 64; ++i) {
                    float a, b;
                    split_f32x2(fma2(make_f32x2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1])), scale2, negm2),
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
                warp_arrive_cluster(lbar(L::bPFull + x));
                m = m_use;
            }
            if (!ok) break;
            // The next item's record, loaded here so that its latency passes
            // during the epilogue rather than before the next item's first pass.
            {
                const int tn = item_at(rnd + 1, pair_id, n_pairs);
                if (tn < n_items) it_next = load_item(items, tn);
            }
            if (nX == 0) continue;  // tile B past the request's last row
            // epilogue: the tile's last O update must have completed.
            ok = __all_sync(0xFFFFFFFFu,
                            wait_or_abort<kDiag>(bar(L::bOFull + x), ophase, flag_addr, p.status, p.wait_cycles));
            ophase ^= 1u;
            if (!ok) break;
            tc_fence_after();
            const float inv = valid_row && l > 0.f ? vsc / l : 0.f;
            const size_t orow = (size_t)(qo0 + t0 + tok) * p.num_qo_heads + (size_t)it.hk * g + hh;
            if (t0 + TQ <= qo_len) {
                // A full tile: O normalized into this tile's staging (both 64-dim
                // halves), then two bulk tensor stores by thread 0, which first
                // made sure the previous stores from this staging have read it.
                const uint32_t stg = base + L::ostage + (uint32_t)x * L::kStage;
                if (issuer) {
                    bulk_wait_read_all();
                    mbar_arrive(bar(L::bStageFree + x));
                }
                ok = __all_sync(0xFFFFFFFFu, wait_or_abort<kDiag>(bar(L::bStageFree + x), stage_round & 1u, flag_addr,
                                                                  p.status, p.wait_cycles));
                if (!ok) break;
                const f32x2 inv2 = make_f32x2(inv, inv);
                // 32 columns (dims) at a time: 16 packed words, four 16-byte chunks
                // of this row in dim half q >> 1.
#pragma unroll 1
                for (int q = 0; q < 4; ++q) {
                    uint32_t v[32];
                    tc_ld32(tO + 32 * q, v);
                    tc_wait_ld();
                    if (q == 3) {
                        // O_X is read: release it to the next item's first PV.
                        tc_fence_before();
                        warp_arrive_cluster(lbar(L::bOEmpty + x));
                    }
                    uint32_t w[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        float a0, a1;
                        split_f32x2(mul2(make_f32x2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1])), inv2),
                                    a0, a1);
                        w[i] = pack_out2(a0, a1, p.o_dtype);
                    }
                    const uint32_t row = stg + (uint32_t)(q >> 1) * kHalfTile + (uint32_t)r * 128u;
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const int chunk = 4 * (q & 1) + c;
                        sts128(row + ((chunk ^ (r & 7)) << 4), w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
                    }
                }
                fence_async_smem();
                mbar_arrive(bar(L::bStageReady + x));
                if (issuer) {
                    ok = wait_or_abort<kDiag>(bar(L::bStageReady + x), stage_round & 1u, flag_addr, p.status,
                                              p.wait_cycles);
                    if (ok) {
                        tma_store_3d(&tmo, stg, 0, it.hk * g, qo0 + t0);
                        tma_store_3d(&tmo, stg + kHalfTile, 64, it.hk * g, qo0 + t0);
                        bulk_commit();
                    }
                }
                ok = __all_sync(0xFFFFFFFFu, ok);
                ++stage_round;
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
                        split_f32x2(mul2(make_f32x2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1])), inv2), a,
                                    b);
                        w[i] = pack_out2(a, b, p.o_dtype);
                    }
                    uint16_t* dst = static_cast<uint16_t*>(p.o) + orow * DH + 32 * c;
                    if (o_32b) {
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
            warp_arrive_cluster(lbar(L::bOEmpty + x));
        }
    }

    // Neither CTA frees its TMEM or shared memory while the pair's MMAs or
    // copies may still touch them: the leader's MMA thread has drained, its
    // producer has seen both CTAs' copies land, and each tile's store issuer
    // waits for its bulk stores here.
    if ((warp == 4 || warp == 8) && lane == 0) bulk_wait_all();
    __syncwarp();
    tc_fence_before();
    cluster_sync_all();
    if (warp == 13) {
        tc_fence_after();
        tc_dealloc_pair(tmem, kTmemCols);
    }
}

template <int KT, bool kDiag, bool kSlots>
cudaError_t launch_pair_t(const PrefillParams& p, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                          const CUtensorMap& to, int num_ctas, cudaStream_t stream) {
    auto kern = prefill_pair_kernel<KT, kDiag, kSlots>;
    const size_t smem = 1024 + PairLayout::bytes;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int pairs = max(1, num_ctas / 2);
    cfg.gridDim = dim3(2 * pairs, 1, 1);
    // The pairs are persistent: no more of them than fit on the device at
    // once (a pair takes two SMs of one GPC), or the rest would start only
    // when a resident pair has finished all its items.  Queried once per
    // device and instantiation.
    static int max_pairs[16] = {};
    int dev = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    int& mp = max_pairs[dev & 15];
    if (mp == 0) {
        int n = 0;
        if ((e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg)) != cudaSuccess) return e;
        mp = max(1, n);
    }
    if (pairs > mp) {
        pairs = mp;
        cfg.gridDim = dim3(2 * pairs, 1, 1);
    }
    return cudaLaunchKernelEx(&cfg, kern, p, tq, tk, tv, to);
}

// A 2-byte cache at head_dim 128 (the query has the cache's dtype).  The
// diagnostic instantiation runs only under a shortened wait bound; pages of
// 16 tokens and of 16 m tokens have one each.
template <int KT>
cudaError_t launch_pair_one(const PrefillParams& p, const CUtensorMap& tq, const CUtensorMap& tk,
                            const CUtensorMap& tv, const CUtensorMap& to, int num_ctas, cudaStream_t stream) {
    if (p.wait_cycles < kWaitCyclesDefault) return launch_pair_t<KT, true, true>(p, tq, tk, tv, to, num_ctas, stream);
    return p.page_mult != 1 ? launch_pair_t<KT, false, true>(p, tq, tk, tv, to, num_ctas, stream)
                            : launch_pair_t<KT, false, false>(p, tq, tk, tv, to, num_ctas, stream);
}

inline cudaError_t launch_prefill_pair(const PrefillParams& p, const CUtensorMap& tmap_q, const CUtensorMap& tmap_k,
                                       const CUtensorMap& tmap_v, const CUtensorMap& tmap_o, int num_ctas,
                                       cudaStream_t stream) {
    switch (p.kv_dtype) {
        case PAFP8_F16: return launch_pair_one<PAFP8_F16>(p, tmap_q, tmap_k, tmap_v, tmap_o, num_ctas, stream);
        case PAFP8_BF16: return launch_pair_one<PAFP8_BF16>(p, tmap_q, tmap_k, tmap_v, tmap_o, num_ctas, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace
}  // namespace pafp8
