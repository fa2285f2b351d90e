// internal.h -- declarations shared by the host code and the kernels of
// libpafp8 (not part of the public ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/pafp8.h"

namespace pafp8 {

constexpr int kHeadDim = 128;   // head_dim served by this library
constexpr int kPageSize = 16;   // page_size served by this library
constexpr int kMaxGroupDecode = 8;
constexpr int kMaxGroupPrefill = 16;
constexpr int kTileRows = 128;   // prefill query rows (token x head) per tile
constexpr int kTileKeys = 128;   // prefill keys per KV tile (8 pages)
// Default bound of a kernel's pipeline waits, in SM clock cycles (~1 s).
constexpr long long kWaitCyclesDefault = 2000000000LL;

// Layout of the int32 partition metadata that the plan builds on the host and
// uploads to the head of the workspace.  Word offsets of the variable-length
// arrays are stored in the header.
enum MetaHeader : int {
    kMetaMagic = 0,      // 0x38464150 ("PAF8" little-endian)
    kMetaMode,           // 0 decode, 1 prefill
    kMetaBatch,
    kMetaHeadBlocks,     // number of KV-head blocks (nhb)
    kMetaHeadsPerCta,    // KV heads per block (hpc)
    kMetaGroup,          // query heads per KV head
    kMetaNumCtas,        // persistent CTAs of the main kernel (0: no launch)
    kMetaNumSegs,
    kMetaNumPartials,
    kMetaNumMerge,
    kMetaOffReqPage,     // int32[batch]   first entry of the request in kv_indices
    kMetaOffReqKvLen,    // int32[batch]   kv_len of the request
    kMetaOffCtaSeg,      // int32[num_ctas+1] CSR of segments per CTA
    kMetaOffSeg,         // int32[4*num_segs] (row, page_begin, page_end, out_slot)
    kMetaOffMergePtr,    // int32[num_merge+1]
    kMetaOffMergeRow,    // int32[num_merge]
    kMetaOffMergeSlot,   // int32[num_partials]
    kMetaOffReqQo,       // int32[batch+1] qo_indptr (prefill)
    kMetaNumTiles,       // prefill tiles
    kMetaOffTile,        // int32[8*num_tiles] prefill items: b, hk, t0, nkv, qo_begin, qo_len, kv_len, page_begin
    kMetaTileRows,       // packed query rows per prefill tile
    kMetaOffRowMerge,    // int32[rows] merge entry of each decode row, or -1
    kMetaNumChunks,      // decode pages handed out at run time, in chunks
    kMetaOffChunk,       // int32[4*num_chunks] (row, page_begin, page_end, out_slot)
    kMetaHeaderWords = 32
};

// Decode work handed out at run time: the last 1/kDynDiv of every row's
// pages, cut into chunks of about 1/kDynChunksPerCta of a CTA's share of
// them, when the batch has at least kDynMinPagesPerCta pages per CTA and at
// least one row per kDynMinRowsDiv CTAs (with fewer, longer rows the chunks
// would add many partial states to each row and slow its merge).  Each CTA
// takes chunks from a counter in the workspace after its own pages; a row's
// chunks add one or two partial states to it.
constexpr int kDynDiv = 16;
constexpr int kDynChunksPerCta = 1;
constexpr int kDynMinChunk = 4;
constexpr int kDynMinPagesPerCta = 16;
constexpr int kDynMinRowsDiv = 4;
// Word offsets in the workspace's 256-byte status block: the status word,
// the chunk counter and the count of CTAs done with chunks (both reset by the
// last CTA of each launch).
constexpr int kStatusWord = 0, kChunkCounterWord = 32, kChunkDoneWord = 48;
constexpr int32_t kMetaMagicValue = 0x38464150;

// log2-domain softmax scale of one head from per-head scales, folded in
// double in the same order as the host folds the per-tensor ones, so equal
// scales give the same float.
__device__ __forceinline__ float fold_scale_log2(float sm_scale, float q_scale, float k_scale) {
    return (float)((double)sm_scale * (double)q_scale * (double)k_scale * 1.4426950408889634);
}

// A request's 16-token sub-page vp (a page of 16 m tokens is m of them) as
// TMA coordinates: the pool page holding it and its first token slot there
// (the cache maps span whole pages, page_size slots; sub-page j of a page
// starts at slot 16 j).  A page id outside [0, num_pages) reads page 0 and
// sets `bad`.
struct SubPageAt {
    int slot, page;
};
__device__ __forceinline__ SubPageAt sub_page(const int32_t* idx, int vp, int m, int num_pages, bool& bad) {
    const int e = m == 1 ? vp : vp / m;
    const int pg = __ldg(idx + e);
    bad = pg < 0 || pg >= num_pages;
    return SubPageAt{(vp - e * m) * kPageSize, bad ? 0 : pg};
}

// Status word bits written by the kernels into the workspace.
enum : uint32_t {
    kStatusBounds = 1u,   // a page index outside [0, num_pages)
    kStatusTimeout = 2u,  // a bounded mbarrier wait expired
};

struct DecodeParams {
    const void* q;           // [batch, Hq, D]
    const int32_t* kv_indices;
    void* o;                 // [batch, Hq, D]
    float* lse;              // [batch, Hq] or nullptr
    const int32_t* meta;     // device copy of the metadata words
    float* part_o;           // [num_partials, hpc*group, D]
    float* part_lse;         // [num_partials, hpc*group] (log2 domain)
    uint32_t* status;        // status block: status word, chunk counter, CTAs done
    int head_dim;            // 128 or 64
    int q_dtype, kv_dtype, o_dtype;
    int num_qo_heads, num_kv_heads, num_pages;
    int page_mult;           // page_size / 16: a page is read as page_mult 16-token sub-pages
    float sm_scale_log2;     // sm_scale * q_scale * k_scale * log2(e)
    float v_scale;
    // Per-head scale tensors (device arrays) instead of the per-tensor scales
    // folded above, when k_scales is not null: q_scales [Hq] (or null: 1),
    // k_scales and v_scales [Hkv]; the kernels fold sm_scale with them.
    const float* q_scales;
    const float* k_scales;
    const float* v_scales;
    float sm_scale;
    long long wait_cycles;   // bound of a pipeline wait (SM clock cycles)
};

struct AppendParams {
    const void* k_new;       // [nnz, Hkv, D] of src_dtype
    const void* v_new;
    const int32_t* batch_indices;  // [nnz]
    const int32_t* positions;      // [nnz]
    const int32_t* kv_indptr;      // [batch + 1]
    const int32_t* kv_indices;
    void* k_cache;           // [num_pages, page_size, Hkv, D] of kv_dtype (fp8)
    void* v_cache;
    uint32_t* status;        // or nullptr
    long long nnz;
    int num_kv_heads, batch, num_pages;
    int src_dtype, kv_dtype;
    int hnd;                 // cache layout: 0 [page][slot][head][d], 1 [page][head][slot][d]
    int page_size;
    int head_dim;            // 128 or 64
    float k_inv, v_inv;      // fp32(1 / scale)
};

struct PrefillParams {
    const void* q;           // [nnz_qo, Hq, D]
    int head_dim;            // D: 128 or 64
    const int32_t* kv_indices;
    void* o;                 // [nnz_qo, Hq, D]
    float* lse;              // [nnz_qo, Hq] or nullptr
    const int32_t* meta;     // device copy of the metadata words
    uint32_t* status;
    int q_dtype, kv_dtype, o_dtype;
    int num_qo_heads, num_kv_heads, num_pages;
    int page_mult;           // page_size / 16: a page is read as page_mult 16-token sub-pages
    int group;               // query heads per KV head
    int tile_tokens;         // query tokens per 128-row tile (128 / group)
    float sm_scale_log2;     // sm_scale * q_scale * k_scale * log2(e)
    float v_scale;
    // Per-head scale tensors (device arrays) instead of the per-tensor scales
    // folded above, when k_scales is not null: q_scales [Hq] (or null: 1),
    // k_scales and v_scales [Hkv]; the kernels fold sm_scale with them.
    const float* q_scales;
    const float* k_scales;
    const float* v_scales;
    float sm_scale;
    long long wait_cycles;   // bound of a pipeline wait (SM clock cycles)
};

// Launchers (decode.cu, prefill_d128.cu / prefill_d64.cu).  Return the launch's cudaError_t.
// heads_per_box: KV heads covered by one TMA box of the cache maps (the
// whole head block when the page-wide map could be encoded, else 1).
cudaError_t launch_decode(const DecodeParams& p, const CUtensorMap& tmap_k,
                          const CUtensorMap& tmap_v, int num_ctas, int heads_per_cta,
                          int group, int heads_per_box, cudaStream_t stream);
cudaError_t launch_append(const AppendParams& p, cudaStream_t stream);
// Size of the built-in scratch of the no-allocation decode entry point, and
// the device ordinals it serves.
constexpr size_t kNoAllocScratchBytes = PAFP8_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;
// Device address of the built-in scratch on the current device (looked up
// once per device; decode.cu).
cudaError_t noalloc_scratch(void** ptr);

cudaError_t launch_merge(const DecodeParams& p, int num_merge, int heads_per_cta, int group,
                         cudaStream_t stream);
// tmap_o: map over o with the 2-byte query tile's box (the fp8-query kernel
// writes full output tiles with bulk tensor stores through it).  One
// translation unit per head size (prefill_d128.cu, prefill_d64.cu).
cudaError_t launch_prefill_d128(const PrefillParams& p, const CUtensorMap& tmap_q,
                                const CUtensorMap& tmap_k, const CUtensorMap& tmap_v,
                                const CUtensorMap& tmap_o, int num_ctas, cudaStream_t stream);
cudaError_t launch_prefill_d64(const PrefillParams& p, const CUtensorMap& tmap_q,
                               const CUtensorMap& tmap_k, const CUtensorMap& tmap_v,
                               const CUtensorMap& tmap_o, int num_ctas, cudaStream_t stream);
inline cudaError_t launch_prefill(const PrefillParams& p, const CUtensorMap& tmap_q,
                                  const CUtensorMap& tmap_k, const CUtensorMap& tmap_v,
                                  const CUtensorMap& tmap_o, int num_ctas, cudaStream_t stream) {
    return p.head_dim == 64 ? launch_prefill_d64(p, tmap_q, tmap_k, tmap_v, tmap_o, num_ctas, stream)
                            : launch_prefill_d128(p, tmap_q, tmap_k, tmap_v, tmap_o, num_ctas, stream);
}

}  // namespace pafp8
