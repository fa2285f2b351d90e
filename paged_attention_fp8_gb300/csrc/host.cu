// host.cu -- the C ABI of libpafp8: validation and refusal sentences, the
// split-KV plan scheduler, metadata upload and kernel dispatch.
//
// Refusals follow "fp8 KV cache in the in-tree prefill kernel", What changed /
// Refusals and Test plan (refusals): every combination the kernels cannot
// serve returns a status with a sentence naming the dtypes, k and v dtypes
// must match at every run, and integer caches are refused rather than read as
// values.  The o_data_type contract (fixed at plan, checked at run; fp8
// outputs refused) follows "Enable Hopper FA3 FP8 attention in decode.py",
// Changes table and the module-validation review note.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "../../include/pafp8.h"
#include "internal.h"

using namespace pafp8;

namespace {

thread_local std::string g_last_error;

pafp8_status fail(pafp8_status st, const char* fmt, ...) {
    char buf[1024];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return st;
}

const char* dtype_name(int32_t dt) {
    switch (dt) {
        case PAFP8_F16: return "float16";
        case PAFP8_BF16: return "bfloat16";
        case PAFP8_E4M3FN: return "float8_e4m3fn";
        case PAFP8_E5M2: return "float8_e5m2";
        case PAFP8_F32: return "float32";
        case PAFP8_INT8: return "int8";
        case PAFP8_UINT8: return "uint8";
        case PAFP8_DTYPE_DEFAULT: return "default";
        default: return "unknown";
    }
}

bool is_fp8(int32_t dt) { return dt == PAFP8_E4M3FN || dt == PAFP8_E5M2; }
bool is_2byte(int32_t dt) { return dt == PAFP8_F16 || dt == PAFP8_BF16; }

// The cache dtype.  fp8 everywhere; a 2-byte cache (f16/bf16) with a 2-byte
// query: in decode any mix ("fp8 KV cache in the in-tree prefill kernel",
// Test plan: decode is exempt from the rule that the cache matches the
// query), in prefill the query's own dtype; never with an fp8 query.
pafp8_status check_kv_dtype(int32_t kv, const char* what, int32_t mode, int32_t q) {
    if (is_fp8(kv)) return PAFP8_OK;
    if (is_2byte(kv)) {
        if (is_fp8(q))
            return fail(PAFP8_ERR_DTYPE,
                        "%s has dtype %s but q is %s: an fp8 query needs an fp8 cache (the QK "
                        "product runs on the tensor cores in one operand type)",
                        what, dtype_name(kv), dtype_name(q));
        if (mode == PAFP8_MODE_PREFILL && kv != q)
            return fail(PAFP8_ERR_DTYPE,
                        "%s has dtype %s but q is %s: prefill takes a 2-byte cache only of the "
                        "query's own dtype (decode accepts either mix)",
                        what, dtype_name(kv), dtype_name(q));
        return PAFP8_OK;
    }
    if (kv == PAFP8_INT8 || kv == PAFP8_UINT8)
        return fail(PAFP8_ERR_DTYPE,
                    "%s has dtype %s: an integer cache has no floating-point reading, and this "
                    "library refuses it rather than reading its bytes as fp8 or as 0..255 values; "
                    "the cache must be float8_e4m3fn or float8_e5m2",
                    what, dtype_name(kv));
    if (kv == PAFP8_F32)
        return fail(PAFP8_ERR_DTYPE,
                    "%s has dtype float32, which is not served; the cache must be "
                    "float8_e4m3fn or float8_e5m2",
                    what);
    return fail(PAFP8_ERR_DTYPE, "%s has an unknown dtype code %d", what, (int)kv);
}

pafp8_status check_q_dtype(int32_t q) {
    if (is_2byte(q) || is_fp8(q)) return PAFP8_OK;
    if (q == PAFP8_INT8 || q == PAFP8_UINT8 || q == PAFP8_F32)
        return fail(PAFP8_ERR_DTYPE,
                    "q has dtype %s, which is not served; the query must be float16, bfloat16, "
                    "float8_e4m3fn or float8_e5m2",
                    dtype_name(q));
    return fail(PAFP8_ERR_DTYPE, "q has an unknown dtype code %d", (int)q);
}

pafp8_status check_o_dtype(int32_t o, int32_t q) {
    if (is_2byte(o)) return PAFP8_OK;
    if (is_fp8(o))
        return fail(PAFP8_ERR_DTYPE,
                    "o_data_type %s is refused: fp8 outputs are not produced; with q %s and an "
                    "fp8 cache the output must be float16 or bfloat16",
                    dtype_name(o), dtype_name(q));
    return fail(PAFP8_ERR_DTYPE,
                "o_data_type %s is not served; the output must be float16 or bfloat16",
                dtype_name(o));
}

int heads_per_cta_for(int hkv) {
    int best = 1;
    for (int d = 1; d <= 8; ++d)
        if (hkv % d == 0) best = d;
    return best;
}

}  // namespace

struct pafp8_plan {
    pafp8_plan_desc desc;    // with defaults resolved
    std::vector<int32_t> kv_indptr, last_page_len, qo_indptr;
    std::vector<int32_t> meta;
    int64_t nnz_pages = 0, nnz_qo = 0;
    int heads_per_cta = 1, head_blocks = 1, group = 1;
    // Pages of page_size = 16 * page_mult tokens are read as page_mult
    // consecutive 16-token sub-pages; vptr is the CSR of sub-pages per
    // request (ceil(kv_len / 16)), the unit of the decode partition.
    int page_mult = 1;
    std::vector<int32_t> vptr;
    int num_ctas = 0, num_partials = 0, num_merge = 0;
    size_t meta_bytes = 0, part_o_off = 0, part_lse_off = 0, status_off = 0, ws_bytes = 0;
    void* uploaded_ws = nullptr;
    // Side stream and fork/join events of pafp8_run_pod for a decode plan,
    // created by its first call.
    mutable cudaStream_t pod_stream = nullptr;
    mutable cudaEvent_t pod_fork = nullptr, pod_join = nullptr;
    ~pafp8_plan() {
        if (pod_join != nullptr) cudaEventDestroy(pod_join);
        if (pod_fork != nullptr) cudaEventDestroy(pod_fork);
        if (pod_stream != nullptr) cudaStreamDestroy(pod_stream);
    }
};

namespace {

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Device staging of pafp8_run_host, after the plan's own workspace bytes: q,
// kv_indices, o and lse, each 256-byte aligned.
struct HostStaging {
    size_t q, idx, o, lse, end;
    size_t q_bytes, idx_bytes, o_bytes, lse_bytes;
};
HostStaging host_staging(const pafp8_plan* plan, int32_t q_dtype) {
    const pafp8_plan_desc& d = plan->desc;
    HostStaging h{};
    const size_t rows = (size_t)plan->nnz_qo * (size_t)d.num_qo_heads;
    h.q_bytes = rows * (size_t)d.head_dim * (is_fp8(q_dtype) ? 1 : 2);
    h.idx_bytes = plan->kv_indptr.empty() ? 0 : (size_t)plan->kv_indptr.back() * 4;
    h.o_bytes = rows * (size_t)d.head_dim * 2;
    h.lse_bytes = rows * 4;
    h.q = align_up(plan->ws_bytes, 256);
    h.idx = align_up(h.q + h.q_bytes, 256);
    h.o = align_up(h.idx + h.idx_bytes, 256);
    h.lse = align_up(h.o + h.o_bytes, 256);
    h.end = h.lse + h.lse_bytes;
    return h;
}

// Decode partition.  Rows are (request b, KV-head block hb), row r = b*nhb + hb,
// each holding the npages[b] pages of its request.  The rule:
//   disable_split_kv: one segment per non-empty row; CTA i takes segments
//                     i, i+G, i+2G, ... (G = min(num_ctas, #segments));
//   fixed_split_pages c: rows cut into chunks of c pages, dealt the same way;
//   balanced (default): with T the total pages over all rows and
//                     G = min(num_ctas, T), CTA i takes the global page range
//                     [floor(i*T/G), floor((i+1)*T/G)) of the rows laid end to
//                     end, cut at row boundaries into segments.
// Rows with no pages get a zero-page segment (written as o = 0, lse = -inf)
// dealt round-robin after the other segments, and each CTA runs its partial
// segments first.  A segment spanning its whole row writes the final output
// (slot -1); every other segment writes a partial state to the next free slot
// (in final segment order); a merge kernel combines the partial states of
// every row with two or more segments.
void build_decode_meta(pafp8_plan* pl) {
    const int B = pl->desc.batch;
    const int nhb = pl->head_blocks;
    const int R = B * nhb;
    std::vector<int32_t> np((size_t)R);
    std::vector<int32_t> empty;  // rows with no pages, ascending
    int64_t T = 0;
    for (int b = 0; b < B; ++b)
        for (int hb = 0; hb < nhb; ++hb) {
            const int32_t n = pl->vptr[b + 1] - pl->vptr[b];
            np[(size_t)b * nhb + hb] = n;
            T += n;
            if (n == 0) empty.push_back(b * nhb + hb);
        }

    // Segments in their final order, CTA after CTA (cta_ptr is the CSR).  A
    // segment's slot is -1 while it covers its whole row (it writes the final
    // output; zero-page rows too) and 0 for a part, numbered below.
    struct Seg { int32_t row, p0, p1, slot; };
    auto seg_of = [&](int32_t r, int64_t a, int64_t e) {
        return Seg{r, (int32_t)a, (int32_t)e, (a == 0 && e == np[r]) ? -1 : 0};
    };
    std::vector<Seg> segs, chunks;
    std::vector<int32_t> cta_ptr(1, 0);
    const int64_t target = pl->desc.num_ctas;
    int64_t G = 0;
    auto add_empties = [&](int64_t i, int64_t gt) {
        for (size_t k = (size_t)i; k < empty.size(); k += (size_t)gt) segs.push_back({empty[k], 0, 0, -1});
    };
    if (pl->desc.disable_split_kv || pl->desc.fixed_split_pages > 0) {
        std::vector<Seg> all;  // the chunks in row order, dealt round-robin
        for (int r = 0; r < R; ++r) {
            const int64_t c = pl->desc.disable_split_kv ? np[r] : pl->desc.fixed_split_pages;
            for (int64_t a = 0; a < np[r]; a += c)
                all.push_back(seg_of(r, a, std::min<int64_t>(a + c, np[r])));
        }
        G = std::min<int64_t>(target, (int64_t)all.size());
        const int64_t gt = G > 0 ? G : (empty.empty() ? 0 : 1);
        cta_ptr.reserve((size_t)gt + 1);
        segs.reserve(all.size() + empty.size());
        for (int64_t i = 0; i < gt; ++i) {
            for (size_t k = (size_t)i; G > 0 && k < all.size(); k += (size_t)G) segs.push_back(all[k]);
            add_empties(i, gt);
            cta_ptr.push_back((int32_t)segs.size());
        }
        G = gt;
    } else {
        G = std::min<int64_t>(target, T);
        // Each row's last np / kDynDiv pages are handed out at run time in
        // chunks (when the batch qualifies); the rows' first ns pages, laid
        // end to end, are split statically.
        const bool dyn = G > 0 && T >= (int64_t)kDynMinPagesPerCta * G && (int64_t)R * kDynMinRowsDiv >= G;
        std::vector<int32_t> ns((size_t)R);
        int64_t Ts = 0;
        for (int rr = 0; rr < R; ++rr) {
            ns[rr] = dyn ? np[rr] - np[rr] / kDynDiv : np[rr];
            Ts += ns[rr];
        }
        const int64_t Td = T - Ts;
        const int64_t gt = G > 0 ? G : (empty.empty() ? 0 : 1);
        cta_ptr.reserve((size_t)gt + 1);
        segs.reserve((size_t)(G + R + empty.size()));
        int64_t start = 0;  // first global static page of row r
        int r = 0;
        // hi = floor((i + 1) Ts / G) kept as quotient and remainder, one step per CTA
        const int64_t dq = G > 0 ? Ts / G : 0, dr = G > 0 ? Ts % G : 0;
        int64_t hq = 0, hr = 0;
        for (int64_t i = 0; i < gt; ++i) {
            if (G > 0) {
                const int64_t lo = hq;
                hq += dq;
                hr += dr;
                if (hr >= G) {
                    ++hq;
                    hr -= G;
                }
                const int64_t hi = hq;
                while (r < R && start + ns[r] <= lo) start += ns[r++];
                int64_t rs = start;
                for (int rr = r; rr < R && rs < hi; rs += ns[rr++]) {
                    const int64_t a = std::max(lo, rs) - rs;
                    const int64_t e = std::min(hi, rs + ns[rr]) - rs;
                    if (e > a) segs.push_back(seg_of(rr, a, e));
                }
            }
            add_empties(i, gt);
            cta_ptr.push_back((int32_t)segs.size());
        }
        G = gt;
        if (Td > 0) {
            const int64_t per = (int64_t)kDynChunksPerCta * G;
            const int64_t c = std::max<int64_t>(kDynMinChunk, (Td + per - 1) / per);
            for (int rr = 0; rr < R; ++rr)
                for (int64_t a = ns[rr]; a < np[rr]; a += c)
                    chunks.push_back(seg_of(rr, a, std::min<int64_t>(a + c, np[rr])));
        }
    }

    // Within a CTA, segments covering part of their row run first, so the
    // merges of split rows happen early rather than in the kernel's tail.
    auto partial = [](const Seg& sg) { return sg.slot == 0; };
    std::vector<Seg> tmp;
    for (int64_t i = 0; i < G; ++i) {
        Seg* a = segs.data() + cta_ptr[i];
        Seg* e = segs.data() + cta_ptr[i + 1];
        if (e - a < 2) continue;
        tmp.clear();
        for (Seg* x = a; x != e; ++x)
            if (partial(*x)) tmp.push_back(*x);
        for (Seg* x = a; x != e; ++x)
            if (!partial(*x)) tmp.push_back(*x);
        std::copy(tmp.begin(), tmp.end(), a);
    }

    // Chunks follow the static segments (records after cta_ptr[G]) and are
    // numbered with them.
    const int32_t nseg_static = (int32_t)segs.size();
    segs.insert(segs.end(), chunks.begin(), chunks.end());

    // Output slots and the merge lists.  A row cut into two or more segments
    // has only partial ones; its partial states are numbered merge row by
    // merge row (ascending), each row's by first page, so a row's slots are
    // consecutive and the merge reads them without an index list.  Whole-row
    // segments (and zero-page ones) write the final output (slot -1).
    // Bucketed by row (a counting sort), then by first page within each row
    // (insertion sort: a row's segments mostly arrive in page order already).
    std::vector<int32_t> first((size_t)R + 1, 0);
    for (const Seg& sg : segs)
        if (partial(sg)) first[(size_t)sg.row + 1]++;
    for (int r = 0; r < R; ++r) first[(size_t)r + 1] += first[r];
    const int32_t nslot = first[R];
    std::vector<int32_t> parts((size_t)nslot), fill(first.begin(), first.end() - 1);
    for (size_t k = 0; k < segs.size(); ++k)
        if (segs[k].slot == 0) parts[(size_t)fill[segs[k].row]++] = (int32_t)k;
    for (int r = 0; r < R; ++r)
        for (int32_t j = first[r] + 1; j < first[(size_t)r + 1]; ++j)
            for (int32_t i = j; i > first[r] && segs[parts[i - 1]].p0 > segs[parts[i]].p0; --i)
                std::swap(parts[i - 1], parts[i]);
    std::vector<int32_t> merge_rows, merge_ptr(1, 0), row_merge((size_t)R, -1);
    for (int32_t k = 0; k < nslot; ++k) {
        Seg& sg = segs[parts[k]];
        sg.slot = k;
        if (k == 0 || segs[parts[k - 1]].row != sg.row) {
            row_merge[sg.row] = (int32_t)merge_rows.size();
            merge_rows.push_back(sg.row);
        }
        if (k + 1 == nslot || segs[parts[k + 1]].row != sg.row) merge_ptr.push_back(k + 1);
    }
    const int32_t nmerge = (int32_t)merge_rows.size();
    const int32_t nseg = nseg_static;
    const int32_t nchunk = (int32_t)chunks.size();

    std::vector<int32_t>& m = pl->meta;
    m.assign(kMetaHeaderWords, 0);
    m.reserve((size_t)kMetaHeaderWords + 2 * (size_t)B + (size_t)G + 1 + 4 * (size_t)nseg + 2 * (size_t)nmerge + 1 +
              (size_t)nslot + (size_t)R);
    m[kMetaMagic] = kMetaMagicValue;
    m[kMetaMode] = PAFP8_MODE_DECODE;
    m[kMetaBatch] = B;
    m[kMetaHeadBlocks] = nhb;
    m[kMetaHeadsPerCta] = pl->heads_per_cta;
    m[kMetaGroup] = pl->group;
    m[kMetaNumCtas] = (int32_t)G;
    m[kMetaNumSegs] = nseg;
    m[kMetaNumPartials] = nslot;
    m[kMetaNumMerge] = nmerge;
    m[kMetaOffReqPage] = (int32_t)m.size();
    for (int b = 0; b < B; ++b) m.push_back(pl->kv_indptr[b]);
    m[kMetaOffReqKvLen] = (int32_t)m.size();
    for (int b = 0; b < B; ++b) {
        const int32_t n = pl->kv_indptr[b + 1] - pl->kv_indptr[b];
        m.push_back(n > 0 ? (n - 1) * pl->desc.page_size + pl->last_page_len[b] : 0);
    }
    m[kMetaOffCtaSeg] = (int32_t)m.size();
    m.insert(m.end(), cta_ptr.begin(), cta_ptr.end());
    m[kMetaOffSeg] = (int32_t)m.size();
    for (int32_t k = 0; k < nseg; ++k) {
        const Seg& sg = segs[(size_t)k];
        m.push_back(sg.row);
        m.push_back(sg.p0);
        m.push_back(sg.p1);
        m.push_back(sg.slot);
    }
    m[kMetaOffMergePtr] = (int32_t)m.size();
    m.insert(m.end(), merge_ptr.begin(), merge_ptr.end());
    m[kMetaOffMergeRow] = (int32_t)m.size();
    m.insert(m.end(), merge_rows.begin(), merge_rows.end());
    m[kMetaOffMergeSlot] = (int32_t)m.size();
    for (int32_t k = 0; k < nslot; ++k) m.push_back(k);
    m[kMetaOffRowMerge] = (int32_t)m.size();
    m.insert(m.end(), row_merge.begin(), row_merge.end());
    m[kMetaNumChunks] = nchunk;
    m[kMetaOffChunk] = (int32_t)m.size();
    for (int32_t k = nseg; k < nseg + nchunk; ++k) {
        const Seg& sg = segs[(size_t)k];
        m.push_back(sg.row);
        m.push_back(sg.p0);
        m.push_back(sg.p1);
        m.push_back(sg.slot);
    }

    pl->num_ctas = (int)G;
    pl->num_partials = nslot;
    pl->num_merge = nmerge;
}

// Prefill work items: for every request b, KV head hk and block of 2 * TQ
// consecutive new tokens starting at t0 (TQ = 128 / group), one item of two
// query tiles of TQ * group packed rows each.  n_kv = the KV tiles of 128 keys
// the item's last token may see (bottom-right causal).  Items are ordered
// longest first (stable); the kernels deal them to the G persistent CTAs (or
// CTA pairs) in snake order: round r gives worker i item r G + i for even r
// and r G + G - 1 - i for odd r.
// (G = min(num_ctas, #items)).
void build_prefill_meta(pafp8_plan* pl) {
    const int B = pl->desc.batch;
    const int g = pl->group;
    const int TQ = kTileRows / g;
    // A 2-byte cache at head_dim 128 runs on CTA pairs: a query tile is 2 TQ
    // tokens (TQ per CTA), an item two such tiles; the rest on single CTAs
    // (tiles of TQ).
    const bool pair = pl->desc.head_dim == kHeadDim && is_2byte(pl->desc.kv_dtype);
    const int span = (pair ? 4 : 2) * TQ;
    struct T { int32_t b, hk, t0, nkv; };
    std::vector<T> tiles;
    std::vector<int32_t> req_page(B), req_kv(B);
    for (int b = 0; b < B; ++b) {
        req_page[b] = pl->kv_indptr[b];
        const int32_t n = pl->kv_indptr[b + 1] - pl->kv_indptr[b];
        req_kv[b] = n > 0 ? (n - 1) * pl->desc.page_size + pl->last_page_len[b] : 0;
        const int qo = pl->qo_indptr[b + 1] - pl->qo_indptr[b];
        for (int hk = 0; hk < pl->desc.num_kv_heads; ++hk)
            for (int t0 = 0; t0 < qo; t0 += span) {
                // An item is two query tiles, A starting at t0 and B right
                // after; its KV tiles are those of its last token.
                const int last = std::min(t0 + span, qo) - 1;
                const int lim = last + req_kv[b] - qo;
                const int nkv = std::min((req_kv[b] + kTileKeys - 1) / kTileKeys, lim / kTileKeys + 1);
                tiles.push_back({b, hk, t0, nkv});
            }
    }
    std::stable_sort(tiles.begin(), tiles.end(), [](const T& a, const T& c) { return a.nkv > c.nkv; });
    const int G = pair ? 2 * (int)std::min<int64_t>(std::max<int64_t>(1, pl->desc.num_ctas / 2), (int64_t)tiles.size())
                       : (int)std::min<int64_t>(pl->desc.num_ctas, (int64_t)tiles.size());

    std::vector<int32_t>& m = pl->meta;
    m.assign(kMetaHeaderWords, 0);
    auto put = [&](int field, const std::vector<int32_t>& arr) {
        m[field] = (int32_t)m.size();
        m.insert(m.end(), arr.begin(), arr.end());
    };
    m[kMetaMagic] = kMetaMagicValue;
    m[kMetaMode] = PAFP8_MODE_PREFILL;
    m[kMetaBatch] = B;
    m[kMetaHeadBlocks] = pl->desc.num_kv_heads;
    m[kMetaHeadsPerCta] = 1;
    m[kMetaGroup] = g;
    m[kMetaNumCtas] = G;
    m[kMetaNumTiles] = (int32_t)tiles.size();
    m[kMetaTileRows] = TQ;
    put(kMetaOffReqPage, req_page);
    put(kMetaOffReqKvLen, req_kv);
    put(kMetaOffReqQo, pl->qo_indptr);
    // Each item record carries the request fields the kernel needs, so a CTA
    // reads one record per item and no dependent loads.
    std::vector<int32_t> tw;
    for (auto& t : tiles) {
        tw.push_back(t.b);
        tw.push_back(t.hk);
        tw.push_back(t.t0);
        tw.push_back(t.nkv);
        tw.push_back(pl->qo_indptr[t.b]);
        tw.push_back(pl->qo_indptr[t.b + 1] - pl->qo_indptr[t.b]);
        tw.push_back(req_kv[t.b]);
        tw.push_back(req_page[t.b]);
    }
    put(kMetaOffTile, tw);
    pl->num_ctas = G;
    pl->num_partials = 0;
    pl->num_merge = 0;
}

void layout_workspace(pafp8_plan* pl) {
    const size_t heads = (size_t)pl->heads_per_cta * pl->group;
    pl->meta_bytes = align_up(pl->meta.size() * sizeof(int32_t), 256);
    pl->part_o_off = pl->meta_bytes;
    pl->part_lse_off = align_up(pl->part_o_off + (size_t)pl->num_partials * heads * pl->desc.head_dim * 4, 256);
    pl->status_off = align_up(pl->part_lse_off + (size_t)pl->num_partials * heads * 4, 256);
    pl->ws_bytes = pl->status_off + 256;
}

PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (PFN_cuTensorMapEncodeTiled_v12000)p;
    }
    return fn;
}

// Byte strides of a cache tensor [num_pages, page_size, Hkv, D] (NHD) or
// [num_pages, Hkv, page_size, D] (HND) with esz-byte elements.  Every TMA map
// below names the same dimensions (dims, token slot, head, page) and only
// these strides differ, so the boxes land in shared memory the same way for
// both.  The token-slot dimension spans the whole page (page_size slots); a
// box covers 16 of them, and the kernels address the 16-token sub-page j of a
// page by the slot coordinate 16 j.
struct KvStrides {
    cuuint64_t token, head, page;
};
KvStrides kv_strides(int layout, int hkv, int esz, int head_dim, int page_size) {
    const cuuint64_t row = (cuuint64_t)head_dim * esz;
    const cuuint64_t page = (cuuint64_t)page_size * hkv * row;
    if (layout == PAFP8_LAYOUT_HND) return KvStrides{row, (cuuint64_t)page_size * row, page};
    return KvStrides{(cuuint64_t)hkv * row, row, page};
}

// Map over an fp8 cache (bytes; the prefill's, and decode's when it takes one
// box per head), dims listed innermost first: (d, kv head, token slot, page).
// One box is one KV head of one page, 16 tokens x
// head_dim bytes, landing in shared memory as [16][head_dim] with the 128-byte
// swizzle (16-byte chunk c of token row t stored at c ^ (t & 7)), or the
// 64-byte one for 64-byte rows.
pafp8_status encode_cache_map(CUtensorMap* map, const void* base, int num_pages, int hkv, int layout,
                              int head_dim, int page_size) {
    auto enc = get_encode();
    if (!enc) return fail(PAFP8_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    const KvStrides ks = kv_strides(layout, hkv, 1, head_dim, page_size);
    cuuint64_t dims[4] = {(cuuint64_t)head_dim, (cuuint64_t)hkv, (cuuint64_t)page_size,
                          (cuuint64_t)num_pages};
    cuuint64_t strides[3] = {ks.head, ks.token, ks.page};
    cuuint32_t box[4] = {(cuuint32_t)head_dim, 1, (cuuint32_t)kPageSize, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(base), dims, strides,
                     box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     head_dim == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(PAFP8_ERR_CUDA, "cuTensorMapEncodeTiled failed for the KV cache (CUresult %d)",
                    (int)r);
    return PAFP8_OK;
}

// Prefill map over a 2-byte cache: dims (d % 64, d / 64, token, head, page);
// one box is one page of one KV head for one 64-dim half, {64, 1, 16, 1, 1},
// landing as 16 swizzled rows of 128 B (one per token).
pafp8_status encode_cache_map_2byte(CUtensorMap* map, const void* base, int num_pages, int hkv, int layout,
                                    int head_dim, int page_size) {
    auto enc = get_encode();
    if (!enc) return fail(PAFP8_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    const KvStrides ks = kv_strides(layout, hkv, 2, head_dim, page_size);
    cuuint64_t dims[5] = {64, (cuuint64_t)(head_dim / 64), (cuuint64_t)page_size, (cuuint64_t)hkv,
                          (cuuint64_t)num_pages};
    cuuint64_t strides[4] = {128, ks.token, ks.head, ks.page};
    cuuint32_t box[5] = {64, 1, (cuuint32_t)kPageSize, 1, 1};
    cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 5, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(PAFP8_ERR_CUDA, "cuTensorMapEncodeTiled failed for the 2-byte KV cache (CUresult %d)",
                    (int)r);
    return PAFP8_OK;
}

// 3-D map over q [nnz_qo, Hq, D]: dims (d, head, row), innermost first.  One
// box is the query tile of one KV head: `rows` consecutive new tokens x the
// group's heads x 64 elements (2-byte q, one box per 64-dim half of the tile)
// or D elements (fp8 q), landing as [rows*group][128 bytes] under the
// 128-byte swizzle, or [rows*group][64 bytes] under the 64-byte one for an
// fp8 query of head_dim 64.
pafp8_status encode_q_map(CUtensorMap* map, const void* base, int nnz_qo, int hq, int group,
                          int rows, bool fp8, int head_dim) {
    auto enc = get_encode();
    if (!enc) return fail(PAFP8_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    const cuuint64_t es = fp8 ? 1 : 2;
    cuuint64_t dims[3] = {(cuuint64_t)head_dim, (cuuint64_t)hq, (cuuint64_t)nnz_qo};
    cuuint64_t strides[2] = {(cuuint64_t)head_dim * es, (cuuint64_t)hq * head_dim * es};
    cuuint32_t box[3] = {fp8 ? (cuuint32_t)head_dim : 64u, (cuuint32_t)group, (cuuint32_t)rows};
    cuuint32_t estr[3] = {1, 1, 1};
    const bool rows64 = fp8 && head_dim == 64;
    CUresult r = enc(map, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_UINT16, 3,
                     const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     rows64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(PAFP8_ERR_CUDA, "cuTensorMapEncodeTiled failed for q (CUresult %d)", (int)r);
    return PAFP8_OK;
}

// Decode maps over one cache tensor.  First choice: dims (d, token, head,
// page) with a box of {128, 16, hpc, 1}, so one TMA box brings a whole page
// of the head block, landing head-major ([head][token][128 B]).  If the
// driver does not accept that dimension order, fall back to one box per head
// (encode_cache_map); the shared-memory layout is the same either way.
// A 2-byte cache row (128 elements, 256 B) is split into two 128-B halves so
// that the 128-byte swizzle applies: dims (d % 64, d / 64, token, head, page)
// with a box of {64, 2, 16, hpc, 1}, landing per head as 32 rows of 128 B
// (row 2 * token + half); the fallback is one box per head with dims (d % 64,
// d / 64, head, token, page) and the same layout.
pafp8_status encode_decode_maps_2byte(CUtensorMap* tk, CUtensorMap* tv, const void* k, const void* v,
                                      int num_pages, int hkv, int hpc, int* heads_per_box, int layout,
                                      int head_dim, int page_size) {
    auto enc = get_encode();
    if (!enc) return fail(PAFP8_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    const KvStrides ks = kv_strides(layout, hkv, 2, head_dim, page_size);
    const cuuint32_t halves = (cuuint32_t)(head_dim / 64);  // 128-B halves of a row
    cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    {
        cuuint64_t dims[5] = {64, halves, (cuuint64_t)page_size, (cuuint64_t)hkv, (cuuint64_t)num_pages};
        cuuint64_t strides[4] = {128, ks.token, ks.head, ks.page};
        cuuint32_t box[5] = {64, halves, (cuuint32_t)kPageSize, (cuuint32_t)hpc, 1};
        CUresult rk = enc(tk, CU_TENSOR_MAP_DATA_TYPE_UINT16, 5, const_cast<void*>(k), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        CUresult rv = enc(tv, CU_TENSOR_MAP_DATA_TYPE_UINT16, 5, const_cast<void*>(v), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (rk == CUDA_SUCCESS && rv == CUDA_SUCCESS) {
            *heads_per_box = hpc;
            return PAFP8_OK;
        }
    }
    cuuint64_t dims[5] = {64, halves, (cuuint64_t)hkv, (cuuint64_t)page_size, (cuuint64_t)num_pages};
    cuuint64_t strides[4] = {128, ks.head, ks.token, ks.page};
    cuuint32_t box[5] = {64, halves, 1, (cuuint32_t)kPageSize, 1};
    CUresult rk = enc(tk, CU_TENSOR_MAP_DATA_TYPE_UINT16, 5, const_cast<void*>(k), dims, strides, box, estr,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    CUresult rv = enc(tv, CU_TENSOR_MAP_DATA_TYPE_UINT16, 5, const_cast<void*>(v), dims, strides, box, estr,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (rk != CUDA_SUCCESS || rv != CUDA_SUCCESS)
        return fail(PAFP8_ERR_CUDA, "cuTensorMapEncodeTiled failed for the 2-byte KV cache (CUresult %d, %d)",
                    (int)rk, (int)rv);
    *heads_per_box = 1;
    return PAFP8_OK;
}

pafp8_status encode_decode_maps(CUtensorMap* tk, CUtensorMap* tv, const void* k, const void* v,
                                int num_pages, int hkv, int hpc, int* heads_per_box, bool two_byte, int layout,
                                int head_dim, int page_size) {
    if (num_pages == 0 || k == nullptr || v == nullptr) {
        // No request has pages: the kernel issues no copy, the maps are unused.
        memset(tk, 0, sizeof(*tk));
        memset(tv, 0, sizeof(*tv));
        *heads_per_box = 1;
        return PAFP8_OK;
    }
    if (two_byte)
        return encode_decode_maps_2byte(tk, tv, k, v, num_pages, hkv, hpc, heads_per_box, layout, head_dim,
                                        page_size);
    auto enc = get_encode();
    if (!enc) return fail(PAFP8_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    const KvStrides ks = kv_strides(layout, hkv, 1, head_dim, page_size);
    // 128-B rows take the 128-byte swizzle, 64-B rows (head_dim 64) the 64-byte one.
    const CUtensorMapSwizzle swz = head_dim == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B;
    cuuint64_t dims[4] = {(cuuint64_t)head_dim, (cuuint64_t)page_size, (cuuint64_t)hkv,
                          (cuuint64_t)num_pages};
    cuuint64_t strides[3] = {ks.token, ks.head, ks.page};
    cuuint32_t box[4] = {(cuuint32_t)head_dim, (cuuint32_t)kPageSize, (cuuint32_t)hpc, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult rk = enc(tk, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(k), dims, strides, box,
                      estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    CUresult rv = enc(tv, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(v), dims, strides, box,
                      estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (rk == CUDA_SUCCESS && rv == CUDA_SUCCESS) {
        *heads_per_box = hpc;
        return PAFP8_OK;
    }
    pafp8_status st;
    if ((st = encode_cache_map(tk, k, num_pages, hkv, layout, head_dim, page_size)) != PAFP8_OK) return st;
    if ((st = encode_cache_map(tv, v, num_pages, hkv, layout, head_dim, page_size)) != PAFP8_OK) return st;
    *heads_per_box = 1;
    return PAFP8_OK;
}

bool scale_ok(float s) { return std::isfinite(s) && s > 0.0f; }

// Page-locked staging ring for metadata uploads, one per device: a copy from
// page-locked memory is a plain DMA, where one from the plan's pageable
// memory first goes through a driver bounce buffer.  A slot is reused once
// the copy that last read it has run (an event recorded after it); slots are
// allocated, and grow, on first use.  Copies `bytes` from `src` to device
// `dst` on `s` through the next slot; *done is false when no slot could be
// used (the caller then copies directly).
constexpr int kStageSlots = 4;
struct StageSlot {
    void* buf = nullptr;
    size_t cap = 0;
    cudaEvent_t ev = nullptr;
    bool pending = false;
};
std::mutex g_stage_mu;
StageSlot g_stage[kMaxDevices][kStageSlots];
int g_stage_next[kMaxDevices] = {};

cudaError_t staged_copy(void* dst, const void* src, size_t bytes, cudaStream_t s, bool* done) {
    *done = false;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaSuccess;
    std::lock_guard<std::mutex> lock(g_stage_mu);
    StageSlot& sl = g_stage[dev][g_stage_next[dev]];
    g_stage_next[dev] = (g_stage_next[dev] + 1) % kStageSlots;
    if (sl.pending && (e = cudaEventSynchronize(sl.ev)) != cudaSuccess) return e;
    sl.pending = false;
    if (sl.ev == nullptr && (e = cudaEventCreateWithFlags(&sl.ev, cudaEventDisableTiming)) != cudaSuccess) {
        sl.ev = nullptr;
        return e;
    }
    if (sl.cap < bytes) {
        if (sl.buf != nullptr) cudaFreeHost(sl.buf);
        sl.buf = nullptr;
        sl.cap = 0;
        const size_t cap = std::max<size_t>(bytes, 64 << 10);
        if ((e = cudaHostAlloc(&sl.buf, cap, cudaHostAllocPortable)) != cudaSuccess) {
            sl.buf = nullptr;
            return e;
        }
        sl.cap = cap;
    }
    std::memcpy(sl.buf, src, bytes);
    if ((e = cudaMemcpyAsync(dst, sl.buf, bytes, cudaMemcpyHostToDevice, s)) != cudaSuccess) return e;
    *done = true;
    e = cudaEventRecord(sl.ev, s);
    sl.pending = e == cudaSuccess;
    return e;
}

// Bound of the kernels' pipeline waits: PAFP8_WAIT_CYCLES (a positive integer,
// SM clock cycles) when set, else about one second.  A diagnostic setting: a
// short bound makes a pipeline wait expire on purpose, which the kernels
// report as PAFP8_ERR_TIMEOUT after winding down; their final waits for their
// own copies in flight keep the long bound.
long long wait_cycles() {
    const char* v = std::getenv("PAFP8_WAIT_CYCLES");
    if (v == nullptr || v[0] == '\0') return kWaitCyclesDefault;
    char* end = nullptr;
    const long long n = std::strtoll(v, &end, 10);
    return (end != v && *end == '\0' && n > 0) ? n : kWaitCyclesDefault;
}

}  // namespace

extern "C" {

int32_t pafp8_abi_version(void) { return PAFP8_ABI_VERSION; }

const char* pafp8_last_error(void) { return g_last_error.c_str(); }

pafp8_status pafp8_plan_create(const pafp8_plan_desc* desc_in, const int32_t* kv_indptr_h,
                               const int32_t* last_page_len_h, const int32_t* qo_indptr_h,
                               pafp8_plan** out) {
    if (out == nullptr) return fail(PAFP8_ERR_ARG, "out (plan pointer) is NULL");
    *out = nullptr;
    if (desc_in == nullptr) return fail(PAFP8_ERR_ARG, "plan description is NULL");
    pafp8_plan_desc d = *desc_in;

    if (d.mode != PAFP8_MODE_DECODE && d.mode != PAFP8_MODE_PREFILL)
        return fail(PAFP8_ERR_ARG, "mode %d is neither decode (0) nor prefill (1)", (int)d.mode);

    pafp8_status st;
    if ((st = check_q_dtype(d.q_dtype)) != PAFP8_OK) return st;
    if ((st = check_kv_dtype(d.kv_dtype, "the KV cache", d.mode, d.q_dtype)) != PAFP8_OK) return st;
    if (d.o_dtype == PAFP8_DTYPE_DEFAULT) d.o_dtype = is_2byte(d.q_dtype) ? d.q_dtype : PAFP8_BF16;
    if ((st = check_o_dtype(d.o_dtype, d.q_dtype)) != PAFP8_OK) return st;

    if (d.batch < 0) return fail(PAFP8_ERR_SHAPE, "batch %d is negative", (int)d.batch);
    if (d.num_qo_heads <= 0 || d.num_kv_heads <= 0)
        return fail(PAFP8_ERR_SHAPE, "head counts must be positive (num_qo_heads %d, num_kv_heads %d)",
                    (int)d.num_qo_heads, (int)d.num_kv_heads);
    if (d.num_qo_heads % d.num_kv_heads != 0)
        return fail(PAFP8_ERR_SHAPE, "num_qo_heads %d is not a multiple of num_kv_heads %d",
                    (int)d.num_qo_heads, (int)d.num_kv_heads);
    const int group = d.num_qo_heads / d.num_kv_heads;
    const int max_group = d.mode == PAFP8_MODE_DECODE ? kMaxGroupDecode : kMaxGroupPrefill;
    if (group > max_group)
        return fail(PAFP8_ERR_UNSUPPORTED,
                    "%s serves up to %d query heads per KV head; got %d (%d / %d)",
                    d.mode == PAFP8_MODE_DECODE ? "decode" : "prefill", max_group, group,
                    (int)d.num_qo_heads, (int)d.num_kv_heads);
    if (d.head_dim != kHeadDim && d.head_dim != 64)
        return fail(PAFP8_ERR_UNSUPPORTED, "head_dim %d is not served by this library (%d or 64)",
                    (int)d.head_dim, kHeadDim);
    if (d.num_pages < 0) return fail(PAFP8_ERR_SHAPE, "num_pages %d is negative", (int)d.num_pages);
    if (d.kv_layout != PAFP8_LAYOUT_NHD && d.kv_layout != PAFP8_LAYOUT_HND)
        return fail(PAFP8_ERR_ARG, "kv_layout %d is neither NHD (0) nor HND (1)", (int)d.kv_layout);
    if (d.page_size <= 0 || d.page_size % kPageSize != 0 ||
        (int64_t)d.num_pages * (d.page_size / kPageSize) > INT32_MAX)
        return fail(PAFP8_ERR_UNSUPPORTED,
                    "page_size %d is not served by this library (a multiple of %d tokens, with "
                    "num_pages * page_size / %d below 2^31)",
                    (int)d.page_size, kPageSize, kPageSize);
    if (std::isnan(d.sm_scale) || std::isinf(d.sm_scale))
        return fail(PAFP8_ERR_ARG, "sm_scale is not finite");
    if (d.sm_scale <= 0.0f) d.sm_scale = 1.0f / std::sqrt((float)d.head_dim);
    if (d.fixed_split_pages < 0)
        return fail(PAFP8_ERR_ARG, "fixed_split_pages %d is negative", (int)d.fixed_split_pages);
    if (d.num_ctas < 0) return fail(PAFP8_ERR_ARG, "num_ctas %d is negative", (int)d.num_ctas);
    if (d.batch > 0 && (kv_indptr_h == nullptr || last_page_len_h == nullptr))
        return fail(PAFP8_ERR_ARG, "kv_indptr and last_page_len host arrays are required");
    if (d.mode == PAFP8_MODE_DECODE && qo_indptr_h != nullptr)
        return fail(PAFP8_ERR_ARG, "decode takes no qo_indptr (one query row per request)");
    if (d.mode == PAFP8_MODE_PREFILL && d.batch > 0 && qo_indptr_h == nullptr)
        return fail(PAFP8_ERR_ARG, "prefill needs the qo_indptr host array");

    if (d.batch > 0 && kv_indptr_h[0] != 0)
        return fail(PAFP8_ERR_SHAPE, "kv_indptr[0] is %d, not 0", (int)kv_indptr_h[0]);
    for (int b = 0; b < d.batch; ++b) {
        const int64_t n = (int64_t)kv_indptr_h[b + 1] - kv_indptr_h[b];
        if (n < 0)
            return fail(PAFP8_ERR_SHAPE, "kv_indptr decreases at request %d (%d -> %d)", b,
                        (int)kv_indptr_h[b], (int)kv_indptr_h[b + 1]);
        if (n > 0 && (last_page_len_h[b] < 1 || last_page_len_h[b] > d.page_size))
            return fail(PAFP8_ERR_SHAPE, "last_page_len[%d] = %d is outside [1, %d]", b,
                        (int)last_page_len_h[b], (int)d.page_size);
        if (n > 0 && d.num_pages == 0)
            return fail(PAFP8_ERR_SHAPE, "request %d has pages but num_pages is 0", b);
        if (d.mode == PAFP8_MODE_PREFILL) {
            if (b == 0 && qo_indptr_h[0] != 0)
                return fail(PAFP8_ERR_SHAPE, "qo_indptr[0] is %d, not 0", (int)qo_indptr_h[0]);
            const int64_t qo = (int64_t)qo_indptr_h[b + 1] - qo_indptr_h[b];
            const int64_t kv = n > 0 ? (n - 1) * d.page_size + last_page_len_h[b] : 0;
            if (qo < 0)
                return fail(PAFP8_ERR_SHAPE, "qo_indptr decreases at request %d (%d -> %d)", b,
                            (int)qo_indptr_h[b], (int)qo_indptr_h[b + 1]);
            if (qo > kv)
                return fail(PAFP8_ERR_SHAPE,
                            "request %d has qo_len %lld > kv_len %lld: the new rows must be the "
                            "last qo_len tokens of the KV sequence",
                            b, (long long)qo, (long long)kv);
        }
    }

    if (d.num_ctas == 0) {
        int dev = 0, sms = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            sms <= 0) {
            cudaGetLastError();
            return fail(PAFP8_ERR_CUDA,
                        "num_ctas is 0 and the SM count of the current device is unavailable");
        }
        d.num_ctas = sms;
    }

    pafp8_plan* pl = new pafp8_plan();
    pl->desc = d;
    pl->group = group;
    pl->heads_per_cta = heads_per_cta_for(d.num_kv_heads);
    pl->head_blocks = d.num_kv_heads / pl->heads_per_cta;
    if (d.batch > 0) {
        pl->kv_indptr.assign(kv_indptr_h, kv_indptr_h + d.batch + 1);
        pl->last_page_len.assign(last_page_len_h, last_page_len_h + d.batch);
    } else {
        pl->kv_indptr.assign(1, 0);
    }
    pl->nnz_pages = pl->kv_indptr.back();
    pl->page_mult = d.page_size / kPageSize;
    pl->vptr.assign((size_t)d.batch + 1, 0);
    for (int b = 0; b < d.batch; ++b) {
        const int64_t n = (int64_t)pl->kv_indptr[b + 1] - pl->kv_indptr[b];
        const int64_t kv = n > 0 ? (n - 1) * d.page_size + pl->last_page_len[b] : 0;
        pl->vptr[b + 1] = pl->vptr[b] + (int32_t)((kv + kPageSize - 1) / kPageSize);
    }
    if (d.mode == PAFP8_MODE_PREFILL) {
        if (d.batch > 0)
            pl->qo_indptr.assign(qo_indptr_h, qo_indptr_h + d.batch + 1);
        else
            pl->qo_indptr.assign(1, 0);
        pl->nnz_qo = pl->qo_indptr.back();
        build_prefill_meta(pl);
    } else {
        pl->nnz_qo = d.batch;
        build_decode_meta(pl);
    }
    layout_workspace(pl);
    *out = pl;
    return PAFP8_OK;
}

void pafp8_plan_destroy(pafp8_plan* plan) { delete plan; }

size_t pafp8_workspace_bytes(const pafp8_plan* plan) { return plan ? plan->ws_bytes : 0; }

pafp8_status pafp8_plan_metadata(const pafp8_plan* plan, const int32_t** words, size_t* count) {
    if (plan == nullptr || words == nullptr || count == nullptr)
        return fail(PAFP8_ERR_ARG, "plan, words and count must be non-NULL");
    *words = plan->meta.data();
    *count = plan->meta.size();
    return PAFP8_OK;
}

pafp8_status pafp8_plan_upload(pafp8_plan* plan, void* workspace, size_t workspace_bytes,
                               void* stream) {
    if (plan == nullptr) return fail(PAFP8_ERR_ARG, "plan is NULL");
    if (workspace == nullptr) return fail(PAFP8_ERR_ARG, "workspace is NULL");
    if ((uintptr_t)workspace % 256 != 0)
        return fail(PAFP8_ERR_WORKSPACE, "workspace must be 256-byte aligned");
    if (workspace_bytes < plan->ws_bytes)
        return fail(PAFP8_ERR_WORKSPACE, "workspace has %zu bytes; the plan needs %zu",
                    workspace_bytes, plan->ws_bytes);
    cudaStream_t s = (cudaStream_t)stream;
    const size_t bytes = plan->meta.size() * 4;
    // Through the page-locked staging ring when the stream is not being
    // captured (a captured copy would read the staging buffer at replay,
    // after later uploads reused it); from the plan's own memory otherwise.
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    cudaError_t e = cudaStreamIsCapturing(s, &cap);
    bool done = false;
    if (e == cudaSuccess && cap == cudaStreamCaptureStatusNone) e = staged_copy(workspace, plan->meta.data(), bytes, s, &done);
    if (e == cudaSuccess && !done)
        e = cudaMemcpyAsync(workspace, plan->meta.data(), bytes, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess)
        e = cudaMemsetAsync((char*)workspace + plan->status_off, 0, plan->ws_bytes - plan->status_off, s);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(PAFP8_ERR_CUDA, "metadata upload failed: %s", cudaGetErrorString(e));
    }
    plan->uploaded_ws = workspace;
    return PAFP8_OK;
}

}  // extern "C"

namespace {

// Checks and launches of the run entry points.  Per-head scale tensors
// (device arrays) replace the per-tensor scales when k_scales is not NULL.
// With launch false only the checks run.
pafp8_status run_body(const pafp8_plan* plan, int32_t stage, int32_t q_dtype, const void* q,
                      int32_t k_dtype, const void* k_cache, int32_t v_dtype, const void* v_cache,
                      const int32_t* kv_indices, float q_scale, float k_scale, float v_scale,
                      const float* q_scales, const float* k_scales, const float* v_scales,
                      int32_t o_dtype, void* o, float* lse, void* workspace, size_t workspace_bytes,
                      void* stream, bool launch) {
    if (plan == nullptr) return fail(PAFP8_ERR_ARG, "plan is NULL");
    if (stage < 0 || stage > 2) return fail(PAFP8_ERR_ARG, "stage %d is not 0, 1 or 2", (int)stage);
    const pafp8_plan_desc& d = plan->desc;
    pafp8_status st;
    if (k_dtype != v_dtype)
        return fail(PAFP8_ERR_DTYPE, "k_cache has dtype %s but v_cache has %s",
                    dtype_name(k_dtype), dtype_name(v_dtype));
    if ((st = check_kv_dtype(k_dtype, "k_cache", d.mode, q_dtype)) != PAFP8_OK) return st;
    if ((st = check_q_dtype(q_dtype)) != PAFP8_OK) return st;
    if ((st = check_o_dtype(o_dtype, q_dtype)) != PAFP8_OK) return st;
    if (q_dtype != d.q_dtype)
        return fail(PAFP8_ERR_DTYPE, "q has dtype %s but the plan was made for %s",
                    dtype_name(q_dtype), dtype_name(d.q_dtype));
    if (k_dtype != d.kv_dtype)
        return fail(PAFP8_ERR_DTYPE, "the KV cache has dtype %s but the plan was made for %s",
                    dtype_name(k_dtype), dtype_name(d.kv_dtype));
    if (o_dtype != d.o_dtype)
        return fail(PAFP8_ERR_DTYPE, "o has dtype %s but the plan fixed o_data_type %s",
                    dtype_name(o_dtype), dtype_name(d.o_dtype));
    if (!scale_ok(q_scale) || !scale_ok(k_scale) || !scale_ok(v_scale))
        return fail(PAFP8_ERR_ARG, "scales must be finite and > 0 (q %g, k %g, v %g)",
                    (double)q_scale, (double)k_scale, (double)v_scale);
    if (is_2byte(q_dtype) && q_scale != 1.0f)
        return fail(PAFP8_ERR_ARG,
                    "q_scale %g given with a %s query: only an fp8 query is dequantized by "
                    "q_scale, so it would be silently ignored",
                    (double)q_scale, dtype_name(q_dtype));
    if (k_scales != nullptr) {
        if (v_scales == nullptr)
            return fail(PAFP8_ERR_ARG, "per-head scales need both k_scales and v_scales");
        if (is_2byte(q_dtype) && q_scales != nullptr)
            return fail(PAFP8_ERR_ARG,
                        "q_scales given with a %s query: only an fp8 query is dequantized by its "
                        "scales, so they would be silently ignored",
                        dtype_name(q_dtype));
        if (((uintptr_t)q_scales | (uintptr_t)k_scales | (uintptr_t)v_scales) % 4 != 0)
            return fail(PAFP8_ERR_ARG, "q_scales, k_scales and v_scales must be 4-byte aligned");
    }
    if (workspace == nullptr || workspace != plan->uploaded_ws)
        return fail(PAFP8_ERR_WORKSPACE,
                    "workspace %p is not the one this plan's metadata was uploaded to (%p)",
                    workspace, plan->uploaded_ws);
    if (workspace_bytes < plan->ws_bytes)
        return fail(PAFP8_ERR_WORKSPACE, "workspace has %zu bytes; the plan needs %zu",
                    workspace_bytes, plan->ws_bytes);
    if (plan->nnz_qo > 0 && (q == nullptr || o == nullptr))
        return fail(PAFP8_ERR_ARG, "q and o must be non-NULL");
    if (plan->nnz_pages > 0 && (k_cache == nullptr || v_cache == nullptr || kv_indices == nullptr))
        return fail(PAFP8_ERR_ARG, "k_cache, v_cache and kv_indices must be non-NULL");
    if (((uintptr_t)q | (uintptr_t)o | (uintptr_t)k_cache | (uintptr_t)v_cache) % 16 != 0)
        return fail(PAFP8_ERR_ARG, "q, o, k_cache and v_cache must be 16-byte aligned");
    if ((uintptr_t)lse % 4 != 0 || (uintptr_t)kv_indices % 4 != 0)
        return fail(PAFP8_ERR_ARG, "lse and kv_indices must be 4-byte aligned");
    if (!launch) return PAFP8_OK;

    cudaStream_t s = (cudaStream_t)stream;
    char* ws = (char*)workspace;
    const float sm_log2 = (float)((double)d.sm_scale * (is_fp8(q_dtype) ? (double)q_scale : 1.0) *
                                  (double)k_scale * 1.4426950408889634);
    if (d.mode == PAFP8_MODE_PREFILL) {
        if (stage == 2 || plan->num_ctas == 0) return PAFP8_OK;  // prefill has no merge stage
        PrefillParams pp{};
        pp.q = q;
        pp.head_dim = d.head_dim;
        pp.kv_indices = kv_indices;
        pp.o = o;
        pp.lse = lse;
        pp.meta = (const int32_t*)ws;
        pp.status = (uint32_t*)(ws + plan->status_off);
        pp.q_dtype = q_dtype;
        pp.kv_dtype = k_dtype;
        pp.o_dtype = o_dtype;
        pp.num_qo_heads = d.num_qo_heads;
        pp.num_kv_heads = d.num_kv_heads;
        pp.num_pages = d.num_pages;
        pp.page_mult = plan->page_mult;
        pp.group = plan->group;
        pp.tile_tokens = kTileRows / plan->group;
        pp.sm_scale_log2 = sm_log2;
        pp.v_scale = v_scale;
        pp.q_scales = k_scales != nullptr ? q_scales : nullptr;
        pp.k_scales = k_scales;
        pp.v_scales = k_scales != nullptr ? v_scales : nullptr;
        pp.sm_scale = d.sm_scale;
        pp.wait_cycles = wait_cycles();
        CUtensorMap tq, tk, tv;
        if ((st = encode_q_map(&tq, q, (int)plan->nnz_qo, d.num_qo_heads, plan->group,
                               pp.tile_tokens, is_fp8(q_dtype), d.head_dim)) != PAFP8_OK)
            return st;
        if (is_2byte(k_dtype)) {
            if ((st = encode_cache_map_2byte(&tk, k_cache, d.num_pages, d.num_kv_heads, d.kv_layout, d.head_dim,
                                             d.page_size)) !=
                PAFP8_OK)
                return st;
            if ((st = encode_cache_map_2byte(&tv, v_cache, d.num_pages, d.num_kv_heads, d.kv_layout, d.head_dim,
                                             d.page_size)) !=
                PAFP8_OK)
                return st;
        } else {
            if ((st = encode_cache_map(&tk, k_cache, d.num_pages, d.num_kv_heads, d.kv_layout, d.head_dim,
                                       d.page_size)) != PAFP8_OK)
                return st;
            if ((st = encode_cache_map(&tv, v_cache, d.num_pages, d.num_kv_heads, d.kv_layout, d.head_dim,
                                       d.page_size)) != PAFP8_OK)
                return st;
        }
        CUtensorMap to;
        if ((st = encode_q_map(&to, o, (int)plan->nnz_qo, d.num_qo_heads, plan->group, pp.tile_tokens,
                               false, d.head_dim)) != PAFP8_OK)
            return st;
        cudaError_t e = launch_prefill(pp, tq, tk, tv, to, plan->num_ctas, s);
        if (e != cudaSuccess) {
            cudaGetLastError();
            return fail(PAFP8_ERR_CUDA, "kernel launch failed: %s", cudaGetErrorString(e));
        }
        return PAFP8_OK;
    }
    DecodeParams p{};
    p.q = q;
    p.kv_indices = kv_indices;
    p.o = o;
    p.lse = lse;
    p.meta = (const int32_t*)ws;
    p.part_o = (float*)(ws + plan->part_o_off);
    p.part_lse = (float*)(ws + plan->part_lse_off);
    p.status = (uint32_t*)(ws + plan->status_off);
    p.q_dtype = q_dtype;
    p.kv_dtype = k_dtype;
    p.o_dtype = o_dtype;
    p.num_qo_heads = d.num_qo_heads;
    p.num_kv_heads = d.num_kv_heads;
    p.num_pages = d.num_pages;
    p.page_mult = plan->page_mult;
    p.head_dim = d.head_dim;
    p.sm_scale_log2 = sm_log2;
    p.v_scale = v_scale;
    p.q_scales = k_scales != nullptr ? q_scales : nullptr;
    p.k_scales = k_scales;
    p.v_scales = k_scales != nullptr ? v_scales : nullptr;
    p.sm_scale = d.sm_scale;
    p.wait_cycles = wait_cycles();

    cudaError_t e = cudaSuccess;
    if (stage != 2 && plan->num_ctas > 0) {
        CUtensorMap tk, tv;
        int hpb = 1;
        if ((st = encode_decode_maps(&tk, &tv, k_cache, v_cache, d.num_pages, d.num_kv_heads,
                                     plan->heads_per_cta, &hpb, is_2byte(k_dtype), d.kv_layout, d.head_dim,
                                     d.page_size)) != PAFP8_OK)
            return st;
        e = launch_decode(p, tk, tv, plan->num_ctas, plan->heads_per_cta, plan->group, hpb, s);
    }
    if (e == cudaSuccess && stage != 1 && plan->num_merge > 0)
        e = launch_merge(p, plan->num_merge, plan->heads_per_cta, plan->group, s);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(PAFP8_ERR_CUDA, "kernel launch failed: %s", cudaGetErrorString(e));
    }
    return PAFP8_OK;
}

}  // namespace

namespace {

// PAFP8_DEBUG set to anything but "0" in the environment: every launching
// run call synchronizes its stream and returns the kernels' status (what
// pafp8_device_status would report), so that a bad page index or an expired
// wait surfaces at the call that caused it.  Not for use under stream capture.
bool debug_sync() {
    const char* v = std::getenv("PAFP8_DEBUG");
    return v != nullptr && v[0] != '\0' && !(v[0] == '0' && v[1] == '\0');
}

pafp8_status run_impl(const pafp8_plan* plan, int32_t stage, int32_t q_dtype, const void* q,
                      int32_t k_dtype, const void* k_cache, int32_t v_dtype, const void* v_cache,
                      const int32_t* kv_indices, float q_scale, float k_scale, float v_scale,
                      const float* q_scales, const float* k_scales, const float* v_scales,
                      int32_t o_dtype, void* o, float* lse, void* workspace, size_t workspace_bytes,
                      void* stream, bool launch = true) {
    const pafp8_status st = run_body(plan, stage, q_dtype, q, k_dtype, k_cache, v_dtype, v_cache, kv_indices,
                                     q_scale, k_scale, v_scale, q_scales, k_scales, v_scales, o_dtype, o, lse,
                                     workspace, workspace_bytes, stream, launch);
    if (st != PAFP8_OK || !launch || !debug_sync()) return st;
    return pafp8_device_status(plan, workspace, stream);
}

}  // namespace

extern "C" {

pafp8_status pafp8_run(const pafp8_plan* plan, int32_t q_dtype, const void* q, int32_t k_dtype,
                       const void* k_cache, int32_t v_dtype, const void* v_cache,
                       const int32_t* kv_indices, float q_scale, float k_scale, float v_scale,
                       int32_t o_dtype, void* o, float* lse, void* workspace,
                       size_t workspace_bytes, void* stream) {
    return run_impl(plan, 0, q_dtype, q, k_dtype, k_cache, v_dtype, v_cache, kv_indices, q_scale, k_scale,
                    v_scale, nullptr, nullptr, nullptr, o_dtype, o, lse, workspace, workspace_bytes, stream);
}

size_t pafp8_host_workspace_bytes(const pafp8_plan* plan, int32_t q_dtype) {
    return plan ? host_staging(plan, q_dtype).end : 0;
}

pafp8_status pafp8_run_host(pafp8_plan* plan, int32_t q_dtype, const void* q_h, int32_t k_dtype,
                            const void* k_cache, int32_t v_dtype, const void* v_cache,
                            const int32_t* kv_indices_h, float q_scale, float k_scale, float v_scale,
                            int32_t o_dtype, void* o_h, float* lse_h, void* workspace,
                            size_t workspace_bytes, void* stream) {
    if (plan == nullptr) return fail(PAFP8_ERR_ARG, "plan is NULL");
    const HostStaging hs = host_staging(plan, q_dtype);
    if (workspace_bytes < hs.end)
        return fail(PAFP8_ERR_WORKSPACE, "workspace has %zu bytes; a host-buffer step of this plan needs %zu",
                    workspace_bytes, hs.end);
    if (hs.q_bytes > 0 && (q_h == nullptr || o_h == nullptr))
        return fail(PAFP8_ERR_ARG, "q_h and o_h must be non-NULL");
    if (hs.idx_bytes > 0 && kv_indices_h == nullptr) return fail(PAFP8_ERR_ARG, "kv_indices_h must be non-NULL");
    pafp8_status st = pafp8_plan_upload(plan, workspace, workspace_bytes, stream);
    if (st != PAFP8_OK) return st;
    char* ws = (char*)workspace;
    void* q_d = ws + hs.q;
    void* o_d = ws + hs.o;
    const int32_t* idx_d = (const int32_t*)(ws + hs.idx);
    float* lse_d = lse_h != nullptr ? (float*)(ws + hs.lse) : nullptr;
    if ((st = run_impl(plan, 0, q_dtype, q_d, k_dtype, k_cache, v_dtype, v_cache, idx_d, q_scale, k_scale,
                       v_scale, nullptr, nullptr, nullptr, o_dtype, o_d, lse_d, workspace, workspace_bytes, stream,
                       false)) != PAFP8_OK)
        return st;
    cudaStream_t s = (cudaStream_t)stream;
    cudaError_t e = cudaSuccess;
    if (hs.q_bytes > 0) e = cudaMemcpyAsync(q_d, q_h, hs.q_bytes, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess && hs.idx_bytes > 0)
        e = cudaMemcpyAsync(ws + hs.idx, kv_indices_h, hs.idx_bytes, cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(PAFP8_ERR_CUDA, "copying q and kv_indices to the device failed: %s", cudaGetErrorString(e));
    }
    if ((st = run_impl(plan, 0, q_dtype, q_d, k_dtype, k_cache, v_dtype, v_cache, idx_d, q_scale, k_scale,
                       v_scale, nullptr, nullptr, nullptr, o_dtype, o_d, lse_d, workspace, workspace_bytes,
                       stream)) != PAFP8_OK)
        return st;
    if (hs.o_bytes > 0) e = cudaMemcpyAsync(o_h, o_d, hs.o_bytes, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess && lse_h != nullptr && hs.lse_bytes > 0)
        e = cudaMemcpyAsync(lse_h, lse_d, hs.lse_bytes, cudaMemcpyDeviceToHost, s);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(PAFP8_ERR_CUDA, "copying o and lse to the host failed: %s", cudaGetErrorString(e));
    }
    return PAFP8_OK;
}

pafp8_status pafp8_run_stage(const pafp8_plan* plan, int32_t stage, int32_t q_dtype, const void* q,
                             int32_t k_dtype, const void* k_cache, int32_t v_dtype,
                             const void* v_cache, const int32_t* kv_indices, float q_scale,
                             float k_scale, float v_scale, int32_t o_dtype, void* o, float* lse,
                             void* workspace, size_t workspace_bytes, void* stream) {
    return run_impl(plan, stage, q_dtype, q, k_dtype, k_cache, v_dtype, v_cache, kv_indices, q_scale,
                    k_scale, v_scale, nullptr, nullptr, nullptr, o_dtype, o, lse, workspace,
                    workspace_bytes, stream);
}

pafp8_status pafp8_run_head_scales(const pafp8_plan* plan, int32_t q_dtype, const void* q,
                                   int32_t k_dtype, const void* k_cache, int32_t v_dtype,
                                   const void* v_cache, const int32_t* kv_indices, const float* q_scales,
                                   const float* k_scales, const float* v_scales, int32_t o_dtype, void* o,
                                   float* lse, void* workspace, size_t workspace_bytes, void* stream) {
    if (k_scales == nullptr || v_scales == nullptr)
        return fail(PAFP8_ERR_ARG, "k_scales and v_scales (device arrays of num_kv_heads floats) are required");
    return run_impl(plan, 0, q_dtype, q, k_dtype, k_cache, v_dtype, v_cache, kv_indices, 1.0f, 1.0f, 1.0f,
                    q_scales, k_scales, v_scales, o_dtype, o, lse, workspace, workspace_bytes, stream);
}

pafp8_status pafp8_device_status(const pafp8_plan* plan, void* workspace, void* stream) {
    if (plan == nullptr || workspace == nullptr) return fail(PAFP8_ERR_ARG, "plan and workspace are required");
    cudaStream_t s = (cudaStream_t)stream;
    uint32_t word = 0;
    char* st_ptr = (char*)workspace + plan->status_off;
    cudaError_t e = cudaMemcpyAsync(&word, st_ptr, 4, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e == cudaSuccess) e = cudaMemsetAsync(st_ptr, 0, 4, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(PAFP8_ERR_CUDA, "reading the device status failed: %s", cudaGetErrorString(e));
    }
    if (word & kStatusTimeout)
        return fail(PAFP8_ERR_TIMEOUT, "a kernel's bounded pipeline wait expired (status 0x%x)", word);
    if (word & kStatusBounds)
        return fail(PAFP8_ERR_BOUNDS, "a page index outside [0, num_pages) was skipped (status 0x%x)",
                    word);
    return PAFP8_OK;
}

// Decode without a caller-supplied workspace: the library's built-in scratch
// (noalloc_scratch) takes its place.  Nothing here allocates device memory.
pafp8_status pafp8_run_decode_noalloc(const pafp8_plan* plan, int32_t q_dtype, const void* q,
                                      int32_t k_dtype, const void* k_cache, int32_t v_dtype,
                                      const void* v_cache, const int32_t* kv_indices,
                                      float q_scale, float k_scale, float v_scale,
                                      int32_t o_dtype, void* o, float* lse, void* stream) {
    if (plan == nullptr) return fail(PAFP8_ERR_ARG, "plan is NULL");
    const pafp8_plan_desc& d = plan->desc;
    if (d.mode != PAFP8_MODE_DECODE)
        return fail(PAFP8_ERR_ARG, "pafp8_run_decode_noalloc serves decode plans only");
    if (plan->ws_bytes > kNoAllocScratchBytes)
        return fail(PAFP8_ERR_WORKSPACE,
                    "the plan needs %zu bytes of scratch but the built-in scratch holds %zu; "
                    "use pafp8_run with a workspace, or plan with fewer CTAs or splits",
                    plan->ws_bytes, kNoAllocScratchBytes);
    pafp8_status st;
    if (k_dtype != v_dtype)
        return fail(PAFP8_ERR_DTYPE, "k_cache has dtype %s but v_cache has %s",
                    dtype_name(k_dtype), dtype_name(v_dtype));
    if ((st = check_kv_dtype(k_dtype, "k_cache", d.mode, q_dtype)) != PAFP8_OK) return st;
    if ((st = check_q_dtype(q_dtype)) != PAFP8_OK) return st;
    if ((st = check_o_dtype(o_dtype, q_dtype)) != PAFP8_OK) return st;
    if (q_dtype != d.q_dtype || k_dtype != d.kv_dtype || o_dtype != d.o_dtype)
        return fail(PAFP8_ERR_DTYPE,
                    "dtypes q %s, kv %s, o %s differ from the plan's q %s, kv %s, o %s",
                    dtype_name(q_dtype), dtype_name(k_dtype), dtype_name(o_dtype),
                    dtype_name(d.q_dtype), dtype_name(d.kv_dtype), dtype_name(d.o_dtype));
    if (!scale_ok(q_scale) || !scale_ok(k_scale) || !scale_ok(v_scale))
        return fail(PAFP8_ERR_ARG, "scales must be finite and > 0 (q %g, k %g, v %g)",
                    (double)q_scale, (double)k_scale, (double)v_scale);
    if (is_2byte(q_dtype) && q_scale != 1.0f)
        return fail(PAFP8_ERR_ARG,
                    "q_scale %g given with a %s query: only an fp8 query is dequantized by "
                    "q_scale, so it would be silently ignored",
                    (double)q_scale, dtype_name(q_dtype));
    if (plan->nnz_qo > 0 && (q == nullptr || o == nullptr))
        return fail(PAFP8_ERR_ARG, "q and o must be non-NULL");
    if (plan->nnz_pages > 0 && (k_cache == nullptr || v_cache == nullptr || kv_indices == nullptr))
        return fail(PAFP8_ERR_ARG, "k_cache, v_cache and kv_indices must be non-NULL");
    if (((uintptr_t)q | (uintptr_t)o | (uintptr_t)k_cache | (uintptr_t)v_cache) % 16 != 0)
        return fail(PAFP8_ERR_ARG, "q, o, k_cache and v_cache must be 16-byte aligned");
    if ((uintptr_t)lse % 4 != 0 || (uintptr_t)kv_indices % 4 != 0)
        return fail(PAFP8_ERR_ARG, "lse and kv_indices must be 4-byte aligned");

    void* scratch = nullptr;
    cudaError_t e = noalloc_scratch(&scratch);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(PAFP8_ERR_CUDA, "looking up the built-in scratch failed: %s",
                    cudaGetErrorString(e));
    }
    cudaStream_t s = (cudaStream_t)stream;
    char* ws = (char*)scratch;
    // The scratch keeps the previous call's bytes: load this plan's metadata
    // and clear the status word; partial states are written before read.
    e = cudaMemcpyAsync(ws, plan->meta.data(), plan->meta.size() * 4, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(ws + plan->status_off, 0, plan->ws_bytes - plan->status_off, s);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(PAFP8_ERR_CUDA, "loading the plan into the built-in scratch failed: %s",
                    cudaGetErrorString(e));
    }
    DecodeParams p{};
    p.q = q;
    p.kv_indices = kv_indices;
    p.o = o;
    p.lse = lse;
    p.meta = (const int32_t*)ws;
    p.part_o = (float*)(ws + plan->part_o_off);
    p.part_lse = (float*)(ws + plan->part_lse_off);
    p.status = (uint32_t*)(ws + plan->status_off);
    p.q_dtype = q_dtype;
    p.kv_dtype = k_dtype;
    p.o_dtype = o_dtype;
    p.num_qo_heads = d.num_qo_heads;
    p.num_kv_heads = d.num_kv_heads;
    p.num_pages = d.num_pages;
    p.page_mult = plan->page_mult;
    p.head_dim = d.head_dim;
    p.sm_scale_log2 = (float)((double)d.sm_scale * (is_fp8(q_dtype) ? (double)q_scale : 1.0) *
                              (double)k_scale * 1.4426950408889634);
    p.v_scale = v_scale;
    p.wait_cycles = wait_cycles();
    if (plan->num_ctas > 0) {
        CUtensorMap tk, tv;
        int hpb = 1;
        if ((st = encode_decode_maps(&tk, &tv, k_cache, v_cache, d.num_pages, d.num_kv_heads,
                                     plan->heads_per_cta, &hpb, is_2byte(k_dtype), d.kv_layout, d.head_dim,
                                     d.page_size)) != PAFP8_OK)
            return st;
        e = launch_decode(p, tk, tv, plan->num_ctas, plan->heads_per_cta, plan->group, hpb, s);
    }
    if (e == cudaSuccess && plan->num_merge > 0)
        e = launch_merge(p, plan->num_merge, plan->heads_per_cta, plan->group, s);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(PAFP8_ERR_CUDA, "kernel launch failed: %s", cudaGetErrorString(e));
    }
    // Under PAFP8_DEBUG the call reports the kernels' status word, as the
    // workspace entry points do.
    if (debug_sync()) return pafp8_device_status(plan, scratch, stream);
    return PAFP8_OK;
}

// Prefill and decode phases of one call on disjoint SMs: the decode grid on
// the decode plan's side stream (highest priority, forked from and joined to
// `stream`), the prefill grid on `stream`.  The plans' num_ctas split the SMs.
pafp8_status pafp8_run_pod(const pafp8_pod_phase* prefill, const pafp8_pod_phase* decode, int32_t q_dtype,
                           int32_t k_dtype, const void* k_cache, int32_t v_dtype, const void* v_cache,
                           float q_scale, float k_scale, float v_scale, int32_t o_dtype, void* stream) {
    if (prefill == nullptr || decode == nullptr || prefill->plan == nullptr || decode->plan == nullptr)
        return fail(PAFP8_ERR_ARG, "both phases and their plans are required");
    const pafp8_plan_desc& a = prefill->plan->desc;
    const pafp8_plan_desc& b = decode->plan->desc;
    if (a.mode != PAFP8_MODE_PREFILL) return fail(PAFP8_ERR_ARG, "the prefill phase's plan is a decode plan");
    if (b.mode != PAFP8_MODE_DECODE) return fail(PAFP8_ERR_ARG, "the decode phase's plan is a prefill plan");
    if (a.num_pages != b.num_pages || a.page_size != b.page_size || a.num_kv_heads != b.num_kv_heads ||
        a.head_dim != b.head_dim || a.kv_layout != b.kv_layout)
        return fail(PAFP8_ERR_SHAPE,
                    "the two plans describe different caches: prefill num_pages %d page_size %d "
                    "num_kv_heads %d head_dim %d layout %d, decode %d %d %d %d %d",
                    (int)a.num_pages, (int)a.page_size, (int)a.num_kv_heads, (int)a.head_dim,
                    (int)a.kv_layout, (int)b.num_pages, (int)b.page_size, (int)b.num_kv_heads,
                    (int)b.head_dim, (int)b.kv_layout);
    const uintptr_t w0 = (uintptr_t)prefill->workspace, w1 = (uintptr_t)decode->workspace;
    if (w0 != 0 && w1 != 0 && w0 < w1 + decode->workspace_bytes && w1 < w0 + prefill->workspace_bytes)
        return fail(PAFP8_ERR_WORKSPACE, "the prefill and decode workspaces overlap");
    pafp8_status st;
    const pafp8_pod_phase* ph[2] = {decode, prefill};
    for (const pafp8_pod_phase* x : ph) {
        if ((st = run_impl(x->plan, 0, q_dtype, x->q, k_dtype, k_cache, v_dtype, v_cache, x->kv_indices,
                           q_scale, k_scale, v_scale, nullptr, nullptr, nullptr, o_dtype, x->o, x->lse,
                           x->workspace, x->workspace_bytes, stream, false)) != PAFP8_OK)
            return st;
    }
    const pafp8_plan* dp = decode->plan;
    if (dp->pod_stream == nullptr) {
        int lo = 0, hi = 0;
        cudaError_t e = cudaDeviceGetStreamPriorityRange(&lo, &hi);
        cudaStream_t side = nullptr;
        cudaEvent_t fork = nullptr, join = nullptr;
        if (e == cudaSuccess) e = cudaStreamCreateWithPriority(&side, cudaStreamNonBlocking, hi);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&fork, cudaEventDisableTiming);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&join, cudaEventDisableTiming);
        if (e != cudaSuccess) {
            cudaGetLastError();
            if (join != nullptr) cudaEventDestroy(join);
            if (fork != nullptr) cudaEventDestroy(fork);
            if (side != nullptr) cudaStreamDestroy(side);
            return fail(PAFP8_ERR_CUDA, "creating the side stream failed: %s", cudaGetErrorString(e));
        }
        dp->pod_stream = side;
        dp->pod_fork = fork;
        dp->pod_join = join;
    }
    cudaStream_t s = (cudaStream_t)stream;
    cudaError_t e = cudaEventRecord(dp->pod_fork, s);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(dp->pod_stream, dp->pod_fork, 0);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(PAFP8_ERR_CUDA, "forking the side stream failed: %s", cudaGetErrorString(e));
    }
    // Decode first, so that its CTAs are dispatched first when both grids are
    // ready; its stream priority keeps them ahead of the prefill CTAs.
    const pafp8_status sd = run_impl(dp, 0, q_dtype, decode->q, k_dtype, k_cache, v_dtype, v_cache,
                                     decode->kv_indices, q_scale, k_scale, v_scale, nullptr, nullptr, nullptr,
                                     o_dtype, decode->o, decode->lse, decode->workspace,
                                     decode->workspace_bytes, dp->pod_stream);
    const pafp8_status sp =
        sd != PAFP8_OK ? sd
                       : run_impl(prefill->plan, 0, q_dtype, prefill->q, k_dtype, k_cache, v_dtype, v_cache,
                                  prefill->kv_indices, q_scale, k_scale, v_scale, nullptr, nullptr, nullptr,
                                  o_dtype, prefill->o, prefill->lse, prefill->workspace,
                                  prefill->workspace_bytes, s);
    // Join even after a failed launch, so that `stream` never runs ahead of
    // work already queued on the side stream.
    e = cudaEventRecord(dp->pod_join, dp->pod_stream);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(s, dp->pod_join, 0);
    if (sd != PAFP8_OK) return sd;
    if (sp != PAFP8_OK) return sp;
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(PAFP8_ERR_CUDA, "joining the side stream failed: %s", cudaGetErrorString(e));
    }
    return PAFP8_OK;
}

pafp8_status pafp8_append_kv(int32_t src_dtype, const void* k_new, const void* v_new, int64_t nnz,
                             int32_t num_kv_heads, int32_t head_dim, const int32_t* batch_indices,
                             const int32_t* positions, int32_t batch, const int32_t* kv_indptr,
                             const int32_t* kv_indices, int32_t kv_dtype, int32_t kv_layout,
                             void* k_cache, void* v_cache, int32_t num_pages, int32_t page_size,
                             float k_scale, float v_scale, uint32_t* status, void* stream) {
    if (src_dtype != PAFP8_F16 && src_dtype != PAFP8_BF16 && src_dtype != PAFP8_F32)
        return fail(PAFP8_ERR_DTYPE, "new tokens of dtype %s: append takes f16, bf16 or f32 rows",
                    dtype_name(src_dtype));
    if (!is_fp8(kv_dtype)) {
        if (is_2byte(kv_dtype))
            return fail(PAFP8_ERR_UNSUPPORTED,
                        "a %s cache holds the new rows as they are; append quantizes into an "
                        "e4m3fn or e5m2 cache only",
                        dtype_name(kv_dtype));
        return fail(PAFP8_ERR_DTYPE, "append writes an e4m3fn or e5m2 cache, not %s",
                    dtype_name(kv_dtype));
    }
    if (kv_layout != PAFP8_LAYOUT_NHD && kv_layout != PAFP8_LAYOUT_HND)
        return fail(PAFP8_ERR_ARG, "kv_layout %d is neither NHD (0) nor HND (1)", (int)kv_layout);
    if (nnz < 0 || batch < 0 || num_pages < 0)
        return fail(PAFP8_ERR_SHAPE, "nnz %lld, batch %d and num_pages %d must not be negative",
                    (long long)nnz, (int)batch, (int)num_pages);
    if (num_kv_heads <= 0)
        return fail(PAFP8_ERR_SHAPE, "num_kv_heads %d must be positive", (int)num_kv_heads);
    if (head_dim != kHeadDim && head_dim != 64)
        return fail(PAFP8_ERR_UNSUPPORTED, "head_dim %d is not served by this library (%d or 64)",
                    (int)head_dim, kHeadDim);
    if (page_size <= 0 || page_size % kPageSize != 0)
        return fail(PAFP8_ERR_UNSUPPORTED, "page_size %d is not served by this library (a multiple of %d)",
                    (int)page_size, kPageSize);
    if (!scale_ok(k_scale) || !scale_ok(v_scale))
        return fail(PAFP8_ERR_ARG, "scales must be finite and > 0 (k %g, v %g)", (double)k_scale,
                    (double)v_scale);
    if (nnz == 0) return PAFP8_OK;
    if (k_new == nullptr || v_new == nullptr || k_cache == nullptr || v_cache == nullptr ||
        batch_indices == nullptr || positions == nullptr || kv_indptr == nullptr || kv_indices == nullptr)
        return fail(PAFP8_ERR_ARG,
                    "k_new, v_new, k_cache, v_cache, batch_indices, positions, kv_indptr and "
                    "kv_indices must be non-NULL");
    if (((uintptr_t)k_new | (uintptr_t)v_new | (uintptr_t)k_cache | (uintptr_t)v_cache) % 16 != 0)
        return fail(PAFP8_ERR_ARG, "k_new, v_new, k_cache and v_cache must be 16-byte aligned");
    if (((uintptr_t)batch_indices | (uintptr_t)positions | (uintptr_t)kv_indptr | (uintptr_t)kv_indices |
         (uintptr_t)status) % 4 != 0)
        return fail(PAFP8_ERR_ARG, "batch_indices, positions, kv_indptr, kv_indices and status must be "
                                   "4-byte aligned");
    AppendParams p{};
    p.k_new = k_new;
    p.v_new = v_new;
    p.batch_indices = batch_indices;
    p.positions = positions;
    p.kv_indptr = kv_indptr;
    p.kv_indices = kv_indices;
    p.k_cache = k_cache;
    p.v_cache = v_cache;
    p.status = status;
    p.nnz = (long long)nnz;
    p.num_kv_heads = num_kv_heads;
    p.batch = batch;
    p.num_pages = num_pages;
    p.src_dtype = src_dtype;
    p.kv_dtype = kv_dtype;
    p.hnd = kv_layout == PAFP8_LAYOUT_HND;
    p.page_size = page_size;
    p.head_dim = head_dim;
    p.k_inv = 1.0f / k_scale;  // IEEE fp32 division: fp32(1/scale)
    p.v_inv = 1.0f / v_scale;
    const cudaError_t e = launch_append(p, (cudaStream_t)stream);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(PAFP8_ERR_CUDA, "append kernel launch failed: %s", cudaGetErrorString(e));
    }
    return PAFP8_OK;
}

}  // extern "C"
