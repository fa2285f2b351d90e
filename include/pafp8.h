/*
 * pafp8.h -- C ABI of libpafp8: batched attention of a query against a paged
 * KV cache stored in fp8 (OCP e4m3fn or e5m2) with per-tensor scales, for
 * NVIDIA GB300 (sm_103a).
 *
 * Two workloads share one plan/run interface:
 *   - decode: one query row per request against its whole KV sequence; the
 *     plan splits long sequences across CTAs and a merge kernel combines the
 *     partial states by their log-sum-exp;
 *   - prefill: a ragged batch of new query rows per request, bottom-right
 *     aligned causal mask (query row i of a request with qo_len new rows and
 *     kv_len keys sees key j iff j <= i + kv_len - qo_len).
 *
 * The plan()/run() split, o_data_type fixed at plan time and checked at run
 * time, and the scale threading follow "Enable Hopper FA3 FP8 attention in
 * decode.py" (flashinfer PR 2148), Changes table and review notes on
 * o_data_type and the FP8 scales.  The dtype refusals follow "fp8 KV cache in
 * the in-tree prefill kernel" (AMD-Ecosystem/flashinfer PR 368), What changed
 * / Refusals and Architecture / design notes.
 *
 * Conventions shared by every entry point:
 *   - Device pointers are plain CUDA device addresses; host pointers are
 *     ordinary host memory.  The caller owns every buffer, the stream and the
 *     workspace; the library owns only the plan object.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default).
 *   - Every function returns a pafp8_status; on failure pafp8_last_error()
 *     returns a sentence naming the offending values (thread-local, valid
 *     until the next failing call on this thread).  Nothing aborts.
 *   - pafp8_run neither allocates nor synchronizes, unless PAFP8_DEBUG is
 *     set in the environment (to anything but "0"): then every run call that
 *     launches (pafp8_run, _stage, _head_scales, _pod) synchronizes its
 *     stream and returns the kernels' status as pafp8_device_status reports
 *     it (PAFP8_ERR_BOUNDS, PAFP8_ERR_TIMEOUT), so a bad page index or an
 *     expired wait surfaces at the call that caused it.  Not for use under
 *     stream capture.
 *   - Every wait inside a kernel is bounded (about one second of SM clock).
 *     On expiry the kernel records PAFP8_ERR_TIMEOUT in the workspace status
 *     word, lets its own copies and MMAs in flight finish, frees its tensor
 *     memory and returns; the workspace and context stay usable.  The
 *     diagnostic setting PAFP8_WAIT_CYCLES (a positive integer, in SM clock
 *     cycles, read by each launching call) shortens the bound of the
 *     pipeline waits, so that a test can make one expire on purpose.
 */
#ifndef PAFP8_H
#define PAFP8_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define PAFP8_ABI_VERSION 1

/* Element types, as int32 codes.  F32, INT8 and UINT8 exist only so that a
 * caller holding such a tensor gets a refusal naming it: an integer cache has
 * no floating-point reading, and reading its bytes as fp8 (or as 0..255) is
 * the silent misread the in-tree prefill page (Architecture / design notes,
 * "kv_smem_type_t keys on the fp8 types") rules out. */
enum {
    PAFP8_DTYPE_DEFAULT = 0, /* only for plan desc o_dtype: see below */
    PAFP8_F16 = 1,
    PAFP8_BF16 = 2,
    PAFP8_E4M3FN = 3,
    PAFP8_E5M2 = 4,
    PAFP8_F32 = 5,
    PAFP8_INT8 = 6,
    PAFP8_UINT8 = 7
};

typedef enum pafp8_status {
    PAFP8_OK = 0,
    PAFP8_ERR_DTYPE = 1,       /* dtype not served, or differs from the plan */
    PAFP8_ERR_SHAPE = 2,       /* head counts, head_dim, page size, lengths  */
    PAFP8_ERR_ARG = 3,         /* NULL pointer, bad scale, bad option        */
    PAFP8_ERR_WORKSPACE = 4,   /* workspace too small / plan not uploaded    */
    PAFP8_ERR_CUDA = 5,        /* a CUDA runtime call failed                 */
    PAFP8_ERR_TIMEOUT = 6,     /* a kernel's bounded wait expired            */
    PAFP8_ERR_BOUNDS = 7,      /* a page index outside [0, num_pages)        */
    PAFP8_ERR_UNSUPPORTED = 8  /* valid request this library does not serve  */
} pafp8_status;

enum { PAFP8_MODE_DECODE = 0, PAFP8_MODE_PREFILL = 1 };

/* Layout of k_cache / v_cache (head_dim is always innermost):
 *   NHD  [num_pages, page_size, num_kv_heads, head_dim]  (token-major page)
 *   HND  [num_pages, num_kv_heads, page_size, head_dim]  (head-major page)
 * The pages fix no layout beyond separate K and V caches with head_dim last
 * ("Enable Hopper FA3 FP8 attention in decode.py", review note on
 * v_cache.shape[-1:]); NHD is the default and HND the head-major variant,
 * read by the same kernels through differently strided tensor maps. */
enum { PAFP8_LAYOUT_NHD = 0, PAFP8_LAYOUT_HND = 1 };

/* Static description of one batch.  Shapes served by this library:
 * head_dim 128 or 64; page_size a multiple of 16 in either layout, a page of 16 m tokens
 * being read as m 16-token sub-pages (token slots 16 j .. 16 j + 15 of every head, so
 * num_pages * page_size / 16 must stay below 2^31); num_qo_heads a multiple of num_kv_heads with
 * group size num_qo_heads/num_kv_heads <= 8 (decode) or <= 16 (prefill).
 *
 * Dtype rules (checked by pafp8_plan_create, re-checked by pafp8_run):
 *   kv_dtype   E4M3FN or E5M2.  Decode also takes an F16 or BF16 cache
 *              with an F16 or BF16 query in any mix ("fp8 KV cache in the
 *              in-tree prefill kernel", Test plan: decode is exempt from the
 *              rule that the cache matches the query); an fp8 query with a
 *              2-byte cache, and a 2-byte cache in prefill, are refused.  An
 *              fp8 cache and its exact f16 widening give bit-identical decode
 *              results.  F32/INT8/UINT8 caches are refused with their own
 *              sentence.
 *   q_dtype    F16 or BF16 (a 2-byte query against the fp8 cache, which is
 *              dequantized on load), or E4M3FN/E5M2 (an fp8 query; q_scale
 *              then folds into sm_scale like the FP8 BMM1 scale).
 *   o_dtype    F16 or BF16.  fp8 outputs are refused (fp8 inputs produce a
 *              16-bit output).  DEFAULT means q_dtype for a 2-byte query and
 *              BF16 for an fp8 query.
 * sm_scale     softmax scale applied to q.k; <= 0 means 1/sqrt(head_dim).
 * Split-KV options (decode; prefill ignores them):
 *   fixed_split_pages > 0  every request is cut into chunks of that many pages;
 *   disable_split_kv != 0  one chunk per request;
 *   otherwise              balanced: the concatenated pages of all
 *                          (request, KV-head block) rows are cut into
 *                          num_ctas equal ranges, one per CTA.
 * num_ctas     persistent CTAs to launch; 0 = the SM count of the device that
 *              is current when the plan is created.
 * kv_layout    NHD (0, also what a zeroed description gives) or HND; the
 *              caches given to pafp8_run are read in that layout. */
typedef struct pafp8_plan_desc {
    int32_t mode;  /* PAFP8_MODE_DECODE or PAFP8_MODE_PREFILL */
    int32_t batch;
    int32_t num_qo_heads;
    int32_t num_kv_heads;
    int32_t head_dim;
    int32_t page_size;
    int32_t num_pages; /* pages in the cache pool (rows of k_cache/v_cache) */
    int32_t q_dtype;
    int32_t kv_dtype;
    int32_t o_dtype;
    float sm_scale;
    int32_t fixed_split_pages;
    int32_t disable_split_kv;
    int32_t num_ctas;
    int32_t kv_layout; /* PAFP8_LAYOUT_NHD (0) or PAFP8_LAYOUT_HND (1) */
} pafp8_plan_desc;

typedef struct pafp8_plan pafp8_plan;

/* ABI version of the loaded library (PAFP8_ABI_VERSION at build time). */
int32_t pafp8_abi_version(void);

/* Thread-local sentence describing the last failure on this thread ("" if
 * none).  The pointer stays valid until the next failing call. */
const char *pafp8_last_error(void);

/* Build a plan on the host.  No device memory is touched.
 *   kv_indptr_h     host int32 [batch+1], non-decreasing, kv_indptr_h[0] = 0;
 *                   request b owns pages kv_indices[kv_indptr_h[b] ..
 *                   kv_indptr_h[b+1]-1], in token order.
 *   last_page_len_h host int32 [batch], in [1, page_size] for a request with
 *                   pages (its kv_len = (npages-1)*page_size + last_page_len);
 *                   ignored for a request with no pages (kv_len 0: output 0,
 *                   lse -inf).
 *   qo_indptr_h     host int32 [batch+1] for prefill (request b owns query
 *                   rows qo_indptr_h[b] .. qo_indptr_h[b+1]-1, with
 *                   qo_len <= kv_len); NULL for decode (row b is request b).
 * The arrays are copied; the caller may free them after the call.  On
 * success *out owns a plan freed by pafp8_plan_destroy.  Planning runs on the
 * calling host thread in time linear in batch, num_ctas and the number of
 * segments (a decode plan for 64 requests on 152 CTAs takes a few
 * microseconds), touches no device memory and, with num_ctas given, makes no
 * CUDA call. */
pafp8_status pafp8_plan_create(const pafp8_plan_desc *desc, const int32_t *kv_indptr_h,
                               const int32_t *last_page_len_h, const int32_t *qo_indptr_h,
                               pafp8_plan **out);

/* Free a plan (NULL is ignored). */
void pafp8_plan_destroy(pafp8_plan *plan);

/* Bytes of device workspace pafp8_run needs for this plan: the uploaded
 * partition metadata, the split-KV partial states and a status word. */
size_t pafp8_workspace_bytes(const pafp8_plan *plan);

/* Read-only host view of the plan's partition metadata, the exact int32 words
 * pafp8_plan_upload copies to the device (layout in the library source).
 * Owned by the plan. */
pafp8_status pafp8_plan_metadata(const pafp8_plan *plan, const int32_t **words, size_t *count);

/* Copy the plan's metadata into the head of `workspace` (device memory of at
 * least pafp8_workspace_bytes) on `stream` and clear its status block.  Must
 * precede pafp8_run with this workspace; the plan records the workspace
 * address and pafp8_run refuses any other.  Outside stream capture the copy
 * goes through a small page-locked staging ring owned by the library (up to
 * four buffers per device, allocated on first use and kept until the process
 * exits; a buffer is reused after the copy that last read it has run), so the
 * host may destroy or re-plan right after the call; under capture it copies
 * from the plan's own memory, which must then outlive the graph. */
pafp8_status pafp8_plan_upload(pafp8_plan *plan, void *workspace, size_t workspace_bytes,
                               void *stream);

/* Launch the attention for the planned batch on `stream`.
 *   q           device, [nnz_qo, num_qo_heads, head_dim] of q_dtype
 *               (nnz_qo = batch for decode, qo_indptr_h[batch] for prefill)
 *   k_cache,
 *   v_cache     device, [num_pages, page_size, num_kv_heads, head_dim] (NHD)
 *               or [num_pages, num_kv_heads, page_size, head_dim] (HND, as
 *               planned) of kv_dtype, 16-byte aligned
 *   kv_indices  device int32 [kv_indptr_h[batch]], each in [0, num_pages)
 *   q_scale     dequantization scale of an fp8 query; must be 1 for a 2-byte
 *               query (it would otherwise be silently ignored)
 *   k_scale,
 *   v_scale     per-tensor dequantization scales of the cache.  k_scale (and
 *               q_scale) fold into sm_scale; v_scale multiplies the output
 *               once, in fp32, before the cast.  Finite and > 0.
 *   o           device, [nnz_qo, num_qo_heads, head_dim] of o_dtype
 *   lse         device float [nnz_qo, num_qo_heads] or NULL: natural-log
 *               log-sum-exp of the scaled logits (sm_scale, q_scale and
 *               k_scale included; v_scale not)
 *   workspace   the buffer given to pafp8_plan_upload for this plan
 * The dtype arguments must equal the planned ones, and k_dtype must equal
 * v_dtype.  A page index out of range is not read (the kernel records it in
 * the workspace status word; see pafp8_device_status). */
pafp8_status pafp8_run(const pafp8_plan *plan, int32_t q_dtype, const void *q,
                       int32_t k_dtype, const void *k_cache, int32_t v_dtype, const void *v_cache,
                       const int32_t *kv_indices, float q_scale, float k_scale, float v_scale,
                       int32_t o_dtype, void *o, float *lse, void *workspace,
                       size_t workspace_bytes, void *stream);

/* One step of the plan from and to host memory, for callers whose q,
 * kv_indices, o and lse live on the host (the same attention as pafp8_run).
 * On `stream`, in this order: the plan's metadata is uploaded to `workspace`
 * (as pafp8_plan_upload), q and kv_indices are copied from host memory into
 * a staging area at the end of `workspace`, the attention runs on them (as
 * pafp8_run), and o and lse are copied back into host memory.  The call
 * returns once all of it is enqueued; o_h and lse_h hold the results when the
 * stream has reached this point (e.g. after cudaStreamSynchronize or an event
 * recorded after the call).
 *   q_h          host, [nnz_qo, num_qo_heads, head_dim] of q_dtype
 *   kv_indices_h host int32 [kv_indptr_h[batch]] (may be NULL if that is 0)
 *   o_h          host, [nnz_qo, num_qo_heads, head_dim] of o_dtype
 *   lse_h        host float [nnz_qo, num_qo_heads] or NULL
 *   workspace    device, 256-byte aligned, at least
 *                pafp8_host_workspace_bytes(plan, q_dtype) bytes; the caller
 *                owns it and must not reuse it (nor the host buffers) until
 *                the stream has passed this call
 * The host buffers should be page-locked (cudaHostAlloc / pinned) for the
 * copies to be asynchronous; pageable memory works but the copies then
 * synchronize with the host.  Other arguments and checks are those of
 * pafp8_run; on a refusal by those checks the metadata upload may already be
 * enqueued, nothing else is. */
size_t pafp8_host_workspace_bytes(const pafp8_plan *plan, int32_t q_dtype);
pafp8_status pafp8_run_host(pafp8_plan *plan, int32_t q_dtype, const void *q_h, int32_t k_dtype,
                            const void *k_cache, int32_t v_dtype, const void *v_cache,
                            const int32_t *kv_indices_h, float q_scale, float k_scale, float v_scale,
                            int32_t o_dtype, void *o_h, float *lse_h, void *workspace,
                            size_t workspace_bytes, void *stream);

/* pafp8_run restricted to one stage of the launch sequence, for callers that
 * time or overlap the stages separately:
 *   stage 0  everything (same as pafp8_run);
 *   stage 1  the attention kernel only (decode: it writes the outputs of
 *            unsplit requests and of requests with no KV, and the partial
 *            states of split ones);
 *   stage 2  the split-KV merge only (decode: combines the partial states
 *            of split requests; launched as a programmatic dependent of the
 *            preceding kernel on the stream); prefill has no stage 2.
 * Running stage 1 then stage 2 on one stream equals stage 0.  Arguments and
 * checks are those of pafp8_run. */
pafp8_status pafp8_run_stage(const pafp8_plan *plan, int32_t stage, int32_t q_dtype, const void *q,
                             int32_t k_dtype, const void *k_cache, int32_t v_dtype,
                             const void *v_cache, const int32_t *kv_indices, float q_scale,
                             float k_scale, float v_scale, int32_t o_dtype, void *o, float *lse,
                             void *workspace, size_t workspace_bytes, void *stream);

/* pafp8_run with per-head scale tensors in place of the per-tensor scales:
 * the "FP8 scale tensors" that "Enable Hopper FA3 FP8 attention in
 * decode.py" threads through the backends (Changes table; review note "FP8
 * scale tensor passing"), read here as one scale per head.
 *   q_scales  device float [num_qo_heads], or NULL (1 for every head).  An
 *             fp8 query only; must be NULL for a 2-byte query.
 *   k_scales,
 *   v_scales  device float [num_kv_heads], required: the dequantization
 *             scales of KV head j's codes.
 * Query head h uses q_scales[h], k_scales[h / group] and v_scales[h / group]
 * the way pafp8_run uses its scalars; the softmax scale is folded per head in
 * double, in the order pafp8_run folds it, so equal entries give pafp8_run's
 * result bit for bit.  The entries must be finite and > 0 (device memory,
 * not checked).  Every other argument and check is pafp8_run's. */
pafp8_status pafp8_run_head_scales(const pafp8_plan *plan, int32_t q_dtype, const void *q,
                                   int32_t k_dtype, const void *k_cache, int32_t v_dtype,
                                   const void *v_cache, const int32_t *kv_indices,
                                   const float *q_scales, const float *k_scales,
                                   const float *v_scales, int32_t o_dtype, void *o, float *lse,
                                   void *workspace, size_t workspace_bytes, void *stream);

/* Synchronize `stream`, read and clear the workspace status word that the
 * kernels set.  Returns PAFP8_OK, PAFP8_ERR_BOUNDS (a page index was out of
 * range) or PAFP8_ERR_TIMEOUT (a bounded pipeline wait expired). */
pafp8_status pafp8_device_status(const pafp8_plan *plan, void *workspace, void *stream);

/* Decode without a workspace argument, for callers that may not allocate
 * device memory themselves: for example an inference engine's plugin or
 * enqueue callback that runs on a stream the host framework owns, where
 * cudaMalloc is off limits because it can synchronize the device and the
 * framework hands out all device memory.  Such callers still pass q, the
 * cache, kv_indices, o and lse (their own buffers); the plan's metadata, the
 * split-KV partial states and the status word go to a scratch array built
 * into the library instead of a caller workspace.  This entry point has no
 * counterpart on the pages the method comes from; it is a deployment
 * convenience of this library.
 *
 * Arguments and checks are those of pafp8_run for a decode plan (prefill
 * plans are refused).  The scratch holds 16 MiB (PAFP8_NOALLOC_SCRATCH_BYTES)
 * on every GPU that loads the library, until the process exits; a plan whose
 * pafp8_workspace_bytes exceeds it is refused with PAFP8_ERR_WORKSPACE
 * (fewer CTAs or splits shrink it).  The first call on a device looks up the
 * scratch's device address (cudaGetSymbolAddress) with that device current,
 * so make it before any stream capture.  No call allocates or frees device
 * memory.  Every call re-loads its plan's metadata into the scratch (a
 * cudaMemcpyAsync on `stream` whose source is the plan's own host memory,
 * which is ordinary pageable memory) and clears the status word (a
 * cudaMemsetAsync on `stream`), so a call never depends on the previous
 * call's contents; but all calls share the one array, so calls that can
 * overlap on the GPU (different streams, or different threads without
 * ordering) race and must be serialized by the caller.  Page-index and
 * timeout reports: with PAFP8_DEBUG set (see pafp8_run) the call synchronizes
 * and returns the kernels' status (PAFP8_ERR_BOUNDS, PAFP8_ERR_TIMEOUT);
 * otherwise the status word stays internal. */
#define PAFP8_NOALLOC_SCRATCH_BYTES (16u << 20)
pafp8_status pafp8_run_decode_noalloc(const pafp8_plan *plan, int32_t q_dtype, const void *q,
                                      int32_t k_dtype, const void *k_cache, int32_t v_dtype,
                                      const void *v_cache, const int32_t *kv_indices,
                                      float q_scale, float k_scale, float v_scale,
                                      int32_t o_dtype, void *o, float *lse, void *stream);

/* Prefill and decode over one paged cache in one call ("POD": the pages'
 * POD and batch-POD kernels, "fp8 KV cache in the in-tree prefill kernel"
 * (AMD-Ecosystem/flashinfer PR 368), Refusals, run a prefill batch and a
 * decode batch together by reusing the prefill kernel's traits, and refuse an
 * fp8 cache).  Here both phases run this library's own kernels, so every
 * cache type pafp8_run serves is served, fp8 included.
 *
 * The prefill kernel is compute-bound on the tensor cores and the decode
 * kernel bound by HBM; run together on disjoint SMs each uses what the other
 * leaves.  The two phases are two grids launched from this one call: the
 * decode kernel (and its split-KV merge) on a side stream of the decode plan,
 * at the device's highest stream priority, forked from `stream` by an event
 * and joined back to it; the prefill kernel on `stream`.  The SM split is the
 * plans' num_ctas: a prefill plan made with num_ctas = Np and a decode plan
 * with Nd run side by side when Np + Nd <= the SM count (152 on GB300); a
 * larger sum is still correct, the CTAs beyond it waiting for free SMs.  On a
 * few SMs the decode phase is bound by its per-SM rate (about 60 GB/s of KV
 * per SM on GB300), so the best Nd balances decode bytes / (Nd * 60 GB/s)
 * against the prefill's time on the other SMs: 20 of 152 for a 304 MB decode
 * batch beside a 236 us prefill.
 *
 *   prefill   the prefill phase: a plan of PAFP8_MODE_PREFILL and its q,
 *             kv_indices, o, lse and uploaded workspace, as pafp8_run takes
 *             them
 *   decode    the decode phase: a plan of PAFP8_MODE_DECODE and its buffers
 *   k_cache,
 *   v_cache   the one cache both phases read; both plans must describe it
 *             alike (num_pages, page_size, num_kv_heads, head_dim, kv_layout)
 * The dtypes and scales apply to both phases, and each phase is checked as
 * pafp8_run checks it, before anything is launched.  The two workspaces must
 * not overlap.  Each phase's results are bit-identical to pafp8_run of its
 * plan alone.  On return `stream` is ordered after both phases.  The first
 * call with a decode plan creates that plan's side stream and two events
 * (make it outside stream capture); pafp8_plan_destroy releases them.  Later
 * calls create nothing; nothing is allocated on the device or synchronized.
 * A plan is not to be used by two threads at once. */
typedef struct pafp8_pod_phase {
    const pafp8_plan *plan;
    const void *q;
    const int32_t *kv_indices;
    void *o;
    float *lse;
    void *workspace;
    size_t workspace_bytes;
} pafp8_pod_phase;

pafp8_status pafp8_run_pod(const pafp8_pod_phase *prefill, const pafp8_pod_phase *decode,
                           int32_t q_dtype, int32_t k_dtype, const void *k_cache, int32_t v_dtype,
                           const void *v_cache, float q_scale, float k_scale, float v_scale,
                           int32_t o_dtype, void *stream);

/* Quantize new K/V tokens into the paged fp8 cache: the step that writes the
 * cache every other entry point reads.  The pages take such a cache as given
 * (fp8 K/V with per-tensor k_scale/v_scale, dequantized as code * scale, "fp8
 * KV cache in the in-tree prefill kernel", What changed and Test plan); the
 * inverse of that dequantization is this library's reading:
 *
 *   code = fp8(RNE, saturating)( fp32(x) * fp32(1 / scale) )
 *
 * in IEEE fp32 (1/scale rounded once, the product rounded once), then rounded
 * to the nearest kv_dtype value with ties to even; magnitudes above the
 * largest finite value (e4m3fn 448, e5m2 57344), infinities included, store
 * that value with their sign; +-0 keep their sign; NaN stores a NaN code.
 *
 *   src_dtype      F16, BF16 or F32: the type of the new tokens
 *   k_new, v_new   device [nnz, num_kv_heads, head_dim] of src_dtype,
 *                  16-byte aligned
 *   nnz            new tokens (0: nothing is launched)
 *   batch_indices  device int32 [nnz]: request of each new token
 *   positions      device int32 [nnz]: the token's position in its request's
 *                  KV sequence; it goes to page kv_indices[kv_indptr[b] +
 *                  pos / page_size], slot pos % page_size
 *   batch          requests in kv_indptr
 *   kv_indptr      device int32 [batch + 1], kv_indices device int32
 *                  [kv_indptr[batch]]: the page table of pafp8_plan_create /
 *                  pafp8_run (already covering the new tokens)
 *   kv_dtype       E4M3FN or E5M2 (the cache's format; 2-byte caches and
 *                  every other dtype are refused)
 *   kv_layout      PAFP8_LAYOUT_NHD or PAFP8_LAYOUT_HND
 *   k_cache,
 *   v_cache        device caches of kv_dtype in that layout, 16-byte aligned;
 *                  only the new tokens' rows are written
 *   k_scale,
 *   v_scale        the per-tensor scales the cache is read with; finite, > 0
 *   status         device uint32 or NULL: the kernel ORs in 1 for a token it
 *                  did not write because its request index, position or page
 *                  index lies outside the table or the pool
 * Shapes served: head_dim 128 or 64; page_size a multiple of 16 (NHD) or 16
 * (HND).  Nothing is allocated or synchronized. */
pafp8_status pafp8_append_kv(int32_t src_dtype, const void *k_new, const void *v_new, int64_t nnz,
                             int32_t num_kv_heads, int32_t head_dim, const int32_t *batch_indices,
                             const int32_t *positions, int32_t batch, const int32_t *kv_indptr,
                             const int32_t *kv_indices, int32_t kv_dtype, int32_t kv_layout,
                             void *k_cache, void *v_cache, int32_t num_pages, int32_t page_size,
                             float k_scale, float v_scale, uint32_t *status, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* PAFP8_H */
