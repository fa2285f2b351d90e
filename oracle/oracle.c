/*
 * oracle.c -- plain, slow, fp64 CPU statement of paged attention over an
 * fp8 KV cache.  TEST INFRASTRUCTURE ONLY: the tests, the package smoke check
 * and the benchmark's CPU-baseline leg call it; the product library never
 * does, and this file shares no code, header or table with the CUDA path.
 *
 * What it computes is "dequantize, then attend", written out literally:
 *
 *   1. fp8 codes are decoded from the OCP format definitions (sign,
 *      exponent, mantissa), never through a library cast.  The two formats
 *      and their exponent biases (e4m3fn bias 7, e5m2 bias 15) are the ones
 *      named on "fp8 KV cache in the in-tree prefill kernel", Architecture /
 *      design notes ("The OCP spellings are refused rather than mapped").
 *   2. K^ = decode(k) * k_scale, V^ = decode(v) * v_scale, Q^ = decode(q) *
 *      q_scale.  Applying the scales to the dequantized values is the
 *      definition that the two folds on "fp8 KV cache in the in-tree prefill
 *      kernel", Test plan (k_scale into sm_scale, v_scale linear on the
 *      output) are equivalent to.  The query scale is the FP8 BMM1 scale of
 *      "Enable Hopper FA3 FP8 attention in decode.py", review note on q_scale.
 *      The scales may instead be per-head scale tensors (the "FP8 scale
 *      tensors" that page threads through): q_scale[h] for query head h,
 *      k_scale[h_kv] and v_scale[h_kv] for KV head h_kv, applied the same way.
 *   3. The KV rows of request b are gathered through the CSR page table
 *      (kv_indptr, kv_indices, last_page_len): token t lives in page
 *      kv_indices[kv_indptr[b] + t / P], slot t % P.
 *   4. Query head h reads KV head h / (Hq / Hkv) (contiguous GQA groups,
 *      "GQA 32/8" in the benchmark section of the in-tree prefill page).
 *   5. s_j = sm_scale * sum_d Q^_d K^_jd over the keys the causal rule
 *      admits: query row i (0-based among the request's qo_len new rows)
 *      sees key j iff j <= i + kv_len - qo_len (bottom-right aligned);
 *      decode is qo_len = 1, which admits every key.
 *   6. m = max_j s_j, l = sum_j exp(s_j - m), o = sum_j exp(s_j - m)/l V^_j,
 *      lse = m + ln l (natural log).  No admissible key: o = 0, lse = -inf.
 *
 * Everything is two-pass and fp64; there is no blocking, fusion, online
 * rescaling or reordering beyond the definition.  OpenMP (when compiled with
 * -fopenmp) only distributes independent (row, head) outputs over threads.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Element encodings the oracle can decode.  These numbers are the oracle's
 * own; its Python wrapper maps dtype names onto them. */
enum {
    ORC_F16 = 1,
    ORC_BF16 = 2,
    ORC_E4M3FN = 3,
    ORC_E5M2 = 4,
};

/* ---- 1. element decoders, from the format definitions ------------------ */

/* OCP FP8 E4M3 ("fn": finite, no infinities).  1 sign, 4 exponent bits with
 * bias 7, 3 mantissa bits.  Exponent field 0 is subnormal (m/8 * 2^-6).
 * S.1111.111 is NaN; every other code is finite, so the largest is
 * 0.1111.110 = 1.75 * 2^8 = 448. */
double orc_decode_e4m3fn(uint8_t code) {
    int s = (code >> 7) & 1;
    int e = (code >> 3) & 0xF;
    int m = code & 0x7;
    double mag;
    if (e == 0xF && m == 0x7) return NAN;
    if (e == 0) mag = ldexp((double)m / 8.0, -6);
    else        mag = ldexp(1.0 + (double)m / 8.0, e - 7);
    return s ? -mag : mag;
}

/* OCP FP8 E5M2.  1 sign, 5 exponent bits with bias 15, 2 mantissa bits,
 * IEEE-style specials: exponent 31 is +-inf (m = 0) or NaN (m != 0);
 * exponent 0 is subnormal (m/4 * 2^-14).  Largest finite: 1.75 * 2^15. */
double orc_decode_e5m2(uint8_t code) {
    int s = (code >> 7) & 1;
    int e = (code >> 2) & 0x1F;
    int m = code & 0x3;
    double mag;
    if (e == 0x1F) {
        if (m != 0) return NAN;
        return s ? -INFINITY : INFINITY;
    }
    if (e == 0) mag = ldexp((double)m / 4.0, -14);
    else        mag = ldexp(1.0 + (double)m / 4.0, e - 15);
    return s ? -mag : mag;
}

/* IEEE binary16: 1 sign, 5 exponent (bias 15), 10 mantissa bits. */
double orc_decode_f16(uint16_t bits) {
    int s = (bits >> 15) & 1;
    int e = (bits >> 10) & 0x1F;
    int m = bits & 0x3FF;
    double mag;
    if (e == 0x1F) {
        if (m != 0) return NAN;
        return s ? -INFINITY : INFINITY;
    }
    if (e == 0) mag = ldexp((double)m / 1024.0, -14);
    else        mag = ldexp(1.0 + (double)m / 1024.0, e - 15);
    return s ? -mag : mag;
}

/* bfloat16: 1 sign, 8 exponent (bias 127), 7 mantissa bits. */
double orc_decode_bf16(uint16_t bits) {
    int s = (bits >> 15) & 1;
    int e = (bits >> 7) & 0xFF;
    int m = bits & 0x7F;
    double mag;
    if (e == 0xFF) {
        if (m != 0) return NAN;
        return s ? -INFINITY : INFINITY;
    }
    if (e == 0) mag = ldexp((double)m / 128.0, -126);
    else        mag = ldexp(1.0 + (double)m / 128.0, e - 127);
    return s ? -mag : mag;
}

static int orc_elem_bytes(int dtype) {
    switch (dtype) {
        case ORC_F16: case ORC_BF16: return 2;
        case ORC_E4M3FN: case ORC_E5M2: return 1;
        default: return 0;
    }
}

static double orc_decode_one(int dtype, const void *base, int64_t idx) {
    switch (dtype) {
        case ORC_F16:    return orc_decode_f16(((const uint16_t *)base)[idx]);
        case ORC_BF16:   return orc_decode_bf16(((const uint16_t *)base)[idx]);
        case ORC_E4M3FN: return orc_decode_e4m3fn(((const uint8_t *)base)[idx]);
        case ORC_E5M2:   return orc_decode_e5m2(((const uint8_t *)base)[idx]);
        default:         return NAN;
    }
}

/* Decode n elements of `dtype` into fp64.  Returns 0, or -1 for an unknown
 * dtype. */
int orc_decode_array(int dtype, const void *src, int64_t n, double *dst) {
    if (orc_elem_bytes(dtype) == 0) return -1;
    for (int64_t i = 0; i < n; ++i) dst[i] = orc_decode_one(dtype, src, i);
    return 0;
}

/* Element offset of the row of (page, slot, KV head) in a cache laid out
 * NHD [num_pages][P][Hkv][D] (kv_layout 0) or HND [num_pages][Hkv][P][D]
 * (kv_layout 1). */
static int64_t orc_row_offset(int kv_layout, int64_t page, int64_t slot, int64_t h, int64_t P,
                              int64_t Hkv, int64_t D) {
    if (kv_layout == 1) return ((page * Hkv + h) * P + slot) * D;
    return ((page * P + slot) * Hkv + h) * D;
}

/* ---- 7. writing new tokens into the cache -----------------------------
 *
 * The inverse of step 2 for K and V.  The pages take the fp8 cache as given
 * (codes whose decoded values times the per-tensor scale are the keys and
 * values); writing a new row is read here as
 *
 *   y    = fl32( fl32(x) * fl32(1 / scale) )          (IEEE single, RNE)
 *   code = the format's value nearest to y, a tie going to the code whose
 *          mantissa LSB is 0; magnitudes above the largest finite value
 *          (e4m3fn 448, e5m2 57344), infinities included, store that value
 *          with their sign; +0 and -0 keep their sign; NaN stores 0x7F,
 *          a NaN code in both formats.
 *
 * The rounding is done on exact doubles: y / spacing is an exact power-of-two
 * scaling, and nearbyint() in the default rounding mode rounds half to even. */
uint8_t orc_encode_fp8(int fmt, float y) {
    const int mbits = fmt == ORC_E4M3FN ? 3 : 2;
    const int bias = fmt == ORC_E4M3FN ? 7 : 15;
    const double maxv = fmt == ORC_E4M3FN ? 448.0 : 57344.0;
    if (isnan(y)) return 0x7F;
    const uint8_t sign = signbit(y) ? 0x80 : 0x00;
    double a = fabs((double)y);
    if (a > maxv) a = maxv; /* saturation; beyond the largest value every value rounds to it or past it */
    /* Spacing of the values around a: 2^(E - mbits) in the binade [2^E, 2^(E+1)) of a normal
     * value, 2^(1 - bias - mbits) below the smallest normal 2^(1 - bias). */
    int E = 1 - bias;
    if (a >= ldexp(1.0, 1 - bias)) {
        frexp(a, &E);
        E -= 1;
    }
    const double step = ldexp(1.0, E - mbits);
    double v = nearbyint(a / step) * step;
    if (v > maxv) v = maxv;
    if (v == 0.0) return sign;
    int ev;
    frexp(v, &ev);
    ev -= 1; /* v = 1.f * 2^ev */
    if (ev < 1 - bias) /* subnormal: exponent field 0, mantissa = v / smallest spacing */
        return (uint8_t)(sign | (uint8_t)(v / ldexp(1.0, 1 - bias - mbits)));
    const int mant = (int)((v / ldexp(1.0, ev) - 1.0) * (double)(1 << mbits));
    return (uint8_t)(sign | (uint8_t)(((ev + bias) << mbits) | mant));
}

/* codes[i] = encode(fl32(x[i] * fl32(1 / scale))).  Returns 0, or -1 for a
 * format that is not fp8. */
int orc_quantize_array(int fmt, const float *x, int64_t n, float scale, uint8_t *codes) {
    if (fmt != ORC_E4M3FN && fmt != ORC_E5M2) return -1;
    const float inv = 1.0f / scale; /* single precision throughout (FLT_EVAL_METHOD 0) */
    for (int64_t i = 0; i < n; ++i) {
        const float y = x[i] * inv;
        codes[i] = orc_encode_fp8(fmt, y);
    }
    return 0;
}

/* Write nnz new tokens (rows [nnz, hkv, d] of k_new and v_new, as fp32) into
 * the paged caches (NHD [num_pages, page_size, hkv, d] for kv_layout 0, HND
 * [num_pages, hkv, page_size, d] for 1) of fp8 codes: token i of
 * request b = batch_idx[i] at position p = pos[i] goes to page
 * kv_indices[kv_indptr[b] + p / page_size], slot p % page_size (the gather of
 * step 3, written instead of read).  A token whose request, position or page
 * is outside the table or the pool is not written.  Returns the number of
 * tokens not written, or -1 for a format that is not fp8. */
int64_t orc_append_kv(int fmt, const float *k_new, const float *v_new, int64_t nnz, int hkv, int d,
                      const int32_t *batch_idx, const int32_t *pos, int batch, const int32_t *kv_indptr,
                      const int32_t *kv_indices, int num_pages, int page_size, int kv_layout,
                      float k_scale, float v_scale, uint8_t *k_cache, uint8_t *v_cache) {
    if (fmt != ORC_E4M3FN && fmt != ORC_E5M2) return -1;
    int64_t skipped = 0;
    const int64_t row = (int64_t)hkv * d;
    for (int64_t i = 0; i < nnz; ++i) {
        const int b = batch_idx[i], p = pos[i];
        if (b < 0 || b >= batch || p < 0) { ++skipped; continue; }
        const int64_t e = (int64_t)kv_indptr[b] + p / page_size;
        if (kv_indptr[b] < 0 || e >= kv_indptr[b + 1]) { ++skipped; continue; }
        const int page = kv_indices[e];
        if (page < 0 || page >= num_pages) { ++skipped; continue; }
        for (int h = 0; h < hkv; ++h) {
            const int64_t dst = orc_row_offset(kv_layout, page, p % page_size, h, page_size, hkv, d);
            orc_quantize_array(fmt, k_new + i * row + (int64_t)h * d, d, k_scale, k_cache + dst);
            orc_quantize_array(fmt, v_new + i * row + (int64_t)h * d, d, v_scale, v_cache + dst);
        }
    }
    return skipped;
}

int orc_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Threads of the OpenMP loop for later calls (the benchmark times the oracle
 * on every host core and on one); returns the count now in effect. */
int orc_set_num_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
    return orc_num_threads();
}

/* ---- 2..6. paged attention ------------------------------------------------
 *
 * Layouts (all row-major, contiguous):
 *   q        [nnz_qo, Hq, D]            elements of q_dtype
 *   k_cache  [num_pages, P, Hkv, D]      elements of kv_dtype
 *   v_cache  [num_pages, P, Hkv, D]
 *   qo_indptr[B+1]   query rows of request b are qo_indptr[b] .. [b+1]-1
 *   kv_indptr[B+1], kv_indices[nnz_pages], last_page_len[B]
 * Output, for each selected (row, head) pair k:
 *   o[k*D + d], lse[k]
 * sel_row/sel_head == NULL means "every (row, head)", in row-major order
 * (k = row*Hq + head).
 * Returns 0, or a negative code for malformed arguments.
 */
int orc_paged_attention(
    int64_t batch, int64_t num_qo_heads, int64_t num_kv_heads,
    int64_t head_dim, int64_t page_size, int64_t num_pages,
    const int32_t *qo_indptr, const int32_t *kv_indptr,
    const int32_t *kv_indices, const int32_t *last_page_len,
    int q_dtype, const void *q, double q_scale,
    int kv_dtype, const void *k_cache, const void *v_cache,
    double k_scale, double v_scale, double sm_scale, int causal, int kv_layout,
    const double *q_scales, const double *k_scales, const double *v_scales,
    int64_t n_sel, const int64_t *sel_row, const int32_t *sel_head,
    double *o, double *lse)
{
    if (batch < 0 || num_qo_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
        page_size <= 0 || num_qo_heads % num_kv_heads != 0)
        return -1;
    if (orc_elem_bytes(q_dtype) == 0 || orc_elem_bytes(kv_dtype) == 0) return -2;

    const int64_t Hq = num_qo_heads, Hkv = num_kv_heads, D = head_dim;
    const int64_t P = page_size;
    const int64_t group = Hq / Hkv;
    const int64_t nnz_qo = batch > 0 ? qo_indptr[batch] : 0;
    const int64_t n_out = (sel_row == NULL) ? nnz_qo * Hq : n_sel;

    /* Longest KV sequence: sizes each thread's score buffer. */
    int64_t max_kv = 1;
    for (int64_t b = 0; b < batch; ++b) {
        int64_t np = kv_indptr[b + 1] - kv_indptr[b];
        if (np < 0) return -3;
        if (np > 0) {
            int64_t lpl = last_page_len[b];
            if (lpl < 1 || lpl > P) return -4;
            int64_t kl = (np - 1) * P + lpl;
            if (kl > max_kv) max_kv = kl;
        }
        for (int64_t j = kv_indptr[b]; j < kv_indptr[b + 1]; ++j)
            if (kv_indices[j] < 0 || kv_indices[j] >= num_pages) return -5;
    }

    int bad = 0;
#ifdef _OPENMP
#pragma omp parallel
#endif
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)max_kv);
        double *qh = (double *)malloc(sizeof(double) * (size_t)D);
        if (s == NULL || qh == NULL) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
            bad = 1;
        }
        /* Every thread reaches the work-sharing loop, even one whose buffers
         * failed to allocate: it then skips its share and the call fails. */
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
        for (int64_t k = 0; k < n_out; ++k) {
            if (s == NULL || qh == NULL) continue;
            const int64_t row = sel_row ? sel_row[k] : k / Hq;
            const int64_t h = sel_head ? sel_head[k] : k % Hq;
            double *ok = o + k * D;

            /* Request that owns this query row. */
            int64_t b = 0;
            while (b < batch && !(row >= qo_indptr[b] && row < qo_indptr[b + 1])) ++b;
            const int64_t qo_len = qo_indptr[b + 1] - qo_indptr[b];
            const int64_t i = row - qo_indptr[b];
            const int64_t np = kv_indptr[b + 1] - kv_indptr[b];
            const int64_t kv_len = np > 0 ? (np - 1) * P + last_page_len[b] : 0;
            const int64_t h_kv = h / group;
            /* Per-tensor scales, or per-head scale tensors (query head h, KV head h_kv). */
            const double qs = q_scales ? q_scales[h] : q_scale;
            const double ks = k_scales ? k_scales[h_kv] : k_scale;
            const double vs = v_scales ? v_scales[h_kv] : v_scale;

            /* Step 2: Q^ for this row and head. */
            for (int64_t d = 0; d < D; ++d)
                qh[d] = orc_decode_one(q_dtype, q, (row * Hq + h) * D + d) * qs;

            /* Admissible keys: j < n_keys. */
            int64_t n_keys = kv_len;
            if (causal) {
                int64_t lim = i + kv_len - qo_len + 1;
                if (lim < n_keys) n_keys = lim;
                if (n_keys < 0) n_keys = 0;
            }

            /* Step 5: logits over the gathered keys. */
            for (int64_t j = 0; j < n_keys; ++j) {
                const int64_t page = kv_indices[kv_indptr[b] + j / P];
                const int64_t slot = j % P;
                const int64_t base = orc_row_offset(kv_layout, page, slot, h_kv, P, Hkv, D);
                double acc = 0.0;
                for (int64_t d = 0; d < D; ++d)
                    acc += qh[d] * (orc_decode_one(kv_dtype, k_cache, base + d) * ks);
                s[j] = sm_scale * acc;
            }

            /* Step 6: softmax and the weighted sum of V rows. */
            for (int64_t d = 0; d < D; ++d) ok[d] = 0.0;
            if (n_keys == 0) {
                lse[k] = -INFINITY;
                continue;
            }
            double m = -INFINITY;
            for (int64_t j = 0; j < n_keys; ++j) if (s[j] > m) m = s[j];
            double l = 0.0;
            for (int64_t j = 0; j < n_keys; ++j) l += exp(s[j] - m);
            for (int64_t j = 0; j < n_keys; ++j) {
                const double p = exp(s[j] - m) / l;
                const int64_t page = kv_indices[kv_indptr[b] + j / P];
                const int64_t slot = j % P;
                const int64_t base = orc_row_offset(kv_layout, page, slot, h_kv, P, Hkv, D);
                for (int64_t d = 0; d < D; ++d)
                    ok[d] += p * (orc_decode_one(kv_dtype, v_cache, base + d) * vs);
            }
            lse[k] = m + log(l);
        }
        free(s);
        free(qh);
    }
    return bad ? -6 : 0;
}

/* ---- attention over dense (already gathered) rows -------------------------
 * q [Hq, D] for one query row; keys/values given densely as fp64 [n, Hkv, D].
 * Used only by the tests, to pin the page-table gather against a plain
 * re-layout of the same rows.  Same definition as above, no paging. */
int orc_dense_attention_row(int64_t num_qo_heads, int64_t num_kv_heads, int64_t head_dim,
                            const double *q, int64_t n_keys, const double *k,
                            const double *v, double sm_scale, double *o, double *lse) {
    const int64_t Hq = num_qo_heads, Hkv = num_kv_heads, D = head_dim;
    if (Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0) return -1;
    const int64_t group = Hq / Hkv;
    double *s = (double *)malloc(sizeof(double) * (size_t)(n_keys > 0 ? n_keys : 1));
    if (s == NULL) return -6;
    for (int64_t h = 0; h < Hq; ++h) {
        const int64_t hk = h / group;
        for (int64_t d = 0; d < D; ++d) o[h * D + d] = 0.0;
        if (n_keys == 0) { lse[h] = -INFINITY; continue; }
        double m = -INFINITY;
        for (int64_t j = 0; j < n_keys; ++j) {
            double acc = 0.0;
            for (int64_t d = 0; d < D; ++d) acc += q[h * D + d] * k[(j * Hkv + hk) * D + d];
            s[j] = sm_scale * acc;
            if (s[j] > m) m = s[j];
        }
        double l = 0.0;
        for (int64_t j = 0; j < n_keys; ++j) l += exp(s[j] - m);
        for (int64_t j = 0; j < n_keys; ++j) {
            const double p = exp(s[j] - m) / l;
            for (int64_t d = 0; d < D; ++d) o[h * D + d] += p * v[(j * Hkv + hk) * D + d];
        }
        lse[h] = m + log(l);
    }
    free(s);
    return 0;
}

/* ---- combining attention states by their log-sum-exp ----------------------
 * n partial states of one (row, head), each the softmax-normalised output
 * O_c [D] over a disjoint key subset with its lse_c.  The combined state over
 * the union of the subsets is
 *   L = ln sum_c exp(lse_c),   o = sum_c exp(lse_c - L) * O_c.
 * States with lse_c = -inf (no keys) contribute nothing; if every state is
 * empty the result is o = 0, lse = -inf. */
void orc_merge_states(int64_t n, int64_t head_dim, const double *o_parts,
                      const double *lse_parts, double *o, double *lse) {
    double m = -INFINITY;
    for (int64_t c = 0; c < n; ++c) if (lse_parts[c] > m) m = lse_parts[c];
    for (int64_t d = 0; d < head_dim; ++d) o[d] = 0.0;
    if (m == -INFINITY) { *lse = -INFINITY; return; }
    double sum = 0.0;
    for (int64_t c = 0; c < n; ++c) sum += exp(lse_parts[c] - m);
    const double L = m + log(sum);
    for (int64_t c = 0; c < n; ++c) {
        const double w = exp(lse_parts[c] - L);
        for (int64_t d = 0; d < head_dim; ++d) o[d] += w * o_parts[c * head_dim + d];
    }
    *lse = L;
}
