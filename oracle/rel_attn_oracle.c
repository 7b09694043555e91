/*
 * Oracle for paged, varlen attention with an additive relative-position bias
 * (Inkling relative attention).  TEST INFRASTRUCTURE ONLY: the tests, the
 * package's smoke check and the benchmark's CPU-baseline leg are the only
 * callers.  It shares no code with the CUDA library and the library never
 * calls it.
 *
 * Plain, slow, fp64.  For each (request b, query head h) it materialises the
 * whole sq_b x sk_b score matrix, applies mask and bias in explicit loops,
 * and forms the softmax-weighted sum of V.  bf16 inputs are widened to fp64
 * exactly (a bf16 is the top 16 bits of an fp32).
 *
 * What it computes, and where each step is stated:
 *  - Shapes: q (T,H,D); key_cache/value_cache (NB,BS,Hk,D) read through the
 *    per-request block_table up to cache_seqlens[b] (seqused_k); rel_logits
 *    (T,H,R).  vLLM API docs, "inkling_fa4_rel_attention", docstring.
 *  - Relative distance d = (q_idx + seqlen_k - seqlen_q) - kv_idx, the bias
 *    row is the global packed token offset_q + q_idx and the query head
 *    h_idx; bias = rel_logits[t,h,d] when 0 <= d < R and exactly 0 otherwise
 *    (the value is zeroed, not clamped).  prhub report on vLLM PR #48858,
 *    "关键源码片段" (source excerpt), score_mod_rel_bias.
 *  - Bias added after the softmax scale: s = scale * q.k + bias.  prhub
 *    report, "实现拆解" (breakdown) item 2, with the scale read as the
 *    softmax_scale argument of the API docs.
 *  - Causal mask aligned bottom-right: query row i sits at key position
 *    i + seqlen_k - seqlen_q (the same offset the bias uses).
 *  - Sliding window (left,right): key j is allowed iff
 *    q_pos - left <= j <= q_pos + right, a negative side meaning unbounded;
 *    (-1,-1) is "no window".  API docs, inkling_fa4_rel_attention
 *    (window_size, and the (-1,-1) -> (None,None) conversion).
 *  - GQA: query head h reads kv head h / (H / Hk).  API docs,
 *    inkling_fa4_num_splits (q_rows = max_query_len * (num_heads // num_kv_heads)).
 *  - A row with no allowed key outputs 0.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

static double bf16_to_f64(uint16_t bits) {
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* rel_logits[idx] as a double: bf16 bits or an fp32 value, both exact. */
static double rel_value(const void* rel, int is_f32, int64_t idx) {
    return is_f32 ? (double)((const float*)rel)[idx] : bf16_to_f64(((const uint16_t*)rel)[idx]);
}

/* Is key j visible from row i of a request with offset off = sk - sq? */
static int key_allowed(int64_t i, int64_t j, int64_t off, int causal, int wl, int wr) {
    int64_t d = i + off - j;
    if (causal && d < 0) return 0;
    if (wl >= 0 && d > wl) return 0;
    if (wr >= 0 && d < -(int64_t)wr) return 0;
    return 1;
}

/* Check the index data once, so that no loop below reads out of bounds. */
static int check_indices(const int32_t* block_table, int64_t max_blocks,
                         const int32_t* cache_seqlens, const int32_t* cu_seqlens_q,
                         int64_t B, int64_t T, int64_t NB, int64_t BS) {
    if (cu_seqlens_q[0] != 0 || cu_seqlens_q[B] != T) return 1;
    for (int64_t b = 0; b < B; ++b) {
        if (cu_seqlens_q[b + 1] < cu_seqlens_q[b]) return 2;
        int64_t sk = cache_seqlens[b];
        if (sk < 0 || sk > max_blocks * BS) return 3;
        for (int64_t j = 0; j < sk; j += BS) {
            int32_t blk = block_table[b * max_blocks + j / BS];
            if (blk < 0 || blk >= NB) return 4;
        }
    }
    return 0;
}

static const uint16_t* cache_row(const uint16_t* cache, const int32_t* block_table,
                                 int64_t max_blocks, int64_t b, int64_t j,
                                 int64_t BS, int64_t Hk, int64_t D, int64_t g) {
    int64_t blk = block_table[b * max_blocks + j / BS];
    int64_t slot = j % BS;
    return cache + ((blk * BS + slot) * Hk + g) * D;
}

/*
 * Full forward.  out is (T,H,D) fp64; lse (T,H) natural-log sum-exp of the
 * allowed scores, -inf for a row with no allowed key (may be NULL).
 * Returns 0, or a nonzero code when the arguments are inconsistent.
 */
int rel_attn_oracle_forward(
    const uint16_t* q, const uint16_t* key_cache, const uint16_t* value_cache,
    const int32_t* block_table, int64_t max_blocks,
    const int32_t* cache_seqlens, const int32_t* cu_seqlens_q,
    int64_t B, int64_t T, int64_t H, int64_t Hk, int64_t D, int64_t NB, int64_t BS,
    double softmax_scale, int causal, int window_left, int window_right,
    int64_t rel_extent, const void* rel_logits, int rel_is_f32,
    double* out, double* lse, int num_threads) {
    if (B < 0 || T < 0 || H <= 0 || Hk <= 0 || D <= 0 || BS <= 0 || H % Hk != 0 || rel_extent < 0)
        return 10;
    int rc = check_indices(block_table, max_blocks, cache_seqlens, cu_seqlens_q, B, T, NB, BS);
    if (rc) return rc;
    const int64_t G = H / Hk;
    int64_t pairs = B * H;
#ifdef _OPENMP
    if (num_threads > 0) omp_set_num_threads(num_threads);
#endif
    int failed = 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t bh = 0; bh < pairs; ++bh) {
        const int64_t b = bh / H, h = bh % H, g = h / G;
        const int64_t q0 = cu_seqlens_q[b];
        const int64_t sq = cu_seqlens_q[b + 1] - q0;
        const int64_t sk = cache_seqlens[b];
        const int64_t off = sk - sq;
        if (sq == 0) continue;
        double* S = (double*)malloc(sizeof(double) * (size_t)(sq * (sk > 0 ? sk : 1)));
        double* qrow = (double*)malloc(sizeof(double) * (size_t)D);
        double* acc = (double*)malloc(sizeof(double) * (size_t)D);
        if (!S || !qrow || !acc) {
            free(S); free(qrow); free(acc);
#pragma omp atomic write
            failed = 1;
            continue;
        }
        /* 1. Scores: scale * q.k + bias, -inf where masked. */
        for (int64_t i = 0; i < sq; ++i) {
            const int64_t t = q0 + i;
            for (int64_t k = 0; k < D; ++k) qrow[k] = bf16_to_f64(q[(t * H + h) * D + k]);
            for (int64_t j = 0; j < sk; ++j) {
                if (!key_allowed(i, j, off, causal, window_left, window_right)) {
                    S[i * sk + j] = -INFINITY;
                    continue;
                }
                const uint16_t* kr = cache_row(key_cache, block_table, max_blocks, b, j, BS, Hk, D, g);
                double dot = 0.0;
                for (int64_t k = 0; k < D; ++k) dot += qrow[k] * bf16_to_f64(kr[k]);
                const int64_t d = i + off - j;
                double bias = 0.0;
                if (d >= 0 && d < rel_extent)
                    bias = rel_value(rel_logits, rel_is_f32, (t * H + h) * rel_extent + d);
                S[i * sk + j] = softmax_scale * dot + bias;
            }
        }
        /* 2. Row softmax and 3. weighted sum of V. */
        for (int64_t i = 0; i < sq; ++i) {
            const int64_t t = q0 + i;
            double m = -INFINITY;
            for (int64_t j = 0; j < sk; ++j)
                if (S[i * sk + j] > m) m = S[i * sk + j];
            double* o = out + (t * H + h) * D;
            if (m == -INFINITY) {
                for (int64_t k = 0; k < D; ++k) o[k] = 0.0;
                if (lse) lse[t * H + h] = -INFINITY;
                continue;
            }
            double l = 0.0;
            for (int64_t k = 0; k < D; ++k) acc[k] = 0.0;
            for (int64_t j = 0; j < sk; ++j) {
                if (S[i * sk + j] == -INFINITY) continue;
                double p = exp(S[i * sk + j] - m);
                l += p;
                const uint16_t* vr = cache_row(value_cache, block_table, max_blocks, b, j, BS, Hk, D, g);
                for (int64_t k = 0; k < D; ++k) acc[k] += p * bf16_to_f64(vr[k]);
            }
            for (int64_t k = 0; k < D; ++k) o[k] = acc[k] / l;
            if (lse) lse[t * H + h] = m + log(l);
        }
        free(S); free(qrow); free(acc);
    }
    return failed ? 11 : 0;
}

/*
 * The same definition for a list of single output rows (t_k, h_k): used to
 * check sampled outputs of workloads too large to run whole.  out_rows is
 * (n, D) fp64.
 */
int rel_attn_oracle_rows(
    const uint16_t* q, const uint16_t* key_cache, const uint16_t* value_cache,
    const int32_t* block_table, int64_t max_blocks,
    const int32_t* cache_seqlens, const int32_t* cu_seqlens_q,
    int64_t B, int64_t T, int64_t H, int64_t Hk, int64_t D, int64_t NB, int64_t BS,
    double softmax_scale, int causal, int window_left, int window_right,
    int64_t rel_extent, const void* rel_logits, int rel_is_f32,
    int64_t n, const int64_t* row_t, const int64_t* row_h, double* out_rows, int num_threads) {
    if (B < 0 || T < 0 || H <= 0 || Hk <= 0 || D <= 0 || BS <= 0 || H % Hk != 0 || rel_extent < 0)
        return 10;
    int rc = check_indices(block_table, max_blocks, cache_seqlens, cu_seqlens_q, B, T, NB, BS);
    if (rc) return rc;
    for (int64_t r = 0; r < n; ++r)
        if (row_t[r] < 0 || row_t[r] >= T || row_h[r] < 0 || row_h[r] >= H) return 12;
    const int64_t G = H / Hk;
#ifdef _OPENMP
    if (num_threads > 0) omp_set_num_threads(num_threads);
#endif
    int failed = 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < n; ++r) {
        const int64_t t = row_t[r], h = row_h[r], g = h / G;
        int64_t b = 0;
        while (b + 1 < B && cu_seqlens_q[b + 1] <= t) ++b;  /* request owning token t */
        const int64_t i = t - cu_seqlens_q[b];
        const int64_t sq = cu_seqlens_q[b + 1] - cu_seqlens_q[b];
        const int64_t sk = cache_seqlens[b];
        const int64_t off = sk - sq;
        double* s = (double*)malloc(sizeof(double) * (size_t)(sk > 0 ? sk : 1));
        double* acc = (double*)calloc((size_t)D, sizeof(double));
        if (!s || !acc) {
            free(s); free(acc);
#pragma omp atomic write
            failed = 1;
            continue;
        }
        double m = -INFINITY;
        for (int64_t j = 0; j < sk; ++j) {
            s[j] = -INFINITY;
            if (!key_allowed(i, j, off, causal, window_left, window_right)) continue;
            const uint16_t* kr = cache_row(key_cache, block_table, max_blocks, b, j, BS, Hk, D, g);
            double dot = 0.0;
            for (int64_t k = 0; k < D; ++k)
                dot += bf16_to_f64(q[(t * H + h) * D + k]) * bf16_to_f64(kr[k]);
            const int64_t d = i + off - j;
            double bias = 0.0;
            if (d >= 0 && d < rel_extent) bias = rel_value(rel_logits, rel_is_f32, (t * H + h) * rel_extent + d);
            s[j] = softmax_scale * dot + bias;
            if (s[j] > m) m = s[j];
        }
        double* o = out_rows + r * D;
        if (m == -INFINITY) {
            for (int64_t k = 0; k < D; ++k) o[k] = 0.0;
        } else {
            double l = 0.0;
            for (int64_t j = 0; j < sk; ++j) {
                if (s[j] == -INFINITY) continue;
                double p = exp(s[j] - m);
                l += p;
                const uint16_t* vr = cache_row(value_cache, block_table, max_blocks, b, j, BS, Hk, D, g);
                for (int64_t k = 0; k < D; ++k) acc[k] += p * bf16_to_f64(vr[k]);
            }
            for (int64_t k = 0; k < D; ++k) o[k] = acc[k] / l;
        }
        free(s); free(acc);
    }
    return failed ? 11 : 0;
}
