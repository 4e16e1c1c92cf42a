/*
 * Reference oracle for grouped-query scaled-dot-product attention.
 *
 * TEST INFRASTRUCTURE ONLY. This file is compiled and called by the test
 * suite, by the smoke check and by the benchmark's CPU-baseline leg. The
 * product library never includes, links or calls it, and it includes nothing
 * from the product library.
 *
 * Everything is plain float64 arithmetic written straight from the definition
 *     O = softmax(scale * Q K^T [+ causal mask]) V
 * with no tiling, no online rescaling and no reordering beyond what the
 * definition states. Sources:
 *   - BootstrapAI evolution log, collab-014 "Kernel 9 GQA": query head h_q
 *     reads K/V head h_kv = h_q / group_size with group_size = H_q / H_kv;
 *     Q is addressed by the query-head stride, K/V by the K/V-head stride.
 *     That entry's CPU reference (standard_gqa_attention_cpu) is a plain
 *     GQA-aware loop of exactly this kind.
 *   - BootstrapAI evolution log, collab-005 "Kernel 2 tiling": the tiled
 *     kernel's online softmax reaches the same result as the two-pass
 *     softmax written here (max, exponentials, sum, weighted average).
 *   - microLLM-rocm optimisation log, Experiment 044: causal GQA attention
 *     with no copying of K/V heads.
 *   - microLLM-rocm optimisation log, Experiments 282-284 (split-sequence
 *     cached attention): partial results over key ranges are merged; the
 *     log-sum-exp merge below is the plain statement of that merge.
 *
 * Readings where the pages are silent (each is listed with the design notes):
 *   - causal alignment when N_q != N_kv is bottom-right: query row i sees key
 *     j iff j <= i + (N_kv - N_q);
 *   - a row that sees no key has O = 0 and lse = -inf;
 *   - decode: one query row per sequence, all seqlens[b] cached rows visible.
 *
 * Parity pins for every function here live in the CPU test suite (closed
 * forms, invariants, hand-derived fixtures and a library special case).
 */
#include <math.h>
#include <stdlib.h>
#include <stddef.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/*
 * One query row q[d] against the first n rows of k[n][d], v[n][d].
 * o[d] receives the attention output, *lse the natural-log sum of
 * exp(scale * q.k_j) over the n visible keys.
 */
void oracle_attend_row(const double *q, const double *k, const double *v,
                       long n, long d, double scale, double *o, double *lse)
{
    long j, c;
    if (n <= 0) {
        for (c = 0; c < d; ++c) o[c] = 0.0;
        if (lse) *lse = -INFINITY;
        return;
    }
    double *s = (double *)malloc((size_t)n * sizeof(double));
    /* scores s_j = scale * sum_c q_c k_jc */
    for (j = 0; j < n; ++j) {
        double acc = 0.0;
        for (c = 0; c < d; ++c) acc += q[c] * k[j * d + c];
        s[j] = scale * acc;
    }
    /* softmax: subtract the maximum, exponentiate, normalise */
    double m = s[0];
    for (j = 1; j < n; ++j) if (s[j] > m) m = s[j];
    double l = 0.0;
    for (j = 0; j < n; ++j) { s[j] = exp(s[j] - m); l += s[j]; }
    /* weighted average of the value rows */
    for (c = 0; c < d; ++c) {
        double acc = 0.0;
        for (j = 0; j < n; ++j) acc += s[j] * v[j * d + c];
        o[c] = acc / l;
    }
    if (lse) *lse = m + log(l);
    free(s);
}

/* Number of keys that query row i sees (bottom-right causal alignment). */
static long visible_keys(long i, long n_q, long n_kv, int causal)
{
    if (!causal) return n_kv;
    long n = i + (n_kv - n_q) + 1;
    if (n < 0) n = 0;
    if (n > n_kv) n = n_kv;
    return n;
}

/*
 * Prefill form. Layouts (row-major, contiguous):
 *   q, o : [B][H_q][N_q][d]      k, v : [B][H_kv][N_kv][d]
 *   lse  : [B][H_q][N_q]         (may be NULL)
 * Only the flattened (b, h_q) heads in [bh_begin, bh_end) are computed, so a
 * caller can time or check a bounded subset. Returns 0, or -1 when H_q is not
 * a multiple of H_kv.
 */
int oracle_prefill(const double *q, const double *k, const double *v,
                   double *o, double *lse,
                   long B, long H_q, long H_kv, long N_q, long N_kv, long d,
                   int causal, double scale, long bh_begin, long bh_end,
                   int n_threads)
{
    if (H_kv <= 0 || H_q % H_kv != 0) return -1;
    const long group = H_q / H_kv;
    long bh;
    if (bh_begin < 0) bh_begin = 0;
    if (bh_end > B * H_q) bh_end = B * H_q;
#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
#pragma omp parallel for schedule(dynamic, 1)
#else
    (void)n_threads;
#endif
    for (bh = bh_begin; bh < bh_end; ++bh) {
        const long b = bh / H_q, h_q = bh % H_q;
        const long h_kv = h_q / group;
        const double *kh = k + (b * H_kv + h_kv) * N_kv * d;
        const double *vh = v + (b * H_kv + h_kv) * N_kv * d;
        for (long i = 0; i < N_q; ++i) {
            const long row = (b * H_q + h_q) * N_q + i;
            oracle_attend_row(q + row * d, kh, vh,
                              visible_keys(i, N_q, N_kv, causal), d, scale,
                              o + row * d, lse ? lse + row : NULL);
        }
    }
    return 0;
}

/*
 * Decode form: one query row per (b, h_q) against a K/V cache.
 *   q, o          : [B][H_q][d]
 *   k_cache, v_cache : [B][H_kv][max_len][d]; rows [0, seqlens[b]) are valid
 *   lse           : [B][H_q] (may be NULL)
 * Returns 0, -1 for a bad head ratio, -2 for a seqlen outside [0, max_len].
 */
int oracle_decode(const double *q, const double *k_cache,
                  const double *v_cache, const int *seqlens, double *o,
                  double *lse, long B, long H_q, long H_kv, long max_len,
                  long d, double scale)
{
    if (H_kv <= 0 || H_q % H_kv != 0) return -1;
    const long group = H_q / H_kv;
    for (long b = 0; b < B; ++b) {
        const long n = seqlens[b];
        if (n < 0 || n > max_len) return -2;
        for (long h_q = 0; h_q < H_q; ++h_q) {
            const long h_kv = h_q / group;
            const long head = b * H_kv + h_kv;
            const long row = b * H_q + h_q;
            oracle_attend_row(q + row * d, k_cache + head * max_len * d,
                              v_cache + head * max_len * d, n, d, scale,
                              o + row * d, lse ? lse + row : NULL);
        }
    }
    return 0;
}

/*
 * Merge of partial attention results over disjoint key ranges.
 *   o_parts [S][d] : each part's normalised output
 *   lse_parts [S]  : each part's log-sum-exp (-inf for an empty part)
 * Writes the merged output o[d] and *lse. Parts with lse = -inf carry no
 * weight; when every part is empty the result is O = 0, lse = -inf.
 */
void oracle_lse_merge(const double *o_parts, const double *lse_parts, long S,
                      long d, double *o, double *lse)
{
    long i, c;
    double m = -INFINITY;
    for (i = 0; i < S; ++i) if (lse_parts[i] > m) m = lse_parts[i];
    if (m == -INFINITY) {
        for (c = 0; c < d; ++c) o[c] = 0.0;
        if (lse) *lse = -INFINITY;
        return;
    }
    double wsum = 0.0;
    for (i = 0; i < S; ++i)
        if (lse_parts[i] > -INFINITY) wsum += exp(lse_parts[i] - m);
    for (c = 0; c < d; ++c) {
        double acc = 0.0;
        for (i = 0; i < S; ++i)
            if (lse_parts[i] > -INFINITY)
                acc += exp(lse_parts[i] - m) * o_parts[i * d + c];
        o[c] = acc / wsum;
    }
    if (lse) *lse = m + log(wsum);
}
