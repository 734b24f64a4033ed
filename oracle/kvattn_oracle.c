/*
 * kvattn_oracle.c -- plain, slow, obviously correct CPU oracle for the
 * generation-phase (decode) attention step over a grouped-query KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file: only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no code, header, table or helper with
 * the CUDA library.
 *
 * What it computes (all arithmetic in IEEE double; bf16 -> double is exact):
 *
 *   KV cache:  "The Basics of Transformer Inference" (How To Scale Your Model,
 *   part 7), the paragraph introducing the KV cache: every token's key and
 *   value projections are written into a cache, and later tokens only form
 *   their q_i . k_j products against it.  The cache of one layer is stored
 *   [B, Hkv, Lmax, D], row-major.
 *
 *   Head grouping: "Tensor Parallelism: Splitting Operations Across GPUs",
 *   section "The GQA ceiling: a worked memory audit" -- 64 query heads share
 *   8 key/value heads, each KV head serving a contiguous group of query heads
 *   ("the original 8-query group sharing that head").  With G = Hq / Hkv the
 *   query head h reads KV head kvh = floor(h / G).  Multi-query attention is
 *   the case Hkv = 1 ("Efficiently Scaling Transformer Inference", section 3
 *   "Attention Layer Partitioning"; "The Basics of Transformer Inference",
 *   the "Grouped multi-query attention" item).
 *
 *   Per head: "Tensor Parallelism ...", section "Splitting attention by head,
 *   and why decode is where it hurts" -- each head forms its own scores, its
 *   own softmax and its own weighted sum of values.  Written out for one
 *   decode query (the plain reading; the pages never print the formula):
 *
 *     s_j        = scale * sum_d q[b,h,d] * K[b,kvh,j,d],   j = 0 .. len_b-1
 *     m          = max_j s_j
 *     p_j        = exp(s_j - m) / sum_i exp(s_i - m)
 *     out[b,h,d] = sum_j p_j * V[b,kvh,j,d]
 *
 *   Ragged lengths: "The Basics of Transformer Inference", the item "Using
 *   ragged HBM reads and Paged Attention" -- only the non-padding part of each
 *   sequence's cache takes part; rows j >= len_b are never read.
 *   len_b = 0 gives an all-zero output row (empty softmax; a reading, the
 *   pages are silent).
 *
 *   KV append: the new token's K and V rows are copied, element by element,
 *   into row seq_lens[b] of the cache (the number of tokens cached before it).
 *
 *   Local (sliding-window) layers: "The Basics of Transformer Inference", the
 *   item on mixing in local attention layers -- a local layer caps how far
 *   back a token attends (a diagonal strip of the attention matrix instead
 *   of a triangle).  For a decode query at position len_b - 1 and a window
 *   of W positions (the token itself included; a reading, the pages give no
 *   formula) the sums above run over j = max(0, len_b - W) .. len_b - 1.
 *   W >= len_b is the full attention.
 *
 *   Several new tokens per sequence (speculative sampling, "The Basics of
 *   Transformer Inference": the big model scores a run of drafted tokens in
 *   one pass, sharing the KV-cache loads among them): the T new tokens sit
 *   at positions len_b - T .. len_b - 1 and token t (0-based) attends
 *   positions 0 .. len_b - T + t, i.e. the cached prefix and the new tokens
 *   up to itself (causal among the new tokens; a reading, the pages give no
 *   formula).  A token with nothing to attend (len_b - T + t < 0) gets a zero
 *   row.  q and out are [B, T, Hq, D].
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <math.h>
#include <pthread.h>

/* bf16 is the upper half of an IEEE binary32; widening to double is exact. */
double oracle_bf16_to_double(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Returns 0 on success, -1 if some seq_lens[b] is outside [0, Lmax). */
int oracle_kv_append(uint16_t *k_cache, uint16_t *v_cache,
                     const uint16_t *k_new, const uint16_t *v_new,
                     const int32_t *seq_lens,
                     int64_t B, int64_t Hkv, int64_t D, int64_t Lmax)
{
    for (int64_t b = 0; b < B; ++b)
        if (seq_lens[b] < 0 || seq_lens[b] >= Lmax)
            return -1;
    for (int64_t b = 0; b < B; ++b) {
        int64_t pos = seq_lens[b];
        for (int64_t kvh = 0; kvh < Hkv; ++kvh) {
            for (int64_t d = 0; d < D; ++d) {
                int64_t dst = ((b * Hkv + kvh) * Lmax + pos) * D + d;
                int64_t src = (b * Hkv + kvh) * D + d;
                k_cache[dst] = k_new[src];
                v_cache[dst] = v_new[src];
            }
        }
    }
    return 0;
}

/* One output row out[b,h,0..D-1], straight from the definition above.
 * s_buf must hold len_b doubles. */
static void oracle_one_head(const uint16_t *q, const uint16_t *k_cache,
                            const uint16_t *v_cache, const int32_t *seq_lens,
                            double *out, int64_t T, int64_t Hq, int64_t Hkv, int64_t D,
                            int64_t Lmax, double scale, int64_t window,
                            int64_t b, int64_t t, int64_t h, double *s_buf)
{
    const int64_t G = Hq / Hkv;
    const int64_t kvh = h / G;
    int64_t len = seq_lens[b] - (T - 1 - t); /* positions this query attends */
    if (len < 0)
        len = 0;
    const int64_t j0 = len > window ? len - window : 0; /* first attended position */
    double *o = out + ((b * T + t) * Hq + h) * D;

    for (int64_t d = 0; d < D; ++d)
        o[d] = 0.0;
    if (len == 0)
        return;

    const uint16_t *qh = q + ((b * T + t) * Hq + h) * D;
    const uint16_t *K = k_cache + (b * Hkv + kvh) * Lmax * D;
    const uint16_t *V = v_cache + (b * Hkv + kvh) * Lmax * D;

    /* scores (s_buf[j - j0] holds s_j) */
    for (int64_t j = j0; j < len; ++j) {
        double dot = 0.0;
        for (int64_t d = 0; d < D; ++d)
            dot += oracle_bf16_to_double(qh[d]) * oracle_bf16_to_double(K[j * D + d]);
        s_buf[j - j0] = scale * dot;
    }
    const int64_t n = len - j0;
    /* max */
    double m = s_buf[0];
    for (int64_t j = 1; j < n; ++j)
        if (s_buf[j] > m)
            m = s_buf[j];
    /* normaliser */
    double denom = 0.0;
    for (int64_t j = 0; j < n; ++j)
        denom += exp(s_buf[j] - m);
    /* weighted sum of values */
    for (int64_t j = 0; j < n; ++j) {
        double p = exp(s_buf[j] - m) / denom;
        for (int64_t d = 0; d < D; ++d)
            o[d] += p * oracle_bf16_to_double(V[(j0 + j) * D + d]);
    }
}

typedef struct {
    const uint16_t *q, *k_cache, *v_cache;
    const int32_t *seq_lens;
    double *out;
    int64_t B, T, Hq, Hkv, D, Lmax;
    double scale;
    int64_t window;
    const int64_t *pairs; /* NULL: all (b,h); else npairs (b,h) pairs */
    int64_t first, last;  /* range of work items (pairs or flat b*Hq+h) */
    int status;
} oracle_job;

static void *oracle_worker(void *arg)
{
    oracle_job *j = (oracle_job *)arg;
    double *s_buf = (double *)malloc((size_t)(j->Lmax > 0 ? j->Lmax : 1) * sizeof(double));
    if (!s_buf) {
        j->status = -2;
        return NULL;
    }
    for (int64_t w = j->first; w < j->last; ++w) {
        int64_t b, t, h;
        if (j->pairs) {
            b = j->pairs[2 * w];
            t = 0;
            h = j->pairs[2 * w + 1];
        } else {
            b = w / (j->T * j->Hq);
            t = (w / j->Hq) % j->T;
            h = w % j->Hq;
        }
        oracle_one_head(j->q, j->k_cache, j->v_cache, j->seq_lens, j->out, j->T,
                        j->Hq, j->Hkv, j->D, j->Lmax, j->scale, j->window, b, t, h, s_buf);
    }
    free(s_buf);
    j->status = 0;
    return NULL;
}

static int oracle_run(const uint16_t *q, const uint16_t *k_cache,
                      const uint16_t *v_cache, const int32_t *seq_lens,
                      double *out, int64_t B, int64_t T, int64_t Hq, int64_t Hkv,
                      int64_t D, int64_t Lmax, double scale, int64_t window,
                      const int64_t *pairs, int64_t nitems, int nthreads)
{
    if (B < 0 || T < 1 || Hq <= 0 || Hkv <= 0 || D <= 0 || Lmax < 0 || Hq % Hkv != 0 ||
        window < 1 || (pairs && T != 1))
        return -1;
    for (int64_t b = 0; b < B; ++b)
        if (seq_lens[b] < 0 || seq_lens[b] > Lmax)
            return -1;
    if (pairs)
        for (int64_t w = 0; w < nitems; ++w)
            if (pairs[2 * w] < 0 || pairs[2 * w] >= B ||
                pairs[2 * w + 1] < 0 || pairs[2 * w + 1] >= Hq)
                return -1;
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > 256)
        nthreads = 256;
    if ((int64_t)nthreads > nitems)
        nthreads = nitems > 0 ? (int)nitems : 1;

    oracle_job jobs[256];
    pthread_t tids[256];
    for (int t = 0; t < nthreads; ++t) {
        oracle_job *j = &jobs[t];
        j->q = q; j->k_cache = k_cache; j->v_cache = v_cache;
        j->seq_lens = seq_lens; j->out = out;
        j->B = B; j->T = T; j->Hq = Hq; j->Hkv = Hkv; j->D = D; j->Lmax = Lmax;
        j->scale = scale; j->window = window; j->pairs = pairs;
        j->first = nitems * t / nthreads;
        j->last = nitems * (t + 1) / nthreads;
        j->status = -3;
    }
    if (nthreads == 1) {
        oracle_worker(&jobs[0]);
    } else {
        int started = 0;
        for (int t = 0; t < nthreads; ++t) {
            if (pthread_create(&tids[t], NULL, oracle_worker, &jobs[t]) != 0)
                break;
            ++started;
        }
        for (int t = 0; t < started; ++t)
            pthread_join(tids[t], NULL);
        for (int t = started; t < nthreads; ++t)
            oracle_worker(&jobs[t]);
    }
    for (int t = 0; t < nthreads; ++t)
        if (jobs[t].status != 0)
            return jobs[t].status;
    return 0;
}

/* Every output row: out is [B, Hq, D] doubles.  Returns 0, or -1 on a bad
 * argument (non-divisible heads, a length outside [0, Lmax]). */
int oracle_gqa_decode(const uint16_t *q, const uint16_t *k_cache,
                      const uint16_t *v_cache, const int32_t *seq_lens,
                      double *out, int64_t B, int64_t Hq, int64_t Hkv,
                      int64_t D, int64_t Lmax, double scale, int nthreads)
{
    return oracle_run(q, k_cache, v_cache, seq_lens, out, B, 1, Hq, Hkv, D, Lmax,
                      scale, Lmax > 0 ? Lmax : 1, NULL, B * Hq, nthreads);
}

/* T new tokens per sequence: q and out are [B, T, Hq, D]; token t attends
 * positions [0, seq_lens[b] - T + 1 + t). */
int oracle_gqa_decode_multi(const uint16_t *q, const uint16_t *k_cache,
                            const uint16_t *v_cache, const int32_t *seq_lens,
                            double *out, int64_t B, int64_t T, int64_t Hq, int64_t Hkv,
                            int64_t D, int64_t Lmax, double scale, int nthreads)
{
    return oracle_run(q, k_cache, v_cache, seq_lens, out, B, T, Hq, Hkv, D, Lmax,
                      scale, Lmax > 0 ? Lmax : 1, NULL, B * T * Hq, nthreads);
}

/* As oracle_gqa_decode, attending only the last `window` positions of each
 * sequence (window >= 1). */
int oracle_gqa_decode_window(const uint16_t *q, const uint16_t *k_cache,
                             const uint16_t *v_cache, const int32_t *seq_lens,
                             double *out, int64_t B, int64_t Hq, int64_t Hkv,
                             int64_t D, int64_t Lmax, double scale, int64_t window,
                             int nthreads)
{
    return oracle_run(q, k_cache, v_cache, seq_lens, out, B, 1, Hq, Hkv, D, Lmax,
                      scale, window, NULL, B * Hq, nthreads);
}

/* Only the listed (b, h) rows: pairs is [npairs, 2] int64; out is still the
 * full [B, Hq, D] doubles and only the listed rows are written. */
int oracle_gqa_decode_pairs(const uint16_t *q, const uint16_t *k_cache,
                            const uint16_t *v_cache, const int32_t *seq_lens,
                            double *out, int64_t B, int64_t Hq, int64_t Hkv,
                            int64_t D, int64_t Lmax, double scale,
                            const int64_t *pairs, int64_t npairs, int nthreads)
{
    return oracle_run(q, k_cache, v_cache, seq_lens, out, B, 1, Hq, Hkv, D, Lmax,
                      scale, Lmax > 0 ? Lmax : 1, pairs, npairs, nthreads);
}
