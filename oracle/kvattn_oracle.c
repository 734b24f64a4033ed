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
 *   row.  q and out are [B, T, Hq, D].  On a local layer each new token
 *   keeps its own window: token t attends the last W positions up to and
 *   including itself, j = max(0, e_t - W) .. e_t - 1 with
 *   e_t = len_b - T + 1 + t (the single-token rule above applied at each
 *   token's own position; a reading, the pages give no formula).
 *
 *   8-bit KV cache: "The Basics of Transformer Inference", the item
 *   "Quantization" (quantizing the KV cache, e.g. to int8, int4 or fp8,
 *   saves memory bandwidth, even post training) and "Machine Learning
 *   Engineering and AI Systems at Scale", section "Quantization" (FP8 E4M3 is
 *   the inference format; quantize the KV cache second).  The pages give no
 *   rule, so the plainest one is taken: each cached row (one position of one
 *   K/V head, D values) is stored as E4M3 codes with one fp32 scale,
 *       scale = absmax(row) / 448 (1 for an all-zero row),
 *       code_d = E4M3(row_d / scale), round to nearest even, saturating,
 *   both divisions in IEEE binary32; the attention then reads
 *       K[b,kvh,j,d] = e4m3_value(code) * k_scale[b,kvh,j]   (V likewise)
 *   in double.  E4M3 is the OCP 8-bit format: sign, 4 exponent bits with
 *   bias 7, 3 mantissa bits, subnormals at exponent 0, no infinities,
 *   S.1111.111 is NaN, largest finite value 448.
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

/* E4M3 code -> value (exact in double); the NaN codes give NaN. */
double oracle_e4m3_to_double(uint8_t code)
{
    const int sign = code >> 7, e = (code >> 3) & 15, m = code & 7;
    double v;
    if (e == 15 && m == 7)
        v = NAN;
    else if (e == 0)
        v = ldexp((double)m, -9);                 /* subnormal: m * 2^-9 */
    else
        v = ldexp(1.0 + m / 8.0, e - 7);          /* normal: 1.m * 2^(e-7) */
    return sign ? -v : v;
}

/* A real value (given in double) -> E4M3, round to nearest with ties to
 * even, finite values beyond the largest (448) saturate to +-448,
 * NaN -> 0x7F. */
static uint8_t oracle_e4m3_from_double(double x)
{
    if (isnan(x))
        return 0x7F;
    const uint8_t sign = signbit(x) ? 0x80 : 0x00;
    const double a = fabs(x);
    if (a > 448.0)
        return sign | 0x7E;
    if (a < ldexp(1.0, -6)) {                     /* subnormal range (or zero) */
        const double m = nearbyint(a / ldexp(1.0, -9));   /* ties to even */
        return sign | (uint8_t)m;                 /* m == 8 is the smallest normal */
    }
    int e = (int)floor(log2(a));
    if (ldexp(1.0, e) > a)                        /* guard log2 rounding */
        --e;
    if (ldexp(1.0, e + 1) <= a)
        ++e;
    double m = nearbyint((a / ldexp(1.0, e) - 1.0) * 8.0);
    if (m == 8.0) {                               /* rounded up to the next binade */
        m = 0.0;
        ++e;
    }
    if (e > 8 || (e == 8 && m > 6.0))             /* past 448: saturate */
        return sign | 0x7E;
    return sign | (uint8_t)(((e + 7) << 3) | (int)m);
}

/* binary32 -> E4M3 (every binary32 value is exact in double). */
uint8_t oracle_e4m3_from_float(float x)
{
    return oracle_e4m3_from_double((double)x);
}

/* One row of D bf16 values -> D codes and its scale (see the header). */
void oracle_quantize_row_fp8(const uint16_t *row, int64_t D, uint8_t *codes, float *scale)
{
    float amax = 0.0f;
    for (int64_t d = 0; d < D; ++d) {
        const float a = fabsf((float)oracle_bf16_to_double(row[d]));
        if (a > amax)
            amax = a;
    }
    volatile float s = amax > 0.0f ? amax / 448.0f : 1.0f;  /* binary32 division */
    *scale = s;
    for (int64_t d = 0; d < D; ++d) {
        volatile float x = (float)oracle_bf16_to_double(row[d]) / s;
        codes[d] = oracle_e4m3_from_float(x);
    }
}

/* rows x D bf16 -> codes and per-row scales. */
void oracle_quantize_fp8(const uint16_t *src, uint8_t *codes, float *scales, int64_t rows,
                         int64_t D)
{
    for (int64_t r = 0; r < rows; ++r)
        oracle_quantize_row_fp8(src + r * D, D, codes + r * D, scales + r);
}

/* The append into an 8-bit cache: each new row is quantized and written at
 * position seq_lens[b] with its scale.  0, or -1 if a length is outside
 * [0, Lmax). */
int oracle_kv_append_fp8(uint8_t *k_codes, uint8_t *v_codes, float *k_scale, float *v_scale,
                         const uint16_t *k_new, const uint16_t *v_new,
                         const int32_t *seq_lens, int64_t B, int64_t Hkv, int64_t D,
                         int64_t Lmax)
{
    for (int64_t b = 0; b < B; ++b)
        if (seq_lens[b] < 0 || seq_lens[b] >= Lmax)
            return -1;
    for (int64_t b = 0; b < B; ++b)
        for (int64_t kvh = 0; kvh < Hkv; ++kvh) {
            const int64_t row = (b * Hkv + kvh) * Lmax + seq_lens[b];
            const int64_t src = (b * Hkv + kvh) * D;
            oracle_quantize_row_fp8(k_new + src, D, k_codes + row * D, k_scale + row);
            oracle_quantize_row_fp8(v_new + src, D, v_codes + row * D, v_scale + row);
        }
    return 0;
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
/* The 8-bit cache of a call, or all NULL for a bf16 cache. */
typedef struct {
    const uint8_t *k, *v;
    const float *k_scale, *v_scale;
} oracle_q8;

/* Element d of cached row j (of the (b, kvh) block starting at row0). */
static double oracle_cache_at(const uint16_t *bf16, const uint8_t *codes, const float *scales,
                              int64_t row0, int64_t j, int64_t D, int64_t d)
{
    if (codes)
        return oracle_e4m3_to_double(codes[(row0 + j) * D + d]) * (double)scales[row0 + j];
    return oracle_bf16_to_double(bf16[(row0 + j) * D + d]);
}

static void oracle_one_head(const uint16_t *q, const uint16_t *k_cache,
                            const uint16_t *v_cache, const oracle_q8 *q8,
                            const int32_t *seq_lens,
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
    const int64_t row0 = (b * Hkv + kvh) * Lmax;  /* first row of this (b, kvh) */

    /* scores (s_buf[j - j0] holds s_j) */
    for (int64_t j = j0; j < len; ++j) {
        double dot = 0.0;
        for (int64_t d = 0; d < D; ++d)
            dot += oracle_bf16_to_double(qh[d]) *
                   oracle_cache_at(k_cache, q8->k, q8->k_scale, row0, j, D, d);
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
            o[d] += p * oracle_cache_at(v_cache, q8->v, q8->v_scale, row0, j0 + j, D, d);
    }
}

typedef struct {
    const uint16_t *q, *k_cache, *v_cache;
    oracle_q8 q8;
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
        oracle_one_head(j->q, j->k_cache, j->v_cache, &j->q8, j->seq_lens, j->out, j->T,
                        j->Hq, j->Hkv, j->D, j->Lmax, j->scale, j->window, b, t, h, s_buf);
    }
    free(s_buf);
    j->status = 0;
    return NULL;
}

static int oracle_run(const uint16_t *q, const uint16_t *k_cache,
                      const uint16_t *v_cache, const oracle_q8 *q8, const int32_t *seq_lens,
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
        j->q = q; j->k_cache = k_cache; j->v_cache = v_cache; j->q8 = *q8;
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

static const oracle_q8 no_q8 = {NULL, NULL, NULL, NULL};

/* Every output row: out is [B, Hq, D] doubles.  Returns 0, or -1 on a bad
 * argument (non-divisible heads, a length outside [0, Lmax]). */
int oracle_gqa_decode(const uint16_t *q, const uint16_t *k_cache,
                      const uint16_t *v_cache, const int32_t *seq_lens,
                      double *out, int64_t B, int64_t Hq, int64_t Hkv,
                      int64_t D, int64_t Lmax, double scale, int nthreads)
{
    return oracle_run(q, k_cache, v_cache, &no_q8, seq_lens, out, B, 1, Hq, Hkv, D, Lmax,
                      scale, Lmax > 0 ? Lmax : 1, NULL, B * Hq, nthreads);
}

/* T new tokens per sequence: q and out are [B, T, Hq, D]; token t attends
 * positions [0, seq_lens[b] - T + 1 + t). */
int oracle_gqa_decode_multi(const uint16_t *q, const uint16_t *k_cache,
                            const uint16_t *v_cache, const int32_t *seq_lens,
                            double *out, int64_t B, int64_t T, int64_t Hq, int64_t Hkv,
                            int64_t D, int64_t Lmax, double scale, int nthreads)
{
    return oracle_run(q, k_cache, v_cache, &no_q8, seq_lens, out, B, T, Hq, Hkv, D, Lmax,
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
    return oracle_run(q, k_cache, v_cache, &no_q8, seq_lens, out, B, 1, Hq, Hkv, D, Lmax,
                      scale, window, NULL, B * Hq, nthreads);
}

/* T new tokens on a local layer: token t attends the last `window`
 * positions up to itself (window >= 1).  q and out are [B, T, Hq, D]. */
int oracle_gqa_decode_multi_window(const uint16_t *q, const uint16_t *k_cache,
                                   const uint16_t *v_cache, const int32_t *seq_lens,
                                   double *out, int64_t B, int64_t T, int64_t Hq, int64_t Hkv,
                                   int64_t D, int64_t Lmax, double scale, int64_t window,
                                   int nthreads)
{
    return oracle_run(q, k_cache, v_cache, &no_q8, seq_lens, out, B, T, Hq, Hkv, D, Lmax,
                      scale, window, NULL, B * T * Hq, nthreads);
}

/* Only the listed (b, h) rows: pairs is [npairs, 2] int64; out is still the
 * full [B, Hq, D] doubles and only the listed rows are written. */
int oracle_gqa_decode_pairs(const uint16_t *q, const uint16_t *k_cache,
                            const uint16_t *v_cache, const int32_t *seq_lens,
                            double *out, int64_t B, int64_t Hq, int64_t Hkv,
                            int64_t D, int64_t Lmax, double scale,
                            const int64_t *pairs, int64_t npairs, int nthreads)
{
    return oracle_run(q, k_cache, v_cache, &no_q8, seq_lens, out, B, 1, Hq, Hkv, D, Lmax,
                      scale, Lmax > 0 ? Lmax : 1, pairs, npairs, nthreads);
}

/* Every output row over an 8-bit cache: k_codes, v_codes [B, Hkv, Lmax, D]
 * E4M3 codes, k_scale, v_scale [B, Hkv, Lmax] fp32 (see the header). */
int oracle_gqa_decode_fp8(const uint16_t *q, const uint8_t *k_codes, const uint8_t *v_codes,
                          const float *k_scale, const float *v_scale,
                          const int32_t *seq_lens, double *out, int64_t B, int64_t Hq,
                          int64_t Hkv, int64_t D, int64_t Lmax, double scale, int nthreads)
{
    if (!k_codes || !v_codes || !k_scale || !v_scale)
        return -1;
    const oracle_q8 q8 = {k_codes, v_codes, k_scale, v_scale};
    return oracle_run(q, NULL, NULL, &q8, seq_lens, out, B, 1, Hq, Hkv, D, Lmax, scale,
                      Lmax > 0 ? Lmax : 1, NULL, B * Hq, nthreads);
}

/* Vector helpers for the tests: n floats -> codes, n codes -> doubles. */
void oracle_e4m3_encode_n(const float *x, uint8_t *codes, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        codes[i] = oracle_e4m3_from_float(x[i]);
}

void oracle_e4m3_decode_n(const uint8_t *codes, double *x, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        x[i] = oracle_e4m3_to_double(codes[i]);
}
