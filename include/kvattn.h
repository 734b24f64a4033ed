/*
 * kvattn.h -- C ABI of libkvattn: the generation-phase (decode) attention
 * step over a grouped-query / multi-query KV cache, for NVIDIA GB300
 * (sm_103a).
 *
 * The operation.  During generation each sequence adds one token per step.
 * Its key and value projections are written into a per-layer KV cache, and
 * its query then forms q_i . k_j products against every cached key without
 * recomputing earlier tokens ("The Basics of Transformer Inference" -- How To
 * Scale Your Model, part 7 -- the paragraph that introduces the KV cache).
 * Each query head runs its own softmax and its own weighted sum of values
 * ("Tensor Parallelism: Splitting Operations Across GPUs", section
 * "Splitting attention by head, and why decode is where it hurts").  Query
 * heads are grouped onto shared K/V heads in contiguous groups of
 * G = Hq / Hkv ("Tensor Parallelism ...", section "The GQA ceiling: a worked
 * memory audit"; multi-query attention, Hkv = 1, in "Efficiently Scaling
 * Transformer Inference", section 3 "Attention Layer Partitioning"):
 *
 *     kvh        = h / G
 *     s_j        = scale * sum_d q[b,h,d] * K[b,kvh,j,d],  0 <= j < seq_lens[b]
 *     out[b,h,:] = sum_j softmax_j(s) * V[b,kvh,j,:]
 *
 * Only the non-padding part of each sequence's cache is read ("The Basics of
 * Transformer Inference", item "Using ragged HBM reads and Paged Attention").
 *
 * Conventions for every call below.
 *  - All tensor arguments are DEVICE pointers to contiguous row-major memory
 *    owned by the caller.  The library never frees or retains them beyond the
 *    call's stream work.
 *  - bf16 is IEEE binary32's upper 16 bits (passed as void*); fp32 is float.
 *  - Every pointer must be 16-byte aligned.
 *  - Calls are asynchronous on `stream` (0 = legacy default stream) and do
 *    not synchronise the host, except that the first attention call on a
 *    (device, stream) pair, or a call needing a larger workspace than any
 *    before on that pair, allocates device memory (cudaMalloc; it may
 *    serialise with other device work).  Make such a first call before
 *    capturing a stream into a CUDA graph.  An outgrown workspace is not
 *    freed until kvattn_release(), so graphs captured with it stay valid.
 *  - Host-detected errors return a non-zero kvattn_status and launch nothing;
 *    kvattn_last_error() then gives a one-line reason (thread-local).
 *  - Device-detected errors (a length outside the cache) never fault or trap:
 *    the offending sequence is skipped and a sticky per-device error word is
 *    set, read and cleared by kvattn_check_device_error().
 *  - Thread-safe: internal caches are guarded by a mutex.  Calls on the same
 *    stream run in order; calls on different streams use separate
 *    workspaces.
 */
#ifndef KVATTN_H
#define KVATTN_H

#include <stdint.h>

#if defined(__GNUC__)
#define KVATTN_API __attribute__((visibility("default")))
#else
#define KVATTN_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t / CUstream, spelled without CUDA headers. */
typedef struct CUstream_st *kvattn_stream_t;

typedef enum {
    KVATTN_OK = 0,
    KVATTN_ERR_INVALID_ARG = 1,   /* null/misaligned pointer, bad size, Hq % Hkv != 0, non-finite scale */
    KVATTN_ERR_UNSUPPORTED = 2,   /* D not in {64, 128, 256}, or sizes beyond the library's limits */
    KVATTN_ERR_CUDA = 3,          /* a CUDA runtime/driver call failed (see kvattn_last_error) */
    KVATTN_ERR_OOM = 4,           /* workspace allocation failed */
    KVATTN_ERR_DEVICE_BOUNDS = 5, /* device saw seq_lens[b] outside the cache (sticky word) */
    KVATTN_ERR_TIMEOUT = 6        /* a bounded device wait gave up (sticky word) */
} kvattn_status;

/*
 * kv_append -- write this step's new key/value rows into the cache.
 *
 * Follows "The Basics of Transformer Inference", the KV-cache paragraph:
 * each token's key and value projections are written into the cache once.
 *
 *   k_cache, v_cache : bf16 [B, Hkv, Lmax, D], modified in place
 *   k_new, v_new     : bf16 [B, Hkv, D], the new token's rows
 *   seq_lens         : int32 [B] (device), the number of tokens cached
 *                      BEFORE this one; row seq_lens[b] is written.  The
 *                      array is not modified -- the caller advances it.
 *   B, Hkv, D, Lmax  : sizes; D in {64, 128, 256}
 *
 * Bit-exact copy; nothing outside row seq_lens[b] of each (b, kvh) changes.
 * A sequence with seq_lens[b] < 0 or >= Lmax is skipped on the device and
 * sets KVATTN_ERR_DEVICE_BOUNDS in the sticky error word.
 */
KVATTN_API int kv_append(void *k_cache, void *v_cache, const void *k_new,
              const void *v_new, const int32_t *seq_lens, int B, int Hkv,
              int D, int Lmax, kvattn_stream_t stream);

/*
 * gqa_decode_attn -- one decode step of grouped-query attention.
 *
 * Computes, for every sequence b and query head h (kvh = h / (Hq / Hkv)),
 *   out[b,h,:] = softmax_j(scale * q[b,h,:] . K[b,kvh,j,:]) . V[b,kvh,j,:]
 * over positions 0 <= j < seq_lens[b] (see the header comment for the
 * passages this follows).
 *
 *   q                : bf16 [B, Hq, D]
 *   k_cache, v_cache : bf16 [B, Hkv, Lmax, D]
 *   seq_lens         : int32 [B] (device), positions attended per sequence,
 *                      0 <= seq_lens[b] <= Lmax (after this step's append)
 *   out              : fp32 [B, Hq, D], written in full
 *   B, Hq, Hkv, D    : sizes; Hq % Hkv == 0; D in {64, 128, 256}
 *   Lmax             : positions allocated per (b, kvh) in the caches
 *   scale            : finite softmax scale (typically 1/sqrt(D))
 *
 * A sequence with seq_lens[b] == 0 gets an all-zero output row.  One with
 * seq_lens[b] outside [0, Lmax] gets an all-zero row and sets
 * KVATTN_ERR_DEVICE_BOUNDS in the sticky error word.
 * Limits: B <= 65535, Hkv <= 4096, Hq <= 8192, Lmax <= 2^24.
 */
KVATTN_API int gqa_decode_attn(const void *q, const void *k_cache, const void *v_cache,
                    const int32_t *seq_lens, float *out, int B, int Hq,
                    int Hkv, int D, int Lmax, float scale,
                    kvattn_stream_t stream);

/*
 * gqa_decode_step -- one whole decode step in one call: kv_append followed
 * by gqa_decode_attn, fused into the attention kernel.
 *
 * Follows the same passages as the two calls it fuses: the new token's key
 * and value are written into the cache, then its query attends over every
 * cached position including its own ("The Basics of Transformer
 * Inference", the KV-cache paragraph).
 *
 *   q                : bf16 [B, Hq, D]
 *   k_new, v_new     : bf16 [B, Hkv, D], this step's key/value rows
 *   k_cache, v_cache : bf16 [B, Hkv, Lmax, D]; row seq_lens[b] is written
 *   seq_lens         : int32 [B] (device), tokens cached BEFORE this step
 *                      (0 <= seq_lens[b] < Lmax); not modified -- the
 *                      attention covers positions [0, seq_lens[b] + 1)
 *   out              : fp32 [B, Hq, D]
 *
 * Results are identical to kv_append then gqa_decode_attn with lengths
 * seq_lens + 1.  A sequence with seq_lens[b] outside [0, Lmax) is neither
 * appended nor attended (zero output row) and sets KVATTN_ERR_DEVICE_BOUNDS.
 */
KVATTN_API int gqa_decode_step(const void *q, const void *k_new, const void *v_new,
                               void *k_cache, void *v_cache, const int32_t *seq_lens,
                               float *out, int B, int Hq, int Hkv, int D, int Lmax,
                               float scale, kvattn_stream_t stream);

/*
 * kv_append_multi -- kv_append for T new tokens per sequence (the drafted
 * tokens of speculative sampling): token t's rows go into row
 * seq_lens[b] + t.
 *
 *   k_new, v_new : bf16 [B, T, Hkv, D]
 *   seq_lens     : int32 [B] (device), tokens cached before the T new ones;
 *                  not modified
 *   T            : 1 .. 64 (KVATTN_ERR_INVALID_ARG otherwise)
 * The rest as for kv_append; a sequence whose T rows do not all fit
 * (seq_lens[b] + T > Lmax, or seq_lens[b] < 0) is left untouched and sets
 * KVATTN_ERR_DEVICE_BOUNDS.  Bit-exact.
 */
KVATTN_API int kv_append_multi(void *k_cache, void *v_cache, const void *k_new,
                               const void *v_new, const int32_t *seq_lens, int B, int T,
                               int Hkv, int D, int Lmax, kvattn_stream_t stream);

/*
 * gqa_decode_attn_multi -- attention for T new tokens per sequence, causal
 * among themselves: the scoring pass of speculative sampling ("The Basics of
 * Transformer Inference": the big model scores a run of drafted tokens in
 * one pass, sharing the KV-cache loads among them).  The tokens' K/V rows
 * are already in the cache at positions seq_lens[b] - T .. seq_lens[b] - 1;
 * token t attends positions [0, seq_lens[b] - T + 1 + t) -- the cached prefix
 * and the new tokens up to itself -- and gets a zero row when that is empty.
 * A pass of the kernel takes hpg of a K/V head's G query heads for all T
 * tokens (hpg x T query rows, at most 64) and reads each K/V tile once for
 * all of them; when G x T rows do not fit one pass, the heads are split over
 * ceil(G / floor(64 / T)) passes of nearly equal size, each of which reads
 * the K/V head's tiles again (e.g. 48 heads sharing one K/V head: 2 passes
 * of 24 heads for T = 2, 3 of 16 for T = 4, 6 of 8 for T = 8).
 *
 *   q        : bf16 [B, T, Hq, D]
 *   k_cache, v_cache, seq_lens : as for gqa_decode_attn (seq_lens counts the
 *              new tokens too)
 *   out      : fp32 [B, T, Hq, D]
 *   T        : 1 .. 64 (one pass's rows); needs D in {128, 256}, else
 *              KVATTN_ERR_UNSUPPORTED.
 *              T = 1 is gqa_decode_attn.
 * Ownership, streams and device-side errors are those of gqa_decode_attn.
 */
KVATTN_API int gqa_decode_attn_multi(const void *q, const void *k_cache, const void *v_cache,
                                     const int32_t *seq_lens, float *out, int B, int T, int Hq,
                                     int Hkv, int D, int Lmax, float scale,
                                     kvattn_stream_t stream);

/*
 * gqa_decode_attn_window, gqa_decode_step_window -- the same two calls for a
 * local (sliding-window) attention layer: the query at position len_b - 1
 * attends only positions [max(0, len_b - window), len_b), the token itself
 * included ("The Basics of Transformer Inference", item on mixing in local
 * attention layers: a local layer caps how far back a token attends).
 *
 * Arguments, layouts, ownership and errors are those of gqa_decode_attn and
 * gqa_decode_step, plus
 *   window : positions attended at most, >= 1 (KVATTN_ERR_INVALID_ARG
 *            otherwise); window >= Lmax is the full attention.
 * Only the attended rows are read from HBM.  Cache rows in [0, len_b) must
 * hold finite values (the last tile may load rows just before the window,
 * which are then masked); rows at and past len_b may hold anything.
 */
KVATTN_API int gqa_decode_attn_window(const void *q, const void *k_cache, const void *v_cache,
                                      const int32_t *seq_lens, float *out, int B, int Hq,
                                      int Hkv, int D, int Lmax, float scale, int window,
                                      kvattn_stream_t stream);
KVATTN_API int gqa_decode_step_window(const void *q, const void *k_new, const void *v_new,
                                      void *k_cache, void *v_cache, const int32_t *seq_lens,
                                      float *out, int B, int Hq, int Hkv, int D, int Lmax,
                                      float scale, int window, kvattn_stream_t stream);

/*
 * gqa_decode_attn_multi_window -- gqa_decode_attn_multi on a local layer:
 * each of the T new tokens keeps its own window, so token t (at position
 * e_t - 1, e_t = seq_lens[b] - T + 1 + t) attends positions
 * [max(0, e_t - window), e_t), and gets a zero row when e_t <= 0.  The
 * tiles cover the union of the T windows, window + T - 1 positions, read
 * once for all tokens.  Arguments as for gqa_decode_attn_multi, plus window
 * as for gqa_decode_attn_window (>= 1; >= Lmax is gqa_decode_attn_multi).
 * Rows in [0, seq_lens[b]) must hold finite values.
 */
KVATTN_API int gqa_decode_attn_multi_window(const void *q, const void *k_cache,
                                            const void *v_cache, const int32_t *seq_lens,
                                            float *out, int B, int T, int Hq, int Hkv, int D,
                                            int Lmax, float scale, int window,
                                            kvattn_stream_t stream);

/*
 * Paged KV cache.  Instead of one contiguous [Lmax] run of rows per sequence,
 * the cache is a pool of fixed-size blocks and each sequence keeps a block
 * table mapping its logical positions to physical blocks; sequences that
 * share a prefix may point at the same blocks ("Machine Learning
 * Engineering and AI Systems at Scale", section "The key and value cache",
 * on PagedAttention; "The Basics of Transformer Inference", item "Using
 * ragged HBM reads and Paged Attention").  Position j of sequence b is row
 * j % block_size of block block_table[b, j / block_size]:
 *
 *   k_pool, v_pool : bf16 [num_blocks, Hkv, block_size, D]
 *   block_table    : int32 [B, max_blocks] (device, 4-byte aligned); a
 *                    sequence may use max_blocks * block_size positions
 *   block_size     : a power of two in [16, 2^20] (vLLM-style 16-position
 *                    blocks as well as blocks of a few hundred positions)
 *   max_blocks * block_size <= 2^24; num_blocks * Hkv < 2^31
 *
 * Table entries of blocks wholly past a sequence's length are never read;
 * pool rows at and past the length in its last block are never read either
 * (they may hold anything).  A table entry that is read and lies outside
 * [0, num_blocks) sets KVATTN_ERR_DEVICE_BOUNDS in the sticky word; that
 * block then reads as zeros (attention) or is not written (append) -- the
 * sequence's output is then meaningless but no memory outside the pool is
 * touched.  Results are those of the contiguous calls on the cache the
 * table describes.  The attention calls need D in {128, 256} (the
 * tensor-core kernel; KVATTN_ERR_UNSUPPORTED otherwise);
 * gqa_decode_attn_paged and gqa_decode_step_paged attend every position,
 * their _window forms a local window.
 */

/*
 * kv_append_paged -- kv_append / kv_append_multi into a paged pool: token t
 * of sequence b goes to position seq_lens[b] + t.
 *
 *   k_new, v_new : bf16 [B, T, Hkv, D]; T in [1, 64]
 *   seq_lens     : int32 [B] (device), tokens cached before the T new ones
 * A sequence whose T rows do not all fit in max_blocks * block_size
 * positions is left untouched and sets KVATTN_ERR_DEVICE_BOUNDS.  Bit-exact.
 */
KVATTN_API int kv_append_paged(void *k_pool, void *v_pool, const void *k_new,
                               const void *v_new, const int32_t *block_table,
                               const int32_t *seq_lens, int B, int T, int Hkv, int D,
                               int num_blocks, int block_size, int max_blocks,
                               kvattn_stream_t stream);

/*
 * gqa_decode_attn_paged -- gqa_decode_attn (T = 1) or gqa_decode_attn_multi
 * (T new tokens, causal among themselves) over a paged pool.
 *
 *   q        : bf16 [B, T, Hq, D]
 *   seq_lens : int32 [B] (device), positions attended per sequence,
 *              0 <= seq_lens[b] <= max_blocks * block_size (for T > 1 they
 *              count the new tokens too)
 *   out      : fp32 [B, T, Hq, D]
 * The rest as for gqa_decode_attn / gqa_decode_attn_multi.
 */
KVATTN_API int gqa_decode_attn_paged(const void *q, const void *k_pool, const void *v_pool,
                                     const int32_t *block_table, const int32_t *seq_lens,
                                     float *out, int B, int T, int Hq, int Hkv, int D,
                                     int num_blocks, int block_size, int max_blocks,
                                     float scale, kvattn_stream_t stream);

/*
 * gqa_decode_step_paged -- gqa_decode_step over a paged pool: the new
 * token's rows go to position seq_lens[b] (through the block table), then
 * its query attends positions [0, seq_lens[b] + 1).  Arguments as for
 * gqa_decode_step, with the pools and table above in place of the caches.
 */
KVATTN_API int gqa_decode_step_paged(const void *q, const void *k_new, const void *v_new,
                                     void *k_pool, void *v_pool, const int32_t *block_table,
                                     const int32_t *seq_lens, float *out, int B, int Hq,
                                     int Hkv, int D, int num_blocks, int block_size,
                                     int max_blocks, float scale, kvattn_stream_t stream);

/*
 * gqa_decode_attn_paged_window, gqa_decode_step_paged_window -- the two
 * paged calls on a local layer ("The Basics of Transformer Inference", the
 * items on local attention layers and on ragged reads with Paged
 * Attention): the queries attend what gqa_decode_attn_multi_window (T new
 * tokens) and gqa_decode_step_window (one new token, appended first) attend,
 * through the block table.  Arguments as for gqa_decode_attn_paged and
 * gqa_decode_step_paged, plus
 *   window : positions one query attends at most, >= 1
 *            (KVATTN_ERR_INVALID_ARG otherwise); >= max_blocks * block_size
 *            is the full attention.
 * A tile of a paged cache starts on a block boundary, so the first tile
 * read starts at the 128-position boundary at or before the window and its
 * rows before the window are masked: up to 127 positions before each
 * window are read (not attended), and their table entries must be valid
 * and their rows finite.
 */
KVATTN_API int gqa_decode_attn_paged_window(const void *q, const void *k_pool,
                                            const void *v_pool, const int32_t *block_table,
                                            const int32_t *seq_lens, float *out, int B, int T,
                                            int Hq, int Hkv, int D, int num_blocks,
                                            int block_size, int max_blocks, float scale,
                                            int window, kvattn_stream_t stream);
KVATTN_API int gqa_decode_step_paged_window(const void *q, const void *k_new, const void *v_new,
                                            void *k_pool, void *v_pool,
                                            const int32_t *block_table, const int32_t *seq_lens,
                                            float *out, int B, int Hq, int Hkv, int D,
                                            int num_blocks, int block_size, int max_blocks,
                                            float scale, int window, kvattn_stream_t stream);

/*
 * 8-bit KV cache (FP8 E4M3 codes with one fp32 scale per cached row).
 * Quantizing the KV cache to int8 / fp8 saves memory bandwidth and capacity
 * ("The Basics of Transformer Inference", item "Quantization"; "Machine
 * Learning Engineering and AI Systems at Scale", section "Quantization":
 * E4M3 is the inference format, the KV cache is the second thing to
 * quantize).  The pages give no rule; this library's: each cached row (one
 * position of one K/V head, D values) is stored as
 *     scale  = absmax(row) / 448          (1 for an all-zero row)
 *     code_d = E4M3(row_d / scale)        nearest, ties to even, saturating
 * with both divisions in IEEE binary32, and read as code value x scale.
 * E4M3: sign, 4 exponent bits (bias 7), 3 mantissa bits, subnormals, no
 * infinities, largest finite 448 (the OCP 8-bit format).  Rows must be
 * finite.
 *
 *   codes  : uint8 [B, Hkv, Lmax, D] (K and V separately)
 *   scales : fp32  [B, Hkv, Lmax]    (K and V separately)
 */

/* kv_quantize_fp8 -- quantize `rows` rows of D bf16 values (src [rows, D])
 * into codes [rows, D] and scales [rows] by the rule above: e.g. a whole
 * prefilled bf16 cache viewed as B*Hkv*Lmax rows.  D in {64, 128, 256}.
 * Bit-exact. */
KVATTN_API int kv_quantize_fp8(const void *src, void *codes, float *scales, long long rows,
                               int D, kvattn_stream_t stream);

/* kv_append_fp8 -- kv_append into an 8-bit cache: the new token's K and V
 * rows (bf16 [B, Hkv, D]) are quantized into position seq_lens[b], codes and
 * scale.  Errors as for kv_append.  Bit-exact. */
KVATTN_API int kv_append_fp8(void *k_codes, void *v_codes, float *k_scale, float *v_scale,
                             const void *k_new, const void *v_new, const int32_t *seq_lens,
                             int B, int Hkv, int D, int Lmax, kvattn_stream_t stream);

/* gqa_decode_attn_fp8 -- gqa_decode_attn over an 8-bit cache: K[b,kvh,j,:] =
 * E4M3(k_codes[b,kvh,j,:]) * k_scale[b,kvh,j], V likewise.  The cache read
 * per position and K/V head is 2 (D + 4) bytes instead of 4 D.  q bf16
 * [B, Hq, D] (any finite value: each head enters the 8-bit products as two
 * E4M3 parts under a power-of-two scale, exact for a bf16 value), out fp32
 * [B, Hq, D]; lengths, errors and ownership as gqa_decode_attn.
 * Needs D = 128 or 256: the kernel copies each position's codes in rows of
 * 128 (one 128-byte swizzled TMA box per 128 head dims); D = 64 is
 * KVATTN_ERR_UNSUPPORTED (not built: its 64-byte rows would need a layout
 * of their own).  Rows at and past seq_lens[b], codes and scales, are never
 * read. */
KVATTN_API int gqa_decode_attn_fp8(const void *q, const void *k_codes, const void *v_codes,
                                   const float *k_scale, const float *v_scale,
                                   const int32_t *seq_lens, float *out, int B, int Hq, int Hkv,
                                   int D, int Lmax, float scale, kvattn_stream_t stream);

/* gqa_decode_step_fp8 -- kv_append_fp8 followed by gqa_decode_attn_fp8 over
 * seq_lens[b] + 1 positions, in one pass over the 8-bit cache (the decode
 * step of "The Basics of Transformer Inference", KV-cache paragraph: write
 * this token's K/V, then attend, itself included): the attention kernel's
 * copy warp quantizes the new rows (the rule above, bit for bit the bytes
 * kv_append_fp8 writes) into position seq_lens[b] just before it copies the
 * tile that holds that position, so the step is one kernel launch (plus the
 * combine when a sequence is split) instead of two.  k_new, v_new: bf16
 * [B, Hkv, D], 16-byte aligned; seq_lens counts the tokens cached before
 * this step and is not modified.  A sequence with seq_lens[b] outside
 * [0, Lmax - 1] gets no append and a zero output row, and sets
 * KVATTN_ERR_DEVICE_BOUNDS.  D = 128 or 256; other arguments, errors and
 * ownership as gqa_decode_attn_fp8. */
KVATTN_API int gqa_decode_step_fp8(const void *q, const void *k_new, const void *v_new,
                                   void *k_codes, void *v_codes, float *k_scale, float *v_scale,
                                   const int32_t *seq_lens, float *out, int B, int Hq, int Hkv,
                                   int D, int Lmax, float scale, kvattn_stream_t stream);

/*
 * gqa_decode_attn_noalloc -- the same computation as gqa_decode_attn, for
 * callers that must not have the library allocate device memory (for
 * example a server that gives all free GPU memory to its own pool at
 * start-up, or a loop that cannot afford the device synchronisation a
 * cudaFree brings).  The paper has no counterpart: this is a property of
 * the library, not of the method.
 *
 * Same arguments, layouts and errors as gqa_decode_attn.  It always runs the
 * CUDA-core split-KV kernel and keeps the partial results of split sequences
 * in a fixed 4 MiB device array that is part of the library (one per GPU,
 * held until the process exits); it never calls cudaMalloc or cudaFree.
 * The array's address is looked up on the first call made on each device
 * (with that device current); make that first call before capturing work on
 * the device into anything.  All calls on a device share the array: calls
 * whose GPU work overlaps (different streams with no ordering) race and may
 * return wrong results.  A call whose partials would not fit (2 x grid CTAs x
 * heads per pass x (D + 2) floats > 4 MiB, e.g. after kvattn_set_tuning
 * forced a very large grid) returns KVATTN_ERR_UNSUPPORTED and launches
 * nothing.
 */
KVATTN_API int gqa_decode_attn_noalloc(const void *q, const void *k_cache,
                                       const void *v_cache, const int32_t *seq_lens,
                                       float *out, int B, int Hq, int Hkv, int D,
                                       int Lmax, float scale, kvattn_stream_t stream);

/* Static string naming a status code. */
KVATTN_API const char *kvattn_status_string(int status);

/* Detail of the last host-side error on the calling thread ("" if none). */
KVATTN_API const char *kvattn_last_error(void);

/*
 * Synchronises `stream`, then returns and clears the current device's sticky
 * error word (KVATTN_OK if no device-side error was seen since the last
 * check), or KVATTN_ERR_CUDA if synchronisation itself failed.
 */
KVATTN_API int kvattn_check_device_error(kvattn_stream_t stream);

/*
 * Frees every workspace the library holds on every device (after a device
 * synchronisation).  Later calls allocate again on demand.
 */
KVATTN_API void kvattn_release(void);

/*
 * Test and ablation knobs (process-wide; 0 restores the automatic choice).
 *   force_path : 0 auto, 1 CUDA-core FMA kernel, 2 tensor-core kernel
 *   num_ctas   : 0 auto, else the persistent grid size of the attention
 *                kernel (a small value forces long multi-CTA splits)
 * Returns KVATTN_ERR_INVALID_ARG for values out of range.
 */
KVATTN_API int kvattn_set_tuning(int force_path, int num_ctas);

/*
 * Test knob for the failure handling (process-wide; 0 restores the default).
 * Every wait inside the tensor-core split-KV kernel is bounded; this sets
 * how many polls its pipeline waits make before giving up -- the softmax
 * threads' waits for scores and for finished P.V products, and the MMA
 * thread's polling while nothing is ready.  A kernel that gives up sets the
 * device error word to KVATTN_ERR_TIMEOUT (read by kvattn_check_device_error),
 * lets every copy and MMA it already issued finish, frees its tensor memory
 * and returns; the output of that call is undefined.  Waits for work already
 * issued keep their default limit.  With a very small value (1) a call is
 * sure to give up, which is how the tests exercise this path.  Always
 * returns KVATTN_OK.
 */
KVATTN_API int kvattn_set_wait_limit(unsigned int polls);

/*
 * Measurement hook (process-wide).  With two events given (cudaEvent_t
 * handles, owned by the caller), every later attention call records
 * `before` on its stream just before its split-KV kernel and `after` just
 * after it, so that cudaEventElapsedTime(before, after) is that kernel's
 * duration alone.  The records sit between the kernel and its neighbours on
 * the stream, so they also end the programmatic overlap with them: use it to
 * time, not in production.  Pass (NULL, NULL) to stop; one NULL alone is
 * KVATTN_ERR_INVALID_ARG.
 */
KVATTN_API int kvattn_set_kernel_events(void *before, void *after);

/* How a call with these sizes would run (host-side planning only; no GPU
 * work).  num_sms <= 0 queries the current device. */
typedef struct {
    int path;            /* 1 FMA, 2 tensor core */
    int tile_positions;  /* positions per pipeline tile */
    int heads_per_cta;   /* query heads one CTA pass serves */
    int head_groups;     /* passes per (b, kvh): ceil(G / heads_per_cta) */
    int stages;          /* shared-memory pipeline depth */
    int threads;         /* threads per CTA */
    int num_ctas;        /* persistent grid size */
    int smem_bytes;      /* dynamic shared memory per CTA */
    int64_t workspace_bytes; /* partial (m, l, o) buffer this call needs */
} kvattn_plan;

KVATTN_API int kvattn_get_plan(int B, int Hq, int Hkv, int D, int Lmax, int num_sms,
                    kvattn_plan *plan);

#ifdef __cplusplus
}
#endif

#endif /* KVATTN_H */
