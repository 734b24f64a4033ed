// internal.h -- declarations shared by the library's translation units
// (host launchers and the parameter blocks the kernels receive).
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace kvattn {

// Error codes written into the sticky per-device word (same values as the
// public kvattn_status enum).
enum : unsigned int { DEV_ERR_BOUNDS = 5u, DEV_ERR_TIMEOUT = 6u };

// One decode-attention call, as the split-KV kernels and the combine see it.
//
// Work decomposition ("segments" and "tiles").  A segment is one
// (sequence b, K/V head kvh, head group hg): the query heads
// [kvh*G + hg*heads_per_seg, ...) that read K/V head kvh.  Segment (b,kvh,hg)
// owns ntiles(b) = max(1, ceil(len_b / tile)) tiles of `tile` consecutive
// cached positions.  All tiles of all segments, in (b, kvh, hg, t) order,
// form one flat list that is cut into num_ctas equal contiguous ranges, one
// per CTA of the persistent grid.  A segment cut by a range boundary is
// computed in pieces whose (m, l, o) partials go to the workspace and are
// merged by the combine kernel.
struct DecodeParams {
    const uint16_t *q;        // bf16 [B, Hq, D]
    const int32_t *seq_lens;  // [B]
    int len_add;              // 1: fused append -- seq_lens count tokens cached before this step
    const uint16_t *k_new;    // fused append only: bf16 [B, Hkv, D] rows written at seq_lens[b]
    const uint16_t *v_new;
    uint16_t *k_cache;        // fused append only: the caches the rows go into
    uint16_t *v_cache;
    float *out;               // [B, Hq, D]
    float *ws_o;              // [2*num_ctas, heads_per_seg, D]  partial o (unnormalised)
    float *ws_ml;             // [2*num_ctas, heads_per_seg, 2]  partial (m, l), m in log2 units
    unsigned int *err;        // sticky device error word
    int *split;               // [grid, 4] per-CTA combine record (b, seg, first slot, pieces)
    int B, Hq, Hkv, D, Lmax;
    int G;                    // Hq / Hkv
    int heads_per_seg;        // query rows one segment serves: heads, or (token, head) pairs
                              // for T new tokens (hpg heads x T tokens)
    int head_groups;          // passes per (b, kvh): ceil(G / hpg)
    int hpg;                  // query heads per pass (T = 1: heads_per_seg)
    int tile;                 // positions per tile
    int window;               // positions the tiles of a sequence span at most (>= Lmax: all):
                              // the union of its T queries' windows, qwin + T - 1
    int T;                    // new tokens (queries) per sequence, >= 1; q and out are
                              // [B, T, Hq, D] and token t attends [0, len - T + 1 + t)
    int q_bytes;              // tensor-core path: bytes of one piece's q load
    int cost_piece;           // schedule cost of starting and finishing a piece, in
                              // units where a tile costs 32
    float scale_log2;         // scale * log2(e)
    // Paged cache (block_table non-null): k_cache/v_cache are pools
    // [num_blocks, Hkv, 2^block_lg, D]; position j of sequence b is row
    // j mod 2^block_lg of block block_table[b * max_blocks + (j >> block_lg)],
    // and Lmax = max_blocks << block_lg.
    const int32_t *block_table;
    int block_lg;
    int max_blocks;
    int num_blocks;
    // 8-bit cache (decode_fp8.cu): one fp32 scale per cached row,
    // [B, Hkv, Lmax] for K and for V; null otherwise
    const float *k_scale;
    const float *v_scale;
    // tensor-core kernel: polls before a pipeline wait gives up (the softmax
    // threads' waits and the MMA thread's idle polling); 0 = the default.
    // Waits for copies and MMAs already issued always keep the default.
    unsigned int wait_limit;
    int qwin;                 // positions one query attends at most (>= Lmax: all)
    int walign;               // 0, or tile - 1 (paged cache): window spans start on a tile
                              // boundary and the rows before a query's window are masked
};

// Host launchers (return cudaError_t of the launch).
// block_table null: contiguous caches [B, Hkv, Lmax, D]; else pools as in
// DecodeParams (Lmax = max_blocks << block_lg).
cudaError_t launch_kv_append(void *k_cache, void *v_cache, const void *k_new, const void *v_new,
                             const int32_t *seq_lens, int B, int T, int Hkv, int D, int Lmax,
                             const int32_t *block_table, int block_lg, int max_blocks,
                             int num_blocks, unsigned int *err, cudaStream_t stream);

// FMA split-KV kernel; heads_per_seg must be the value plan_fma() returned.
cudaError_t launch_decode_fma(const CUtensorMap &tmk, const CUtensorMap &tmv,
                              const DecodeParams &p, int num_ctas, int smem_bytes,
                              cudaStream_t stream);
int fma_heads_per_seg(int G);
int fma_tile(int D);
int fma_stages(int D);
int fma_smem_bytes(int D, int heads_per_seg);
int fma_threads();
cudaError_t fma_prepare(int D, int heads_per_seg, int smem_bytes);

// Tensor-core (tcgen05) split-KV kernel for D in {128, 256}; np = query heads
// per pass rounded up to a multiple of 16 (tc_np).
int tc_np(int G, int D);
int tc_heads_per_seg(int G, int D);
int tc_max_cols_several(int D);
int tc_tile();
int tc_threads(int D, int np);  // threads of a CTA for np columns per pass
int tc_smem_bytes(int D, int np);
int tc_stages(int D, int np);
cudaError_t tc_prepare(int D, int np, bool several_tokens);
cudaError_t launch_decode_tc(const CUtensorMap &tmk, const CUtensorMap &tmv,
                             const CUtensorMap &tmq, const DecodeParams &p, int np, int num_ctas,
                             cudaStream_t stream);
// the one-token 16-column instantiations (compiled in their own unit)
cudaError_t tc_prepare_one16(int D);
cudaError_t launch_decode_tc_one16(const CUtensorMap &tmk, const CUtensorMap &tmv,
                                   const CUtensorMap &tmq, const DecodeParams &p, int num_ctas,
                                   cudaStream_t stream);
// the same kernel reading a paged cache (p.block_table set; the K/V maps are
// over the pools, box rows min(block size, 128))
cudaError_t tc_prepare_paged(int D, int np, bool several_tokens);
cudaError_t launch_decode_tc_paged(const CUtensorMap &tmk, const CUtensorMap &tmv,
                                   const CUtensorMap &tmq, const DecodeParams &p, int np,
                                   int num_ctas, cudaStream_t stream);

cudaError_t launch_combine(const DecodeParams &p, int num_ctas, cudaStream_t stream);

// 8-bit (FP8 E4M3) cache: the attention kernel (D = 128 or 256; np as
// tc_np), the row quantizer and the append.
int q8_smem_bytes(int D, int np);
cudaError_t launch_decode_q8(const CUtensorMap &tmk, const CUtensorMap &tmv,
                             const DecodeParams &p, int np, int num_ctas, cudaStream_t stream);
cudaError_t launch_quantize_fp8(const void *src, void *codes, float *scales, long long rows,
                                int D, cudaStream_t stream);
cudaError_t launch_kv_append_fp8(void *k_codes, void *v_codes, float *k_scale, float *v_scale,
                                 const void *k_new, const void *v_new, const int32_t *seq_lens,
                                 int B, int Hkv, int D, int Lmax, unsigned int *err,
                                 cudaStream_t stream);

// Shared with the allocation-free entry point (defined in api.cu).
int api_fail(int status, const char *msg);
int api_check_args(const void *q, const void *k_cache, const void *v_cache,
                   const int32_t *seq_lens, const float *out, int B, int Hq, int Hkv, int D,
                   int Lmax, float scale);
int api_forced_ctas();
int api_encode_cache_maps(CUtensorMap *tmk, CUtensorMap *tmv, const void *k_cache,
                          const void *v_cache, int D, int Lmax, int BH, int tile);
int api_error_word(unsigned int **word);
int api_cuda_fail(cudaError_t e, const char *what);

}  // namespace kvattn
