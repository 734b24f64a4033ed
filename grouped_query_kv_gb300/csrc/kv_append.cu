// kv_append.cu -- write each sequence's new key/value rows into row
// seq_lens[b] of the cache ("The Basics of Transformer Inference": every
// token's key and value projections are written into the KV cache once), or
// the rows of T new tokens into rows seq_lens[b] .. seq_lens[b] + T - 1.
// With a block table the cache is a pool of fixed-size blocks and position
// j of sequence b lives in block block_table[b][j / block_size]
// ("Machine Learning Engineering and AI Systems at Scale", section "The key
// and value cache", on PagedAttention).
// A bit-exact 16-byte-vector copy; one warp per (b, t, kvh) row pair.
#include "internal.h"

namespace kvattn {

namespace {

__global__ void __launch_bounds__(128)
    kv_append_kernel(uint4 *__restrict__ k_cache, uint4 *__restrict__ v_cache,
                     const uint4 *__restrict__ k_new, const uint4 *__restrict__ v_new,
                     const int32_t *__restrict__ seq_lens, int B, int T, int Hkv, int D,
                     int Lmax, const int32_t *__restrict__ block_table, int block_lg,
                     int max_blocks, int num_blocks, unsigned int *err) {
    // the attention kernel that follows may start its prologue now; it
    // waits for these writes with griddepcontrol.wait before reading
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int row = blockIdx.x * 4 + (threadIdx.x >> 5);  // (b, t, kvh) of k_new
    const int lane = threadIdx.x & 31;
    if (row >= B * T * Hkv) return;
    const int kvh = row % Hkv;
    const int t = (row / Hkv) % T;
    const int b = row / (Hkv * T);
    const int pos = seq_lens[b];
    if (pos < 0 || pos > Lmax - T) {  // every one of the T rows must fit
        if (lane == 0) atomicCAS(err, 0u, (unsigned int)DEV_ERR_BOUNDS);
        return;
    }
    const int vecs = D / 8;  // 16-byte vectors per row
    size_t dst;
    if (block_table) {
        const int j = pos + t;
        const int blk = block_table[(size_t)b * max_blocks + (j >> block_lg)];
        if (blk < 0 || blk >= num_blocks) {  // a block outside the pool: skip the row
            if (lane == 0) atomicCAS(err, 0u, (unsigned int)DEV_ERR_BOUNDS);
            return;
        }
        dst = ((((size_t)blk * Hkv + kvh) << block_lg) + (j & ((1 << block_lg) - 1))) * vecs;
    } else {
        dst = (((size_t)b * Hkv + kvh) * Lmax + pos + t) * vecs;
    }
    const size_t src = (size_t)row * vecs;
    for (int v = lane; v < vecs; v += 32) {
        k_cache[dst + v] = k_new[src + v];
        v_cache[dst + v] = v_new[src + v];
    }
}

}  // namespace

cudaError_t launch_kv_append(void *k_cache, void *v_cache, const void *k_new, const void *v_new,
                             const int32_t *seq_lens, int B, int T, int Hkv, int D, int Lmax,
                             const int32_t *block_table, int block_lg, int max_blocks,
                             int num_blocks, unsigned int *err, cudaStream_t stream) {
    const int rows = B * T * Hkv;
    const int blocks = (rows + 3) / 4;
    kv_append_kernel<<<blocks, 128, 0, stream>>>(
        static_cast<uint4 *>(k_cache), static_cast<uint4 *>(v_cache),
        static_cast<const uint4 *>(k_new), static_cast<const uint4 *>(v_new), seq_lens, B, T, Hkv,
        D, Lmax, block_table, block_lg, max_blocks, num_blocks, err);
    return cudaGetLastError();
}

}  // namespace kvattn
