// decode_tc.cuh -- split-KV decode attention on the 5th-generation tensor
// cores (tcgen05, accumulators in tensor memory), for any query group size
// G when D is 128 or 256.
//
// Grouped-query attention shares each K/V head among G query heads ("The
// Basics of Transformer Inference", item "Grouped multi-query attention";
// "Tensor Parallelism ...", section "The GQA ceiling"), so every cached
// position meets G queries: the score and value products of one tile are
// small dense matrix products, done here as
//     S^T [T x NP]  = K_tile [T x D] . Q^T [D x NP]          (M = 128 positions)
//     O^T [D x NP] += V_tile^T [D x T] . P^T [T x NP]        (M = 128 head dims)
// with NP = G rounded up to a multiple of 16 (at most 64 heads per pass).
//
// Warp roles (320 threads, or 192 where the softmax keeps one group; one
// persistent CTA per SM):
//   warp 0    TMA producer: per segment piece the group's q rows (2-D map,
//             128-byte swizzle, double-buffered), and the K and V tiles of
//             T = 128 positions as 32 KB chunks (two 64-column boxes) into a
//             ring of NCH chunks, each V tile one K tile behind its K tile.
//   warp 1    allocates tensor memory; one thread issues every tcgen05.mma
//             (QK of tile i, then PV of tile i-1) and the commits that release
//             ring chunks, score buffers and probability buffers.
//   warps 2-9 softmax, in two groups of four that each take half of the
//             pass's columns (warps 2-5 alone for the 16-column passes at
//             D = 128; TcGroups): thread r of a group owns tile position r
//             (TMEM lane r): loads its group's scores, masks positions past
//             the length, computes p = 2^(s - m) and writes it as two bf16
//             parts (hi + lo) into shared memory (the B operands of two PV
//             products), and at the end of a piece reads O^T rows (lane =
//             head dim).
// The running max is only moved when a score exceeds it by more than 2^8
// (a vote over all softmax threads); then the exact tile max is taken and
// O, l are rescaled.  Between moves p stays below 2^8, so fp32 sums are safe and
// the result is the same softmax.
#pragma once

#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"
#include "schedule.cuh"

namespace kvattn {

namespace {

constexpr int kT = 128;             // positions per tile
constexpr int kChunk = 32768;       // one ring chunk: 2 boxes of 64 columns x 128 rows
constexpr int kSmemLimit = 232448;  // 227 KB per CTA
constexpr float kTau = 8.0f;        // log2 headroom before the running max must move
constexpr int kBarSoftmax = 1;      // named barrier: all softmax threads (128 or 256)
constexpr int kBarEnd = 2;          // named barrier: all warps before TMEM is freed
constexpr int kBarGroup = 3;        // named barriers 3, 4: softmax group 0, 1 (128 threads each)
constexpr uint32_t kMmaIdleLimit = 1u << 23;  // ~seconds of polling with nothing ready

__host__ __device__ constexpr int pow2_at_least(int x) {
    int p = 32;
    while (p < x) p <<= 1;
    return p;
}

template <int D, int NP>
struct TcCfg {
    static constexpr int KCH = D / 128;               // ring chunks per K (or V) tile
    static constexpr int QB = (D / 64) * NP * 128;    // one q buffer (swizzled, K-major)
    static constexpr int PB = NP * kT * 2;            // one P^T operand (bf16); hi and lo per stage
    static constexpr int NBAR_FIXED = 14;
    static constexpr int FIXED = 2 * QB + 4 * 64 * 4 + 3 * 64 * 4 + 64 +
                                 1024 + (2 * 5 + NBAR_FIXED) * 8;
    // P^T stages (each holding the hi and lo parts): two when the ring still
    // fits one K and one V tile, else one (then tile i's P waits for PV of i-1)
    static constexpr int NCH_2P = (kSmemLimit - FIXED - 2 * 2 * PB) / kChunk;
    static constexpr int PST = NCH_2P >= 2 * KCH ? 2 : 1;
    static constexpr int NCH_FIT = (kSmemLimit - FIXED - PST * 2 * PB) / kChunk;
    static constexpr int NCH = NCH_FIT > 5 ? 5 : NCH_FIT;
    static_assert(NCH >= 2 * KCH, "ring must hold one K and one V tile");

    static constexpr int off_ring = 0;
    static constexpr int off_q = NCH * kChunk;
    static constexpr int off_p = off_q + 2 * QB;
    static constexpr int off_red = off_p + PST * 2 * PB; // float [4][64]
    static constexpr int off_ltot = off_red + 4 * 64 * 4; // float [64]
    static constexpr int off_mref = off_ltot + 64 * 4;    // float [64] running max (log2 units)
    static constexpr int off_alpha = off_mref + 64 * 4;   // float [64] rescale factors
    static constexpr int off_bar = off_alpha + 64 * 4;
    static constexpr int nbar = 2 * NCH + NBAR_FIXED;
    static constexpr int off_misc = off_bar + nbar * 8;  // tmem base, abort flag
    static constexpr int bytes = off_misc + 64;
    static constexpr int alloc = bytes + 1024;

    // TMEM columns: S0, S1 (NP each), then per 128-row head-dim block an O
    // accumulator of 2*NP columns: the V.P_hi products and the V.P_lo products
    static constexpr int TMEM_NEED = 2 * NP + KCH * 2 * NP;
    static constexpr int TMEM_COLS = pow2_at_least(TMEM_NEED);
    static constexpr uint32_t IDESC_QK = idesc_bf16_f32(128, NP, false, false);
    static constexpr uint32_t IDESC_PV = idesc_bf16_f32(128, 2 * NP, true, true);
};

// Softmax warps: two groups of four (each with half of the columns, so two
// softmax warps share each SM sub-partition), or one group for the passes
// of 16 columns at D = 128.  Two groups leave 168 registers a thread (ten
// warps: three on some sub-partitions); the partial-output stores of a split
// piece go 8 columns at a time so that 24 and 32 columns a group fit.
// Measured on GB300 against one group: the 48-head PaLM-540B pass 55.7 ->
// 50.9 us, a 64-head one at D = 128 48.0 -> 37.4 us, the 16-head PaLM-8B
// pass 30.8 -> 30.1 us, the 32-column one 2 % faster, the several-token
// passes of 32 and 48 columns 25 % and 8 %; the 16-column passes at D = 128
// (Llama-70B, the G = 4 sweep, the local window) ran ~1 % slower split.
template <int D, int NP, bool MT>
struct TcGroups {
    static constexpr int SG = (NP >= 32 || D == 256) ? 2 : 1;
    static constexpr int NPH = NP / SG;            // columns of one softmax group
    static constexpr int THREADS = 64 + 128 * SG;
    static constexpr int RS = SG == 1 ? 64 : 32;   // stride of a warp's column totals in red
};

struct Bars {
    uint64_t *chunk_full, *chunk_empty;
    uint64_t *q_full, *q_empty, *s_full, *s_empty, *p_full, *pv_done;
    uint64_t *o_free, *drain;
};

__device__ __forceinline__ void set_error(unsigned int *err, unsigned int code) {
    atomicCAS(err, 0u, code);
}

// Bounded wait that also gives up early once another role has aborted.
__device__ __forceinline__ bool wait_bar(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                         uint32_t limit = KVATTN_SPIN_LIMIT) {
    for (uint32_t it = 0; it < limit; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 255u) == 255u && *abort_flag) return false;
    }
    *abort_flag = 1;
    return false;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sumf(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

struct OpMax {
    __device__ __forceinline__ float operator()(float a, float b) const { return fmaxf(a, b); }
};
struct OpSum {
    __device__ __forceinline__ float operator()(float a, float b) const { return a + b; }
};

// Totals over the warp's 32 lanes of N columns (N = 8, 16 or 32), column
// c's total stored to out[c]: a reduce-scatter in which each butterfly step
// keeps half of a lane's columns and adds its partner's copy of them, so N/2
// + N/4 + ... shuffles instead of 5 per column.  For N < 32, 32 / N lanes
// end with each column (all store it).  (Compile-time steps: every index is a
// constant, so the columns stay in registers.)
template <int M, int O, class Op>
__device__ __forceinline__ void warp_cols_step(float (&a)[32], int lane, int &col, Op op) {
    if constexpr (M > 1) {
        constexpr int H = M / 2;
        const bool up = (lane & O) != 0;  // keeps the upper half of its columns
#pragma unroll
        for (int i = 0; i < H; ++i) {
            const float keep = up ? a[i + H] : a[i];
            const float send = up ? a[i] : a[i + H];
            a[i] = op(keep, __shfl_xor_sync(0xffffffffu, send, O));
        }
        if (up) col += H;
        if constexpr (O > 1) warp_cols_step<H, O / 2>(a, lane, col, op);
    } else {
        a[0] = op(a[0], __shfl_xor_sync(0xffffffffu, a[0], O));
        if constexpr (O > 1) warp_cols_step<1, O / 2>(a, lane, col, op);
    }
}

template <int N, class Op>
__device__ __forceinline__ void warp_cols(const float *v, float *out, int lane, Op op) {
    float a[32];
#pragma unroll
    for (int i = 0; i < N; ++i) a[i] = v[i];
    int col = 0;
    warp_cols_step<N, 16>(a, lane, col, op);
    out[col] = a[0];
}

// N columns (a multiple of 8) of this warp's 32 TMEM lanes from taddr.
template <int N>
__device__ __forceinline__ void tmem_ld_n(uint32_t taddr, float (&v)[N]) {
#pragma unroll
    for (int c = 0; c + 16 <= N; c += 16) {
        float t[16];
        tmem_ld16(taddr + c, t);
#pragma unroll
        for (int k = 0; k < 16; ++k) v[c + k] = t[k];
    }
    if constexpr (N % 16 == 8) {
        float t[8];
        tmem_ld8(taddr + N - 8, t);
#pragma unroll
        for (int k = 0; k < 8; ++k) v[N - 8 + k] = t[k];
    }
}
template <int N>
__device__ __forceinline__ void tmem_st_n(uint32_t taddr, const float (&v)[N]) {
#pragma unroll
    for (int c = 0; c + 16 <= N; c += 16) {
        float t[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) t[k] = v[c + k];
        tmem_st16(taddr + c, t);
    }
    if constexpr (N % 16 == 8) {
        float t[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) t[k] = v[N - 8 + k];
        tmem_st8(taddr + N - 8, t);
    }
}

// Totals over the warp's lanes of N columns (a multiple of 8), column c's
// total stored to out[c] (by every lane that ends with it).
template <int N, class Op>
__device__ __forceinline__ void warp_cols_n(const float (&v)[N], float *out, int lane, Op op) {
#pragma unroll
    for (int c0 = 0; c0 + 32 <= N; c0 += 32) warp_cols<32>(v + c0, out + c0, lane, op);
    if constexpr (N % 32 >= 16) warp_cols<16>(v + N / 32 * 32, out + N / 32 * 32, lane, op);
    if constexpr (N % 16 == 8) warp_cols<8>(v + N - 8, out + N - 8, lane, op);
}

// Ring order of the K/V chunks of a CTA's n tiles (KCH chunks per tile each):
//     K_0, K_1, V_0, K_2, V_1, ..., K_{n-1}, V_{n-2}, V_{n-1}
// V_i goes in behind K_{i+1}: it is needed only after tile i's scores and
// probabilities exist, so issuing it one K tile later shortens the time it
// sits in the ring, and the ring keeps more bytes in flight.
template <int KCH>
__device__ __forceinline__ long long k_chunk(long long i, int c) {
    return (i == 0 ? 0 : (2 * i - 1) * KCH) + c;
}
template <int KCH>
__device__ __forceinline__ long long v_chunk(long long j, int c, long long n) {
    return (j == n - 1 ? (2 * n - 1) * KCH : (2 * j + 2) * KCH) + c;
}
// Whether ring chunk m is a V chunk; if so *tile receives its tile.
template <int KCH>
__device__ __forceinline__ bool chunk_is_v(long long m, long long n, long long *tile) {
    if (m < KCH) return false;
    const long long r = (m - KCH) / (2 * KCH) + 1;
    const long long w = (m - KCH) % (2 * KCH);
    if (r == n || w >= KCH) {
        *tile = r - 1;
        return true;
    }
    return false;
}

// MT: several new tokens per sequence (columns are (token, head), causal
// limits on the last tile); a separate instantiation, so the one-token
// kernel carries none of it.
// PG: a paged cache ("Machine Learning Engineering and AI Systems at Scale",
// section "The key and value cache", on PagedAttention): the K/V maps are
// over pools [num_blocks * Hkv, block_size, D] and each tile's rows come
// through the sequence's block table, one TMA box per block the tile spans
// (block_size >= 128: one box; smaller blocks: 128 / block_size boxes,
// stacked in shared memory exactly as one 128-row box would land).  A
// sequence's last tile ends at its length as in the contiguous cache: for
// blocks of 128 positions or more the box simply starts before the last
// block (rows before it read as zeros); for smaller blocks the last block's
// n rows are loaded to end the tile, after block_size - n zero rows, behind
// the earlier blocks' full rows -- the "hole" rows are masked.  Table
// entries of blocks past the length are never read.
// Box size sets the speed: measured on GB300, tiles made of 16-row boxes
// stream at about 0.70 and of 32-row boxes at 0.88 of what 64-row and larger
// boxes reach (a fixed cost per box in the copy engine), whatever the
// blocks' placement in the pool; 16-byte cp.async copies issued by the one
// producer warp were slower still.
template <int D, int NP, bool MT, bool PG>
__global__ void __launch_bounds__(TcGroups<D, NP, MT>::THREADS, 1)
    decode_tc_kernel(const __grid_constant__ CUtensorMap tmk,
                     const __grid_constant__ CUtensorMap tmv,
                     const __grid_constant__ CUtensorMap tmq, const DecodeParams p) {
    using C = TcCfg<D, NP>;
    using SGC = TcGroups<D, NP, MT>;
    constexpr int KCH = C::KCH;
    constexpr int NCH = C::NCH;

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *ring = smem + C::off_ring;
    uint8_t *qbuf = smem + C::off_q;
    uint8_t *pbuf = smem + C::off_p;
    float *red = reinterpret_cast<float *>(smem + C::off_red);
    float *ltot_s = reinterpret_cast<float *>(smem + C::off_ltot);
    float *mref_s = reinterpret_cast<float *>(smem + C::off_mref);
    float *alpha_s = reinterpret_cast<float *>(smem + C::off_alpha);
    uint64_t *bar_base = reinterpret_cast<uint64_t *>(smem + C::off_bar);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::off_misc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::off_misc + 16);

    Bars bs;
    bs.chunk_full = bar_base;
    bs.chunk_empty = bar_base + NCH;
    bs.q_full = bar_base + 2 * NCH;
    bs.q_empty = bs.q_full + 2;
    bs.s_full = bs.q_empty + 2;
    bs.s_empty = bs.s_full + 2;
    bs.p_full = bs.s_empty + 2;
    bs.pv_done = bs.p_full + 2;
    bs.o_free = bs.pv_done + 2;
    bs.drain = bs.o_free + 1;

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int segs_per_b = p.Hkv * p.head_groups;

    if (tid == 0) {
        for (int s = 0; s < NCH; ++s) {
            mbar_init(&bs.chunk_full[s], 1);
            mbar_init(&bs.chunk_empty[s], 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&bs.q_full[s], 1);
            mbar_init(&bs.q_empty[s], 1);
            mbar_init(&bs.s_full[s], 1);
            mbar_init(&bs.s_empty[s], 4 * SGC::SG);  // one arrival per softmax warp
            mbar_init(&bs.p_full[s], 4 * SGC::SG);
            mbar_init(&bs.pv_done[s], 1);
        }
        mbar_init(bs.o_free, 4 * SGC::SG);
        mbar_init(bs.drain, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tmk);
        prefetch_tmap(&tmv);
        prefetch_tmap(&tmq);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, C::TMEM_COLS);
        tmem_relinquish();
    }
    // everything above overlaps the previous kernel's tail
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    pdl_wait_prior();  // the caches, q and lengths may come from the previous kernel
    // each warp locates the CTA's tile range by itself: no block barrier
    // stands between reading the lengths and the first TMA load
    const LenView lens{p.seq_lens, p.len_add, p.window, PG ? p.walign : 0};  // (only a paged cache aligns)
    const SchedCost wcost{p.cost_piece};
    const SchedStart st = warp_locate(lens, p.B, p.Lmax, kT, segs_per_b, wcost, blockIdx.x, gridDim.x);
    // (a softmax warp writes the record: the producer goes straight to its loads)
    if (warp == 2) sched_split_record(lens, p.B, p.Lmax, kT, segs_per_b, wcost, blockIdx.x, st, p.split);
    if (!st.found) {  // (a range that has a start is never empty)
        if (warp == 1) tmem_dealloc(tmem, C::TMEM_COLS);
        pdl_launch_dependents();
        return;
    }
    const long long ntiles = st.g_end - st.g_begin;
    const uint32_t ring_s = smem_u32(ring);
    const uint32_t qbuf_s = smem_u32(qbuf);
    const uint32_t pbuf_s = smem_u32(pbuf);

    // ================================================================ producer
    // The whole warp walks the tile list (it needs all lanes for the fused
    // append); lane 0 alone waits on ring slots and issues the copies.
    if (warp == 0) {
        const uint64_t pol = l2_policy_evict_first();
        TileIter itk, itv;  // tile of the next K chunks / of the next V chunks
        itk.init(lens, p.B, p.Lmax, kT, segs_per_b, st);
        itv.init(lens, p.B, p.Lmax, kT, segs_per_b, st);
        long long n = 0;
        int piece = 0;
        bool ok = true;
        // paged: boxes per tile (lanes 0 .. nbox-1 issue one each) and the
        // shared-memory bytes of one box's 64 columns
        const int nbox = PG ? (p.block_lg >= 7 ? 1 : kT >> p.block_lg) : 1;
        const int box_bytes = PG ? (p.block_lg >= 7 ? kT : 1 << p.block_lg) * 128 : 0;
        // one ring chunk: two 64-column halves of 128 positions
        auto issue = [&](const void *tm, int c, int y, int z) -> bool {
            const int slot = (int)(n % NCH);
            bool w = true;
            if (lane == 0 && n >= NCH)
                w = wait_bar(&bs.chunk_empty[slot], (uint32_t)(((n / NCH) - 1) & 1), abort_flag);
            if (!__shfl_sync(0xffffffffu, w, 0)) return false;
            if (PG) {
                if (lane == 0) mbar_arrive_expect_tx(&bs.chunk_full[slot], kChunk);
                __syncwarp();
                if (lane < nbox) {
                    uint8_t *dst = ring + slot * kChunk + lane * box_bytes;
                    tma_load_3d(dst, tm, &bs.chunk_full[slot], (2 * c) * 64, y, z, pol);
                    tma_load_3d(dst + 16384, tm, &bs.chunk_full[slot], (2 * c + 1) * 64, y, z, pol);
                }
            } else if (lane == 0) {
                mbar_arrive_expect_tx(&bs.chunk_full[slot], kChunk);
                uint8_t *dst = ring + slot * kChunk;
                tma_load_3d(dst, tm, &bs.chunk_full[slot], (2 * c) * 64, y, z, pol);
                tma_load_3d(dst + 16384, tm, &bs.chunk_full[slot], (2 * c + 1) * 64, y, z, pol);
            }
            ++n;
            return true;
        };
        // paged: this lane's box of tile `it` -- in-block first row y and the
        // table entry of its block (-1: a block before position 0, read as
        // zeros).  The entry is loaded one tile ahead of its use, so its
        // latency hides behind the previous tile's copies.
        auto paged_fetch = [&](const TileIter &it, int &y, int &blk, bool &use) {
            const int lg = p.block_lg;
            const int len = seq_valid_len(it.len, p.Lmax);
            int k;  // logical block
            if (lg >= 7) {
                const int r0 = it.row0();
                k = (r0 + kT - 1) >> lg;  // the block of the tile's last row
                y = r0 - (k << lg);
            } else if (!it.last_tile_of_segment()) {
                k = (it.first_pos() >> lg) + lane;
                y = 0;
            } else {
                const int kend = (len - 1) >> lg;  // -1 for an empty sequence
                k = kend - (nbox - 1 - lane);
                y = lane == nbox - 1 ? len - ((kend + 1) << lg) : 0;
            }
            use = lane < nbox && k >= 0;
            blk = use ? p.block_table[(size_t)it.b * p.max_blocks + k] : -1;
        };
        // the pool row of a fetched entry for K/V head kvh (-1: zeros)
        auto paged_row = [&](int blk, bool use, int kvh) -> int {
            if (!use) return -1;
            if (blk >= 0 && blk < p.num_blocks) return blk * p.Hkv + kvh;
            set_error(p.err, DEV_ERR_BOUNDS);
            return -1;
        };
        int ky = 0, kz = -1, vy = 0, vz = -1;  // paged: boxes of the current K and V tiles
        int ny = 0, nblk = -1;                  // paged: the next K tile's, fetched early
        bool nuse = false;
        if (PG) paged_fetch(itk, ny, nblk, nuse);
        for (long long r = 0; r <= ntiles && ok; ++r) {
            vy = ky;  // V of tile r-1 comes from the blocks of K tile r-1
            vz = kz;
            if (r < ntiles) {  // K of tile r (and the group's q at a piece start)
                const int kvh = itk.seg / p.head_groups;
                const int hg = itk.seg % p.head_groups;
                if (r == 0 || itk.t == 0) {
                    const int qs = piece & 1;
                    bool w = true;
                    if (lane == 0 && piece >= 2)
                        w = wait_bar(&bs.q_empty[qs], ((piece >> 1) - 1) & 1, abort_flag);
                    if (!__shfl_sync(0xffffffffu, w, 0)) {
                        ok = false;
                        break;
                    }
                    if (lane == 0) {
                        // one token: q as (D, B*Hq, 1), the NP rows from the group's
                        // first head; T tokens: q as (D, Hq, B*T), the group's heads
                        // of each of the sequence's T tokens, rows ordered (token, head)
                        mbar_arrive_expect_tx(&bs.q_full[qs], (uint32_t)p.q_bytes);
                        const int h0 = kvh * p.G + hg * p.hpg;
                        const int qy = MT ? h0 : itk.b * p.Hq + h0;
                        const int qz = MT ? itk.b * p.T : 0;
#pragma unroll
                        for (int sl = 0; sl < D / 64; ++sl)
                            tma_load_3d_plain(qbuf + qs * C::QB + sl * NP * 128, &tmq,
                                              &bs.q_full[qs], sl * 64, qy, qz);
                    }
                    ++piece;
                }
                const int z = itk.b * p.Hkv + kvh;
                // fused append: this tile holds the new token's row
                if (p.len_add && itk.last_tile_of_segment() && itk.len >= 1 && itk.len <= p.Lmax) {
                    const int j = itk.len - 1;
                    if (!PG) {
                        append_row_warp(p, z, (size_t)z * p.Lmax + j, D, lane);
                    } else {
                        const int blk = p.block_table[(size_t)itk.b * p.max_blocks + (j >> p.block_lg)];
                        if (blk >= 0 && blk < p.num_blocks)
                            append_row_warp(p, z,
                                            (((size_t)blk * p.Hkv + kvh) << p.block_lg) +
                                                (j & ((1 << p.block_lg) - 1)),
                                            D, lane);
                        else if (lane == 0)
                            set_error(p.err, DEV_ERR_BOUNDS);
                    }
                }
                if (PG) {
                    ky = ny;
                    kz = paged_row(nblk, nuse, kvh);
                }
#pragma unroll
                for (int c = 0; c < KCH && ok; ++c)
                    ok = PG ? issue(&tmk, c, ky, kz) : issue(&tmk, c, itk.row0(), z);
                itk.next();
                if (PG && r + 1 < ntiles) paged_fetch(itk, ny, nblk, nuse);
            }
            if (r >= 1 && ok) {  // V of tile r-1
                const int z = itv.b * p.Hkv + itv.seg / p.head_groups;
#pragma unroll
                for (int c = 0; c < KCH && ok; ++c)
                    ok = PG ? issue(&tmv, c, vy, vz) : issue(&tmv, c, itv.row0(), z);
                itv.next();
            }
        }
        if (!ok && lane == 0) {
            set_error(p.err, DEV_ERR_TIMEOUT);
            *abort_flag = 1;
        }
        // every load of this CTA is issued: the next kernel (the combine) may
        // be scheduled now -- late enough that its waiting blocks do not sit
        // beside this kernel for long, early enough to hide its launch
        pdl_launch_dependents();
        named_bar_sync(kBarEnd, SGC::THREADS);
        if (*abort_flag && lane == 0) {
            // a role gave up, so copies may still be in flight that no one
            // consumed: let them land before the CTA exits -- the last NCH
            // ring chunks and the last two q loads (earlier ones were waited
            // for before their slots were reused)
            volatile int never = 0;
            const long long first = n > NCH ? n - NCH : 0;
            for (long long k = first; k < n; ++k)
                wait_bar(&bs.chunk_full[k % NCH], (uint32_t)((k / NCH) & 1), &never);
            for (int q = piece > 2 ? piece - 2 : 0; q < piece; ++q)
                wait_bar(&bs.q_full[q & 1], (uint32_t)((q >> 1) & 1), &never);
        }
        return;
    }

    // ================================================================== MMA
    // One thread issues both streams -- QK of tile iq (chunk by chunk, as
    // each K chunk lands) and PV of tile ip -- whichever has its inputs ready
    // (non-blocking tests), PV first because it releases ring chunks.  PV
    // multiplies V^T by [P_hi^T | P_lo^T] (N = 2*NP) in one instruction per
    // 16 positions; the two halves of the accumulator are summed at the end.
    if (warp == 1) {
        if (lane == 0) {
            TileIter itq, itp;
            itq.init(lens, p.B, p.Lmax, kT, segs_per_b, st);
            itp.init(lens, p.B, p.Lmax, kT, segs_per_b, st);
            long long iq = 0, ip = 0;
            int qc = 0;  // next K chunk of tile iq
            int piece_q = 0, piece_pv = 0, qcur = 0;
            uint32_t idle = 0;
            bool ok = true;
            while (ip < ntiles) {
                bool did = false;
                if (ip < iq) {
                    const long long j = ip;
                    const int pb = (int)(j & 1);
                    const bool first_pv = (j == 0) || (itp.t == 0);
                    bool ready = mbar_test(&bs.p_full[pb], (uint32_t)((j >> 1) & 1));
                    if (ready && first_pv && piece_pv > 0)
                        ready = mbar_test(bs.o_free, (uint32_t)((piece_pv - 1) & 1));
#pragma unroll
                    for (int db = 0; db < KCH; ++db) {
                        const long long idx = v_chunk<KCH>(j, db, ntiles);
                        if (ready)
                            ready = mbar_test(&bs.chunk_full[idx % NCH], (uint32_t)((idx / NCH) & 1));
                    }
                    if (ready) {
                        if (first_pv) ++piece_pv;
                        tc_fence_after();
                        const uint32_t pstage = pbuf_s + 2 * (int)(j % C::PST) * C::PB;
#pragma unroll
                        for (int db = 0; db < KCH; ++db) {
                            const long long idx = v_chunk<KCH>(j, db, ntiles);
                            const int slot = (int)(idx % NCH);
                            const uint32_t v0 = ring_s + slot * kChunk;
                            const uint32_t d_o = tmem + 2 * NP + db * 2 * NP;
#pragma unroll
                            for (int kk = 0; kk < 8; ++kk) {
                                // V^T: M = head dims (64-column boxes 16 KB apart), K = positions
                                const uint64_t ad = smem_desc(v0 + kk * 2048, 16384, 1024, 2);
                                // [P_hi^T | P_lo^T]: core matrices of 8 positions x 8 heads,
                                // 128 B each; position groups 128 B apart, head groups 2 KB
                                const uint64_t bd =
                                    smem_desc(pstage + kk * 256, 128, (kT / 8) * 128, 0);
                                umma_bf16(d_o, ad, bd, C::IDESC_PV, !(first_pv && kk == 0));
                            }
                            umma_commit(&bs.chunk_empty[slot]);
                        }
                        umma_commit(&bs.pv_done[pb]);
                        if (j < ntiles - 1) itp.next();
                        ++ip;
                        did = true;
                    }
                }
                if (iq < ntiles) {
                    const long long i = iq;
                    const int sb = (int)(i & 1);
                    const bool first_q = (i == 0) || (itq.t == 0);
                    bool ready = true;
                    if (qc == 0) {
                        if (first_q)
                            ready = mbar_test(&bs.q_full[piece_q & 1], (uint32_t)((piece_q >> 1) & 1));
                        if (ready && i >= 2)
                            ready = mbar_test(&bs.s_empty[sb], (uint32_t)(((i >> 1) - 1) & 1));
                    }
                    const long long idx = k_chunk<KCH>(i, qc);
                    const int slot = (int)(idx % NCH);
                    // A parity test is only meaningful once the slot's previous
                    // occupant (chunk idx - NCH) has landed; the QK stream runs
                    // ahead of PV, so that occupant may be a V chunk whose PV has
                    // not been issued yet -- then the slot is simply not ready.
                    if (ready && idx >= NCH) {
                        long long vt;
                        if (chunk_is_v<KCH>(idx - NCH, ntiles, &vt) && vt >= ip) ready = false;
                    }
                    if (ready) ready = mbar_test(&bs.chunk_full[slot], (uint32_t)((idx / NCH) & 1));
                    if (ready) {
                        if (qc == 0 && first_q) {
                            qcur = piece_q & 1;
                            ++piece_q;
                        }
                        tc_fence_after();
                        const uint32_t d_s = tmem + sb * NP;
                        const uint32_t a0 = ring_s + slot * kChunk;
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk) {
                            const int kq = qc * 8 + kk;
                            const uint64_t ad =
                                smem_desc(a0 + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024, 2);
                            const uint64_t bd = smem_desc(
                                qbuf_s + qcur * C::QB + (kq >> 2) * (NP * 128) + (kq & 3) * 32, 16,
                                1024, 2);
                            umma_bf16(d_s, ad, bd, C::IDESC_QK, kq != 0);
                        }
                        umma_commit(&bs.chunk_empty[slot]);
                        if (++qc == KCH) {
                            qc = 0;
                            umma_commit(&bs.s_full[sb]);
                            if (itq.last_tile_of_segment() || i == ntiles - 1)
                                umma_commit(&bs.q_empty[qcur]);
                            if (i < ntiles - 1) itq.next();
                            ++iq;
                        }
                        did = true;
                    }
                }
                if (did) {
                    idle = 0;
                    continue;
                }
                ++idle;
                if ((idle & 255u) == 0 && *abort_flag) {
                    ok = false;
                    break;
                }
                if (idle >= (p.wait_limit ? p.wait_limit : kMmaIdleLimit)) {
                    ok = false;
                    *abort_flag = 1;
                    break;
                }
                if (idle > 16) __nanosleep(64);
            }
            if (!ok) {
                set_error(p.err, DEV_ERR_TIMEOUT);
                *abort_flag = 1;
            }
            // every MMA issued so far has finished before tensor memory is freed
            umma_commit(bs.drain);
            volatile int never = 0;
            wait_bar(bs.drain, 0, &never);
        }
        __syncwarp();
        named_bar_sync(kBarEnd, SGC::THREADS);
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
        return;
    }

    // ============================================================== softmax
    // SG groups of four warps; group sg owns columns [cg0, cg0 + NPH) of the
    // pass for all 128 positions of a tile.  Votes (the running-max refresh,
    // aborts) are taken by every softmax thread, so the groups refresh
    // their maxima in the same tiles; the exchanges stay within a group.
    constexpr int SG = SGC::SG;
    constexpr int NPH = SGC::NPH;
    constexpr int RS = SGC::RS;
    const int sg = SG == 1 ? 0 : (warp - 2) >> 2;
    const int cg0 = sg * NPH;
    const int bar_grp = SG == 1 ? kBarSoftmax : kBarGroup + sg;
    const int q4 = warp & 3;             // TMEM lane quarter this warp may access
    const int row = q4 * 32 + lane;      // tile position / head-dim row in O^T
    const uint32_t lane_base = tmem + ((uint32_t)(q4 * 32) << 16);
    float *redg = red + sg * 4 * RS;     // this group's column totals, RS floats per warp

    TileIter it;
    it.init(lens, p.B, p.Lmax, kT, segs_per_b, st);
    long long i = 0;
    bool first_piece = true;
    bool aborted = false;
    const uint32_t wlim = p.wait_limit ? p.wait_limit : KVATTN_SPIN_LIMIT;
    bool carry_fail = false;  // a failed wait late in a tile is voted on at the next barrier
    float l[NPH];

    while (i < ntiles && !aborted) {
        const int b = it.b;
        const int kvh = it.seg / p.head_groups;
        const int hg = it.seg % p.head_groups;
        const int len = seq_valid_len(it.len, p.Lmax);
        const int t0 = it.t;
        if (row == 0 && q4 == 0 && sg == 0 && t0 == 0 && (it.len < 0 || it.len > p.Lmax))
            set_error(p.err, DEV_ERR_BOUNDS);
        const int h0 = kvh * p.G + hg * p.hpg;
        // columns: (token, head) for T new tokens, heads of one group otherwise;
        // with T tokens a column is valid when its head is one of the pass's
        // hvalid heads (the last pass of a group may hold fewer)
        const int gvalid = MT ? p.heads_per_seg : min(p.heads_per_seg, p.G - hg * p.heads_per_seg);
        const int hvalid = min(p.hpg, p.G - hg * p.hpg);
        const long long i0 = i;
#pragma unroll
        for (int g = 0; g < NPH; ++g) l[g] = 0.f;
        if (row < NPH) mref_s[cg0 + row] = -INFINITY;
        named_bar_sync(bar_grp, 128);

        while (true) {
            const int sb = (int)(i & 1);
            bool fail = carry_fail || !wait_bar(&bs.s_full[sb], (uint32_t)((i >> 1) & 1), abort_flag, wlim);
            tc_fence_after();
            float s[NPH];
            tmem_ld_n<NPH>(lane_base + sb * NP + cg0, s);
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bs.s_empty[sb]);

            // rows of the box before this tile's first new position repeat
            // positions already attended, lie before a local layer's window,
            // or are zeros before row 0
            const int r0 = it.row0();
            int pos = r0 + row;  // the cached position this row holds
            bool valid;
            if (PG && p.block_lg < 7 && it.last_tile_of_segment()) {
                // paged, small blocks: the last block's rows end the tile
                // after hn zero rows (the hole); rows before the hole hold
                // the earlier blocks, hn positions further on
                const int hn = ((((len - 1) >> p.block_lg) + 1) << p.block_lg) - len;
                const int hl = kT - (1 << p.block_lg);
                if (row < hl) pos += hn;
                valid = !(row >= hl && row < hl + hn) && pos >= it.first_pos() && pos < len;
            } else {
                valid = row >= it.first_pos() - r0 && r0 + row < len;
            }
            // paged, one token: the first tile starts at the tile boundary
            // before the local window
            if (PG && !MT) valid = valid && pos >= len - p.qwin;
            bool over = false;
#pragma unroll
            for (int g = 0; g < NPH; g += 4) {
                const float4 m4 = *reinterpret_cast<const float4 *>(mref_s + cg0 + g);
                s[g] = valid ? s[g] * p.scale_log2 : -INFINITY;
                s[g + 1] = valid ? s[g + 1] * p.scale_log2 : -INFINITY;
                s[g + 2] = valid ? s[g + 2] * p.scale_log2 : -INFINITY;
                s[g + 3] = valid ? s[g + 3] * p.scale_log2 : -INFINITY;
                over |= (s[g] > m4.x + kTau) | (s[g + 1] > m4.y + kTau) |
                        (s[g + 2] > m4.z + kTau) | (s[g + 3] > m4.w + kTau);
            }
            if (MT && (r0 + kT - 1 >= len - (p.T - 1) || r0 < len - p.qwin)) {
                // the tile holds new tokens, or rows before the last token's
                // window: token t sees positions [e - qwin, e), e = len - (T-1-t)
                // (a column masked here after voting at most costs an exact max)
                int t = cg0 / p.hpg, gg = cg0 % p.hpg;
#pragma unroll
                for (int g = 0; g < NPH; ++g) {
                    const int e = len - (p.T - 1 - t);
                    if (pos >= e || pos < e - p.qwin) s[g] = -INFINITY;
                    if (++gg == p.hpg) {
                        gg = 0;
                        ++t;
                    }
                }
            }
            if (named_bar_sync_or(kBarSoftmax, 128 * SG, over || fail)) {
                if (named_bar_sync_or(kBarSoftmax, 128 * SG, fail || *abort_flag != 0)) {
                    aborted = true;
                    break;
                }
                // exact tile max per head, then move the running max
                warp_cols_n<NPH>(s, redg + q4 * RS, lane, OpMax());
                named_bar_sync(bar_grp, 128);
                if (row < NPH) {
                    const int g = cg0 + row;
                    const float tmax = fmaxf(fmaxf(redg[row], redg[RS + row]),
                                             fmaxf(redg[2 * RS + row], redg[3 * RS + row]));
                    const float m_old = mref_s[g];
                    const float m_new = fmaxf(m_old, tmax);
                    alpha_s[g] = (m_new == -INFINITY || m_old == m_new) ? 1.f
                                                                         : fast_exp2(m_old - m_new);
                    mref_s[g] = m_new;
                }
                named_bar_sync(bar_grp, 128);
#pragma unroll
                for (int g = 0; g < NPH; ++g) l[g] *= alpha_s[cg0 + g];
                if (i > i0) {
                    // O^T holds this piece's earlier tiles: scale column g by alpha[g]
                    const long long j = i - 1;
                    if (!wait_bar(&bs.pv_done[j & 1], (uint32_t)((j >> 1) & 1), abort_flag, wlim))
                        fail = true;
                    tc_fence_after();
                    if constexpr (SG == 1) {
                        // hi and lo halves side by side: 2 NP columns per block
#pragma unroll
                        for (int db = 0; db < KCH; ++db) {
#pragma unroll
                            for (int c = 0; c < 2 * NP / 16; ++c) {
                                float v[16];
                                const uint32_t a = lane_base + 2 * NP + db * 2 * NP + c * 16;
                                tmem_ld16(a, v);
                                tmem_ld_wait();
#pragma unroll
                                for (int k = 0; k < 16; ++k) v[k] *= alpha_s[(c * 16 + k) % NP];
                                tmem_st16(a, v);
                            }
                        }
                    } else {
#pragma unroll
                    for (int db = 0; db < KCH; ++db) {
#pragma unroll
                        for (int part = 0; part < 2; ++part) {  // the hi half, then the lo half
                            const uint32_t a = lane_base + 2 * NP + db * 2 * NP + part * NP + cg0;
#pragma unroll
                            for (int c = 0; c + 16 <= NPH; c += 16) {
                                float v[16];
                                tmem_ld16(a + c, v);
                                tmem_ld_wait();
#pragma unroll
                                for (int k = 0; k < 16; ++k) v[k] *= alpha_s[cg0 + c + k];
                                tmem_st16(a + c, v);
                            }
                            if constexpr (NPH % 16 == 8) {
                                float v[8];
                                tmem_ld8(a + NPH - 8, v);
                                tmem_ld_wait();
#pragma unroll
                                for (int k = 0; k < 8; ++k) v[k] *= alpha_s[cg0 + NPH - 8 + k];
                                tmem_st8(a + NPH - 8, v);
                            }
                        }
                    }
                    }
                    tmem_st_wait();
                }
            }

            // probabilities as two bf16 parts, p = hi + lo (hi = p rounded to
            // bf16, lo = the remainder rounded to bf16): the P.V products then
            // carry ~16 significant bits of p instead of 8
            uint32_t pk[NPH / 2], pl[NPH / 2];
#pragma unroll
            for (int g4 = 0; g4 < NPH; g4 += 4) {
                const float4 m4 = *reinterpret_cast<const float4 *>(mref_s + cg0 + g4);
                const float mm[4] = {m4.x, m4.y, m4.z, m4.w};
#pragma unroll
                for (int h = 0; h < 4; h += 2) {
                    const int g = g4 + h;
                    const float p0 = (s[g] == -INFINITY) ? 0.f : fast_exp2(s[g] - mm[h]);
                    const float p1 = (s[g + 1] == -INFINITY) ? 0.f : fast_exp2(s[g + 1] - mm[h + 1]);
                    l[g] += p0;
                    l[g + 1] += p1;
                    const __nv_bfloat162 h2 = __floats2bfloat162_rn(p0, p1);
                    const __nv_bfloat162 r2 =
                        __floats2bfloat162_rn(p0 - __low2float(h2), p1 - __high2float(h2));
                    pk[g / 2] = *reinterpret_cast<const uint32_t *>(&h2);
                    pl[g / 2] = *reinterpret_cast<const uint32_t *>(&r2);
                }
            }
            // the P stage written now was last read by PV of tile i - PST
            if (i >= C::PST) {
                const long long jp = i - C::PST;
                if (!wait_bar(&bs.pv_done[jp & 1], (uint32_t)((jp >> 1) & 1), abort_flag, wlim))
                    fail = true;
            }
            // P^T: 8-column groups (core matrices of 8 positions x 8 heads)
            // 2 KB apart; the group's columns start at group cg0 / 8
            uint8_t *pdst = pbuf + 2 * (int)(i % C::PST) * C::PB + (row >> 3) * 128 + (row & 7) * 16 +
                            (cg0 / 8) * (kT / 8) * 128;
#pragma unroll
            for (int c = 0; c < NPH / 8; ++c) {
                *reinterpret_cast<uint4 *>(pdst + c * (kT / 8) * 128) =
                    make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
                *reinterpret_cast<uint4 *>(pdst + C::PB + c * (kT / 8) * 128) =
                    make_uint4(pl[4 * c], pl[4 * c + 1], pl[4 * c + 2], pl[4 * c + 3]);
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bs.p_full[sb]);
            carry_fail = fail;

            ++i;
            if (it.last_tile_of_segment() || i == ntiles) break;
            it.next();
        }
        if (aborted) break;

        // ---- piece end: O^T is complete once the last PV has finished
        const long long e = i - 1;
        bool fail = carry_fail || !wait_bar(&bs.pv_done[e & 1], (uint32_t)((e >> 1) & 1), abort_flag, wlim);
        carry_fail = false;
        tc_fence_after();
        warp_cols_n<NPH>(l, redg + q4 * RS, lane, OpSum());
        named_bar_sync(bar_grp, 128);
        if (row < NPH)
            ltot_s[cg0 + row] = redg[row] + redg[RS + row] + redg[2 * RS + row] + redg[3 * RS + row];
        named_bar_sync(bar_grp, 128);
        const bool complete = (t0 == 0) && it.last_tile_of_segment();
        const size_t slot = 2 * (size_t)blockIdx.x + (first_piece ? 0 : 1);
        if (SG == 2 && !complete) {
            // partial pieces of two groups: 8 columns read and stored at a time
#pragma unroll
            for (int db = 0; db < KCH; ++db) {
                const uint32_t ob = lane_base + 2 * NP + db * 2 * NP + cg0;
                float *dst = p.ws_o + (slot * p.heads_per_seg + cg0) * D + db * 128 + row;
#pragma unroll
                for (int c = 0; c < NPH; c += 8) {
                    float v[8], w[8];
                    tmem_ld8(ob + c, v);
                    tmem_ld8(ob + NP + c, w);
                    tmem_ld_wait();
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        if (cg0 + c + k < gvalid) dst[(c + k) * D] = v[k] + w[k];
                }
            }
        } else
#pragma unroll
        for (int db = 0; db < KCH; ++db) {
            float o[NPH];
            const uint32_t ob = lane_base + 2 * NP + db * 2 * NP + cg0;
#pragma unroll
            for (int c = 0; c + 16 <= NPH; c += 16) {
                float v[16], w[16];
                tmem_ld16(ob + c, v);       // V.P_hi
                tmem_ld16(ob + NP + c, w);  // V.P_lo
                tmem_ld_wait();
#pragma unroll
                for (int k = 0; k < 16; ++k) o[c + k] = v[k] + w[k];
            }
            if constexpr (NPH % 16 == 8) {
                float v[8], w[8];
                tmem_ld8(ob + NPH - 8, v);
                tmem_ld8(ob + NP + NPH - 8, w);
                tmem_ld_wait();
#pragma unroll
                for (int k = 0; k < 8; ++k) o[NPH - 8 + k] = v[k] + w[k];
            }
            const int d = db * 128 + row;
            if (complete && MT) {
                // column (t, gg) -> out row (b*T + t)*Hq + h0 + gg
                int t = cg0 / p.hpg, gg = cg0 % p.hpg;
#pragma unroll
                for (int k = 0; k < NPH; ++k) {
                    const int g = cg0 + k;
                    if (g < gvalid && gg < hvalid) {
                        const float lt = ltot_s[g];
                        p.out[(((size_t)b * p.T + t) * p.Hq + h0 + gg) * D + d] =
                            (lt > 0.f) ? o[k] / lt : 0.f;
                    }
                    if (++gg == p.hpg) {
                        gg = 0;
                        ++t;
                    }
                }
            } else if (complete) {
#pragma unroll
                for (int k = 0; k < NPH; ++k) {
                    const int g = cg0 + k;
                    if (g < gvalid) {
                        const float lt = ltot_s[g];
                        p.out[((size_t)b * p.Hq + h0 + g) * D + d] = (lt > 0.f) ? o[k] / lt : 0.f;
                    }
                }
            } else if constexpr (SG == 1) {
#pragma unroll
                for (int k = 0; k < NPH; ++k) {
                    const int g = cg0 + k;
                    if (g < gvalid) p.ws_o[(slot * p.heads_per_seg + g) * D + d] = o[k];
                }
            } else {
                // one base address, the columns' rows D floats apart
                float *dst = p.ws_o + (slot * p.heads_per_seg + cg0) * D + d;
#pragma unroll
                for (int k = 0; k < NPH; ++k)
                    if (cg0 + k < gvalid) dst[k * D] = o[k];
            }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bs.o_free);
        if (!complete && (SG == 1 ? row < gvalid : (row < NPH && cg0 + row < gvalid))) {
            const int g = cg0 + row;
            p.ws_ml[(slot * p.heads_per_seg + g) * 2 + 0] = mref_s[g];
            p.ws_ml[(slot * p.heads_per_seg + g) * 2 + 1] = ltot_s[g];
        }
        first_piece = false;
        if (named_bar_sync_or(kBarSoftmax, 128 * SG, fail)) {
            *abort_flag = 1;
            aborted = true;
            break;
        }
        if (i < ntiles) it.next();
    }
    if (aborted) set_error(p.err, DEV_ERR_TIMEOUT);
    tc_fence_before();
    named_bar_sync(kBarEnd, SGC::THREADS);
}

template <int D, int NP, bool MT, bool PG>
cudaError_t launch_t(const CUtensorMap &tmk, const CUtensorMap &tmv, const CUtensorMap &tmq,
                     const DecodeParams &p, int num_ctas, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(num_ctas);
    cfg.blockDim = dim3(TcGroups<D, NP, MT>::THREADS);
    cfg.dynamicSmemBytes = TcCfg<D, NP>::alloc;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, decode_tc_kernel<D, NP, MT, PG>, tmk, tmv, tmq, p);
}

template <int D, int NP, bool MT, bool PG>
cudaError_t prepare_t() {
    static int done_for_device[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64 && done_for_device[dev]) return cudaSuccess;
    e = cudaFuncSetAttribute(decode_tc_kernel<D, NP, MT, PG>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             TcCfg<D, NP>::alloc);
    if (e == cudaSuccess && dev >= 0 && dev < 64) done_for_device[dev] = 1;
    return e;
}

}  // namespace

#define KVATTN_TC_DISPATCH(FN, ...)                       \
    switch (D * 1000 + np) {                              \
        case 128 * 1000 + 16: return FN<128, 16>(__VA_ARGS__); \
        case 128 * 1000 + 32: return FN<128, 32>(__VA_ARGS__); \
        case 128 * 1000 + 48: return FN<128, 48>(__VA_ARGS__); \
        case 128 * 1000 + 64: return FN<128, 64>(__VA_ARGS__); \
        case 256 * 1000 + 16: return FN<256, 16>(__VA_ARGS__); \
        case 256 * 1000 + 32: return FN<256, 32>(__VA_ARGS__); \
        case 256 * 1000 + 48: return FN<256, 48>(__VA_ARGS__); \
        case 256 * 1000 + 64: return FN<256, 64>(__VA_ARGS__); \
        default: break;                                   \
    }
// the same, choosing the one-token or the several-token kernel (mt) for a
// contiguous or a paged cache (pg, a constant)
#define KVATTN_TC_CASE_MT(FN, d, n, mt, pg, ...) \
    case d * 1000 + n: return mt ? FN<d, n, true, pg>(__VA_ARGS__) : FN<d, n, false, pg>(__VA_ARGS__);
// the same without the one-token 16-column kernels (contiguous cache: they
// live in decode_tc16.cu, a translation unit of their own)
#define KVATTN_TC_DISPATCH_MT_NOT16(FN, mt, pg, ...)                  \
    switch (D * 1000 + np) {                                         \
        case 128 * 1000 + 16:                                        \
            if (mt) return FN<128, 16, true, pg>(__VA_ARGS__);       \
            break;                                                   \
        KVATTN_TC_CASE_MT(FN, 128, 32, mt, pg, __VA_ARGS__)          \
        KVATTN_TC_CASE_MT(FN, 128, 48, mt, pg, __VA_ARGS__)          \
        KVATTN_TC_CASE_MT(FN, 128, 64, mt, pg, __VA_ARGS__)          \
        case 256 * 1000 + 16:                                        \
            if (mt) return FN<256, 16, true, pg>(__VA_ARGS__);       \
            break;                                                   \
        KVATTN_TC_CASE_MT(FN, 256, 32, mt, pg, __VA_ARGS__)          \
        KVATTN_TC_CASE_MT(FN, 256, 48, mt, pg, __VA_ARGS__)          \
        case 256 * 1000 + 64:                                        \
            if (mt) return FN<256, 64, true, pg>(__VA_ARGS__);       \
            break;                                                   \
        default: break;                                              \
    }
#define KVATTN_TC_DISPATCH_MT(FN, mt, pg, ...)                        \
    switch (D * 1000 + np) {                                         \
        KVATTN_TC_CASE_MT(FN, 128, 16, mt, pg, __VA_ARGS__)          \
        KVATTN_TC_CASE_MT(FN, 128, 32, mt, pg, __VA_ARGS__)          \
        KVATTN_TC_CASE_MT(FN, 128, 48, mt, pg, __VA_ARGS__)          \
        KVATTN_TC_CASE_MT(FN, 128, 64, mt, pg, __VA_ARGS__)          \
        KVATTN_TC_CASE_MT(FN, 256, 16, mt, pg, __VA_ARGS__)          \
        KVATTN_TC_CASE_MT(FN, 256, 32, mt, pg, __VA_ARGS__)          \
        KVATTN_TC_CASE_MT(FN, 256, 48, mt, pg, __VA_ARGS__)          \
        case 256 * 1000 + 64:                                        \
            if (mt) return FN<256, 64, true, pg>(__VA_ARGS__);       \
            break;                                                   \
        default: break;                                              \
    }

}  // namespace kvattn
