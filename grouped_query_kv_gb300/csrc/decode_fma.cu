// decode_fma.cu -- split-KV decode attention on the CUDA cores (FMA): the
// path for D = 64, and a general path for any (D, G) that tests force.
//
// One persistent CTA per SM: warp 4 streams K/V tiles of `T` cached
// positions from HBM into a ring of shared-memory stages with TMA
// (cp.async.bulk.tensor, 128-byte swizzle, one tile = D/64 boxes of
// 64 elements x T rows for K and the same for V); warps 0-3 consume them.
// Each K/V tile is read from HBM once and used by every query head of the
// segment: in grouped-query attention several query heads share one K/V
// head ("The Basics of Transformer Inference", item "Grouped multi-query
// attention").
//
// Per tile, in the consumers:
//   1. scores  s[g][j] = (scale*log2e*q_g) . k_j     one thread per position
//   2. running max per head over the tile (warp shuffles + shared memory)
//   3. p[g][j] = 2^(s - m), running sum l, rescale factor alpha = 2^(m_old - m_new)
//   4. o[g][:] = alpha*o[g][:] + sum_j p[g][j] v_j    lanes split the head dim
// At the end of a segment piece the four warps' o are summed; a complete
// segment writes out = o / l, a piece of a longer segment writes (m, l, o)
// to the workspace for the combine kernel.
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"
#include "schedule.cuh"

namespace kvattn {

namespace {

constexpr int kConsumers = 128;
constexpr int kThreads = kConsumers + 32;
constexpr int kBarConsumers = 1;  // named barrier id for the 128 consumers

template <int D>
struct FmaCfg {
    static constexpr int TPP = (D == 256) ? 2 : 1;      // threads per position in phase 1
    static constexpr int T = kConsumers / TPP;          // positions per tile
    static constexpr int NSLAB = D / 64;                // 128-byte TMA boxes per row
    static constexpr int TILE_BYTES = T * D * 2;        // one of K or V
    static constexpr int STAGES = (D == 64) ? 6 : 3;    // 192 KB of stages in flight
    static constexpr int DL = D / 32;                   // value columns per lane, phase 4
    static constexpr int CHUNKS = D / 8 / TPP;          // 16-byte key chunks per thread
};

template <int D, int GC>
struct FmaSmem {
    using C = FmaCfg<D>;
    static constexpr int stage_bytes = 2 * C::TILE_BYTES;
    static constexpr int off_q = C::STAGES * stage_bytes;
    static constexpr int off_p = off_q + GC * D * 4;
    static constexpr int off_o = off_p + C::T * GC * 4;
    static constexpr int off_redm = off_o + GC * D * 4;
    static constexpr int off_redl = off_redm + 4 * GC * 4;
    static constexpr int off_bar = (off_redl + 4 * GC * 4 + 7) & ~7;
    static constexpr int bytes = off_bar + 2 * C::STAGES * 8;
    static constexpr int alloc = bytes + 1024;  // slack to align the base to 1024 B
};

__device__ __forceinline__ void bf16x2_to_f32(uint32_t w, float &lo, float &hi) {
    lo = __uint_as_float(w << 16);
    hi = __uint_as_float(w & 0xffff0000u);
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

__device__ __forceinline__ void set_error(unsigned int *err, unsigned int code) {
    atomicCAS(err, 0u, code);
}

template <int D, int GC>
__global__ void __launch_bounds__(kThreads, 1)
    decode_fma_kernel(const __grid_constant__ CUtensorMap tmk,
                      const __grid_constant__ CUtensorMap tmv, const DecodeParams p) {
    using C = FmaCfg<D>;
    using S = FmaSmem<D, GC>;
    constexpr int T = C::T;

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float *q_s = reinterpret_cast<float *>(smem + S::off_q);
    float *p_s = reinterpret_cast<float *>(smem + S::off_p);
    float *o_red = reinterpret_cast<float *>(smem + S::off_o);
    float *red_m = reinterpret_cast<float *>(smem + S::off_redm);
    float *red_l = reinterpret_cast<float *>(smem + S::off_redl);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + S::off_bar);
    uint64_t *empty = full + C::STAGES;

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int segs_per_b = p.Hkv * p.head_groups;

    if (tid == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 4);
        }
        fence_barrier_init();
    }
    if (warp == 4 && lane == 0) {
        prefetch_tmap(&tmk);
        prefetch_tmap(&tmv);
    }
    pdl_wait_prior();  // the caches, q and lengths may come from the previous kernel
    const LenView lens{p.seq_lens, p.len_add, p.window, 0};  // contiguous: no window alignment
    const SchedCost wcost{p.cost_piece};
    const SchedStart st = warp_locate(lens, p.B, p.Lmax, T, segs_per_b, wcost, blockIdx.x, gridDim.x);
    if (warp == 0) sched_split_record(lens, p.B, p.Lmax, T, segs_per_b, wcost, blockIdx.x, st, p.split);
    if (!st.found || st.g_begin >= st.g_end) {
        pdl_launch_dependents();
        return;
    }
    const long long ntiles = st.g_end - st.g_begin;

    // ------------------------------------------------------------ producer
    // The whole warp walks the tile list (all lanes copy the fused append's
    // row); lane 0 alone waits on stages and issues the copies.
    if (warp == 4) {
        const uint64_t pol = l2_policy_evict_first();
        TileIter it;
        it.init(lens, p.B, p.Lmax, T, segs_per_b, st);
        for (long long i = 0; i < ntiles; ++i) {
            const int s = (int)(i % C::STAGES);
            bool w = true;
            if (lane == 0 && i >= C::STAGES)
                w = mbar_wait(&empty[s], (uint32_t)((i / C::STAGES - 1) & 1));
            if (!__shfl_sync(0xffffffffu, w, 0)) {
                if (lane == 0) set_error(p.err, DEV_ERR_TIMEOUT);
                break;
            }
            const int kvh = it.seg / p.head_groups;
            const int z = it.b * p.Hkv + kvh;
            const int y = it.first_pos();
            // fused append: this tile holds the new token's row
            if (p.len_add && it.last_tile_of_segment() && it.len >= 1 && it.len <= p.Lmax)
                append_row_warp(p, z, (size_t)z * p.Lmax + (it.len - 1), D, lane);
            if (lane == 0) {
                uint8_t *kdst = smem + s * S::stage_bytes;
                uint8_t *vdst = kdst + C::TILE_BYTES;
                mbar_arrive_expect_tx(&full[s], 2 * C::TILE_BYTES);
#pragma unroll
                for (int sl = 0; sl < C::NSLAB; ++sl) {
                    tma_load_3d(kdst + sl * T * 128, &tmk, &full[s], sl * 64, y, z, pol);
                    tma_load_3d(vdst + sl * T * 128, &tmv, &full[s], sl * 64, y, z, pol);
                }
            }
            it.next();
        }
        // every load is issued: let the combine kernel be scheduled
        pdl_launch_dependents();
        return;
    }

    // ----------------------------------------------------------- consumers
    const int TPP = C::TPP;
    const int jj = tid / TPP;        // position within the tile (phase 1)
    const int half = tid % TPP;
    const int dcol = lane * C::DL;   // first value column of this lane (phase 4)

    TileIter it;
    it.init(lens, p.B, p.Lmax, T, segs_per_b, st);
    long long i = 0;
    bool first_piece = true;
    bool aborted = false;

    float o[GC][C::DL];
    float l_part[GC];
    float m_run[GC];

    while (i < ntiles && !aborted) {
        // ---- piece start: a run of tiles of one segment
        const int b = it.b;
        const int kvh = it.seg / p.head_groups;
        const int hg = it.seg % p.head_groups;
        const int len = seq_valid_len(it.len, p.Lmax);
        const int t0 = it.t;
        if (tid == 0 && t0 == 0 && (it.len < 0 || it.len > p.Lmax)) set_error(p.err, DEV_ERR_BOUNDS);
        const int h0 = kvh * p.G + hg * p.heads_per_seg;
        const int gvalid = min(GC, p.G - hg * p.heads_per_seg);
        for (int x = tid; x < GC * D; x += kConsumers) {
            const int g = x / D, d = x % D;
            float v = 0.f;
            if (g < gvalid) {
                const uint16_t raw = p.q[((size_t)b * p.Hq + h0 + g) * D + d];
                v = __uint_as_float((uint32_t)raw << 16) * p.scale_log2;
            }
            q_s[x] = v;
        }
#pragma unroll
        for (int g = 0; g < GC; ++g) {
            m_run[g] = -INFINITY;
            l_part[g] = 0.f;
#pragma unroll
            for (int k = 0; k < C::DL; ++k) o[g][k] = 0.f;
        }
        named_bar_sync(kBarConsumers, kConsumers);

        while (true) {
            const int s = (int)(i % C::STAGES);
            const uint32_t par = (uint32_t)((i / C::STAGES) & 1);
            // a thread whose bounded wait gave up still runs this tile on
            // whatever the stage holds (reads stay inside shared memory);
            // the vote at the next barrier then stops every consumer together
            const bool timed_out = !mbar_wait(&full[s], par);
            const uint8_t *kt = smem + s * S::stage_bytes;
            const uint8_t *vt = kt + C::TILE_BYTES;
            const int pos0 = it.first_pos();
            const int nvalid = max(0, min(T, len - pos0));

            // ---- 1. scores, one position per TPP threads
            float acc[GC];
#pragma unroll
            for (int g = 0; g < GC; ++g) acc[g] = 0.f;
#pragma unroll 4
            for (int c = 0; c < C::CHUNKS; ++c) {
                // the two halves of a D=256 row start 4 chunks apart so that
                // they never hit the same bank in one 8-lane phase
                const int lc = (c + half * 4) % C::CHUNKS;
                const int d0 = half * (D / TPP) + lc * 8;
                const int slab = d0 >> 6, ch = (d0 & 63) >> 3;
                const uint4 raw = *reinterpret_cast<const uint4 *>(
                    kt + slab * T * 128 + jj * 128 + ((ch ^ (jj & 7)) << 4));
                float kf[8];
                bf16x2_to_f32(raw.x, kf[0], kf[1]);
                bf16x2_to_f32(raw.y, kf[2], kf[3]);
                bf16x2_to_f32(raw.z, kf[4], kf[5]);
                bf16x2_to_f32(raw.w, kf[6], kf[7]);
#pragma unroll
                for (int g = 0; g < GC; ++g) {
                    const float4 qa = *reinterpret_cast<const float4 *>(q_s + g * D + d0);
                    const float4 qb = *reinterpret_cast<const float4 *>(q_s + g * D + d0 + 4);
                    float a = acc[g];
                    a = fmaf(qa.x, kf[0], a);
                    a = fmaf(qa.y, kf[1], a);
                    a = fmaf(qa.z, kf[2], a);
                    a = fmaf(qa.w, kf[3], a);
                    a = fmaf(qb.x, kf[4], a);
                    a = fmaf(qb.y, kf[5], a);
                    a = fmaf(qb.z, kf[6], a);
                    a = fmaf(qb.w, kf[7], a);
                    acc[g] = a;
                }
            }
            if (TPP == 2) {
#pragma unroll
                for (int g = 0; g < GC; ++g) acc[g] += __shfl_xor_sync(0xffffffffu, acc[g], 1);
            }
            const bool valid = jj < nvalid;

            // ---- 2. tile max per head
#pragma unroll
            for (int g = 0; g < GC; ++g) {
                const float mx = warp_max(valid ? acc[g] : -INFINITY);
                if (lane == 0) red_m[warp * GC + g] = mx;
            }
            if (named_bar_sync_or(kBarConsumers, kConsumers, timed_out)) {
                if (tid == 0) set_error(p.err, DEV_ERR_TIMEOUT);
                aborted = true;
                break;
            }

            // ---- 3. probabilities, running sum, rescale factor
            float alpha[GC];
#pragma unroll
            for (int g = 0; g < GC; ++g) {
                const float mt = fmaxf(fmaxf(red_m[g], red_m[GC + g]),
                                       fmaxf(red_m[2 * GC + g], red_m[3 * GC + g]));
                const float m_new = fmaxf(m_run[g], mt);
                // all positions so far masked: keep everything at zero
                alpha[g] = (m_new == -INFINITY) ? 1.f : fast_exp2(m_run[g] - m_new);
                const float pr = (valid && m_new != -INFINITY) ? fast_exp2(acc[g] - m_new) : 0.f;
                if (half == 0) {
                    l_part[g] = l_part[g] * alpha[g] + pr;
                    p_s[jj * GC + g] = pr;
                }
                m_run[g] = m_new;
            }
            named_bar_sync(kBarConsumers, kConsumers);

            // ---- 4. o = alpha * o + P V ; warp w takes positions w, w+4, ...
#pragma unroll
            for (int g = 0; g < GC; ++g)
#pragma unroll
                for (int k = 0; k < C::DL; ++k) o[g][k] *= alpha[g];
            {
                const int slab = dcol >> 6, ch = (dcol & 63) >> 3, sub = (dcol & 7) * 2;
                for (int j = warp; j < nvalid; j += 4) {
                    const uint8_t *row = vt + slab * T * 128 + j * 128 + ((ch ^ (j & 7)) << 4) + sub;
                    float vf[C::DL];
                    if constexpr (C::DL == 8) {
                        const uint4 r = *reinterpret_cast<const uint4 *>(row);
                        bf16x2_to_f32(r.x, vf[0], vf[1]);
                        bf16x2_to_f32(r.y, vf[2], vf[3]);
                        bf16x2_to_f32(r.z, vf[4], vf[5]);
                        bf16x2_to_f32(r.w, vf[6], vf[7]);
                    } else if constexpr (C::DL == 4) {
                        const uint2 r = *reinterpret_cast<const uint2 *>(row);
                        bf16x2_to_f32(r.x, vf[0], vf[1]);
                        bf16x2_to_f32(r.y, vf[2], vf[3]);
                    } else {
                        const uint32_t r = *reinterpret_cast<const uint32_t *>(row);
                        bf16x2_to_f32(r, vf[0], vf[1]);
                    }
                    float pj[GC];
#pragma unroll
                    for (int g = 0; g < GC; ++g) pj[g] = p_s[j * GC + g];
#pragma unroll
                    for (int g = 0; g < GC; ++g)
#pragma unroll
                        for (int k = 0; k < C::DL; ++k) o[g][k] = fmaf(pj[g], vf[k], o[g][k]);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);

            ++i;
            if (it.last_tile_of_segment() || i == ntiles) break;
            it.next();
        }
        if (aborted) break;

        // ---- piece end: reduce l and o over the four warps
        const bool complete = (t0 == 0) && it.last_tile_of_segment();
#pragma unroll
        for (int g = 0; g < GC; ++g) {
            const float ls = warp_sumf(l_part[g]);
            if (lane == 0) red_l[warp * GC + g] = ls;
        }
        // fixed summation order (warp 0, then 1, 2, 3): bitwise reproducible
#pragma unroll 1
        for (int w = 0; w < 4; ++w) {
            if (warp == w) {
#pragma unroll
                for (int g = 0; g < GC; ++g)
#pragma unroll
                    for (int k = 0; k < C::DL; ++k) {
                        float *dst = &o_red[g * D + dcol + k];
                        *dst = (w == 0) ? o[g][k] : *dst + o[g][k];
                    }
            }
            named_bar_sync(kBarConsumers, kConsumers);
        }
        if (complete) {
            for (int x = tid; x < gvalid * D; x += kConsumers) {
                const int g = x / D, d = x % D;
                const float l = red_l[g] + red_l[GC + g] + red_l[2 * GC + g] + red_l[3 * GC + g];
                p.out[((size_t)b * p.Hq + h0 + g) * D + d] = (l > 0.f) ? o_red[x] / l : 0.f;
            }
        } else {
            const size_t slot = 2 * (size_t)blockIdx.x + (first_piece ? 0 : 1);
            for (int x = tid; x < gvalid * D; x += kConsumers)
                p.ws_o[slot * p.heads_per_seg * D + x] = o_red[x];
            if (tid < gvalid) {
                const int g = tid;
                const float l = red_l[g] + red_l[GC + g] + red_l[2 * GC + g] + red_l[3 * GC + g];
                p.ws_ml[(slot * p.heads_per_seg + g) * 2 + 0] = m_run[g];
                p.ws_ml[(slot * p.heads_per_seg + g) * 2 + 1] = l;
            }
        }
        first_piece = false;
        named_bar_sync(kBarConsumers, kConsumers);  // o_red, red_l, q_s free again
        if (i < ntiles) it.next();
    }
}

template <int D, int GC>
cudaError_t launch_t(const CUtensorMap &tmk, const CUtensorMap &tmv, const DecodeParams &p,
                     int num_ctas, int smem_bytes, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(num_ctas);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem_bytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, decode_fma_kernel<D, GC>, tmk, tmv, p);
}

// Raises the kernel's dynamic shared-memory limit once per process and
// device (never again later, e.g. inside a stream capture).
template <int D, int GC>
cudaError_t prepare_t(int smem_bytes) {
    static int done_for_device[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64 && done_for_device[dev] >= smem_bytes) return cudaSuccess;
    e = cudaFuncSetAttribute(decode_fma_kernel<D, GC>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
    if (e == cudaSuccess && dev >= 0 && dev < 64) done_for_device[dev] = smem_bytes;
    return e;
}

template <int D>
int smem_for(int gc) {
    switch (gc) {
        case 1: return FmaSmem<D, 1>::alloc;
        case 2: return FmaSmem<D, 2>::alloc;
        case 4: return FmaSmem<D, 4>::alloc;
        default: return FmaSmem<D, 8>::alloc;
    }
}

}  // namespace

int fma_heads_per_seg(int G) { return G <= 1 ? 1 : G <= 2 ? 2 : G <= 4 ? 4 : 8; }
int fma_threads() { return kThreads; }
int fma_tile(int D) { return D == 256 ? FmaCfg<256>::T : D == 128 ? FmaCfg<128>::T : FmaCfg<64>::T; }
int fma_stages(int D) {
    return D == 256 ? FmaCfg<256>::STAGES : D == 128 ? FmaCfg<128>::STAGES : FmaCfg<64>::STAGES;
}
int fma_smem_bytes(int D, int gc) {
    return D == 256 ? smem_for<256>(gc) : D == 128 ? smem_for<128>(gc) : smem_for<64>(gc);
}

#define KVATTN_FMA_DISPATCH(FN, ...)                                  \
    switch (D * 16 + gc) {                                            \
        case 64 * 16 + 1: return FN<64, 1>(__VA_ARGS__);              \
        case 64 * 16 + 2: return FN<64, 2>(__VA_ARGS__);              \
        case 64 * 16 + 4: return FN<64, 4>(__VA_ARGS__);              \
        case 64 * 16 + 8: return FN<64, 8>(__VA_ARGS__);              \
        case 128 * 16 + 1: return FN<128, 1>(__VA_ARGS__);            \
        case 128 * 16 + 2: return FN<128, 2>(__VA_ARGS__);            \
        case 128 * 16 + 4: return FN<128, 4>(__VA_ARGS__);            \
        case 128 * 16 + 8: return FN<128, 8>(__VA_ARGS__);            \
        case 256 * 16 + 1: return FN<256, 1>(__VA_ARGS__);            \
        case 256 * 16 + 2: return FN<256, 2>(__VA_ARGS__);            \
        case 256 * 16 + 4: return FN<256, 4>(__VA_ARGS__);            \
        case 256 * 16 + 8: return FN<256, 8>(__VA_ARGS__);            \
        default: return cudaErrorInvalidValue;                        \
    }

cudaError_t fma_prepare(int D, int gc, int smem_bytes) {
    KVATTN_FMA_DISPATCH(prepare_t, smem_bytes)
}

cudaError_t launch_decode_fma(const CUtensorMap &tmk, const CUtensorMap &tmv,
                              const DecodeParams &p, int num_ctas, int smem_bytes,
                              cudaStream_t stream) {
    const int D = p.D, gc = p.heads_per_seg;
    KVATTN_FMA_DISPATCH(launch_t, tmk, tmv, p, num_ctas, smem_bytes, stream)
}

}  // namespace kvattn
