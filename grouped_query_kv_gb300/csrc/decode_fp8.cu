// decode_fp8.cu -- split-KV decode attention over an 8-bit KV cache: FP8
// E4M3 codes with one fp32 scale per cached row ("The Basics of Transformer
// Inference", item "Quantization": an int8 / fp8 KV cache saves memory
// bandwidth; "Machine Learning Engineering and AI Systems at Scale", section
// "Quantization": E4M3 is the inference format).  Row j of a (b, kvh) block
// stands for K[j, :] = e4m3(code[j, :]) * k_scale[j] (V likewise), so the
// cache read per position is D + 4 bytes for K and as much for V instead of
// 2 D.
//
// The same tiles, schedule, softmax and combine as the bf16 tensor-core
// kernel (decode_tc.cuh).  Both products run on the 8-bit tensor-core path
// (kind::f8f6f4, fp32 accumulation) straight from the staged codes: warp 0
// brings each 128-position tile of K codes and of V codes (16 KB at
// D = 128) into its staging ring with one TMA box, and the MMAs read them
// there -- no widening pass.  A tcgen05 MMA of M = 128 costs the tensor pipe
// about the same time at any N up to 256, so what paces a decode tile is the
// number of MMAs, not their width; this layout takes 8 per tile (4 for
// Q K^T, 4 for P V) where 16-bit operands take 16.
//
//   * Q K^T.  The piece's q rows go in as two E4M3 parts under a per-head
//     power-of-two scale 2^c (c puts the head's largest |q| in [128, 256)):
//     hi = e4m3(q 2^c), lo = e4m3(q 2^c - hi).  A bf16 value has 8
//     significant bits and E4M3 4, and the remainder after rounding to 4
//     bits is a multiple of the bf16 ulp no larger than 8 of them, so
//     hi + lo is q 2^c exactly for entries within 2^9 of the head's
//     largest (smaller ones are off by at most 2^-17 of it: the remainder
//     falls below E4M3's smallest step).  The two parts sit side by side
//     as the 2 NP columns of one B operand (at most 128, and 480 of the 512
//     tensor-memory columns with the O accumulators at NP = 48, D = 256),
//     so Q K^T takes 4 D / 128 MMAs per tile, and the softmax adds the two
//     partial scores 16 columns at a time.  (Running the lo part as 4 more
//     MMAs into the same accumulator, as passes of more than 32 heads once
//     did, took the PaLM-540B-shaped step from 58.0 to 59.4 us.)
//     The last two warps write the parts; the softmax scales the score by
//     2^-c k_scale[j].
//   * P V.  The weight of position j for head g is w = p v_scale[j]
//     (p = 2^(s - m) the unnormalised probability).  Scaled by a
//     power of two 2^cv that the CTA keeps per piece (the largest v_scale
//     met so far times 2^cv in [32, 64)) and with p <= 4 between rescales
//     (the running max is refreshed once a score passes it by 2), w 2^cv
//     stays <= 256, inside E4M3's range.  It is rounded to binary16 (11
//     significant bits, as the f16 P of a widening design) and goes in as
//     three E4M3 parts hi + mid + lo (each the rounded remainder of the
//     previous, taken in binary16, where the remainders are exact), which
//     carry its 11 bits whole (4 + 4 + 3; a remainder below E4M3's
//     smallest step, 2^-9, is lost as before).  The
//     parts sit side by side as the 3 NP columns of the B operand (P stored
//     position-major, no swizzle), so 4 MMAs per tile accumulate three
//     partial O^T blocks; the epilogue adds them and divides by 2^cv.  A
//     tile whose v_scale would break the bound lowers cv first, rescaling
//     the accumulator by the same power of two (with the running-max
//     rescale, in the same step).
// D = 128 or 256.  A 128-position tile of codes is D / 128 TMA boxes of 128
// positions x 128 codes (the 128-byte swizzle's width), side by side in its
// staging slot; the q parts have one 128-code slab per box; Q K^T runs
// 4 D / 128 K-steps of 32 codes, and P V runs one M = 128 block of MMAs per
// 128 head dims, each into its own O^T accumulator.
#include <cuda_fp16.h>

#include "decode_tc.cuh"
#include "fp8_codec.cuh"

namespace kvattn {

namespace {

constexpr int kBox = 16384;      // one TMA box: 128 positions x 128 codes
// Warps: 0 copies, 1 issues the MMAs, then the softmax in SG groups of four
// (group sg = (warp - 2) / 4 takes NP / SG of the pass's columns, so SG
// softmax warps share each SM sub-partition), then two that write the q
// parts (Q8Cfg: SG, THREADS).
constexpr int kQWarps = 2;
constexpr int kBarQ8All = 1;     // named barrier: all softmax threads
constexpr int kBarQ8Grp = 3;     // named barriers 3, 4, ...: the 128 threads of group 0, 1, ...
constexpr float kTauQ8 = 2.f;    // rescale once a score passes the running max by 2 (log2 units)
constexpr float kVHi = 64.f;     // v_scale[j] 2^cv stays <= 64
constexpr int kCvNone = 1 << 20; // cv not chosen yet (piece start)

template <int D, int NP>
struct Q8Cfg {
    static constexpr int SL = D / 128;        // 128-code slabs per row
    static constexpr int kStage = SL * kBox;  // one staged tile: 128 positions x D codes
    static constexpr int QSL = 2 * NP * 128;  // one slab of a q buffer: NP hi rows, NP lo rows
    static constexpr int QB = SL * QSL;       // one q buffer (E4M3, swizzled, K-major)
    static constexpr int PB = 3 * NP * kT;    // one P stage: 3 NP E4M3 columns x 128 positions
    static constexpr int PST = 2;
    static constexpr int NS_MAX = 12;
    static constexpr int NBAR_MAX = 2 * NS_MAX + 14;
    static constexpr int FIXED = 2 * QB + PST * PB + (NP == 48 ? 3 : 2) * 4 * 64 * 4 +
                                 3 * 64 * 4 + 2 * 64 * 4 + 64 + 64 + 1024 + NBAR_MAX * 8;
    static constexpr int NS_FIT = (kSmemLimit - FIXED) / kStage;
    static constexpr int NS = NS_FIT > NS_MAX ? NS_MAX : NS_FIT;   // staging slots, both rings
    static constexpr int NSK = NS / 2;                             // K staging slots
    static constexpr int NSV = NS - NSK;                           // V staging slots
    static_assert(NSV >= 2 && NSK >= 2, "staging rings must hold two tiles each");
    static_assert(NP % (4 * kQWarps) == 0, "the q warps convert four heads at a time each");
    // softmax groups: three at 48 columns (16 each), else two
    static constexpr int SG = NP == 48 ? 3 : 2;
    static constexpr int NPH = NP / SG;  // columns of one softmax group
    static_assert(NPH % 8 == 0, "a group's columns come in tensor-memory loads of 8");
    static constexpr int SOFTW = 4 * SG;              // softmax warps
    static constexpr int QWARP0 = 2 + SOFTW;          // first q-part warp
    static constexpr int THREADS = 32 * (QWARP0 + kQWarps);
    static constexpr int END_THREADS = 32 * QWARP0;   // warps that meet before TMEM is freed

    static constexpr int off_kst = 0;
    static constexpr int off_vst = off_kst + NSK * kStage;
    static constexpr int off_q = off_vst + NSV * kStage;
    static constexpr int off_p = off_q + 2 * QB;
    static constexpr int off_red = off_p + PST * PB;      // float [groups][4][64]
    static constexpr int off_ltot = off_red + (NP == 48 ? 3 : 2) * 4 * 64 * 4;
    static constexpr int off_mref = off_ltot + 64 * 4;
    static constexpr int off_alpha = off_mref + 64 * 4;
    static constexpr int off_qinv = off_alpha + 64 * 4;   // float [2][64]: 2^-c per head
    static constexpr int off_vred = off_qinv + 2 * 64 * 4;  // float [groups][4]: a tile's largest v_scale
    static constexpr int off_bar = off_vred + 64;
    static constexpr int nbar = 2 * NS + 14;
    static constexpr int off_misc = off_bar + nbar * 8;
    static constexpr int bytes = off_misc + 64;
    static constexpr int alloc = bytes + 1024;
    static_assert(alloc <= kSmemLimit, "shared memory");
    static_assert(off_q % 1024 == 0 && off_p % 1024 == 0 && QB % 1024 == 0, "swizzle atoms");

    // TMEM: S0, S1 (side by side: 2 NP columns each, hi part then lo part),
    // then per 128 head dims an O^T accumulator (3 NP columns: hi, mid, lo
    // parts of P)
    static constexpr bool SBS = true;
    static constexpr int SW = SBS ? 2 * NP : NP;
    static constexpr int OA = 2 * SW;
    static constexpr int TMEM_COLS = pow2_at_least(OA + SL * 3 * NP);
    static constexpr uint32_t IDESC_QK = idesc_e4m3_f32(128, SW, false, false);
    static constexpr uint32_t IDESC_PV = idesc_e4m3_f32(128, 3 * NP, true, true);
};

// Two E4M3 codes (low byte first) -> f16x2 (low half first); exact.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t two) {
    uint32_t r;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(two));
    return r;
}

// Two binary32 values -> two E4M3 codes (nearest, ties to even,
// saturating), a in the low byte.
__device__ __forceinline__ uint16_t e4m3x2_of(float a, float b) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(b), "f"(a));
    return r;
}

// Two binary32 values -> f16x2 (a in the low half), nearest even.
__device__ __forceinline__ uint32_t f16x2_of(float a, float b) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(b), "f"(a));
    return r;
}

// f16x2 -> two E4M3 codes (nearest, ties to even, saturating), the low
// half in the low byte.
__device__ __forceinline__ uint16_t e4m3x2_of_f16x2(uint32_t h) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f16x2 %0, %1;" : "=h"(r) : "r"(h));
    return r;
}

// a - b in f16x2 arithmetic (exact for the remainders it is used on).
__device__ __forceinline__ uint32_t f16x2_sub(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

__device__ __forceinline__ float2 e4m3x2_value(uint16_t two) {
    const uint32_t h = e4m3x2_to_f16x2(two);
    return __half22float2(*reinterpret_cast<const __half2 *>(&h));
}

// 2^e as a binary32 value, e in [-126, 127].
__device__ __forceinline__ float pow2i(int e) { return __uint_as_float((uint32_t)(127 + e) << 23); }

template <int D, int NP>
__global__ void __launch_bounds__(Q8Cfg<D, NP>::THREADS, 1)
    decode_q8_kernel(const __grid_constant__ CUtensorMap tmk,
                     const __grid_constant__ CUtensorMap tmv, const DecodeParams p) {
    using C = Q8Cfg<D, NP>;
    constexpr int SL = C::SL;
    constexpr int kStage = C::kStage;
    constexpr int NSK = C::NSK;
    constexpr int NSV = C::NSV;

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *kst = smem + C::off_kst;
    uint8_t *vst = smem + C::off_vst;
    uint8_t *qbuf = smem + C::off_q;
    uint8_t *pbuf = smem + C::off_p;
    float *red = reinterpret_cast<float *>(smem + C::off_red);
    float *ltot_s = reinterpret_cast<float *>(smem + C::off_ltot);
    float *mref_s = reinterpret_cast<float *>(smem + C::off_mref);
    float *alpha_s = reinterpret_cast<float *>(smem + C::off_alpha);
    float *qinv_s = reinterpret_cast<float *>(smem + C::off_qinv);
    float *vred_s = reinterpret_cast<float *>(smem + C::off_vred);
    uint64_t *bar_base = reinterpret_cast<uint64_t *>(smem + C::off_bar);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::off_misc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::off_misc + 16);

    // kst_*: the K staging ring (TMA -> Q K^T); vst_*: the V staging ring
    // (TMA -> P V); q_full/q_empty: the q parts and 2^-c (written by the q
    // warps, freed by the last Q K^T of the piece and the softmax warps)
    uint64_t *kst_full = bar_base, *kst_empty = kst_full + NSK;
    uint64_t *vst_full = kst_empty + NSK, *vst_empty = vst_full + NSV;
    uint64_t *q_full = vst_empty + NSV, *q_empty = q_full + 2;
    uint64_t *s_full = q_empty + 2, *s_empty = s_full + 2;
    uint64_t *p_full = s_empty + 2, *pv_done = p_full + 2;
    uint64_t *o_free = pv_done + 2, *drain = o_free + 1;

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int segs_per_b = p.Hkv * p.head_groups;

    if (tid == 0) {
        for (int s = 0; s < NSK; ++s) {
            mbar_init(&kst_full[s], 1);
            mbar_init(&kst_empty[s], 1);
        }
        for (int s = 0; s < NSV; ++s) {
            mbar_init(&vst_full[s], 1);
            mbar_init(&vst_empty[s], 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&q_full[s], kQWarps);
            mbar_init(&q_empty[s], 1 + C::SOFTW);  // the MMA commit and the softmax warps
            mbar_init(&s_full[s], 1);
            mbar_init(&s_empty[s], C::SOFTW);
            mbar_init(&p_full[s], C::SOFTW);
            mbar_init(&pv_done[s], 1);
        }
        mbar_init(o_free, C::SOFTW);
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tmk);
        prefetch_tmap(&tmv);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    pdl_wait_prior();
    const LenView lens{p.seq_lens, p.len_add, p.window, 0};  // contiguous: no window alignment
    const SchedCost wcost{p.cost_piece};
    const SchedStart st = warp_locate(lens, p.B, p.Lmax, kT, segs_per_b, wcost, blockIdx.x, gridDim.x);
    if (warp == 2) sched_split_record(lens, p.B, p.Lmax, kT, segs_per_b, wcost, blockIdx.x, st, p.split);
    if (!st.found) {
        if (warp == 1) tmem_dealloc(tmem, C::TMEM_COLS);
        pdl_launch_dependents();
        return;
    }
    const long long ntiles = st.g_end - st.g_begin;
    const uint32_t kst_s = smem_u32(kst);
    const uint32_t vst_s = smem_u32(vst);
    const uint32_t qbuf_s = smem_u32(qbuf);
    const uint32_t pbuf_s = smem_u32(pbuf);

    // ================================================================ producer
    // Issue order K_0, K_1, V_0, K_2, V_1, ... (each ring in its own order).
    // The whole warp walks the tiles (the fused append quantizes a row with
    // all 32 lanes); lane 0 alone waits on staging slots and issues copies.
    if (warp == 0) {
        long long nk = 0, nv = 0;  // K and V stage copies issued
        const uint64_t pol = l2_policy_evict_first();
        TileIter itk, itv;
        itk.init(lens, p.B, p.Lmax, kT, segs_per_b, st);
        itv.init(lens, p.B, p.Lmax, kT, segs_per_b, st);
        bool ok = true;
        auto issue = [&](const void *tm, const TileIter &it, uint8_t *base, uint64_t *full,
                         uint64_t *empty, int ns, long long &n) -> bool {
            const int slot = (int)(n % ns);
            bool w = true;
            if (lane == 0 && n >= ns) w = wait_bar(&empty[slot], (uint32_t)(((n / ns) - 1) & 1), abort_flag);
            if (!__shfl_sync(0xffffffffu, w, 0)) return false;
            if (lane == 0) {
                mbar_arrive_expect_tx(&full[slot], kStage);
                const int z = it.b * p.Hkv + it.seg / p.head_groups;
#pragma unroll
                for (int sl = 0; sl < SL; ++sl)
                    tma_load_3d(base + slot * kStage + sl * kBox, tm, &full[slot], sl * 128,
                                it.row0(), z, pol);
            }
            ++n;
            return true;
        };
        for (long long r = 0; r <= ntiles && ok; ++r) {
            if (r < ntiles) {
                // fused append: this tile holds the new token's row -- its
                // codes and scales are written (and made visible to the
                // copies and to every SM) before the tile's copies go out
                if (p.len_add && itk.last_tile_of_segment() && itk.len >= 1 && itk.len <= p.Lmax) {
                    const int z = itk.b * p.Hkv + itk.seg / p.head_groups;
                    const size_t dst = (size_t)z * p.Lmax + (itk.len - 1);
                    uint8_t *kc = reinterpret_cast<uint8_t *>(p.k_cache);
                    uint8_t *vc = reinterpret_cast<uint8_t *>(p.v_cache);
                    quantize_row_warp<D / 32>(p.k_new + (size_t)z * D, kc + dst * D,
                                              const_cast<float *>(p.k_scale) + dst, lane);
                    quantize_row_warp<D / 32>(p.v_new + (size_t)z * D, vc + dst * D,
                                              const_cast<float *>(p.v_scale) + dst, lane);
                    asm volatile("fence.proxy.async.global;" ::: "memory");
                    __threadfence();
                    __syncwarp();
                }
                ok = issue(&tmk, itk, kst, kst_full, kst_empty, NSK, nk);
                itk.next();
            }
            if (r >= 1 && ok) {
                ok = issue(&tmv, itv, vst, vst_full, vst_empty, NSV, nv);
                itv.next();
            }
        }
        if (!ok && lane == 0) {
            set_error(p.err, DEV_ERR_TIMEOUT);
            *abort_flag = 1;
        }
        __syncwarp();
        pdl_launch_dependents();
        named_bar_sync(kBarEnd, C::END_THREADS);
        if (*abort_flag && lane == 0) {
            // a role gave up, so copies may still be in flight that no one
            // consumed: let them land before the CTA exits
            volatile int never = 0;
            for (long long k = nk > NSK ? nk - NSK : 0; k < nk; ++k)
                wait_bar(&kst_full[k % NSK], (uint32_t)((k / NSK) & 1), &never);
            for (long long k = nv > NSV ? nv - NSV : 0; k < nv; ++k)
                wait_bar(&vst_full[k % NSV], (uint32_t)((k / NSV) & 1), &never);
        }
        return;
    }

    // ======================================================== q parts (6, 7)
    if (warp >= C::QWARP0) {
        const int qw = warp - C::QWARP0;
        TileIter itq;
        itq.init(lens, p.B, p.Lmax, kT, segs_per_b, st);
        int piece = 0;
        bool ok = true;
        // the piece's q rows as E4M3 hi / lo parts, swizzled K-major rows
        // (hi of head g in row g, lo in row NP + g), and 2^-c per head
        for (long long r = 0; r < ntiles && ok; ++r) {
            if (r == 0 || itq.t == 0) {
                const int qs = piece & 1;
                if (piece >= 2) {
                    bool w = true;
                    if (lane == 0) w = wait_bar(&q_empty[qs], (uint32_t)(((piece >> 1) - 1) & 1), abort_flag);
                    ok = __shfl_sync(0xffffffffu, w, 0);
                    if (!ok) break;
                }
                const int kvh = itq.seg / p.head_groups, hg = itq.seg % p.head_groups;
                const int h0 = kvh * p.G + hg * p.heads_per_seg;
                const int gvalid = min(p.heads_per_seg, p.G - hg * p.heads_per_seg);
                uint8_t *qb = qbuf + qs * C::QB;
                // eight lanes per head, each with VPL consecutive head dims;
                // a warp converts four heads at a time and first loads every
                // head it converts, so their reads overlap
                constexpr int VPL = D / 8;              // head dims per lane
                constexpr int NV = VPL / 8;             // 16-byte loads per lane and head
                constexpr int HPW = NP / kQWarps;       // heads per warp
                constexpr int NIT = HPW / 4;            // four heads per pass of the warp
                const int sub = lane & 7, d0 = sub * VPL;
                uint4 raw[NIT][NV];
#pragma unroll
                for (int it4 = 0; it4 < NIT; ++it4) {
                    const int g = (it4 * kQWarps + qw) * 4 + (lane >> 3);
#pragma unroll
                    for (int v = 0; v < NV; ++v) raw[it4][v] = make_uint4(0u, 0u, 0u, 0u);
                    if (g < gvalid) {
                        const uint4 *src = reinterpret_cast<const uint4 *>(
                            p.q + ((size_t)itq.b * p.Hq + h0 + g) * D + d0);
#pragma unroll
                        for (int v = 0; v < NV; ++v) raw[it4][v] = __ldg(src + v);
                    }
                }
#pragma unroll
                for (int it4 = 0; it4 < NIT; ++it4) {
                    const int g = (it4 * kQWarps + qw) * 4 + (lane >> 3);
                    float x[VPL];
#pragma unroll
                    for (int v = 0; v < NV; ++v) {
                        const uint32_t w[4] = {raw[it4][v].x, raw[it4][v].y, raw[it4][v].z,
                                               raw[it4][v].w};
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            x[8 * v + 2 * u] = __uint_as_float(w[u] << 16);
                            x[8 * v + 2 * u + 1] = __uint_as_float(w[u] & 0xFFFF0000u);
                        }
                    }
                    float amax = 0.f;
#pragma unroll
                    for (int k = 0; k < VPL; ++k) amax = fmaxf(amax, fabsf(x[k]));
#pragma unroll
                    for (int o = 4; o > 0; o >>= 1)  // over the head's eight lanes
                        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
                    // c = 7 - floor(log2 amax), kept where 2^c and 2^-c are normal
                    int e = (int)((__float_as_uint(amax) >> 23) & 0xFF) - 127;
                    e = max(-119, min(e, 120));
                    const float sc = pow2i(7 - e);
                    // this lane's 16-code chunks of the head's row: slab d0 / 128,
                    // 16-byte chunk (d0 mod 128) / 16 + j, swizzled by the row
                    uint8_t *qs_b = qb + (d0 >> 7) * C::QSL;
#pragma unroll
                    for (int j = 0; j < VPL / 16; ++j) {
                        uint32_t hw[4], lw[4];
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            const float a0 = x[16 * j + 4 * u] * sc, a1 = x[16 * j + 4 * u + 1] * sc;
                            const float a2 = x[16 * j + 4 * u + 2] * sc, a3 = x[16 * j + 4 * u + 3] * sc;
                            const uint16_t h01 = e4m3x2_of(a0, a1), h23 = e4m3x2_of(a2, a3);
                            const float2 v01 = e4m3x2_value(h01), v23 = e4m3x2_value(h23);
                            const uint16_t l01 = e4m3x2_of(a0 - v01.x, a1 - v01.y);
                            const uint16_t l23 = e4m3x2_of(a2 - v23.x, a3 - v23.y);
                            hw[u] = (uint32_t)h01 | ((uint32_t)h23 << 16);
                            lw[u] = (uint32_t)l01 | ((uint32_t)l23 << 16);
                        }
                        const int chunk = (((d0 & 127) >> 4) + j) ^ (g & 7);
                        *reinterpret_cast<uint4 *>(qs_b + g * 128 + (chunk << 4)) =
                            make_uint4(hw[0], hw[1], hw[2], hw[3]);
                        *reinterpret_cast<uint4 *>(qs_b + (NP + g) * 128 + (chunk << 4)) =
                            make_uint4(lw[0], lw[1], lw[2], lw[3]);
                    }
                    if (sub == 0) qinv_s[qs * 64 + g] = (g < gvalid) ? pow2i(e - 7) : 0.f;
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&q_full[qs]);
                ++piece;
            }
            itq.next();
        }
        if (!ok && lane == 0) {
            set_error(p.err, DEV_ERR_TIMEOUT);
            *abort_flag = 1;
        }
        return;
    }

    // ================================================================== MMA
    if (warp == 1) {
        if (lane == 0) {
            TileIter itq, itp;
            itq.init(lens, p.B, p.Lmax, kT, segs_per_b, st);
            itp.init(lens, p.B, p.Lmax, kT, segs_per_b, st);
            long long iq = 0, ip = 0;
            int piece_q = 0, piece_pv = 0, qcur = 0;
            uint32_t idle = 0;
            bool ok = true;
            while (ip < ntiles) {
                bool did = false;
                if (ip < iq) {  // P V of tile ip: 32 positions per MMA, the 3 P parts side by side
                    const long long j = ip;
                    const int pb = (int)(j & 1);
                    const bool first_pv = (j == 0) || (itp.t == 0);
                    bool ready = mbar_test(&p_full[pb], (uint32_t)((j >> 1) & 1));
                    if (ready && first_pv && piece_pv > 0)
                        ready = mbar_test(o_free, (uint32_t)((piece_pv - 1) & 1));
                    const int slot = (int)(j % NSV);
                    if (ready) ready = mbar_test(&vst_full[slot], (uint32_t)((j / NSV) & 1));
                    if (ready) {
                        if (first_pv) ++piece_pv;
                        tc_fence_after();
                        const uint32_t pstage = pbuf_s + (int)(j % C::PST) * C::PB;
                        const uint32_t v0 = vst_s + slot * kStage;
#pragma unroll
                        for (int sl = 0; sl < SL; ++sl) {  // head dims 128 sl .. 128 sl + 127
#pragma unroll
                            for (int kk = 0; kk < 4; ++kk) {
                                // A = V^T: the staged box read position-major (SW128);
                                // B = P: position-major, no swizzle, 16-column blocks
                                const uint64_t ad = smem_desc(v0 + sl * kBox + kk * 4096, 16384, 1024, 2);
                                const uint64_t bd = smem_desc(pstage + kk * 512, 128, 2048, 0);
                                umma_f8(tmem + C::OA + sl * 3 * NP, ad, bd, C::IDESC_PV,
                                        !(first_pv && kk == 0));
                            }
                        }
                        umma_commit(&vst_empty[slot]);
                        umma_commit(&pv_done[pb]);
                        if (j < ntiles - 1) itp.next();
                        ++ip;
                        did = true;
                    }
                }
                if (iq < ntiles) {  // Q K^T of tile iq
                    const long long i = iq;
                    const int sb = (int)(i & 1);
                    const bool first_q = (i == 0) || (itq.t == 0);
                    bool ready = true;
                    if (first_q) ready = mbar_test(&q_full[piece_q & 1], (uint32_t)((piece_q >> 1) & 1));
                    if (ready && i >= 2) ready = mbar_test(&s_empty[sb], (uint32_t)(((i >> 1) - 1) & 1));
                    const int slot = (int)(i % NSK);
                    if (ready) ready = mbar_test(&kst_full[slot], (uint32_t)((i / NSK) & 1));
                    if (ready) {
                        if (first_q) {
                            qcur = piece_q & 1;
                            ++piece_q;
                        }
                        tc_fence_after();
                        const uint32_t a0 = kst_s + slot * kStage;
                        const uint32_t b0 = qbuf_s + qcur * C::QB;
                        // 32 codes per MMA; side by side the hi and lo rows are one
                        // operand of 2 NP rows, else the lo part follows the hi part
#pragma unroll
                        for (int part = 0; part < (C::SBS ? 1 : 2); ++part)
#pragma unroll
                            for (int sl = 0; sl < SL; ++sl)
#pragma unroll
                                for (int kk = 0; kk < 4; ++kk) {
                                    const uint64_t ad = smem_desc(a0 + sl * kBox + kk * 32, 16, 1024, 2);
                                    const uint64_t bd = smem_desc(
                                        b0 + sl * C::QSL + part * (NP * 128) + kk * 32, 16, 1024, 2);
                                    umma_f8(tmem + sb * C::SW, ad, bd, C::IDESC_QK,
                                            part != 0 || sl != 0 || kk != 0);
                                }
                        umma_commit(&kst_empty[slot]);
                        umma_commit(&s_full[sb]);
                        if (itq.last_tile_of_segment() || i == ntiles - 1) umma_commit(&q_empty[qcur]);
                        if (i < ntiles - 1) itq.next();
                        ++iq;
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
                if (idle >= kMmaIdleLimit) {
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
            umma_commit(drain);
            volatile int never = 0;
            wait_bar(drain, 0, &never);
        }
        __syncwarp();
        named_bar_sync(kBarEnd, C::END_THREADS);
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
        return;
    }

    // ============================================================== softmax
    // SG groups of four warps; group sg owns columns [cg0, cg0 + NPH) of
    // the pass (heads cg0 .. cg0 + NPH - 1) for all 128 positions of a tile.
    // Votes (the running-max refresh, aborts) are taken by all softmax
    // threads, so the groups move their maxima and the V unit together.
    constexpr int NPH = C::NPH;
    const int sg = (warp - 2) >> 2;
    const int cg0 = sg * NPH;
    const int bar_grp = kBarQ8Grp + sg;
    const int q4 = warp & 3;
    const int row = q4 * 32 + lane;
    const uint32_t lane_base = tmem + ((uint32_t)(q4 * 32) << 16);
    float *redg = red + sg * 256;
    float *vredg = vred_s + sg * 4;

    TileIter it;
    it.init(lens, p.B, p.Lmax, kT, segs_per_b, st);
    long long i = 0;
    int spiece = 0;
    bool first_piece = true;
    bool aborted = false;
    bool carry_fail = false;
    float l[NPH];

    while (i < ntiles && !aborted) {
        const int b = it.b;
        const int kvh = it.seg / p.head_groups;
        const int hg = it.seg % p.head_groups;
        const int len = seq_valid_len(it.len, p.Lmax);
        const int t0 = it.t;
        if (row == 0 && q4 == 0 && sg == 0 && t0 == 0 && (it.len < 0 || it.len > p.Lmax))
            set_error(p.err, DEV_ERR_BOUNDS);
        const int h0 = kvh * p.G + hg * p.heads_per_seg;
        const int gvalid = min(p.heads_per_seg, p.G - hg * p.heads_per_seg);
        const size_t zrow = ((size_t)b * p.Hkv + kvh) * p.Lmax;  // first scale of this block
        const long long i0 = i;
        const int qs = spiece & 1;
        const float *qinv = qinv_s + qs * 64 + cg0;
        int cv = kCvNone;  // the piece's V weights run in units of 2^-cv (same in every thread)
        float vsf = 0.f;   // 2^cv
#pragma unroll
        for (int g = 0; g < NPH; ++g) l[g] = 0.f;
        if (row < NPH) mref_s[cg0 + row] = -INFINITY;
        // the piece's 2^-c (written by the q warps)
        carry_fail = carry_fail || !wait_bar(&q_full[qs], (uint32_t)((spiece >> 1) & 1), abort_flag);
        named_bar_sync(bar_grp, 128);

        while (true) {
            const int sb = (int)(i & 1);
            const int r0 = it.row0();
            const int pos = r0 + row;
            const bool valid = row >= it.first_pos() - r0 && pos < len;
            // this row's scales, loaded while the scores are made -- except
            // in a segment's last tile when this call appends: that tile may
            // hold the row the copy warp has just written, so its scales are
            // read once the tile's scores exist (the copy warp fenced its
            // stores before issuing the tile's copies), past L1 (which may
            // hold the line from the tile before)
            const bool late = p.len_add && it.last_tile_of_segment();
            float ksc = 0.f, vsc = 0.f;
            if (valid && !late) {
                ksc = p.k_scale[zrow + pos];
                vsc = p.v_scale[zrow + pos];
            }
            bool fail = carry_fail || !wait_bar(&s_full[sb], (uint32_t)((i >> 1) & 1), abort_flag);
            if (valid && late) {
                ksc = __ldcg(p.k_scale + zrow + pos);
                vsc = __ldcg(p.v_scale + zrow + pos);
            }
            tc_fence_after();
            // the group's scores: hi-part plus lo-part columns
            float s[NPH];
            tmem_ld_n<NPH>(lane_base + sb * C::SW + cg0, s);
            tmem_ld_wait();
#pragma unroll
            for (int c = 0; c + 16 <= NPH; c += 16) {
                float v[16];
                tmem_ld16(lane_base + sb * C::SW + NP + cg0 + c, v);
                tmem_ld_wait();
#pragma unroll
                for (int k = 0; k < 16; ++k) s[c + k] += v[k];
            }
            if constexpr (NPH % 16 == 8) {
                float v[8];
                tmem_ld8(lane_base + sb * C::SW + NP + cg0 + NPH - 8, v);
                tmem_ld_wait();
#pragma unroll
                for (int k = 0; k < 8; ++k) s[NPH - 8 + k] += v[k];
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&s_empty[sb]);

            const float sl = p.scale_log2 * ksc;
            bool over = vsc * vsf > kVHi;
#pragma unroll
            for (int g = 0; g < NPH; g += 4) {
                const float4 m4 = *reinterpret_cast<const float4 *>(mref_s + cg0 + g);
                const float4 c4 = *reinterpret_cast<const float4 *>(qinv + g);
                s[g] = valid ? s[g] * (c4.x * sl) : -INFINITY;
                s[g + 1] = valid ? s[g + 1] * (c4.y * sl) : -INFINITY;
                s[g + 2] = valid ? s[g + 2] * (c4.z * sl) : -INFINITY;
                s[g + 3] = valid ? s[g + 3] * (c4.w * sl) : -INFINITY;
                over |= (s[g] > m4.x + kTauQ8) | (s[g + 1] > m4.y + kTauQ8) |
                        (s[g + 2] > m4.z + kTauQ8) | (s[g + 3] > m4.w + kTauQ8);
            }
            if (named_bar_sync_or(kBarQ8All, 128 * C::SG, over || fail)) {
                if (named_bar_sync_or(kBarQ8All, 128 * C::SG, fail || *abort_flag != 0)) {
                    aborted = true;
                    break;
                }
                warp_cols_n<NPH>(s, redg + q4 * 64, lane, OpMax());
                const float vm = warp_max(vsc);  // 0 on rows past the length
                if (lane == 0) vredg[q4] = vm;
                named_bar_sync(bar_grp, 128);
                if (row < NPH) {
                    const int g = cg0 + row;
                    const float tmax = fmaxf(fmaxf(redg[row], redg[64 + row]),
                                             fmaxf(redg[128 + row], redg[192 + row]));
                    const float m_old = mref_s[g];
                    const float m_new = fmaxf(m_old, tmax);
                    alpha_s[g] = (m_new == -INFINITY || m_old == m_new) ? 1.f
                                                                         : fast_exp2(m_old - m_new);
                    mref_s[g] = m_new;
                }
                // the V unit: the tile's largest v_scale times 2^cv in [32, 64),
                // lowered only (the accumulator follows by the same power of
                // two); both groups see the same rows, so they agree on it
                const float tv = fmaxf(fmaxf(vredg[0], vredg[1]), fmaxf(vredg[2], vredg[3]));
                float fv = 1.f;
                if (tv > 0.f) {
                    int e = (int)((__float_as_uint(tv) >> 23) & 0xFF) - 127;
                    e = max(-120, min(e, 127));
                    const int cn = 5 - e;
                    if (cv == kCvNone) {
                        cv = cn;
                    } else if (cn < cv) {
                        fv = ldexpf(1.f, cn - cv);
                        cv = cn;
                    }
                } else if (cv == kCvNone) {
                    cv = 0;
                }
                vsf = pow2i(cv);
                named_bar_sync(bar_grp, 128);
#pragma unroll
                for (int g = 0; g < NPH; ++g) l[g] *= alpha_s[cg0 + g];
                if (i > i0) {
                    const long long j = i - 1;
                    if (!wait_bar(&pv_done[j & 1], (uint32_t)((j >> 1) & 1), abort_flag))
                        fail = true;
                    tc_fence_after();
                    // the group's columns of every part of every O^T block
#pragma unroll
                    for (int blk = 0; blk < SL * 3; ++blk) {
                        float v[NPH];
                        const uint32_t a = lane_base + C::OA + blk * NP + cg0;
                        tmem_ld_n<NPH>(a, v);
                        tmem_ld_wait();
#pragma unroll
                        for (int k = 0; k < NPH; ++k) v[k] *= alpha_s[cg0 + k] * fv;
                        tmem_st_n<NPH>(a, v);
                    }
                    tmem_st_wait();
                }
            }

            // probabilities p (summed into l); the weights p v_scale 2^cv in
            // binary16 as three E4M3 parts, each the rounded remainder of the
            // previous
            const float vs2 = vsc * vsf;
            uint32_t ph[NPH / 4], pm[NPH / 4], pl[NPH / 4];
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
                    // w rounded to binary16; its 11 significant bits split
                    // exactly into three 4-bit E4M3 parts (each remainder is
                    // a binary16 value, so the subtractions are exact)
                    const uint32_t w = f16x2_of(p0 * vs2, p1 * vs2);
                    const uint16_t c1 = e4m3x2_of_f16x2(w);
                    const uint32_t r1 = f16x2_sub(w, e4m3x2_to_f16x2(c1));
                    const uint16_t c2 = e4m3x2_of_f16x2(r1);
                    const uint16_t c3 = e4m3x2_of_f16x2(f16x2_sub(r1, e4m3x2_to_f16x2(c2)));
                    if (h == 0) {
                        ph[g4 / 4] = c1;
                        pm[g4 / 4] = c2;
                        pl[g4 / 4] = c3;
                    } else {
                        ph[g4 / 4] |= (uint32_t)c1 << 16;
                        pm[g4 / 4] |= (uint32_t)c2 << 16;
                        pl[g4 / 4] |= (uint32_t)c3 << 16;
                    }
                }
            }
            if (i >= C::PST) {
                const long long jp = i - C::PST;
                if (!wait_bar(&pv_done[jp & 1], (uint32_t)((jp >> 1) & 1), abort_flag))
                    fail = true;
            }
            // P stage: column n's byte at 2048 (n / 16) + n mod 16 of its
            // position row, rows at 128 (row / 8) + 16 (row mod 8); columns
            // hi 0..NP-1, mid NP.., lo 2 NP..; the group's columns go in as
            // 8-byte runs (column starts are multiples of 8)
            uint8_t *pdst = pbuf + (int)(i % C::PST) * C::PB + (row >> 3) * 128 + (row & 7) * 16;
#pragma unroll
            for (int u = 0; u < NPH / 8; ++u) {
                const int ch = cg0 + 8 * u, cm = NP + cg0 + 8 * u, cl = 2 * NP + cg0 + 8 * u;
                *reinterpret_cast<uint2 *>(pdst + (ch >> 4) * 2048 + (ch & 15)) =
                    make_uint2(ph[2 * u], ph[2 * u + 1]);
                *reinterpret_cast<uint2 *>(pdst + (cm >> 4) * 2048 + (cm & 15)) =
                    make_uint2(pm[2 * u], pm[2 * u + 1]);
                *reinterpret_cast<uint2 *>(pdst + (cl >> 4) * 2048 + (cl & 15)) =
                    make_uint2(pl[2 * u], pl[2 * u + 1]);
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&p_full[sb]);
            carry_fail = fail;

            ++i;
            if (it.last_tile_of_segment() || i == ntiles) break;
            it.next();
        }
        if (aborted) break;
        // this warp is done with the piece's 2^-c
        __syncwarp();
        if (lane == 0) mbar_arrive(&q_empty[qs]);
        ++spiece;

        // ---- piece end
        const long long e = i - 1;
        bool fail = carry_fail || !wait_bar(&pv_done[e & 1], (uint32_t)((e >> 1) & 1), abort_flag);
        carry_fail = false;
        tc_fence_after();
        warp_cols_n<NPH>(l, redg + q4 * 64, lane, OpSum());
        named_bar_sync(bar_grp, 128);
        if (row < NPH)
            ltot_s[cg0 + row] = redg[row] + redg[64 + row] + redg[128 + row] + redg[192 + row];
        named_bar_sync(bar_grp, 128);
        const bool complete = (t0 == 0) && it.last_tile_of_segment();
        const size_t slot = 2 * (size_t)blockIdx.x + (first_piece ? 0 : 1);
        const float vinv = (cv == kCvNone) ? 1.f : ldexpf(1.f, -cv);
        if (D == 256 && NP == 48 && !complete) {
            // (the 48-column pass at D = 256) a split piece's partial outputs, 8 columns
            // read and stored at a time from one base address (the heads'
            // rows D floats apart): fewer registers live than the loop below
#pragma unroll
            for (int sl = 0; sl < SL; ++sl) {
                const uint32_t oa = lane_base + C::OA + sl * 3 * NP + cg0;
                float *dst = p.ws_o + (slot * p.heads_per_seg + cg0) * D + sl * 128 + row;
#pragma unroll
                for (int c = 0; c < NPH; c += 8) {
                    float v[8], w[8], x[8];
                    tmem_ld8(oa + c, v);
                    tmem_ld8(oa + NP + c, w);
                    tmem_ld8(oa + 2 * NP + c, x);
                    tmem_ld_wait();
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        if (cg0 + c + k < gvalid) dst[(c + k) * D] = (v[k] + w[k] + x[k]) * vinv;
                }
            }
        } else
#pragma unroll
        for (int sl = 0; sl < SL; ++sl) {  // head dims 128 sl + row
            const uint32_t oa = lane_base + C::OA + sl * 3 * NP + cg0;
            float o[NPH];
#pragma unroll
            for (int c = 0; c + 16 <= NPH; c += 16) {  // O^T = (hi + mid + lo parts) 2^-cv
                float v[16], w[16], x[16];
                tmem_ld16(oa + c, v);
                tmem_ld16(oa + NP + c, w);
                tmem_ld16(oa + 2 * NP + c, x);
                tmem_ld_wait();
#pragma unroll
                for (int k = 0; k < 16; ++k) o[c + k] = (v[k] + w[k] + x[k]) * vinv;
            }
            if constexpr (NPH % 16 == 8) {
                float v[8], w[8], x[8];
                tmem_ld8(oa + NPH - 8, v);
                tmem_ld8(oa + NP + NPH - 8, w);
                tmem_ld8(oa + 2 * NP + NPH - 8, x);
                tmem_ld_wait();
#pragma unroll
                for (int k = 0; k < 8; ++k) o[NPH - 8 + k] = (v[k] + w[k] + x[k]) * vinv;
            }
            const int d = sl * 128 + row;
            if (complete) {
#pragma unroll
                for (int k = 0; k < NPH; ++k) {
                    const int g = cg0 + k;
                    if (g < gvalid) {
                        const float lt = ltot_s[g];
                        p.out[((size_t)b * p.Hq + h0 + g) * D + d] = (lt > 0.f) ? o[k] / lt : 0.f;
                    }
                }
            } else {
#pragma unroll
                for (int k = 0; k < NPH; ++k) {
                    const int g = cg0 + k;
                    if (g < gvalid) p.ws_o[(slot * p.heads_per_seg + g) * D + d] = o[k];
                }
            }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(o_free);
        if (!complete && row < NPH && cg0 + row < gvalid) {
            const int g = cg0 + row;
            p.ws_ml[(slot * p.heads_per_seg + g) * 2 + 0] = mref_s[g];
            p.ws_ml[(slot * p.heads_per_seg + g) * 2 + 1] = ltot_s[g];
        }
        first_piece = false;
        if (named_bar_sync_or(kBarQ8All, 128 * C::SG, fail)) {
            *abort_flag = 1;
            aborted = true;
            break;
        }
        if (i < ntiles) it.next();
    }
    if (aborted) set_error(p.err, DEV_ERR_TIMEOUT);
    tc_fence_before();
    named_bar_sync(kBarEnd, C::END_THREADS);
}

template <int D, int NP>
cudaError_t launch_q8(const CUtensorMap &tmk, const CUtensorMap &tmv, const DecodeParams &p,
                      int num_ctas, cudaStream_t stream) {
    static int done_for_device[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (!(dev >= 0 && dev < 64 && done_for_device[dev])) {
        e = cudaFuncSetAttribute(decode_q8_kernel<D, NP>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, Q8Cfg<D, NP>::alloc);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) done_for_device[dev] = 1;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(num_ctas);
    cfg.blockDim = dim3(Q8Cfg<D, NP>::THREADS);
    cfg.dynamicSmemBytes = Q8Cfg<D, NP>::alloc;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, decode_q8_kernel<D, NP>, tmk, tmv, p);
}

}  // namespace

int q8_smem_bytes(int D, int np) {
    switch (D * 1000 + np) {
        case 128016: return Q8Cfg<128, 16>::alloc;
        case 128032: return Q8Cfg<128, 32>::alloc;
        case 128048: return Q8Cfg<128, 48>::alloc;
        case 128064: return Q8Cfg<128, 64>::alloc;
        case 256016: return Q8Cfg<256, 16>::alloc;
        case 256032: return Q8Cfg<256, 32>::alloc;
        case 256048: return Q8Cfg<256, 48>::alloc;
        default: return -1;
    }
}

cudaError_t launch_decode_q8(const CUtensorMap &tmk, const CUtensorMap &tmv,
                             const DecodeParams &p, int np, int num_ctas, cudaStream_t stream) {
    switch (p.D * 1000 + np) {
        case 128016: return launch_q8<128, 16>(tmk, tmv, p, num_ctas, stream);
        case 128032: return launch_q8<128, 32>(tmk, tmv, p, num_ctas, stream);
        case 128048: return launch_q8<128, 48>(tmk, tmv, p, num_ctas, stream);
        case 128064: return launch_q8<128, 64>(tmk, tmv, p, num_ctas, stream);
        case 256016: return launch_q8<256, 16>(tmk, tmv, p, num_ctas, stream);
        case 256032: return launch_q8<256, 32>(tmk, tmv, p, num_ctas, stream);
        case 256048: return launch_q8<256, 48>(tmk, tmv, p, num_ctas, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace kvattn
