// combine.cu -- merge the (m, l, o) partials of segments that the persistent
// grid cut into several pieces (flash-decoding's cross-split log-sum-exp
// combine):  m* = max_s m_s,  w_s = 2^(m_s - m*),
//            out = sum_s w_s o_s / sum_s w_s l_s.
// Block (c, y) owns the segment containing CTA c's range start when that
// start lies strictly inside a segment and CTA c-1's start does not (c is
// the first cut inside it); y picks a slice of the segment's heads.
#include "internal.h"
#include "schedule.cuh"

namespace kvattn {

namespace {

constexpr int kThreads = 128;

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__global__ void __launch_bounds__(kThreads)
    combine_kernel(const DecodeParams p, int heads_per_block) {
    __shared__ SchedScratch sched;
    const int c = blockIdx.x;
    const int segs_per_b = p.Hkv * p.head_groups;
    sched_locate(p.seq_lens, p.B, p.Lmax, p.tile, segs_per_b, c, gridDim.x, &sched);
    const SchedStart st = sched.res;
    if (c == 0 || !st.found || st.t == 0) return;   // range starts on a segment start
    const long long S0 = st.g_begin - st.t;          // the segment's first tile
    const long long total = st.total;
    const int C = st.ctas_eff;
    const long long g_prev = (long long)(c - 1) * total / C;
    if (g_prev > S0) return;                          // an earlier cut owns this segment
    const int nt = seq_ntiles(p.seq_lens[st.b], p.Lmax, p.tile);
    const long long S1 = S0 + nt;
    const int c_last = (int)((S1 * C - 1) / total);   // CTA holding tile S1-1

    const int kvh = st.seg / p.head_groups;
    const int hg = st.seg % p.head_groups;
    const int h0 = kvh * p.G + hg * p.heads_per_seg;
    const int gvalid = min(p.heads_per_seg, p.G - hg * p.heads_per_seg);
    const int gb = blockIdx.y * heads_per_block;
    const int ge = min(gvalid, gb + heads_per_block);
    const int D = p.D;
    const int first_slot = (g_prev == S0) ? 2 * (c - 1) : 2 * (c - 1) + 1;
    const int npieces = 1 + (c_last - c + 1);

    for (int x = threadIdx.x; x < (ge - gb) * D; x += kThreads) {
        const int g = gb + x / D, d = x % D;
        float mstar = -INFINITY;
        for (int k = 0; k < npieces; ++k) {
            const int slot = (k == 0) ? first_slot : 2 * (c + k - 1);
            mstar = fmaxf(mstar, p.ws_ml[((size_t)slot * p.heads_per_seg + g) * 2]);
        }
        float num = 0.f, den = 0.f;
        if (mstar != -INFINITY) {
            for (int k = 0; k < npieces; ++k) {
                const int slot = (k == 0) ? first_slot : 2 * (c + k - 1);
                const size_t ml = ((size_t)slot * p.heads_per_seg + g) * 2;
                const float w = ex2(p.ws_ml[ml] - mstar);
                den = fmaf(w, p.ws_ml[ml + 1], den);
                num = fmaf(w, p.ws_o[((size_t)slot * p.heads_per_seg + g) * D + d], num);
            }
        }
        p.out[((size_t)st.b * p.Hq + h0 + g) * D + d] = (den > 0.f) ? num / den : 0.f;
    }
}

}  // namespace

cudaError_t launch_combine(const DecodeParams &p, int num_ctas, cudaStream_t stream) {
    const int hpb = p.heads_per_seg <= 8 ? p.heads_per_seg : 4;
    dim3 grid(num_ctas, (p.heads_per_seg + hpb - 1) / hpb);
    combine_kernel<<<grid, kThreads, 0, stream>>>(p, hpb);
    return cudaGetLastError();
}

}  // namespace kvattn
