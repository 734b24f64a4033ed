// combine.cu -- merge the (m, l, o) partials of segments that the persistent
// grid cut into several pieces (flash-decoding's cross-split log-sum-exp
// combine):  m* = max_s m_s,  w_s = 2^(m_s - m*),
//            out = sum_s w_s o_s / sum_s w_s l_s.
// Block (c, y) owns the segment containing CTA c's range start when that
// start lies strictly inside a segment and CTA c-1's start does not (c is
// the first cut inside it); y picks a slice of kOutPerBlock of the segment's
// heads x D outputs, one output per thread, so the partial loads of many
// outputs are in flight at once.
#include "internal.h"
#include "schedule.cuh"

namespace kvattn {

namespace {

constexpr int kThreads = 256;
constexpr int kOutPerBlock = kThreads;

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__global__ void __launch_bounds__(kThreads) combine_kernel(const DecodeParams p) {
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
    const int D = p.D;
    const int first_slot = (g_prev == S0) ? 2 * (c - 1) : 2 * (c - 1) + 1;
    const int npieces = 1 + (c_last - c + 1);
    const int x = blockIdx.y * kOutPerBlock + threadIdx.x;   // output index within segment
    if (blockIdx.y * kOutPerBlock >= gvalid * D) return;      // uniform per block
    const int g = x / D, d = x % D;
    const bool active = x < gvalid * D;

    // each thread forms its own weights; the (m, l) loads are shared by the
    // D consecutive threads of one head and served as broadcasts
    float num = 0.f, den = 0.f;
    float mstar = -INFINITY;
    for (int k = 0; k < npieces; ++k) {
        const int slot = (k == 0) ? first_slot : 2 * (c + k - 1);
        if (active) mstar = fmaxf(mstar, p.ws_ml[((size_t)slot * p.heads_per_seg + g) * 2]);
    }
    if (active && mstar != -INFINITY) {
#pragma unroll 4
        for (int k = 0; k < npieces; ++k) {
            const int slot = (k == 0) ? first_slot : 2 * (c + k - 1);
            const size_t ml = ((size_t)slot * p.heads_per_seg + g) * 2;
            const float w = ex2(p.ws_ml[ml] - mstar);
            den = fmaf(w, p.ws_ml[ml + 1], den);
            num = fmaf(w, p.ws_o[((size_t)slot * p.heads_per_seg + g) * D + d], num);
        }
    }
    if (active) p.out[((size_t)st.b * p.Hq + h0 + g) * D + d] = (den > 0.f) ? num / den : 0.f;
}

}  // namespace

cudaError_t launch_combine(const DecodeParams &p, int num_ctas, cudaStream_t stream) {
    dim3 grid(num_ctas, (p.heads_per_seg * p.D + kOutPerBlock - 1) / kOutPerBlock);
    combine_kernel<<<grid, kThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace kvattn
