// combine.cu -- merge the (m, l, o) partials of segments that the persistent
// grid cut into several pieces (flash-decoding's cross-split log-sum-exp
// combine):  m* = max_s m_s,  w_s = 2^(m_s - m*),
//            out = sum_s w_s o_s / sum_s w_s l_s.
// The split-KV kernel leaves one record per CTA; CTA c's record names a
// segment when c is the first cut inside it.  Block (x, y) merges the
// segment of the x-th such record (found with a block-wide ballot over the
// records), y picks a slice of kThreads of the segment's heads x D outputs
// (one output per thread).  For each head in the slice one warp weighs the
// pieces once -- w_s = 2^(m_s - m*), and the denominator -- into shared
// memory; every thread then only streams its o_s values, independent loads
// that can all be in flight.  The grid has at most min(CTAs, segments) rows.
// Launched
// with programmatic serialisation: it waits on the split-KV kernel with
// griddepcontrol.wait instead of a full launch gap.
#include "internal.h"
#include "ptx.cuh"

namespace kvattn {

namespace {

constexpr int kThreads = 256;       // one output (head, d) per thread
constexpr int kMaxPieces = 64;      // pieces weighed per batch (per head, in shared memory)
constexpr int kMaxHeadsPerBlock = kThreads / 64;  // D >= 64

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__global__ void __launch_bounds__(kThreads) combine_kernel(const DecodeParams p, int num_ctas) {
    __shared__ int s_wcount[kThreads / 32];
    __shared__ int s_owner;
    __shared__ float s_w[kMaxHeadsPerBlock][kMaxPieces];
    __shared__ float s_m[kMaxHeadsPerBlock], s_den[kMaxHeadsPerBlock], s_scale[kMaxHeadsPerBlock];
    // the next kernel in the stream may start its prologue while this one
    // runs; it waits for these writes with its own griddepcontrol.wait
    pdl_launch_dependents();
    pdl_wait_prior();  // partials and records come from the split-KV kernel just before
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int4 *recs = reinterpret_cast<const int4 *>(p.split);

    // the blockIdx.x-th CTA whose record names a segment
    if (tid == 0) s_owner = -1;
    int seen = 0;
    for (int base = 0; base < num_ctas; base += kThreads) {
        const int c = base + tid;
        const bool own = c < num_ctas && recs[c].x >= 0;
        const unsigned m = __ballot_sync(0xffffffffu, own);
        if (lane == 0) s_wcount[warp] = __popc(m);
        __syncthreads();
        int before = seen, total = 0;
        for (int w = 0; w < kThreads / 32; ++w) {
            if (w < warp) before += s_wcount[w];
            total += s_wcount[w];
        }
        if (own && before + __popc(m & ((1u << lane) - 1u)) == (int)blockIdx.x) s_owner = c;
        __syncthreads();
        seen += total;
        if (seen > (int)blockIdx.x) break;
    }
    const int c = s_owner;
    if (c < 0) return;

    const int4 rec = recs[c];
    const int b = rec.x, seg = rec.y, first_slot = rec.z, npieces = rec.w;
    const int kvh = seg / p.head_groups;
    const int hg = seg % p.head_groups;
    const int h0 = kvh * p.G + hg * p.heads_per_seg;
    const int gvalid = min(p.heads_per_seg, p.G - hg * p.heads_per_seg);
    const int D = p.D;
    // this block's heads: kThreads consecutive (head, d) outputs
    const int x0 = blockIdx.y * kThreads;
    const int g_lo = x0 / D;
    const int g_hi = min(gvalid - 1, (x0 + kThreads - 1) / D);
    if (g_lo >= gvalid) return;

    // warp w (< heads in the block) forms its head's weights: lane k takes
    // pieces k, k+32, ...; the max is a warp reduction
    const int x = x0 + tid;
    const int g = x / D, d = x % D;
    float num = 0.f;
    for (int k0 = 0; k0 < npieces; k0 += kMaxPieces) {
        const int nk = min(kMaxPieces, npieces - k0);
        if (warp <= g_hi - g_lo) {
            const int gw = g_lo + warp;
            float mk[kMaxPieces / 32], lk[kMaxPieces / 32];
            float mx = -INFINITY;
#pragma unroll
            for (int u = 0; u < kMaxPieces / 32; ++u) {
                const int k = u * 32 + lane;
                mk[u] = -INFINITY;
                lk[u] = 0.f;
                if (k < nk) {
                    const int kk = k0 + k;
                    const size_t slot = (kk == 0) ? first_slot : 2 * (c + kk - 1);
                    const size_t ml = (slot * p.heads_per_seg + gw) * 2;
                    mk[u] = p.ws_ml[ml];
                    lk[u] = p.ws_ml[ml + 1];
                }
                mx = fmaxf(mx, mk[u]);
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            // fold the previous batches into this batch's reference
            const float m_prev = (k0 == 0) ? -INFINITY : s_m[warp];
            const float m_new = fmaxf(m_prev, mx);
            float dsum = 0.f;
#pragma unroll
            for (int u = 0; u < kMaxPieces / 32; ++u) {
                const int k = u * 32 + lane;
                const float w = (m_new == -INFINITY || mk[u] == -INFINITY) ? 0.f : ex2(mk[u] - m_new);
                if (k < nk) s_w[warp][k] = w;
                dsum = fmaf(w, lk[u], dsum);
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) dsum += __shfl_xor_sync(0xffffffffu, dsum, o);
            if (lane == 0) {
                const float a = (m_prev == -INFINITY || m_new == -INFINITY) ? 0.f : ex2(m_prev - m_new);
                s_scale[warp] = a;
                s_den[warp] = ((k0 == 0) ? 0.f : s_den[warp] * a) + dsum;
                s_m[warp] = m_new;
            }
        }
        __syncthreads();
        if (g < gvalid) {
            const int wi = g - g_lo;
            float acc = num * s_scale[wi];
#pragma unroll 8
            for (int k = 0; k < nk; ++k) {
                const int kk = k0 + k;
                const size_t slot = (kk == 0) ? first_slot : 2 * (c + kk - 1);
                acc = fmaf(s_w[wi][k], p.ws_o[(slot * p.heads_per_seg + g) * D + d], acc);
            }
            num = acc;
        }
        __syncthreads();
    }
    if (g < gvalid) {
        const float den = s_den[g - g_lo];
        p.out[((size_t)b * p.Hq + h0 + g) * D + d] = (den > 0.f) ? num / den : 0.f;
    }
}

}  // namespace

cudaError_t launch_combine(const DecodeParams &p, int num_ctas, cudaStream_t stream) {
    // at most one owner per segment, and at most one per CTA
    const long long segs = (long long)p.B * p.Hkv * p.head_groups;
    const int rows = (int)(segs < num_ctas ? segs : num_ctas);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(rows, (p.heads_per_seg * p.D + kThreads - 1) / kThreads);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, combine_kernel, p, num_ctas);
}

}  // namespace kvattn
