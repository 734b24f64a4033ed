// combine.cu -- merge the (m, l, o) partials of segments that the persistent
// grid cut into several pieces (flash-decoding's cross-split log-sum-exp
// combine):  m* = max_s m_s,  w_s = 2^(m_s - m*),
//            out = sum_s w_s o_s / sum_s w_s l_s.
// Block (c, y) merges the segment named by CTA c's combine record (written by
// the split-KV kernel: present when c is the first cut inside a segment); y
// picks a slice of kOutPerBlock of the segment's heads x D outputs, one
// output per thread, so the partial loads of many outputs are in flight at
// once.  Launched with programmatic serialisation: it waits on the split-KV
// kernel with griddepcontrol.wait instead of a full launch gap.
#include "internal.h"
#include "ptx.cuh"

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
    pdl_wait_prior();  // partials and records come from the split-KV kernel just before
    const int c = blockIdx.x;
    const int4 rec = reinterpret_cast<const int4 *>(p.split)[c];
    if (rec.x < 0) return;  // c is not the first cut inside a segment
    const int b = rec.x, seg = rec.y, first_slot = rec.z, npieces = rec.w;
    const int kvh = seg / p.head_groups;
    const int hg = seg % p.head_groups;
    const int h0 = kvh * p.G + hg * p.heads_per_seg;
    const int gvalid = min(p.heads_per_seg, p.G - hg * p.heads_per_seg);
    const int D = p.D;
    const int x = blockIdx.y * kOutPerBlock + threadIdx.x;   // output index within segment
    if (x >= gvalid * D) return;
    const int g = x / D, d = x % D;

    // each thread forms its own weights; the (m, l) loads are shared by the
    // D consecutive threads of one head and served as broadcasts
    float mstar = -INFINITY;
    for (int k = 0; k < npieces; ++k) {
        const int slot = (k == 0) ? first_slot : 2 * (c + k - 1);
        mstar = fmaxf(mstar, p.ws_ml[((size_t)slot * p.heads_per_seg + g) * 2]);
    }
    float num = 0.f, den = 0.f;
    if (mstar != -INFINITY) {
#pragma unroll 4
        for (int k = 0; k < npieces; ++k) {
            const int slot = (k == 0) ? first_slot : 2 * (c + k - 1);
            const size_t ml = ((size_t)slot * p.heads_per_seg + g) * 2;
            const float w = ex2(p.ws_ml[ml] - mstar);
            den = fmaf(w, p.ws_ml[ml + 1], den);
            num = fmaf(w, p.ws_o[((size_t)slot * p.heads_per_seg + g) * D + d], num);
        }
    }
    p.out[((size_t)b * p.Hq + h0 + g) * D + d] = (den > 0.f) ? num / den : 0.f;
}

}  // namespace

cudaError_t launch_combine(const DecodeParams &p, int num_ctas, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(num_ctas, (p.heads_per_seg * p.D + kOutPerBlock - 1) / kOutPerBlock);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, combine_kernel, p);
}

}  // namespace kvattn
