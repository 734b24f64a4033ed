// combine.cu -- merge the (m, l, o) partials of segments that the persistent
// grid cut into several pieces (flash-decoding's cross-split log-sum-exp
// combine):  m* = max_s m_s,  w_s = 2^(m_s - m*),
//            out = sum_s w_s o_s / sum_s w_s l_s.
// The split-KV kernel leaves one record per CTA; CTA c's record names a
// segment when c is the first cut inside it.  Block (x, y) merges the
// segment of record x, or of the x-th record that names one (found with a
// block-wide ballot over the records), y picks a slice of 4 x kThreads of the segment's heads x D
// outputs (four consecutive d per thread, as float4).  Each thread loads its
// head's (m_s, l_s) and its own o_s for a batch of pieces at once -- all
// independent loads, one round trip -- and forms the weights itself (the
// (m, l) loads of a warp hit one or two addresses).  Batches after the first
// fold in with an online rescale.  The grid has at most min(CTAs, segments)
// rows, and few blocks: a large grid takes microseconds just to be placed.  Launched with programmatic
// serialisation: it waits on the split-KV kernel with griddepcontrol.wait
// instead of a full launch gap.
#include "internal.h"
#include "ptx.cuh"

namespace kvattn {

namespace {

constexpr int kThreads = 256;  // four outputs (head, d..d+3) per thread
constexpr int kBatch = 8;      // pieces whose loads are in flight together

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// direct: block row c merges the segment CTA c's record names (rows whose
// record names none exit at once); else block row x finds the x-th record
// that names a segment.  The host takes direct rows unless they would mean
// many more blocks (few long segments): placing blocks costs microseconds.
__global__ void __launch_bounds__(kThreads) combine_kernel(const DecodeParams p, int num_ctas,
                                                           int direct) {
    __shared__ int s_wcount[kThreads / 32];
    __shared__ int s_owner;
    // the next kernel in the stream may start its prologue while this one
    // runs; it waits for these writes with its own griddepcontrol.wait
    pdl_launch_dependents();
    pdl_wait_prior();  // partials and records come from the split-KV kernel just before
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int4 *recs = reinterpret_cast<const int4 *>(p.split);

    int c = (int)blockIdx.x;
    if (direct) {
        if (recs[c].x < 0) return;
    } else {
        // the blockIdx.x-th CTA whose record names a segment
        if (tid == 0) s_owner = -1;
        int seen = 0;
        for (int base = 0; base < num_ctas; base += kThreads) {
            const int cc = base + tid;
            const bool own = cc < num_ctas && recs[cc].x >= 0;
            const unsigned m = __ballot_sync(0xffffffffu, own);
            if (lane == 0) s_wcount[warp] = __popc(m);
            __syncthreads();
            int before = seen, total = 0;
            for (int w = 0; w < kThreads / 32; ++w) {
                if (w < warp) before += s_wcount[w];
                total += s_wcount[w];
            }
            if (own && before + __popc(m & ((1u << lane) - 1u)) == (int)blockIdx.x) s_owner = cc;
            __syncthreads();
            seen += total;
            if (seen > (int)blockIdx.x) break;
        }
        c = s_owner;
        if (c < 0) return;
    }

    const int4 rec = recs[c];
    const int b = rec.x, seg = rec.y, first_slot = rec.z, npieces = rec.w;
    const int kvh = seg / p.head_groups;
    const int hg = seg % p.head_groups;
    const int h0 = kvh * p.G + hg * p.heads_per_seg;
    const int gvalid = p.T == 1 ? min(p.heads_per_seg, p.G - hg * p.heads_per_seg)
                                : p.heads_per_seg;  // (token, head) columns
    const int D = p.D;
    const int x = (blockIdx.y * kThreads + tid) * 4;
    const int g = x / D, d = x % D;
    if (g >= gvalid) return;

    // piece k's workspace slot: the first piece is the last piece of CTA
    // c-1 (or its first), piece k >= 1 is the first piece of CTA c + k - 1
    float mrun = -INFINITY, den = 0.f;
    float4 num = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int k0 = 0; k0 < npieces; k0 += kBatch) {
        const int nk = min(kBatch, npieces - k0);
        float mk[kBatch], lk[kBatch];
        float4 ok[kBatch];
#pragma unroll
        for (int k = 0; k < kBatch; ++k) {
            mk[k] = -INFINITY;
            lk[k] = 0.f;
            ok[k] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (k < nk) {
                const int kk = k0 + k;
                const size_t slot = (kk == 0) ? first_slot : 2 * (size_t)(c + kk - 1);
                const size_t hs = slot * p.heads_per_seg + g;
                const float2 ml = *reinterpret_cast<const float2 *>(p.ws_ml + hs * 2);
                mk[k] = ml.x;
                lk[k] = ml.y;
                ok[k] = *reinterpret_cast<const float4 *>(p.ws_o + hs * D + d);
            }
        }
        float mx = mrun;
#pragma unroll
        for (int k = 0; k < kBatch; ++k) mx = fmaxf(mx, mk[k]);
        if (mx == -INFINITY) continue;  // nothing but empty pieces so far
        const float a = (mrun == -INFINITY) ? 0.f : ex2(mrun - mx);
        num.x *= a;
        num.y *= a;
        num.z *= a;
        num.w *= a;
        den *= a;
#pragma unroll
        for (int k = 0; k < kBatch; ++k) {
            const float w = (mk[k] == -INFINITY) ? 0.f : ex2(mk[k] - mx);
            num.x = fmaf(w, ok[k].x, num.x);
            num.y = fmaf(w, ok[k].y, num.y);
            num.z = fmaf(w, ok[k].z, num.z);
            num.w = fmaf(w, ok[k].w, num.w);
            den = fmaf(w, lk[k], den);
        }
        mrun = mx;
    }
    const float inv = (den > 0.f) ? 1.f / den : 0.f;
    const int t = p.T == 1 ? 0 : g / p.G, gg = p.T == 1 ? g : g % p.G;
    *reinterpret_cast<float4 *>(p.out + (((size_t)b * p.T + t) * p.Hq + h0 + gg) * D + d) =
        make_float4(num.x * inv, num.y * inv, num.z * inv, num.w * inv);
}

}  // namespace

cudaError_t launch_combine(const DecodeParams &p, int num_ctas, cudaStream_t stream) {
    // at most one owner per segment, and at most one per CTA
    const long long segs = (long long)p.B * p.Hkv * p.head_groups;
    const int ycount = (p.heads_per_seg * p.D / 4 + kThreads - 1) / kThreads;
    const int direct = (segs >= num_ctas || (long long)num_ctas * ycount <= 1024) ? 1 : 0;
    const int rows = direct ? num_ctas : (int)(segs < num_ctas ? segs : num_ctas);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(rows, ycount);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, combine_kernel, p, num_ctas, direct);
}

}  // namespace kvattn
