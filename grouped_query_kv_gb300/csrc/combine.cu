// combine.cu -- merge the (m, l, o) partials of segments that the persistent
// grid cut into several pieces (flash-decoding's cross-split log-sum-exp
// combine):  m* = max_s m_s,  w_s = 2^(m_s - m*),
//            out = sum_s w_s o_s / sum_s w_s l_s.
// Block (x, y) merges one split segment: with fewer segments than CTAs, row
// x is segment x, located from the lengths by the split-KV kernel's own cost
// arithmetic before the wait on that kernel; otherwise row x reads CTA x's
// record, which names a segment when x is the first cut inside it.  y picks
// a slice of 4 x kThreads of the segment's heads x D outputs (four
// consecutive d per thread, as float4).  Each thread loads its head's
// (m_s, l_s) and its own o_s for a batch of pieces at once -- all independent
// loads, one round trip -- and forms the weights itself (the (m, l) loads of
// a warp hit one or two addresses).  Batches after the first fold in with an
// online rescale.  The grid has at most min(CTAs, segments) rows, and few
// blocks: a large grid takes microseconds just to be placed.  Launched with
// programmatic serialisation: it waits on the split-KV kernel with
// griddepcontrol.wait instead of a full launch gap.
#include "internal.h"
#include "ptx.cuh"
#include "schedule.cuh"

namespace kvattn {

namespace {

constexpr int kThreads = 128;  // four outputs (head, d..d+3) per thread
constexpr int kBatch = 8;      // pieces whose loads are in flight together

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Where the split-KV kernel put segment s's pieces, from the lengths alone,
// with the same cost arithmetic as its schedule (schedule.cuh): the first
// contributing CTA c0, the number of pieces n (1: the segment was not split)
// and the workspace slot of piece 0 -- 2 c0 when c0's range starts at the
// segment's first tile, else 2 c0 + 1 (its last piece).  Called by a whole
// warp; every lane gets the results.
__device__ inline void segment_pieces(const DecodeParams &p, int s, int grid, int *c0, int *n,
                                      int *first_slot) {
    const int lane = threadIdx.x & 31;
    const LenView lens{p.seq_lens, p.len_add, p.window, p.walign};
    const int segs_per_b = p.Hkv * p.head_groups;
    const SchedCost w{p.cost_piece};
    long long total, cost;
    int ctas_eff;
    sched_totals(lens, p.B, p.Lmax, p.tile, segs_per_b, w, grid, &total, &cost, &ctas_eff);
    const int b = s / segs_per_b, sg = s % segs_per_b;
    int before = 0;  // tiles of one segment of every sequence before b
    for (int bb = lane; bb < b; bb += 32) before += seq_ntiles(lens[bb], p.Lmax, p.tile, lens.window, lens.walign);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) before += __shfl_xor_sync(0xffffffffu, before, o);
    const int nt = seq_ntiles(lens[b], p.Lmax, p.tile, lens.window, lens.walign);
    const long long cost0 = (long long)segs_per_b * ((long long)before * kCostTile + (long long)w.P * b) +
                            (long long)sg * ((long long)nt * kCostTile + w.P);
    const long long last = cost0 + (nt == 1 ? 0 : w.P + (long long)kCostTile * (nt - 1));
    const int c = sched_owner(cost0, cost, ctas_eff);
    bool starts = true;  // c's range starts at this segment's first tile
    if (s > 0) {
        // the tile before: the last of the previous segment
        const int ntp = sg > 0 ? nt : seq_ntiles(lens[b - 1], p.Lmax, p.tile, lens.window, lens.walign);
        const long long prev = cost0 - kCostTile - (ntp == 1 ? w.P : 0);
        starts = prev < sched_bound(cost, ctas_eff, c);
    }
    *c0 = c;
    *n = sched_owner(last, cost, ctas_eff) - c + 1;
    *first_slot = 2 * c + (starts ? 0 : 1);
}

// by_segment: block row s merges segment s, whose pieces it locates from the
// lengths before waiting on the split-KV kernel (the lengths are an input of
// the call, written before that kernel started, so only the partials are
// waited for); else block row c merges the segment CTA c's record names
// (rows whose record names none exit at once).  The host takes rows by
// segment when there are fewer segments than CTAs: few rows, and no record
// load between the wait and the partials' loads.
__global__ void __launch_bounds__(kThreads) combine_kernel(const DecodeParams p, int num_ctas,
                                                           int by_segment) {
    // the next kernel in the stream may start its prologue while this one
    // runs; it waits for these writes with its own griddepcontrol.wait
    pdl_launch_dependents();
    const int tid = threadIdx.x;
    const int4 *recs = reinterpret_cast<const int4 *>(p.split);

    int c = (int)blockIdx.x;
    int4 rec;
    if (by_segment) {
        int c0, n, fs;
        segment_pieces(p, (int)blockIdx.x, num_ctas, &c0, &n, &fs);
        if (n <= 1) return;  // not split: the split-KV kernel wrote this segment's rows
        const int segs_per_b = p.Hkv * p.head_groups;
        rec = make_int4((int)blockIdx.x / segs_per_b, (int)blockIdx.x % segs_per_b, fs, n);
        c = c0 + 1;
        pdl_wait_prior();  // the partials come from the split-KV kernel just before
    } else {
        pdl_wait_prior();  // partials and records come from the split-KV kernel just before
        if (recs[c].x < 0) return;  // CTA c is not the first cut inside a segment
        rec = recs[c];
    }
    const int b = rec.x, seg = rec.y, first_slot = rec.z, npieces = rec.w;
    const int kvh = seg / p.head_groups;
    const int hg = seg % p.head_groups;
    const int h0 = kvh * p.G + hg * p.hpg;
    // columns: heads, or (token, head) pairs of the pass's hpg heads for T
    // new tokens, of which the first hvalid heads exist
    const int gvalid = p.T == 1 ? min(p.heads_per_seg, p.G - hg * p.heads_per_seg)
                                : p.heads_per_seg;
    const int hvalid = min(p.hpg, p.G - hg * p.hpg);
    const int D = p.D;
    const int x = (blockIdx.y * kThreads + tid) * 4;
    const int g = x / D, d = x % D;
    const int t = p.T == 1 ? 0 : g / p.hpg, gg = p.T == 1 ? g : g % p.hpg;
    if (g >= gvalid || gg >= hvalid) return;

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
    *reinterpret_cast<float4 *>(p.out + (((size_t)b * p.T + t) * p.Hq + h0 + gg) * D + d) =
        make_float4(num.x * inv, num.y * inv, num.z * inv, num.w * inv);
}

}  // namespace

cudaError_t launch_combine(const DecodeParams &p, int num_ctas, cudaStream_t stream) {
    // rows: one per segment when segments are fewer than CTAs, else one per
    // CTA record (at most one owner per segment, and at most one per CTA)
    const long long segs = (long long)p.B * p.Hkv * p.head_groups;
    const int ycount = (p.heads_per_seg * p.D / 4 + kThreads - 1) / kThreads;
    const int by_segment = segs < num_ctas ? 1 : 0;
    const int rows = by_segment ? (int)segs : num_ctas;
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
    return cudaLaunchKernelEx(&cfg, combine_kernel, p, num_ctas, by_segment);
}

}  // namespace kvattn
