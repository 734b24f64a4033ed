// schedule.cuh -- the persistent grid's split of the flat tile list.
//
// Every segment (b, kvh, hg) owns ntiles(len_b) tiles; the list of all tiles
// in (b, kvh, hg, t) order is cut into contiguous CTA ranges of equal COST.
// A segment of nt tiles costs nt * W + P: W per tile, and P for the fixed
// work of starting and finishing a piece (its q load, the first tile's exact
// max, reading out and storing the output), charged at its first tile.  So
// tile t of a segment whose cost starts at B0 starts at cost B0 for t = 0 and
// at B0 + P + W t for t >= 1, and with TC the total cost and C the CTAs,
//     CTA c owns the tiles whose start cost s has  T(c) <= s < T(c + 1),
//     T(c) = ceil(c TC / C).
// C = min(gridDim.x, tiles, TC / (W + P)): every share is then at least as
// long as the costliest tile, and consecutive start costs are at most W + P
// apart, so no range is empty.  With P = 0 this is the plain equal split.
// Lengths live on the device, so each CTA locates its own range with a
// warp-level scan over seq_lens (no host synchronisation).
#pragma once

#include <cstdint>
#include "internal.h"

namespace kvattn {

// Lengths as the kernels see them.  For the fused append-then-attend step the
// array holds the number of tokens cached BEFORE this step's token, and the
// attention covers one more position; a negative entry stays invalid.  A
// local (sliding-window) layer attends only the last `window` positions
// ("The Basics of Transformer Inference", item on mixing in local attention
// layers); window >= Lmax is the full attention.  A paged cache's tiles
// must start on block boundaries, so there the window's first tile starts
// at the tile boundary at or before the window (walign = tile - 1; the
// rows before the window are masked); elsewhere it starts at the window.
struct LenView {
    const int32_t *p;
    int add;     // 0: attention lengths as given; 1: cached-before counts (+1)
    int window;  // positions attended at most, >= 1
    int walign;  // 0, or tile - 1: window starts rounded down to a tile boundary
    __device__ __forceinline__ int operator[](int b) const {
        const int r = p[b];
        return add ? (r < 0 ? -1 : r + 1) : r;
    }
};

// A sequence whose length is outside [1, Lmax] still owns one tile, with no
// valid positions (zero output row; out-of-range lengths also raise the
// device error word).  Otherwise its tiles cover the min(len, window)
// attended positions, and with walign = tile - 1 the positions from the
// tile boundary before the window's start.
__device__ __forceinline__ int seq_ntiles(int len, int Lmax, int tile, int window, int walign) {
    // (len - window) & walign: the rows between that boundary and the window
    // (a span of at least len when len <= window, so the min stays len)
    const int span = window + ((len - window) & walign);
    // tiles are a power of two positions (64 or 128): a shift, not a division
    return (len <= 0 || len > Lmax) ? 1 : ((len < span ? len : span) + tile - 1) >> (__ffs(tile) - 1);
}

__device__ __forceinline__ int seq_valid_len(int len, int Lmax) {
    return (len < 0 || len > Lmax) ? 0 : len;
}

// First position the tiles of a sequence of (valid) length len cover.
__device__ __forceinline__ int seq_window_start(int len, int window, int walign) {
    return len > window ? (len - window) & ~walign : 0;
}

// The cost model's weights: W = kCostTile per tile (a power of two, so the
// kernels divide by shifting) and P = DecodeParams::cost_piece per segment.
constexpr int kCostTile = 32;
constexpr int kCostTileShift = 5;
struct SchedCost {
    int P;
};

struct SchedStart {
    long long total;    // tiles in the whole call
    long long cost;     // total cost TC
    long long g_begin;  // this CTA's first tile
    long long g_end;    // one past its last tile
    long long cost0;    // start cost of the segment that holds g_begin
    int ctas_eff;
    int found;          // 1 if this CTA has work
    int b, seg, t;      // coordinates of g_begin: sequence, segment within b, tile
};

__device__ __forceinline__ long long warp_sum_ll(long long v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ int warp_incl_scan(int v) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += n;
    }
    return v;
}

// A tile found by its start cost.
struct SchedHit {
    long long g;      // tile index (the total if the cost is past the end)
    long long cost0;  // start cost of its segment
    int b, seg, t;
};

// Where cost T falls in a sequence whose cost starts at ec (segments of segc,
// nt tiles each): the tile, its segment's start cost and coordinates.
__device__ __forceinline__ SchedHit sched_hit_in(long long T, long long ec, int segc, int nt,
                                                 long long tiles_before, int b, int segs_per_b,
                                                 int P) {
    const unsigned long long rb = (unsigned long long)(T - ec);
    int seg = (int)(rb <= 0xffffffffull ? (unsigned)rb / (unsigned)segc
                                        : rb / (unsigned long long)segc);
    const int rem = (int)(rb - (unsigned long long)seg * segc);
    int t = rem == 0 ? 0 : max(1, (rem - P + kCostTile - 1) >> kCostTileShift);
    SchedHit h;
    h.g = tiles_before + (long long)seg * nt + t;
    h.cost0 = ec + (long long)seg * segc;
    h.b = b;
    if (t >= nt) {  // the next segment's first tile
        t = 0;
        h.cost0 += segc;
        if (++seg == segs_per_b) {
            seg = 0;
            ++h.b;
        }
    }
    h.seg = seg;
    h.t = t;
    return h;
}

__device__ __forceinline__ void sched_take(SchedHit *h, const SchedHit &mine, int src) {
    h->g = __shfl_sync(0xffffffffu, mine.g, src);
    h->cost0 = __shfl_sync(0xffffffffu, mine.cost0, src);
    h->b = __shfl_sync(0xffffffffu, mine.b, src);
    h->seg = __shfl_sync(0xffffffffu, mine.seg, src);
    h->t = __shfl_sync(0xffffffffu, mine.t, src);
}

// Called by a whole warp: the first tiles whose start costs are >= T0 and
// (NT = 2) >= T1, T0 <= T1.  The cost before sequence b is
// segs_per_b * (W * (tiles of the sequences before b) + P * b).  Every lane
// evaluates its own sequence for both bounds at once; a ballot picks the
// lane that holds each.
template <int NT>
__device__ inline void sched_find(LenView lens, int B, int Lmax, int tile, int segs_per_b,
                                  SchedCost w, long long T0, long long T1, long long total,
                                  SchedHit *h0, SchedHit *h1) {
    const int lane = threadIdx.x & 31;
    h0->g = h1->g = total;
    h0->cost0 = h1->cost0 = 0;
    h0->b = h0->seg = h0->t = h1->b = h1->seg = h1->t = 0;
    bool got0 = false, got1 = NT < 2;
    int tcarry = 0;  // tiles of one segment of every sequence so far
    for (int base = 0; base < B && !(got0 && got1); base += 32) {
        const int b = base + lane;
        const int nt = (b < B) ? seq_ntiles(lens[b], Lmax, tile, lens.window, lens.walign) : 0;
        const int incl = warp_incl_scan(nt);
        const int before = tcarry + incl - nt;
        const int segc = nt * kCostTile + w.P;  // one segment of sequence b
        const long long ec = (long long)segs_per_b * ((long long)before * kCostTile + (long long)w.P * b);
        const long long vc = (b < B) ? (long long)segs_per_b * segc : 0;
        const long long tb = (long long)before * segs_per_b;
        const bool in0 = (b < B) && ec <= T0 && T0 < ec + vc;
        const bool in1 = NT > 1 && (b < B) && ec <= T1 && T1 < ec + vc;
        const SchedHit m0 = sched_hit_in(in0 ? T0 : ec, ec, segc > 0 ? segc : 1, nt, tb, b,
                                         segs_per_b, w.P);
        SchedHit m1 = m0;
        if (NT > 1) m1 = sched_hit_in(in1 ? T1 : ec, ec, segc > 0 ? segc : 1, nt, tb, b, segs_per_b, w.P);
        const unsigned b0 = __ballot_sync(0xffffffffu, in0);
        const unsigned b1 = __ballot_sync(0xffffffffu, in1);
        if (b0 && !got0) {
            sched_take(h0, m0, __ffs(b0) - 1);
            got0 = true;
        }
        if (NT > 1 && b1 && !got1) {
            sched_take(h1, m1, __ffs(b1) - 1);
            got1 = true;
        }
        tcarry += __shfl_sync(0xffffffffu, incl, 31);
    }
}

// Called by a whole warp: totals (tiles, cost) and the CTA count that the
// split uses.
__device__ inline void sched_totals(LenView lens, int B, int Lmax, int tile, int segs_per_b,
                                    SchedCost w, int grid, long long *total, long long *cost,
                                    int *ctas_eff) {
    const int lane = threadIdx.x & 31;
    int nt_lane = 0;
    for (int b = lane; b < B; b += 32) nt_lane += seq_ntiles(lens[b], Lmax, tile, lens.window, lens.walign);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) nt_lane += __shfl_xor_sync(0xffffffffu, nt_lane, o);
    const long long nt_sum = nt_lane;  // tiles of one segment of every sequence
    *total = nt_sum * segs_per_b;
    *cost = (long long)segs_per_b * (nt_sum * kCostTile + (long long)w.P * B);
    long long ce = *total < (long long)grid ? *total : (long long)grid;
    if (*cost < (long long)(kCostTile + w.P) * ce) ce = *cost / (kCostTile + w.P);
    *ctas_eff = (int)(ce < 1 ? 1 : ce);
}

// Owner of a tile with start cost s.
__device__ __forceinline__ int sched_owner(long long s, long long cost, int ctas_eff) {
    const long long c = s * ctas_eff / cost;
    return (int)(c < ctas_eff - 1 ? c : ctas_eff - 1);
}

// T(c) = ceil(c TC / C) = c q + ceil(c rem / C) with TC = q C + rem (the
// last part in 32 bits: C <= 65535).
__device__ __forceinline__ long long sched_bound(long long cost, int ctas_eff, int c) {
    const long long q = cost / ctas_eff;
    const unsigned rem = (unsigned)(cost - q * ctas_eff);
    const unsigned C = (unsigned)ctas_eff;
    return (long long)c * q + ((unsigned)c * rem + C - 1) / C;
}

// Locate CTA `c`'s tile range; called by a whole warp (every warp of a CTA
// can do it on its own, so the TMA producer starts as soon as the lengths
// have been read).
__device__ inline SchedStart warp_locate(LenView lens, int B, int Lmax, int tile,
                                         int segs_per_b, SchedCost w, int c, int grid) {
    SchedStart r;
    sched_totals(lens, B, Lmax, tile, segs_per_b, w, grid, &r.total, &r.cost, &r.ctas_eff);
    r.found = 0;
    r.b = r.seg = r.t = 0;
    r.g_begin = r.g_end = r.total;
    r.cost0 = 0;
    if (c >= r.ctas_eff) return r;
    const long long T0 = sched_bound(r.cost, r.ctas_eff, c);
    const long long T1 = sched_bound(r.cost, r.ctas_eff, c + 1);
    SchedHit h0, h1;
    sched_find<2>(lens, B, Lmax, tile, segs_per_b, w, T0, T1, r.total, &h0, &h1);
    r.g_end = h1.g;
    r.g_begin = h0.g;
    r.cost0 = h0.cost0;
    r.b = h0.b;
    r.seg = h0.seg;
    r.t = h0.t;
    r.found = h0.g < r.total ? 1 : 0;
    return r;
}

// The combine record of CTA c, written by lane 0 of a whole calling warp:
// when c's range starts strictly inside a segment and c-1's range starts at
// or before that segment's start, c owns the merge of the segment's pieces
// -- the last piece of CTA c-1 (or its first, if c-1 started exactly at the
// segment start) and the first pieces of CTAs c .. c_last.  Written as
// {b, seg, first_slot, pieces}, or b = -1.
__device__ inline void sched_split_record(LenView lens, int B, int Lmax, int tile,
                                          int segs_per_b, SchedCost w, int c,
                                          const SchedStart &st, int *rec) {
    const int lane = threadIdx.x & 31;
    int r0 = -1, r1 = 0, r2 = 0, r3 = 0;
    if (st.found && c > 0 && st.t > 0 && c < st.ctas_eff) {
        const long long S0 = st.g_begin - st.t;  // the segment's first tile
        // CTA c-1 holds the segment's start iff that start's cost is not
        // below T(c-1)
        const long long Tp = sched_bound(st.cost, st.ctas_eff, c - 1);
        if (st.cost0 >= Tp) {
            SchedHit hp, unused;
            sched_find<1>(lens, B, Lmax, tile, segs_per_b, w, Tp, Tp, st.total, &hp, &unused);
            const int nt = seq_ntiles(lens[st.b], Lmax, tile, lens.window, lens.walign);
            const long long last_cost = st.cost0 + (nt == 1 ? 0 : w.P + (long long)kCostTile * (nt - 1));
            const int c_last = sched_owner(last_cost, st.cost, st.ctas_eff);
            r0 = st.b;
            r1 = st.seg;
            r2 = (hp.g == S0) ? 2 * (c - 1) : 2 * (c - 1) + 1;
            r3 = 1 + (c_last - c + 1);
        }
    }
    if (lane == 0) reinterpret_cast<int4 *>(rec)[c] = make_int4(r0, r1, r2, r3);
}

// Fused append, called by all 32 lanes of the producer warp before any TMA
// copy of the tile that holds row `pos`: write this step's K and V rows of
// (b, kvh) = z into that row of the caches, and make the writes visible to
// the tensor-copy (async) proxy.  Every CTA that loads the tile writes the
// row itself (head groups of one K/V head write identical bytes), so no
// reader depends on another CTA's write.
// Row src (b * Hkv + kvh) of k_new/v_new goes into cache row dst (a row
// index of the [.., D] view of the cache or pool).
__device__ __forceinline__ void append_row_warp(const DecodeParams &p, int src, size_t dst, int D,
                                                int lane) {
    const int vecs = D / 8;  // 16-byte vectors per row
    const uint4 *ks = reinterpret_cast<const uint4 *>(p.k_new) + (size_t)src * vecs;
    const uint4 *vs = reinterpret_cast<const uint4 *>(p.v_new) + (size_t)src * vecs;
    uint4 *kd = reinterpret_cast<uint4 *>(p.k_cache) + dst * vecs;
    uint4 *vd = reinterpret_cast<uint4 *>(p.v_cache) + dst * vecs;
    for (int i = lane; i < vecs; i += 32) {
        kd[i] = ks[i];
        vd[i] = vs[i];
    }
    asm volatile("fence.proxy.async.global;" ::: "memory");
    __syncwarp();
}

// Walks the tile list in the same order in every thread that uses it.
struct TileIter {
    LenView lens;
    int B, Lmax, tile, segs_per_b;
    int b, seg, t, nt, len;

    __device__ __forceinline__ void init(LenView lens_, int B_, int Lmax_, int tile_,
                                         int segs_per_b_, const SchedStart &s) {
        lens = lens_; B = B_; Lmax = Lmax_; tile = tile_; segs_per_b = segs_per_b_;
        b = s.b; seg = s.seg; t = s.t;
        len = lens[b];
        nt = seq_ntiles(len, Lmax, tile, lens.window, lens.walign);
    }
    __device__ __forceinline__ bool last_tile_of_segment() const { return t == nt - 1; }
    // First attended position of the current sequence, and the first
    // position that tile t adds.
    __device__ __forceinline__ int start() const {
        return seq_window_start(seq_valid_len(len, Lmax), lens.window, lens.walign);
    }
    __device__ __forceinline__ int first_pos() const { return start() + t * tile; }
    // First cache row of the tile's box.  A segment's last tile is moved back
    // to end exactly at the length (rows before 0 read as zeros; rows before
    // the tile's first new position are masked), so no tile ever covers rows
    // past the length: padding is never loaded.
    __device__ __forceinline__ int row0() const {
        return (t == nt - 1) ? seq_valid_len(len, Lmax) - tile : first_pos();
    }
    __device__ __forceinline__ void next() {
        if (++t < nt) return;
        t = 0;
        if (++seg < segs_per_b) return;
        seg = 0;
        if (++b < B) {
            len = lens[b];
            nt = seq_ntiles(len, Lmax, tile, lens.window, lens.walign);
        }
    }
};

}  // namespace kvattn
