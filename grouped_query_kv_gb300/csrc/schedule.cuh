// schedule.cuh -- the persistent grid's split of the flat tile list.
//
// Every segment (b, kvh, hg) owns ntiles(len_b) tiles; the list of all tiles
// in (b, kvh, hg, t) order is cut into ctas_eff = min(gridDim.x, total)
// contiguous ranges [c*total/ctas_eff, (c+1)*total/ctas_eff).  Because
// ctas_eff <= total, every range is non-empty.  Lengths live on the device,
// so each CTA locates its own start with a block-wide scan over seq_lens (no
// host synchronisation; ragged batches balance to within one tile per CTA).
#pragma once

#include <cstdint>
#include "internal.h"

namespace kvattn {

// Lengths as the kernels see them.  For the fused append-then-attend step the
// array holds the number of tokens cached BEFORE this step's token, and the
// attention covers one more position; a negative entry stays invalid.
struct LenView {
    const int32_t *p;
    int add;  // 0: attention lengths as given; 1: cached-before counts (+1)
    __device__ __forceinline__ int operator[](int b) const {
        const int r = p[b];
        return add ? (r < 0 ? -1 : r + 1) : r;
    }
};

// A sequence whose length is outside [1, Lmax] still owns one tile, with no
// valid positions (zero output row; out-of-range lengths also raise the
// device error word).
__device__ __forceinline__ int seq_ntiles(int len, int Lmax, int tile) {
    return (len <= 0 || len > Lmax) ? 1 : (len + tile - 1) / tile;
}

__device__ __forceinline__ int seq_valid_len(int len, int Lmax) {
    return (len < 0 || len > Lmax) ? 0 : len;
}

struct SchedStart {
    long long total;    // tiles in the whole call
    long long g_begin;  // this CTA's first tile
    long long g_end;    // one past its last tile
    int ctas_eff;
    int found;          // 1 if this CTA has work
    int b, seg, t;      // coordinates of g_begin: sequence, segment within b, tile
};

struct SchedScratch {
    long long part[32];
    SchedStart res;
};

__device__ __forceinline__ long long warp_sum_ll(long long v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ long long warp_incl_scan_ll(long long v) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        long long n = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += n;
    }
    return v;
}

// Locate CTA `c`'s tile range.  Every thread of the block must call it
// (blockDim.x a multiple of 32, at most 1024); the result is left in sh->res.
__device__ inline void sched_locate(LenView lens, int B, int Lmax, int tile,
                             int segs_per_b, int c, int grid, SchedScratch *sh) {
    const int tid = threadIdx.x, nthr = blockDim.x;
    const int lane = tid & 31, warp = tid >> 5, nwarps = nthr >> 5;

    long long mine = 0;
    for (int b = tid; b < B; b += nthr) mine += seq_ntiles(lens[b], Lmax, tile);
    mine = warp_sum_ll(mine);
    if (lane == 0) sh->part[warp] = mine;
    __syncthreads();
    if (tid == 0) {
        long long tot = 0;
        for (int w = 0; w < nwarps; ++w) tot += sh->part[w];
        tot *= segs_per_b;
        SchedStart r;
        r.total = tot;
        r.ctas_eff = (int)(tot < (long long)grid ? tot : (long long)grid);
        r.found = 0;
        r.b = r.seg = r.t = 0;
        if (c < r.ctas_eff) {
            r.g_begin = (long long)c * tot / r.ctas_eff;
            r.g_end = (long long)(c + 1) * tot / r.ctas_eff;
        } else {
            r.g_begin = r.g_end = tot;
        }
        sh->res = r;
    }
    __syncthreads();
    const long long g_begin = sh->res.g_begin;
    const bool active = c < sh->res.ctas_eff;
    __syncthreads();
    if (!active) return;

    long long carry = 0;
    for (int base = 0; base < B; base += nthr) {
        const int b = base + tid;
        const int nt = (b < B) ? seq_ntiles(lens[b], Lmax, tile) : 0;
        const long long v = (long long)nt * segs_per_b;
        const long long incl = warp_incl_scan_ll(v);
        if (lane == 31) sh->part[warp] = incl;
        __syncthreads();
        long long woff = 0, chunk = 0;
        for (int w = 0; w < nwarps; ++w) {
            const long long pw = sh->part[w];
            if (w < warp) woff += pw;
            chunk += pw;
        }
        const long long excl = carry + woff + incl - v;
        if (b < B && excl <= g_begin && g_begin < excl + v) {
            const long long rem = g_begin - excl;
            sh->res.b = b;
            sh->res.seg = (int)(rem / nt);
            sh->res.t = (int)(rem % nt);
            sh->res.found = 1;
        }
        __syncthreads();
        carry += chunk;
        if (carry > g_begin) break;  // uniform: carry is the same in every thread
    }
    __syncthreads();
}

// Warp-level variant of sched_locate: every warp of a CTA can locate the
// CTA's range on its own, without block barriers, so the TMA producer can
// start as soon as the lengths have been read.  Same result as sched_locate.
__device__ inline SchedStart warp_locate(LenView lens, int B, int Lmax,
                                         int tile, int segs_per_b, int c, int grid) {
    const int lane = threadIdx.x & 31;
    long long mine = 0;
    for (int b = lane; b < B; b += 32) mine += seq_ntiles(lens[b], Lmax, tile);
    const long long tot = warp_sum_ll(mine) * segs_per_b;
    SchedStart r;
    r.total = tot;
    r.ctas_eff = (int)(tot < (long long)grid ? tot : (long long)grid);
    r.found = 0;
    r.b = r.seg = r.t = 0;
    r.g_begin = r.g_end = tot;
    if (c >= r.ctas_eff) return r;
    r.g_begin = (long long)c * tot / r.ctas_eff;
    r.g_end = (long long)(c + 1) * tot / r.ctas_eff;
    long long carry = 0;
    for (int base = 0; base < B; base += 32) {
        const int b = base + lane;
        const int nt = (b < B) ? seq_ntiles(lens[b], Lmax, tile) : 0;
        const long long v = (long long)nt * segs_per_b;
        const long long incl = warp_incl_scan_ll(v);
        const long long excl = carry + incl - v;
        const bool hit = (b < B) && excl <= r.g_begin && r.g_begin < excl + v;
        const unsigned m = __ballot_sync(0xffffffffu, hit);
        if (m) {
            const int src = __ffs(m) - 1;
            const long long rem = __shfl_sync(0xffffffffu, r.g_begin - excl, src);
            const int ntb = __shfl_sync(0xffffffffu, nt, src);
            r.b = base + src;
            r.seg = (int)(rem / ntb);
            r.t = (int)(rem % ntb);
            r.found = 1;
            break;
        }
        carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    return r;
}

// The combine record of CTA c: when c's range starts strictly inside a
// segment and c-1's range starts at or before that segment's start, c owns
// the merge of the segment's pieces -- the last piece of CTA c-1 (or its
// first, if c-1 started exactly at the segment start) and the first pieces
// of CTAs c .. c_last.  Written as {b, seg, first_slot, pieces}, or b = -1.
__device__ inline void sched_split_record(LenView lens, int Lmax, int tile,
                                          int c, const SchedStart &st, int *rec) {
    int r0 = -1, r1 = 0, r2 = 0, r3 = 0;
    if (st.found && c > 0 && st.t > 0 && c < st.ctas_eff) {
        const long long S0 = st.g_begin - st.t;
        const long long g_prev = (long long)(c - 1) * st.total / st.ctas_eff;
        if (g_prev <= S0) {
            const long long S1 = S0 + seq_ntiles(lens[st.b], Lmax, tile);
            const int c_last = (int)((S1 * st.ctas_eff - 1) / st.total);
            r0 = st.b;
            r1 = st.seg;
            r2 = (g_prev == S0) ? 2 * (c - 1) : 2 * (c - 1) + 1;
            r3 = 1 + (c_last - c + 1);
        }
    }
    reinterpret_cast<int4 *>(rec)[c] = make_int4(r0, r1, r2, r3);
}

// Fused append, called by all 32 lanes of the producer warp before any TMA
// copy of the tile that holds row `pos`: write this step's K and V rows of
// (b, kvh) = z into that row of the caches, and make the writes visible to
// the tensor-copy (async) proxy.  Every CTA that loads the tile writes the
// row itself (head groups of one K/V head write identical bytes), so no
// reader depends on another CTA's write.
__device__ __forceinline__ void append_row_warp(const DecodeParams &p, int z, int pos, int D,
                                                int lane) {
    const int vecs = D / 8;  // 16-byte vectors per row
    const uint4 *ks = reinterpret_cast<const uint4 *>(p.k_new) + (size_t)z * vecs;
    const uint4 *vs = reinterpret_cast<const uint4 *>(p.v_new) + (size_t)z * vecs;
    uint4 *kd = reinterpret_cast<uint4 *>(p.k_cache) + ((size_t)z * p.Lmax + pos) * vecs;
    uint4 *vd = reinterpret_cast<uint4 *>(p.v_cache) + ((size_t)z * p.Lmax + pos) * vecs;
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
        nt = seq_ntiles(len, Lmax, tile);
    }
    __device__ __forceinline__ bool last_tile_of_segment() const { return t == nt - 1; }
    // First cache row of the tile's box.  A segment's last tile is moved back
    // to end exactly at the length (rows before 0 read as zeros), so no tile
    // ever covers rows past the length: padding is never loaded.
    __device__ __forceinline__ int row0() const {
        return (t == nt - 1) ? seq_valid_len(len, Lmax) - tile : t * tile;
    }
    __device__ __forceinline__ void next() {
        if (++t < nt) return;
        t = 0;
        if (++seg < segs_per_b) return;
        seg = 0;
        if (++b < B) {
            len = lens[b];
            nt = seq_ntiles(len, Lmax, tile);
        }
    }
};

}  // namespace kvattn
