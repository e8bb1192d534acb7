// tile_walk.cuh -- the static tile order of the block-scaled expert GEMMs,
// walked incrementally.
//
// The tiles of one launch are (group g, weight tile m, token tile nt).  Groups
// with several token tiles ("hot") and with one ("cold") form two lists: hs[g]
// and cs[g] are the exclusive prefix sums of hot and cold token-tile counts
// (hs[GG], cs[GG] the totals), each list enumerated as (g, m, nt) with nt
// fastest, so the token tiles of a hot weight tile are consecutive.  Position t
// of the order (0 <= t < N, N = (hs[GG] + cs[GG]) * MT, H = hs[GG] * MT) is hot
// iff floor((t + 1) H / N) > floor(t H / N); then it is hot tile floor(t H / N),
// else cold tile t - floor(t H / N).  So every stretch of positions mixes
// tensor-bound and weight-streaming tiles in proportion.
//
// A CTA pair takes positions first, first + step, ...: the walker keeps
// floor(t H / N) and the remainder, and a cursor into each list, so a step
// costs a 32-bit division and a few comparisons instead of a 64-bit division
// and two binary searches.  Host and device code (tested on the host against
// the direct formula).
#pragma once

#include <cstdint>

#ifndef __CUDACC__
#define __host__
#define __device__
#define __forceinline__ inline
#endif

namespace moe {

struct TileWalk {
    int t;          // current position, -1 past the end
    uint32_t q, r;  // floor(t H / N), t H mod N
    int gh, gc;     // cursors: current group of the hot and of the cold list
};

struct TileOrder {
    const int* hs;  // [GG + 1]
    const int* cs;  // [GG + 1]
    int GG, MT;
    uint32_t H, N;  // hot positions, all positions
};

struct TilePos {
    int g, m, nt;
    bool hot;  // from the hot list (the group has several token tiles)
};

__host__ __device__ __forceinline__ TileWalk tile_walk_begin(int first, const TileOrder& o) {
    TileWalk w;
    w.gh = 0;
    w.gc = 0;
    if (first < 0 || static_cast<uint32_t>(first) >= o.N) {
        w.t = -1;
        w.q = w.r = 0;
        return w;
    }
    const uint64_t th = static_cast<uint64_t>(first) * o.H;
    w.t = first;
    w.q = static_cast<uint32_t>(th / o.N);
    w.r = static_cast<uint32_t>(th - static_cast<uint64_t>(w.q) * o.N);
    return w;
}

// Requires step * H + N < 2^32.
__host__ __device__ __forceinline__ void tile_walk_next(TileWalk& w, int step, const TileOrder& o) {
    if (w.t < 0) return;
    const int64_t nt = static_cast<int64_t>(w.t) + step;
    if (nt >= static_cast<int64_t>(o.N)) {
        w.t = -1;
        return;
    }
    const uint32_t rr = w.r + static_cast<uint32_t>(step) * o.H;
    w.q += rr / o.N;
    w.r = rr % o.N;
    w.t = static_cast<int>(nt);
}

// Moves the walker forward to position t (t >= its position; -1 or t >= N end
// it), for tiles handed out in increasing order with arbitrary gaps.
__host__ __device__ __forceinline__ void tile_walk_to(TileWalk& w, int t, const TileOrder& o) {
    if (t < 0 || static_cast<uint32_t>(t) >= o.N) {
        w.t = -1;
        return;
    }
    if (w.t < 0) {
        const int gh = w.gh, gc = w.gc;
        w = tile_walk_begin(t, o);
        w.gh = gh;
        w.gc = gc;
        return;
    }
    const uint64_t rr = w.r + static_cast<uint64_t>(t - w.t) * o.H;
    if (rr < (static_cast<uint64_t>(1) << 32)) {
        const uint32_t r32 = static_cast<uint32_t>(rr);
        w.q += r32 / o.N;
        w.r = r32 % o.N;
    } else {
        w.q += static_cast<uint32_t>(rr / o.N);
        w.r = static_cast<uint32_t>(rr % o.N);
    }
    w.t = t;
}

// The (group, weight tile, token tile) of the walker's position; moves the
// list cursors forward (positions must be visited in increasing order).
__host__ __device__ __forceinline__ TilePos tile_walk_pos(TileWalk& w, const TileOrder& o) {
    TilePos p;
    if (w.r + o.H >= o.N) {  // hot: hot tile q
        const int j = static_cast<int>(w.q);
        const int x = j / o.MT;
        while (w.gh + 1 < o.GG && o.hs[w.gh + 1] <= x) ++w.gh;
        const int ntg = o.hs[w.gh + 1] - o.hs[w.gh];
        const int l = j - o.hs[w.gh] * o.MT;
        p.g = w.gh;
        p.m = l / ntg;
        p.nt = l - p.m * ntg;
        p.hot = true;
    } else {  // cold: cold tile t - q
        const int j = w.t - static_cast<int>(w.q);
        const int x = j / o.MT;
        while (w.gc + 1 < o.GG && o.cs[w.gc + 1] <= x) ++w.gc;
        p.g = w.gc;
        p.m = j - o.cs[w.gc] * o.MT;
        p.nt = 0;
        p.hot = false;
    }
    return p;
}

}  // namespace moe
