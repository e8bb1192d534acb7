// dispatch.cu -- deterministic stable counting sort of the (token, slot) pairs
// by expert id, and the gather of token rows into expert order.
//
// On one GPU the token dispatch of the Composer 2 Technical Report, §6.1
// "Training infrastructure" (tokens dispatched to their experts, combined back
// afterwards) is a grouping of the pairs i = t*k + s by expert.  Positions are
// a pure function of the ids: dst(i) = off[e] + #{i' < i : id(i') = e}, built
// from per-segment histograms, a segment-order scan and in-order ranks from
// warp match masks -- no position ever depends on the order of atomics.
#include <cstdint>

#include "moe_internal.h"

namespace moe {
namespace {

constexpr int kSegPairs = 4096;  // pairs per segment (one CTA)
constexpr int kSegWarps = 8;     // each warp ranks 512 consecutive pairs
constexpr int kWarpPairs = kSegPairs / kSegWarps;
constexpr int kMaxE = 512;

// Pass 1: per-segment, per-warp histograms.  hist[seg][w][e].
__global__ void __launch_bounds__(32 * kSegWarps) seg_hist_kernel(const int32_t* __restrict__ ids,
                                                                  int64_t n, int E,
                                                                  int32_t* __restrict__ hist) {
    __shared__ int32_t h[kSegWarps][kMaxE];
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int i = threadIdx.x; i < kSegWarps * kMaxE; i += blockDim.x) (&h[0][0])[i] = 0;
    __syncthreads();
    const int64_t base = static_cast<int64_t>(blockIdx.x) * kSegPairs + w * kWarpPairs;
    for (int r = 0; r < kWarpPairs; r += 32) {
        const int64_t i = base + r + lane;
        const bool in = i < n;
        const int key = in ? ids[i] : -1;
        const uint32_t act = __ballot_sync(0xffffffffu, in);
        if (in) {
            const uint32_t peers = __match_any_sync(act, key);
            if ((__ffs(peers) - 1) == lane) h[w][key] += __popc(peers);
        }
        __syncwarp();
    }
    __syncthreads();
    int32_t* out = hist + static_cast<int64_t>(blockIdx.x) * kSegWarps * E;
    for (int i = threadIdx.x; i < kSegWarps * E; i += blockDim.x) out[i] = h[i / E][i % E];
}

// Pass 2 (one CTA): cnt[e], off[e] (exclusive over e), and each (segment, warp)
// base position base[seg][w][e] = off[e] + pairs of e in earlier (seg, w).
__global__ void __launch_bounds__(kMaxE) seg_scan_kernel(int32_t* __restrict__ hist, int nseg, int E,
                                                         int32_t* __restrict__ cnt,
                                                         int32_t* __restrict__ off) {
    __shared__ int32_t tot[kMaxE];
    __shared__ int32_t warp_sums[kMaxE / 32];
    const int e = threadIdx.x;
    int32_t run = 0;
    // nseg * kSegWarps entries per expert, a multiple of kSegWarps: eight loads
    // are issued before their eight stores, the running sum kept in order
    if (e < E) {
        for (int sw0 = 0; sw0 < nseg * kSegWarps; sw0 += kSegWarps) {
            int32_t c[kSegWarps];
#pragma unroll
            for (int u = 0; u < kSegWarps; ++u) c[u] = hist[static_cast<int64_t>(sw0 + u) * E + e];
#pragma unroll
            for (int u = 0; u < kSegWarps; ++u) {
                hist[static_cast<int64_t>(sw0 + u) * E + e] = run;
                run += c[u];
            }
        }
    }
    tot[e] = e < E ? run : 0;
    __syncthreads();
    // exclusive scan of tot over e (E <= 512): warp scans, then warp totals
    const int lane = e & 31, w = e >> 5;
    int32_t incl = tot[e];
#pragma unroll
    for (int s = 1; s < 32; s <<= 1) {
        const int32_t v = __shfl_up_sync(0xffffffffu, incl, s);
        if (lane >= s) incl += v;
    }
    if (lane == 31) warp_sums[w] = incl;
    __syncthreads();
    int32_t wbase = 0;
    for (int i = 0; i < w; ++i) wbase += warp_sums[i];
    const int32_t excl = wbase + incl - tot[e];
    if (e < E) {
        cnt[e] = tot[e];
        off[e] = excl;
        if (e == E - 1) off[E] = excl + tot[e];
        for (int sw0 = 0; sw0 < nseg * kSegWarps; sw0 += kSegWarps) {
            int32_t c[kSegWarps];
#pragma unroll
            for (int u = 0; u < kSegWarps; ++u) c[u] = hist[static_cast<int64_t>(sw0 + u) * E + e];
#pragma unroll
            for (int u = 0; u < kSegWarps; ++u) hist[static_cast<int64_t>(sw0 + u) * E + e] = c[u] + excl;
        }
    }
}

// Pass 3: in-order ranks inside each warp's 512 pairs; perm[dst] = i, inv[i] = dst.
__global__ void __launch_bounds__(32 * kSegWarps) seg_scatter_kernel(
    const int32_t* __restrict__ ids, int64_t n, int E, const int32_t* __restrict__ base_pos,
    int32_t* __restrict__ perm, int32_t* __restrict__ inv) {
    __shared__ int32_t pos[kSegWarps][kMaxE];
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int32_t* b = base_pos + static_cast<int64_t>(blockIdx.x) * kSegWarps * E;
    for (int i = threadIdx.x; i < kSegWarps * E; i += blockDim.x) pos[i / E][i % E] = b[i];
    __syncthreads();
    const int64_t base = static_cast<int64_t>(blockIdx.x) * kSegPairs + w * kWarpPairs;
    for (int r = 0; r < kWarpPairs; r += 32) {
        const int64_t i = base + r + lane;
        const bool in = i < n;
        const int key = in ? ids[i] : -1;
        const uint32_t act = __ballot_sync(0xffffffffu, in);
        if (in) {
            const uint32_t peers = __match_any_sync(act, key);
            const int rank = __popc(peers & ((1u << lane) - 1u));
            const int32_t dst = pos[w][key] + rank;
            perm[dst] = static_cast<int32_t>(i);
            inv[i] = dst;
            __syncwarp(act);
            if ((__ffs(peers) - 1) == lane) pos[w][key] += __popc(peers);
        }
        __syncwarp();
    }
}

// All three passes in one CTA, for at most one segment of pairs (n <= 4096):
// the decode-sized case, where three launches would cost more than the work.
__global__ void __launch_bounds__(32 * kSegWarps) dispatch_small_kernel(
    const int32_t* __restrict__ ids, int64_t n, int E, int32_t* __restrict__ cnt,
    int32_t* __restrict__ off, int32_t* __restrict__ perm, int32_t* __restrict__ inv) {
    __shared__ int32_t h[kSegWarps][kMaxE];
    __shared__ int32_t warp_tot[kSegWarps];
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int i = threadIdx.x; i < kSegWarps * kMaxE; i += blockDim.x) (&h[0][0])[i] = 0;
    __syncthreads();
    // each warp takes an equal run of consecutive pairs (a multiple of 32):
    // both passes below use the same runs, in warp order, so ranks stay in
    // pair order
    const int per = static_cast<int>((n + 32 * kSegWarps - 1) / (32 * kSegWarps)) * 32;
    const int64_t base = static_cast<int64_t>(w) * per;
    for (int r = 0; r < per; r += 32) {  // per-warp histograms
        const int64_t i = base + r + lane;
        const bool in = i < n;
        const int key = in ? ids[i] : -1;
        const uint32_t act = __ballot_sync(0xffffffffu, in);
        if (in) {
            const uint32_t peers = __match_any_sync(act, key);
            if ((__ffs(peers) - 1) == lane) h[w][key] += __popc(peers);
        }
        __syncwarp();
    }
    __syncthreads();
    // exclusive scan over experts: thread handles experts 2*tid, 2*tid + 1
    const int e0 = 2 * threadIdx.x;
    int32_t c0 = 0, c1 = 0;
    for (int ww = 0; ww < kSegWarps; ++ww) {
        if (e0 < E) c0 += h[ww][e0];
        if (e0 + 1 < E) c1 += h[ww][e0 + 1];
    }
    int32_t incl = c0 + c1;
#pragma unroll
    for (int s = 1; s < 32; s <<= 1) {
        const int32_t v = __shfl_up_sync(0xffffffffu, incl, s);
        if (lane >= s) incl += v;
    }
    if (lane == 31) warp_tot[w] = incl;
    __syncthreads();
    int32_t wbase = 0;
    for (int ww = 0; ww < w; ++ww) wbase += warp_tot[ww];
    const int32_t ex0 = wbase + incl - c0 - c1;
    const int32_t ex1 = ex0 + c0;
    __syncthreads();
    // per (warp, expert) start positions, in place of the histograms
    for (int j = 0; j < 2; ++j) {
        const int e = e0 + j;
        if (e >= E) continue;
        int32_t run = j ? ex1 : ex0;
        cnt[e] = j ? c1 : c0;
        off[e] = run;
        if (e == E - 1) off[E] = run + (j ? c1 : c0);
        for (int ww = 0; ww < kSegWarps; ++ww) {
            const int32_t c = h[ww][e];
            h[ww][e] = run;
            run += c;
        }
    }
    __syncthreads();
    for (int r = 0; r < per; r += 32) {  // in-order ranks
        const int64_t i = base + r + lane;
        const bool in = i < n;
        const int key = in ? ids[i] : -1;
        const uint32_t act = __ballot_sync(0xffffffffu, in);
        if (in) {
            const uint32_t peers = __match_any_sync(act, key);
            const int rank = __popc(peers & ((1u << lane) - 1u));
            const int32_t dst = h[w][key] + rank;
            perm[dst] = static_cast<int32_t>(i);
            inv[i] = dst;
            __syncwarp(act);
            if ((__ffs(peers) - 1) == lane) h[w][key] += __popc(peers);
        }
        __syncwarp();
    }
}

// Gather, in token order: token t's row of x is read once and stored to
// xp[inv[t*k + s]] for s = 0 .. k-1 (its rows in expert order) and, for the
// shared expert, to xp[T*k + t].  16-byte vectors; d % 8 == 0.  scale_out
// (NVFP4) receives the token's scale at the same rows.
constexpr int kGatherMaxK = 16;

__global__ void __launch_bounds__(256) gather_rows_kernel(
    const uint4* __restrict__ x, const int32_t* __restrict__ inv, int64_t T, int k,
    int vec_per_row, int n_shared, uint4* __restrict__ xp, const float* __restrict__ scale_in,
    float* __restrict__ scale_out) {
    __shared__ int64_t dst[kGatherMaxK + 1];
    const int64_t Tk = T * k;
    const int nd = k + (n_shared ? 1 : 0);
    for (int64_t t = blockIdx.x; t < T; t += gridDim.x) {
        if (threadIdx.x < nd)
            dst[threadIdx.x] = threadIdx.x < k ? static_cast<int64_t>(inv[t * k + threadIdx.x])
                                               : Tk + t;
        __syncthreads();
        const uint4* src = x + t * vec_per_row;
        for (int v = threadIdx.x; v < vec_per_row; v += blockDim.x) {
            const uint4 val = src[v];
            for (int j = 0; j < nd; ++j) xp[dst[j] * vec_per_row + v] = val;
        }
        if (scale_out && threadIdx.x < nd) scale_out[dst[threadIdx.x]] = scale_in[t];
        __syncthreads();
    }
}

}  // namespace

size_t dispatch_scratch_bytes(int64_t n_pairs, int E) {
    const int64_t nseg = (n_pairs + kSegPairs - 1) / kSegPairs;
    return static_cast<size_t>((nseg > 0 ? nseg : 1) * kSegWarps * E) * sizeof(int32_t);
}

cudaError_t launch_dispatch(const int32_t* ids, int64_t T, int k, int E, int32_t* cnt,
                            int32_t* off, int32_t* perm, int32_t* inv, int32_t* scratch,
                            cudaStream_t s) {
    if (E > kMaxE) return cudaErrorInvalidValue;
    const int64_t n = T * k;
    const int nseg = static_cast<int>((n + kSegPairs - 1) / kSegPairs);
    if (nseg == 1) {
        dispatch_small_kernel<<<1, 32 * kSegWarps, 0, s>>>(ids, n, E, cnt, off, perm, inv);
        return cudaGetLastError();
    }
    if (nseg > 0) {
        seg_hist_kernel<<<nseg, 32 * kSegWarps, 0, s>>>(ids, n, E, scratch);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    seg_scan_kernel<<<1, kMaxE, 0, s>>>(scratch, nseg, E, cnt, off);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || nseg == 0) return e;
    seg_scatter_kernel<<<nseg, 32 * kSegWarps, 0, s>>>(ids, n, E, scratch, perm, inv);
    return cudaGetLastError();
}

cudaError_t launch_gather(const uint16_t* x, const int32_t* inv, int64_t T, int k, int d,
                          int n_shared, uint16_t* xp, cudaStream_t s, const float* scale_in,
                          float* scale_out) {
    if (k > kGatherMaxK || d % 8) return cudaErrorInvalidValue;
    if (T == 0) return cudaSuccess;
    const int vpr = d / 8;
    const int64_t grid = T < 148 * 16 ? T : 148 * 16;
    gather_rows_kernel<<<static_cast<unsigned>(grid), 256, 0, s>>>(
        reinterpret_cast<const uint4*>(x), inv, T, k, vpr, n_shared, reinterpret_cast<uint4*>(xp),
        scale_in, scale_out);
    return cudaGetLastError();
}

namespace {

// One thread per 16 bytes of the packed output: packed row ((g * F/64 + b) * 128
// + i) is row 64 b + (i % 64) of gate[g] (i < 64) or of up[g] (i >= 64).
__global__ void __launch_bounds__(256) pack_gate_up_kernel(const uint4* __restrict__ gate,
                                                           const uint4* __restrict__ up,
                                                           uint4* __restrict__ out, int64_t nmat,
                                                           int F, int d) {
    const int q = d / 8;  // uint4 per row
    const int64_t rows = nmat * 2 * F;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < rows * q;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t prow = i / q;
        const int c = static_cast<int>(i % q);
        const int64_t blk = prow / 128;   // g * F/64 + b
        const int r = static_cast<int>(prow % 128);
        const int64_t g = blk / (F / 64);
        const int b = static_cast<int>(blk % (F / 64));
        const int64_t srow = g * F + 64 * b + (r & 63);
        out[i] = (r < 64 ? gate : up)[srow * q + c];
    }
}

}  // namespace

cudaError_t launch_pack_gate_up(const uint16_t* gate, const uint16_t* up, int64_t nmat, int F,
                                int d, uint16_t* packed, cudaStream_t s) {
    if (F % 64 || d % 8) return cudaErrorInvalidValue;
    const int64_t n = nmat * 2 * F * (d / 8);
    if (n == 0) return cudaSuccess;
    int64_t blocks = (n + 255) / 256;
    if (blocks > 65536) blocks = 65536;
    pack_gate_up_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(
        reinterpret_cast<const uint4*>(gate), reinterpret_cast<const uint4*>(up),
        reinterpret_cast<uint4*>(packed), nmat, F, d);
    return cudaGetLastError();
}

}  // namespace moe
