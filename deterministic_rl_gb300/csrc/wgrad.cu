// wgrad.cu -- grouped weight-gradient GEMM of the MoE layer backward: for each
// expert group g,  W'[g][n][m] = sum over the group's tokens j of
//     A[m][j] * B[n][j],
// where A and B are token-major (transposed) activations whose columns are the
// group's tokens in dispatch order, padded with zeros to a multiple of 64 at
// column poff[g].  The contraction length differs per group (ragged K); the
// output shape does not.
//
// Composer 2 Technical Report, §6.1 "Training infrastructure" (Kernels,
// Fig. 10): the grouped expert GEMMs of the MoE training step; the backward's
// GEMM operands are MXFP8 (quantised by backward.cu along the token axis,
// stored as the exact bf16 values), multiplied here on tcgen05 with fp32
// accumulation in TMEM.
//
// Determinism: every output element is produced by one CTA pair, from one MMA
// shape, with its K loop run from the group's first token block to its last;
// no split-K, no atomics.
//
// SM pairs (clusters of 2, tcgen05 cta_group::2): a tile is M = 256 rows of A
// (the output's contiguous axis; 128 per CTA, in its TMEM lanes, so each
// epilogue store of a warp is one 128-byte row segment) by N = 256 rows of B
// (128 loaded by each CTA and read by the pair's MMA from both), so each SM
// takes 32 KB of operands per 64-deep k-block.  Tiles go to the pairs in a
// static order.
//
// Roles per CTA (192 threads, one CTA per SM, persistent):
//   warp 0      TMA producer (one elected lane; both CTAs load their halves,
//               completing on the leader's barrier)
//   warp 1      TMEM owner; MMA issuer in the leader CTA (one elected lane)
//   warps 2..5  epilogue: TMEM -> registers -> global (lane quarter = warp % 4)
#include <cuda_bf16.h>

#include "moe_internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kThreads = 192;
constexpr int WM = 256;          // A rows per pair tile (128 per CTA)
constexpr int WN = 256;          // B rows per pair tile (128 per CTA)
constexpr int kRowsCta = 128;
constexpr uint32_t kABytes = kRowsCta * BK * 2;
constexpr uint32_t kBBytes = kRowsCta * BK * 2;
constexpr uint32_t kStageBytes = kABytes + kBBytes;
constexpr int kStages = 6;
constexpr uint32_t kTmemCols = 2 * WN;
constexpr uint32_t kIdesc = idesc_bf16_f32(WM, WN);

struct WTile {
    int g, mt, nt, kb, k0;
};

__device__ __forceinline__ WTile decode(int t, const WgradParams& p, const int* poff) {
    WTile w;
    const int per = p.MT * p.NT;
    w.g = t / per;
    const int rem = t - w.g * per;
    w.nt = rem / p.MT;
    w.mt = rem - w.nt * p.MT;
    w.k0 = poff[w.g];
    w.kb = (poff[w.g + 1] - w.k0) / BK;
    return w;
}

__device__ __forceinline__ void raise_timeout(const WgradParams& p, volatile int* abort, int where) {
    atomicOr(p.status, STATUS_TIMEOUT);
    atomicMax(p.status + 1, where);
    *abort = 1;
}

__global__ void __launch_bounds__(kThreads, 1) wgrad_kernel(const __grid_constant__ WgradParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * kStageBytes);
    uint64_t* empty = full + kStages;
    uint64_t* tfull = empty + kStages;
    uint64_t* tempty = tfull + 2;
    uint64_t* drain = tempty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);
    int* poff = reinterpret_cast<int*>(tmem_slot + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;

    if (warp == 0) {
        for (int g = lane; g <= p.G; g += 32) poff[g] = p.poff[g];
    } else if (warp == 1) {
        tmem_alloc_pair(tmem_slot, kTmemCols);
        tmem_relinquish_pair();
    } else if (threadIdx.x == 64) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&tfull[a], 1);
            mbar_init(&tempty[a], 8);  // 4 epilogue warps in each of the two CTAs
        }
        mbar_init(drain, 1);
        *abort = 0;
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // barriers of both CTAs initialised before any remote use
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const int total = p.G * p.MT * p.NT;
    const int cid = static_cast<int>(cluster_id_x());
    const int ncl = static_cast<int>(nclusters_x());
    const uint64_t tmo = p.timeout_ns;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer (both CTAs) ----------------
            tma_prefetch_desc(&p.a);
            tma_prefetch_desc(&p.b);
            const uint64_t pol = l2_policy_evict_last();
            int stage = 0;
            uint32_t phase = 0;
            uint32_t issued = 0, last_par = 0;
            bool ok = p.stall_test == 0;
            for (int t = cid; t < total && ok; t += ncl) {
                const WTile w = decode(t, p, poff);
                const int arow = w.mt * WM + static_cast<int>(rank) * kRowsCta;
                const int brow = w.nt * WN + static_cast<int>(rank) * kRowsCta;
                for (int kb = 0; kb < w.kb; ++kb) {
                    if (!mbar_wait(&empty[stage], phase ^ 1u, abort, tmo)) {
                        if (!*abort) raise_timeout(p, abort, 41);
                        ok = false;
                        break;
                    }
                    uint8_t* st = smem + stage * kStageBytes;
                    if (leader) mbar_arrive_expect_tx(&full[stage], 2 * kStageBytes);
                    const uint32_t bar = map_to_rank(&full[stage], 0);
                    tma_load_2d_pair(st, &p.a, bar, w.k0 + kb * BK, arow, pol);
                    tma_load_2d_pair(st + kABytes, &p.b, bar, w.k0 + kb * BK, brow, pol);
                    issued |= 1u << stage;
                    last_par = (last_par & ~(1u << stage)) | (phase << stage);
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            // The leader's full barriers count both CTAs' copies: once they have
            // all completed, no copy of either CTA is in flight.
            if (leader)
                for (int s = 0; s < kStages; ++s)
                    if (issued & (1u << s)) {
                        if (!mbar_wait(&full[s], (last_par >> s) & 1u, nullptr, tmo))
                            raise_timeout(p, abort, 42);
                    }
        }
    } else if (warp == 1) {
        if (lane == 0 && leader) {
            // ---------------- MMA issuer (leader only) ----------------
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            for (int t = cid; t < total && ok; t += ncl) {
                const WTile w = decode(t, p, poff);
                if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, abort, tmo)) {
                    if (!*abort) raise_timeout(p, abort, 43);
                    break;
                }
                tc_fence_after();
                const uint32_t d0 = tmem_base + acc * WN;
                for (int kb = 0; kb < w.kb; ++kb) {
                    if (!mbar_wait(&full[stage], phase, abort, tmo)) {
                        if (!*abort) raise_timeout(p, abort, 44);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = smem_addr(smem + stage * kStageBytes);
                    const uint32_t sb = sa + kABytes;
#pragma unroll
                    for (int k = 0; k < BK / 16; ++k)
                        umma_bf16_pair(d0, sdesc_kmajor_sw128(sa + k * 32),
                                       sdesc_kmajor_sw128(sb + k * 32), kIdesc, (kb | k) != 0);
                    umma_commit_pair(&empty[stage], 0x3);
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                // a group without tokens issues no MMA: its epilogue writes zeros
                umma_commit_pair(&tfull[acc], 0x3);
                if (++acc == 2) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
            }
            umma_commit_pair(drain, 0x1);
            if (!mbar_wait(drain, 0, nullptr, tmo)) raise_timeout(p, abort, 45);
        }
    } else {
        // ---------------- epilogue (warps 2..5, both CTAs) ----------------
        const int q = warp & 3;
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int t = cid; t < total; t += ncl) {
            const WTile w = decode(t, p, poff);
            const bool ready = __all_sync(0xffffffffu, mbar_wait(&tfull[acc], acc_phase, abort, tmo));
            if (!ready) {
                if (lane == 0 && !*abort) raise_timeout(p, abort, 46);
                break;
            }
            tc_fence_after();
            const int m = w.mt * WM + static_cast<int>(rank) * kRowsCta + q * 32 + lane;
            const int n0 = w.nt * WN;
            // the tile lies wholly on one side of n_split (a multiple of WN)
            const bool hi = n0 >= p.n_split;
            const bool routed = w.g < p.G_routed;
            float* base = routed ? (hi ? p.out1 : p.out0) + static_cast<int64_t>(w.g) * p.gstride
                                 : (hi ? p.sout1 : p.sout0);
            float* o = base + static_cast<int64_t>(n0 - (hi ? p.n_split : 0)) * p.M + m;
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * WN;
            for (int c0 = 0; c0 < WN; c0 += 32) {
                float v[32];
                if (w.kb > 0) {
                    tmem_ld32(taddr + c0, v);
                    tmem_ld_wait();
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] = 0.0f;
                }
#pragma unroll
                for (int j = 0; j < 32; ++j) __stcs(o + static_cast<int64_t>(c0 + j) * p.M, v[j]);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(map_to_rank(&tempty[acc], 0));
            if (++acc == 2) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync();  // neither CTA leaves while the pair may still touch its memory
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, kTmemCols);
    }
}

size_t wgrad_smem(int G) {
    return 1024 + kStages * kStageBytes + (2 * kStages + 5) * 8 + 16 +
           static_cast<size_t>(G + 1) * 4;
}

}  // namespace

// grid = CTA pairs (clusters of 2)
cudaError_t launch_wgrad(const WgradParams& p, int clusters, cudaStream_t s) {
    if (p.G <= 0 || p.G > kMaxWgradGroups || clusters <= 0) return cudaErrorInvalidValue;
    if (p.M % WM || p.N != p.NT * WN || p.M != p.MT * WM || p.n_split % WN) return cudaErrorInvalidValue;
    const size_t smem = wgrad_smem(p.G);
    cudaError_t e = cudaFuncSetAttribute(wgrad_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * clusters, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int resident = 0;
    e = cudaOccupancyMaxActiveClusters(&resident, wgrad_kernel, &cfg);
    if (e != cudaSuccess) return e;
    if (resident <= 0) return cudaErrorInvalidConfiguration;
    if (clusters > resident) {
        clusters = resident;
        cfg.gridDim = dim3(2 * clusters, 1, 1);
    }
    return cudaLaunchKernelEx(&cfg, wgrad_kernel, p);
}

int wgrad_tile_m() { return WM; }
int wgrad_tile_n() { return WN; }
int wgrad_box_rows() { return kRowsCta; }

}  // namespace moe
