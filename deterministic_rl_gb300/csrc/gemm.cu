// gemm.cu -- persistent, warp-specialised grouped GEMM on tcgen05/TMEM fed by
// TMA, with three fused epilogues: router logits (+bias, fp32), SwiGLU of the
// gate/up pair (bf16 H), and the down projection (bf16 routed rows, fp32
// shared-expert rows).
//
// The expert FFNs are the grouped GEMMs of the MoE layer in the Composer 2
// Technical Report, §6.1 "Training infrastructure" (Kernels paragraph,
// Fig. 10: one grouped GEMM per projection, experts as groups).  The fixed
// accumulation order asked for by the Training Data No. 94 write-up (section
// "浮点数不守规矩，MoE 火上浇油") is obtained by construction: every output
// element is produced by exactly one CTA, from one MMA instruction shape, with
// the K loop always run from 0 to K in BK steps into one TMEM accumulator;
// no split-K, no atomics, and the same schedule whatever the group sizes.
//
// Roles (192 threads, one CTA per SM, persistent over a static tile order):
//   warp 0      TMA producer (one elected lane)
//   warp 1      TMEM owner + MMA issuer (one elected lane)
//   warps 2..5  epilogue: TMEM -> registers -> global (lane quarter = warp % 4)
// Weights are the MMA's M side (128 rows per tile) and tokens the N side, so
// a weight tile is read once per 128 tokens of its expert.  This one-SM kernel
// serves the router and, for small batches, the expert GEMMs (its stages carry
// 32 KB of gate/up weights, which keeps HBM busy when weights are streamed);
// gemm_pair.cu serves the expert GEMMs of large batches.
#include <cuda_bf16.h>

#include "moe_internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kThreads = 192;
constexpr uint32_t kABytes = BM * BK * 2;
constexpr uint32_t kBBytes = BN * BK * 2;
constexpr uint32_t kBox32Bytes = 32 * BK * 2;
constexpr int kMaxGroups = 1024;

template <int MODE>
struct Cfg {
    static constexpr bool kDual = MODE == GEMM_SWIGLU;
    static constexpr int kStages = kDual ? 4 : 6;
    static constexpr uint32_t kStageBytes = kABytes * (kDual ? 2 : 1) + kBBytes;
    static constexpr int kAccCols = BN * (kDual ? 2 : 1);
    static constexpr uint32_t kTmemCols = kDual ? 512 : 256;
};

constexpr uint32_t kIdesc = idesc_bf16_f32(BM, BN);

struct Tile {
    int m, g, n_valid, brow, arow;
    bool shared;
};

__device__ __forceinline__ Tile decode_tile(int t, const GemmParams& p, const int* tile_start,
                                            const int* gcnt, const int* goff, int GG) {
    Tile tl;
    tl.m = t % p.MT;
    const int j = t / p.MT;
    int lo = 0, hi = GG;  // find g with tile_start[g] <= j < tile_start[g+1]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (tile_start[mid] <= j) lo = mid; else hi = mid;
    }
    tl.g = lo;
    const int nt = j - tile_start[lo];
    tl.n_valid = min(BN, gcnt[lo] - nt * BN);
    tl.brow = goff[lo] + nt * BN;
    tl.shared = lo >= p.G;
    tl.arow = (tl.shared ? 0 : lo * p.M) + tl.m * BM;
    return tl;
}

__device__ __forceinline__ void raise_timeout(const GemmParams& p, volatile int* abort, int where) {
    atomicOr(p.status, STATUS_TIMEOUT);
    atomicMax(p.status + 1, where);
    *abort = 1;
}

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1) grouped_gemm_kernel(const __grid_constant__ GemmParams p) {
    using C = Cfg<MODE>;
    extern __shared__ uint8_t smem_raw[];
    // Offsetting the shared array itself (never through an integer) keeps every
    // derived pointer in the shared address space, so that accesses through
    // them compile to shared-memory loads and stores, not generic ones.
    uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kStages * C::kStageBytes);
    uint64_t* empty = full + C::kStages;
    uint64_t* tfull = empty + C::kStages;
    uint64_t* tempty = tfull + 2;
    uint64_t* drain = tempty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);
    int* tile_start = reinterpret_cast<int*>(tmem_slot + 4);
    const int GG = p.G + p.has_shared;
    int* gcnt = tile_start + GG + 1;
    int* goff = gcnt + GG;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (warp == 0) {
        // Group table: rows, B offset and exclusive prefix of n-tiles per group.
        const int per = (GG + 31) / 32;
        const int g0 = lane * per;
        int local = 0;
        for (int g = g0; g < min(g0 + per, GG); ++g) {
            int c, o;
            if (g < p.G) {
                c = p.cnt ? p.cnt[g] : p.n_single;
                o = p.off ? p.off[g] : 0;
            } else {
                c = p.shared_rows;
                o = p.shared_b_off;
            }
            gcnt[g] = c;
            goff[g] = o;
            local += (c + BN - 1) / BN;
        }
        int incl = local;
#pragma unroll
        for (int s = 1; s < 32; s <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, s);
            if (lane >= s) incl += v;
        }
        int run = incl - local;
        for (int g = g0; g < min(g0 + per, GG); ++g) {
            tile_start[g] = run;
            run += (gcnt[g] + BN - 1) / BN;
        }
        if (lane == 31) tile_start[GG] = incl;
    } else if (warp == 1) {
        tmem_alloc(tmem_slot, C::kTmemCols);
        tmem_relinquish();
    } else if (threadIdx.x == 64) {
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&tfull[a], 1);
            mbar_init(&tempty[a], 4);
        }
        mbar_init(drain, 1);
        *abort = 0;
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // Fixed K split (router): tile t covers K part t % S of output tile t / S.
    const int S = p.ksplit > 1 ? p.ksplit : 1;
    const int KBs = p.KB / S;
    const int total = tile_start[GG] * p.MT * S;
    const uint64_t tmo = p.timeout_ns;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer ----------------
            tma_prefetch_desc(&p.a0);
            tma_prefetch_desc(&p.b);
            if (p.has_shared) tma_prefetch_desc(&p.as0);
            const uint64_t pol_w = l2_policy_evict_first();
            const uint64_t pol_x = l2_policy_evict_last();
            int stage = 0;
            uint32_t phase = 0;
            uint32_t issued = 0, last_par = 0;  // per-stage bit masks
            bool ok = p.stall_test == 0;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
                const Tile tl = decode_tile(t / S, p, tile_start, gcnt, goff, GG);
                const int kb0 = (t % S) * KBs;
                const CUtensorMap* ma0 = tl.shared ? &p.as0 : &p.a0;
                const CUtensorMap* ma1 = tl.shared ? &p.as1 : &p.a1;
                // Token rows: the whole box, or only the 32-row boxes in use.
                const int nbox = (tl.n_valid + 31) >> 5;
                const bool part = p.partial_b && nbox < BN / 32;
                const uint32_t stage_bytes = C::kStageBytes - kBBytes + (part ? nbox * kBox32Bytes : kBBytes);
                for (int kb = kb0; kb < kb0 + KBs; ++kb) {
                    if (!mbar_wait(&empty[stage], phase ^ 1u, abort, tmo)) {
                        if (!*abort) raise_timeout(p, abort, 1);
                        ok = false;
                        break;
                    }
                    uint8_t* st = smem + stage * C::kStageBytes;
                    mbar_arrive_expect_tx(&full[stage], stage_bytes);
                    tma_load_2d(st, ma0, &full[stage], kb * BK, tl.arow, pol_w);
                    if constexpr (C::kDual)
                        tma_load_2d(st + kABytes, ma1, &full[stage], kb * BK, tl.arow, pol_w);
                    uint8_t* sb = st + kABytes * (C::kDual ? 2 : 1);
                    if (part) {
                        for (int i = 0; i < nbox; ++i)
                            tma_load_2d(sb + i * kBox32Bytes, &p.b32, &full[stage], kb * BK,
                                        tl.brow + 32 * i, pol_x);
                    } else {
                        tma_load_2d(sb, &p.b, &full[stage], kb * BK, tl.brow, pol_x);
                    }
                    issued |= 1u << stage;
                    last_par = (last_par & ~(1u << stage)) | (phase << stage);
                    if (++stage == C::kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            // Copies in flight must land before the CTA may exit.
            for (int s = 0; s < C::kStages; ++s)
                if (issued & (1u << s)) {
                    if (!mbar_wait(&full[s], (last_par >> s) & 1u, nullptr, tmo))
                        raise_timeout(p, abort, 2);
                }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------- MMA issuer ----------------
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
                if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, abort, tmo)) {
                    if (!*abort) raise_timeout(p, abort, 3);
                    break;
                }
                tc_fence_after();
                const uint32_t d0 = tmem_base + acc * C::kAccCols;
                for (int kb = 0; kb < KBs; ++kb) {
                    if (!mbar_wait(&full[stage], phase, abort, tmo)) {
                        if (!*abort) raise_timeout(p, abort, 4);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = smem_addr(smem + stage * C::kStageBytes);
                    const uint32_t sb = sa + kABytes * (C::kDual ? 2 : 1);
#pragma unroll
                    for (int k = 0; k < BK / 16; ++k) {
                        const uint32_t accum = (kb | k) != 0;
                        umma_bf16(d0, sdesc_kmajor_sw128(sa + k * 32), sdesc_kmajor_sw128(sb + k * 32),
                                  kIdesc, accum);
                        if constexpr (C::kDual)
                            umma_bf16(d0 + BN, sdesc_kmajor_sw128(sa + kABytes + k * 32),
                                      sdesc_kmajor_sw128(sb + k * 32), kIdesc, accum);
                    }
                    umma_commit(&empty[stage]);
                    if (++stage == C::kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                umma_commit(&tfull[acc]);
                if (++acc == 2) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
            }
            // All MMAs issued by this thread complete before TMEM is freed.
            umma_commit(drain);
            if (!mbar_wait(drain, 0, nullptr, tmo)) raise_timeout(p, abort, 5);
        }
    } else {
        // ---------------- epilogue (warps 2..5) ----------------
        const int q = warp & 3;
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int t = blockIdx.x; t < total; t += gridDim.x) {
            const Tile tl = decode_tile(t / S, p, tile_start, gcnt, goff, GG);
            // The lanes decide together: tcgen05.ld below needs the whole warp.
            const bool ready = __all_sync(0xffffffffu, mbar_wait(&tfull[acc], acc_phase, abort, tmo));
            if (!ready) {
                if (lane == 0 && !*abort) raise_timeout(p, abort, 6);
                break;
            }
            tc_fence_after();
            const int row = tl.m * BM + q * 32 + lane;  // weight row: e, f or i
            const bool row_ok = row < p.M;
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * C::kAccCols;
            for (int c0 = 0; c0 < tl.n_valid; c0 += 32) {
                float v[32];
                tmem_ld32(taddr + c0, v);
                if constexpr (MODE == GEMM_SWIGLU) {
                    float u[32];
                    tmem_ld32(taddr + BN + c0, u);
                    tmem_ld_wait();
                    __nv_bfloat16* H = static_cast<__nv_bfloat16*>(p.out);
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        if (row_ok && c0 + j < tl.n_valid) {
                            const float g = v[j];
                            const float h = swiglu(g, u[j]);
                            H[static_cast<int64_t>(tl.brow + c0 + j) * p.ldo + row] = __float2bfloat16_rn(h);
                        }
                    }
                } else if constexpr (MODE == GEMM_ROUTER) {
                    tmem_ld_wait();
                    float* L = static_cast<float*>(p.out) + (t % S) * p.split_stride;
                    const float b = (row_ok && p.bias) ? p.bias[row] : 0.0f;
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if (row_ok && c0 + j < tl.n_valid)
                            L[static_cast<int64_t>(tl.brow + c0 + j) * p.ldo + row] = v[j] + b;
                } else {
                    tmem_ld_wait();
                    if (tl.shared) {
                        float* Ys = static_cast<float*>(p.out_shared);
                        const int tok0 = tl.brow - p.shared_b_off + c0;
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            if (row_ok && c0 + j < tl.n_valid)
                                Ys[static_cast<int64_t>(tok0 + j) * p.ldo + row] = v[j];
                    } else {
                        __nv_bfloat16* Y = static_cast<__nv_bfloat16*>(p.out);
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            if (row_ok && c0 + j < tl.n_valid)
                                Y[static_cast<int64_t>(tl.brow + c0 + j) * p.ldo + row] =
                                    __float2bfloat16_rn(v[j]);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[acc]);
            if (++acc == 2) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, C::kTmemCols);
    }
}

template <int MODE>
size_t smem_bytes_for(int GG) {
    using C = Cfg<MODE>;
    return 1024 + C::kStages * C::kStageBytes + (2 * C::kStages + 5) * 8 + 16 +
           static_cast<size_t>(3 * GG + 1) * 4;
}

template <int MODE>
cudaError_t launch_mode(const GemmParams& p, int grid, cudaStream_t s) {
    const int GG = p.G + p.has_shared;
    const size_t smem = smem_bytes_for<MODE>(GG);
    cudaError_t e = cudaFuncSetAttribute(grouped_gemm_kernel<MODE>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    grouped_gemm_kernel<MODE><<<grid, kThreads, smem, s>>>(p);
    return cudaGetLastError();
}

}  // namespace

size_t gemm_smem_bytes(int mode, int GG) {
    switch (mode) {
        case GEMM_ROUTER: return smem_bytes_for<GEMM_ROUTER>(GG);
        case GEMM_SWIGLU: return smem_bytes_for<GEMM_SWIGLU>(GG);
        default: return smem_bytes_for<GEMM_DOWN>(GG);
    }
}

cudaError_t launch_grouped_gemm(int mode, const GemmParams& p, int grid, cudaStream_t s) {
    if (p.G + p.has_shared > kMaxGroups || grid <= 0) return cudaErrorInvalidValue;
    switch (mode) {
        case GEMM_ROUTER: return launch_mode<GEMM_ROUTER>(p, grid, s);
        case GEMM_SWIGLU: return launch_mode<GEMM_SWIGLU>(p, grid, s);
        case GEMM_DOWN: return launch_mode<GEMM_DOWN>(p, grid, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace moe
