// gemm_pair.cu -- the expert GEMMs (gate/up + SwiGLU, down) on pairs of SMs:
// tcgen05.mma.cta_group::2 with M = 256 weight rows (128 in each CTA of a
// 2-CTA cluster) and N = 256 tokens (each CTA loads and holds 128 of them).
// Each SM thus loads 16 KB of weights and 16 KB of tokens per 64-wide K step
// for 4.2 MFLOP of MMA work, a third less operand traffic than a one-SM
// 128 x 256 tile, and a 32 KB pipeline stage leaves room for six stages.
//
// These are the grouped expert GEMMs of the Composer 2 Technical Report,
// §6.1 "Training infrastructure" (Fig. 10).  The fixed accumulation order of
// the Training Data No. 94 write-up (section "浮点数不守规矩，MoE 火上浇油")
// holds as in the one-SM kernel: one CTA pair produces each output element
// from one MMA shape (M = 256, N = 256, K = 16 steps in K order, one TMEM
// accumulator); no split-K, no atomics; the same schedule for every group size.
//
// Roles in each CTA (192 threads): warp 0 TMA producer; warp 1 TMEM owner and,
// in the pair's leader (cluster rank 0), the MMA issuer; warps 2..5 epilogue.
// The leader's "full" barrier counts the bytes both CTAs load; the leader's MMA
// completion is multicast to both CTAs' "empty" and "tmem full" barriers; both
// CTAs' epilogues arrive on the leader's "tmem empty" barrier.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "moe_internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kPairN = BN_EXPERT;                // tokens per pair tile (256)
constexpr int kHalfN = kPairN / 2;               // token rows held by each CTA
constexpr uint32_t kABytes = BM * BK * 2;        // 128 weight rows x 64 along K
constexpr uint32_t kBBytes = kHalfN * BK * 2;    // 128 token rows x 64 along K
constexpr uint32_t kBox32Bytes = 32 * BK * 2;
constexpr int kAccCols = kPairN;
constexpr uint32_t kTmemCols = 2 * kAccCols;
constexpr uint32_t kIdesc = idesc_bf16_f32(2 * BM, kPairN);
constexpr int kXPad = 33;
constexpr int kMaxGroups = 1024;

// MX: expert weights stored as MXFP8 (E4M3 bytes + one E8M0 scale per 32
// along K).  Each stage then also holds the CTA's fp8 weight tile and a 16-byte
// scale box per row (8 k-blocks of scales); four converter warps write the
// exactly dequantised bf16 tile into the stage's MMA operand buffer.
template <int MODE, bool MX>
struct PCfg {
    static constexpr bool kPair = MODE == GEMM_SWIGLU;      // 64 gate + 64 up rows per CTA
    static constexpr int kRowsCta = gemm_rows(MODE);        // output weight rows per CTA
    static constexpr int kRowsTile = 2 * kRowsCta;          // per CTA pair
    static constexpr uint32_t kXBytes = kPair ? 2 * 32 * kXPad * 4 : 0;
    static constexpr uint32_t kF8Bytes = MX ? BM * BK : 0;  // fp8 weight tile
    static constexpr uint32_t kScBytes = MX ? BM * 16 : 0;  // scale boxes
    static constexpr uint32_t kStageBytes = kABytes + kBBytes + kF8Bytes + kScBytes;
    static constexpr int kStages = MX ? 4 : 6;
    static constexpr int kThreads = MX ? 320 : 192;
};

struct Tile {
    int m, g, n_valid, brow, arow;
    bool shared;
};

template <int MODE>
__device__ __forceinline__ Tile decode_tile(int t, uint32_t rank, const GemmParams& p,
                                            const int* tile_start, const int* gcnt,
                                            const int* goff, int GG) {
    Tile tl;
    tl.m = t % p.MT;
    const int j = t / p.MT;
    int lo = 0, hi = GG;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (tile_start[mid] <= j) lo = mid; else hi = mid;
    }
    tl.g = lo;
    const int nt = j - tile_start[lo];
    tl.n_valid = min(kPairN, gcnt[lo] - nt * kPairN);
    tl.brow = goff[lo] + nt * kPairN;
    tl.shared = lo >= p.G;
    tl.arow = (tl.shared ? 0 : lo * p.M) + tl.m * 2 * gemm_rows(MODE) + rank * gemm_rows(MODE);
    return tl;
}

// Token-row bytes CTA `rank` loads for a tile with n_valid tokens.
__device__ __forceinline__ uint32_t b_bytes(int n_valid, uint32_t rank, int partial) {
    const int nv = min(max(n_valid - static_cast<int>(rank) * kHalfN, 0), kHalfN);
    const int nbox = (nv + 31) >> 5;
    if (!partial || nbox == kHalfN / 32) return kBBytes;
    return nbox * kBox32Bytes;
}

__device__ __forceinline__ void raise_timeout(const GemmParams& p, volatile int* abort, int where) {
    atomicOr(p.status, STATUS_TIMEOUT);
    atomicMax(p.status + 1, where);
    *abort = 1;
}

// E8M0 scale byte -> 2^(s-127) as fp32 (0xFF is NaN).
__device__ __forceinline__ float e8m0_scale(uint32_t s) {
    if (s == 0) return __int_as_float(0x00400000);   // 2^-127, an fp32 subnormal
    if (s == 255) return __int_as_float(0x7fc00000);
    return __int_as_float(static_cast<int>(s << 23));
}

// Two E4M3 values (low byte first) -> two bf16 of value * scale, packed.
// Exact: E4M3 -> f16 -> f32 are exact, the scale is a power of two, and the
// product has at most 4 significant bits.
__device__ __forceinline__ uint32_t e4m3x2_to_bf16x2(uint32_t two, float scale) {
    const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(two), __NV_E4M3);
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&hr));
    const __nv_bfloat162 b = __floats2bfloat162_rn(f.x * scale, f.y * scale);
    return *reinterpret_cast<const uint32_t*>(&b);
}

// Four E4M3 bytes of one 32-element block (scale byte s) -> four bf16 in two
// words (element 0 in the low half of `lo`).  Exact.  For normal E4M3 inputs
// and 7 <= s <= 246 the bf16 pattern is the E4M3 pattern with its exponent
// re-biased by s - 7 (E4M3 exponent bias 7, bf16 bias 127, scale 2^(s-127)),
// done with integer operations; zero, subnormal or NaN bytes and extreme
// scales take the float route above.
__device__ __forceinline__ void e4m3x4_to_bf16x4(uint32_t w, uint32_t s, uint32_t& lo,
                                                 uint32_t& hi) {
    const uint32_t x7 = w & 0x7F7F7F7Fu;
    const uint32_t ex = (w >> 3) & 0x0F0F0F0Fu;                       // exponent field per byte
    const uint32_t zero_exp = (ex - 0x01010101u) & ~ex & 0x80808080u;  // some byte has exponent 0
    const uint32_t nan = (x7 + 0x01010101u) & 0x80808080u;           // some byte is 0x7F / 0xFF
    if ((zero_exp | nan) == 0u && s >= 7u && s <= 246u) {
        const uint32_t a = __byte_perm(w, 0u, 0x4140);  // bytes 0, 1 -> low halves of two shorts
        const uint32_t b = __byte_perm(w, 0u, 0x4342);  // bytes 2, 3
        const uint32_t k = ((s - 7u) << 7) * 0x00010001u;
        lo = (((a << 4) & 0x07F007F0u) + k) | ((a << 8) & 0x80008000u);
        hi = (((b << 4) & 0x07F007F0u) + k) | ((b << 8) & 0x80008000u);
    } else {
        const float scale = e8m0_scale(s);
        lo = e4m3x2_to_bf16x2(w & 0xFFFFu, scale);
        hi = e4m3x2_to_bf16x2(w >> 16, scale);
    }
}

template <int MODE, bool MX>
__global__ void __launch_bounds__(PCfg<MODE, MX>::kThreads, 1)
    pair_gemm_kernel(const __grid_constant__ GemmParams p) {
    using C = PCfg<MODE, MX>;
    constexpr int kStages = C::kStages;
    constexpr uint32_t kStageBytes = C::kStageBytes;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    float* xbuf = reinterpret_cast<float*>(smem + kStages * kStageBytes);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * kStageBytes + C::kXBytes);
    uint64_t* empty = full + kStages;
    uint64_t* tfull = empty + kStages;
    uint64_t* tempty = tfull + 2;
    uint64_t* drain = tempty + 2;
    uint64_t* xfull = drain + 1;
    uint64_t* xempty = xfull + 2;
    uint64_t* afull = xempty + 2;  // MX: fp8 tile + scales of a stage landed (local)
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(afull + kStages);
    volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);
    int* tile_start = reinterpret_cast<int*>(tmem_slot + 4);
    const int GG = p.G + p.has_shared;
    int* gcnt = tile_start + GG + 1;
    int* goff = gcnt + GG;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;

    if (warp == 0) {
        const int per = (GG + 31) / 32;
        const int g0 = lane * per;
        int local = 0;
        for (int g = g0; g < min(g0 + per, GG); ++g) {
            int c, o;
            if (g < p.G) {
                c = p.cnt[g];
                o = p.off[g];
            } else {
                c = p.shared_rows;
                o = p.shared_b_off;
            }
            gcnt[g] = c;
            goff[g] = o;
            local += (c + kPairN - 1) / kPairN;
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
            run += (gcnt[g] + kPairN - 1) / kPairN;
        }
        if (lane == 31) tile_start[GG] = incl;
    } else if (warp == 1) {
        tmem_alloc_pair(tmem_slot, kTmemCols);
        tmem_relinquish_pair();
    } else if (threadIdx.x == 64) {
        for (int s = 0; s < kStages; ++s) {
            // MX: the leader's full barrier also waits for the 4 converter
            // warps of each CTA.
            mbar_init(&full[s], MX ? 9 : 1);
            mbar_init(&empty[s], 1);
            mbar_init(&afull[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&tfull[a], 1);
            mbar_init(&tempty[a], 8);  // 4 epilogue warps in each of the two CTAs
            mbar_init(&xfull[a], 1);
            mbar_init(&xempty[a], 1);
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
    const int total = tile_start[GG] * p.MT;
    const uint64_t tmo = p.timeout_ns;
    const int cid = static_cast<int>(cluster_id_x());
    const int ncl = static_cast<int>(nclusters_x());

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer (both CTAs) ----------------
            tma_prefetch_desc(&p.a0);
            tma_prefetch_desc(&p.b);
            if (p.has_shared) tma_prefetch_desc(&p.as0);
            const uint64_t pol_w = l2_policy_evict_first();
            const uint64_t pol_x = l2_policy_evict_last();
            int stage = 0;
            uint32_t phase = 0;
            uint32_t issued = 0, last_par = 0;
            bool ok = true;
            for (int t = cid; t < total && ok; t += ncl) {
                const Tile tl = decode_tile<MODE>(t, rank, p, tile_start, gcnt, goff, GG);
                const CUtensorMap* ma0 = tl.shared ? &p.as0 : &p.a0;
                const CUtensorMap* ma1 = tl.shared ? &p.as1 : &p.a1;
                const int nv = min(max(tl.n_valid - static_cast<int>(rank) * kHalfN, 0), kHalfN);
                const int nbox = (nv + 31) >> 5;
                const bool whole = !p.partial_b || nbox == kHalfN / 32;
                const uint32_t expect = (MX ? 0 : 2 * kABytes) + b_bytes(tl.n_valid, 0, p.partial_b) +
                                        b_bytes(tl.n_valid, 1, p.partial_b);
                const int brow = tl.brow + static_cast<int>(rank) * kHalfN;
                for (int kb = 0; kb < p.KB; ++kb) {
                    if (!mbar_wait(&empty[stage], phase ^ 1u, abort, tmo)) {
                        if (!*abort) raise_timeout(p, abort, 11);
                        ok = false;
                        break;
                    }
                    uint8_t* st = smem + stage * kStageBytes;
                    if (leader) mbar_arrive_expect_tx(&full[stage], expect);
                    const uint32_t bar = map_to_rank(&full[stage], 0);
                    if constexpr (MX) {
                        // fp8 tile and its scales into this CTA's staging; the
                        // converter warps turn them into the bf16 operand.
                        uint8_t* f8 = st + kABytes + kBBytes;
                        uint8_t* sc = f8 + C::kF8Bytes;
                        const int sx = (kb & ~7) * 2;  // 8 k-blocks of scales per box
                        mbar_arrive_expect_tx(&afull[stage], C::kF8Bytes + C::kScBytes);
                        if constexpr (C::kPair) {
                            tma_load_2d(f8, &p.a0, &afull[stage], kb * BK, tl.arow, pol_w);
                            tma_load_2d(f8 + C::kF8Bytes / 2, &p.a1, &afull[stage], kb * BK, tl.arow, pol_w);
                            tma_load_2d(sc, &p.sa0, &afull[stage], sx, tl.arow, pol_w);
                            tma_load_2d(sc + C::kScBytes / 2, &p.sa1, &afull[stage], sx, tl.arow, pol_w);
                        } else {
                            tma_load_2d(f8, &p.a0, &afull[stage], kb * BK, tl.arow, pol_w);
                            tma_load_2d(sc, &p.sa0, &afull[stage], sx, tl.arow, pol_w);
                        }
                    } else if constexpr (C::kPair) {
                        tma_load_2d_pair(st, ma0, bar, kb * BK, tl.arow, pol_w);
                        tma_load_2d_pair(st + kABytes / 2, ma1, bar, kb * BK, tl.arow, pol_w);
                    } else {
                        tma_load_2d_pair(st, ma0, bar, kb * BK, tl.arow, pol_w);
                    }
                    uint8_t* sb = st + kABytes;
                    if (whole) {
                        tma_load_2d_pair(sb, &p.b, bar, kb * BK, brow, pol_x);
                    } else {
                        for (int i = 0; i < nbox; ++i)
                            tma_load_2d_pair(sb + i * kBox32Bytes, &p.b32, bar, kb * BK, brow + 32 * i,
                                             pol_x);
                    }
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
                            raise_timeout(p, abort, 12);
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
                if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, abort, tmo)) {
                    if (!*abort) raise_timeout(p, abort, 13);
                    break;
                }
                tc_fence_after();
                const uint32_t d0 = tmem_base + acc * kAccCols;
                for (int kb = 0; kb < p.KB; ++kb) {
                    if (!mbar_wait(&full[stage], phase, abort, tmo)) {
                        if (!*abort) raise_timeout(p, abort, 14);
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
                umma_commit_pair(&tfull[acc], 0x3);
                if (++acc == 2) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
            }
            umma_commit_pair(drain, 0x1);
            if (!mbar_wait(drain, 0, nullptr, tmo)) raise_timeout(p, abort, 15);
        }
    } else if (warp >= 6) {
        if constexpr (MX) {
            // ---------------- converters (warps 6..9, both CTAs) ----------------
            const int ctid = threadIdx.x - 192;
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int t = cid; t < total && ok; t += ncl) {
                for (int kb = 0; kb < p.KB; ++kb) {
                    if (!__all_sync(0xffffffffu, mbar_wait(&afull[stage], phase, abort, tmo))) {
                        if (lane == 0 && !*abort) raise_timeout(p, abort, 19);
                        ok = false;
                        break;
                    }
                    uint8_t* st = smem + stage * kStageBytes;
                    const uint8_t* f8 = st + kABytes + kBBytes;
                    const uint8_t* sc = f8 + C::kF8Bytes;
                    // 128 rows x 8 chunks of 8 values; each chunk becomes one
                    // 16-byte chunk of the 128-byte-swizzled bf16 row.
#pragma unroll 2
                    for (int it = 0; it < 8; ++it) {
                        const int task = it * 128 + ctid;
                        const int r = task >> 3, c = task & 7;
                        const uint2 q = *reinterpret_cast<const uint2*>(f8 + r * 64 + c * 8);
                        const uint32_t sbyte = sc[r * 16 + (kb & 7) * 2 + (c >> 2)];
                        uint4 o;
                        e4m3x4_to_bf16x4(q.x, sbyte, o.x, o.y);
                        e4m3x4_to_bf16x4(q.y, sbyte, o.z, o.w);
                        *reinterpret_cast<uint4*>(st + r * 128 + ((c ^ (r & 7)) << 4)) = o;
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive_cluster(map_to_rank(&full[stage], 0));
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
        }
    } else {
        // ---------------- epilogue (warps 2..5, both CTAs) ----------------
        const int q = warp & 3;
        const int pr = q & 1;
        const bool up_warp = q >= 2;
        int acc = 0;
        uint32_t acc_phase = 0;
        uint32_t xph = 0;
        bool ok = true;
        for (int t = cid; t < total && ok; t += ncl) {
            const Tile tl = decode_tile<MODE>(t, rank, p, tile_start, gcnt, goff, GG);
            const bool ready = __all_sync(0xffffffffu, mbar_wait(&tfull[acc], acc_phase, abort, tmo));
            if (!ready) {
                if (lane == 0 && !*abort) raise_timeout(p, abort, 16);
                break;
            }
            tc_fence_after();
            const int row = tl.m * C::kRowsTile + static_cast<int>(rank) * C::kRowsCta +
                            (C::kPair ? pr : q) * 32 + lane;
            const bool row_ok = row < p.M;
            const uint32_t taddr =
                tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * kAccCols;
            for (int c0 = 0; c0 < tl.n_valid; c0 += 32) {
                float v[32];
                tmem_ld32(taddr + c0, v);
                tmem_ld_wait();
                if constexpr (MODE == GEMM_SWIGLU) {
                    float* xb = xbuf + pr * 32 * kXPad + lane * kXPad;
                    if (up_warp) {
                        if (!__all_sync(0xffffffffu, mbar_wait(&xempty[pr], xph ^ 1u, abort, tmo))) {
                            if (lane == 0 && !*abort) raise_timeout(p, abort, 17);
                            ok = false;
                            break;
                        }
#pragma unroll
                        for (int j = 0; j < 32; ++j) xb[j] = v[j];
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&xfull[pr]);
                    } else {
                        if (!__all_sync(0xffffffffu, mbar_wait(&xfull[pr], xph, abort, tmo))) {
                            if (lane == 0 && !*abort) raise_timeout(p, abort, 18);
                            ok = false;
                            break;
                        }
                        float u[32];
#pragma unroll
                        for (int j = 0; j < 32; ++j) u[j] = xb[j];
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&xempty[pr]);
                        __nv_bfloat16* H = static_cast<__nv_bfloat16*>(p.out);
#pragma unroll
                        for (int j = 0; j < 32; ++j) {
                            if (row_ok && c0 + j < tl.n_valid) {
                                const float g = v[j];
                                const float h = g / (1.0f + expf(-g)) * u[j];
                                H[static_cast<int64_t>(tl.brow + c0 + j) * p.ldo + row] =
                                    __float2bfloat16_rn(h);
                            }
                        }
                    }
                    xph ^= 1u;
                } else {
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
            if (!ok) break;
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

template <int MODE, bool MX>
size_t pair_smem_bytes(int GG) {
    using C = PCfg<MODE, MX>;
    return 1024 + C::kStages * C::kStageBytes + C::kXBytes + (3 * C::kStages + 9) * 8 + 16 +
           static_cast<size_t>(3 * GG + 1) * 4;
}

template <int MODE, bool MX>
cudaError_t launch_pair_mode(const GemmParams& p, int clusters, cudaStream_t s) {
    const int GG = p.G + p.has_shared;
    const size_t smem = pair_smem_bytes<MODE, MX>(GG);
    cudaError_t e = cudaFuncSetAttribute(pair_gemm_kernel<MODE, MX>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * clusters, 1, 1);
    cfg.blockDim = dim3(PCfg<MODE, MX>::kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // Persistent clusters: never more than can be resident at once, so that no
    // cluster's share of the static tile order waits for a second wave.
    int resident = 0;
    e = cudaOccupancyMaxActiveClusters(&resident, pair_gemm_kernel<MODE, MX>, &cfg);
    if (e != cudaSuccess) return e;
    if (resident <= 0) return cudaErrorInvalidConfiguration;
    if (clusters > resident) {
        clusters = resident;
        cfg.gridDim = dim3(2 * clusters, 1, 1);
    }
    return cudaLaunchKernelEx(&cfg, pair_gemm_kernel<MODE, MX>, p);
}

}  // namespace

cudaError_t launch_pair_gemm(int mode, const GemmParams& p, int clusters, cudaStream_t s,
                             int mxfp8) {
    if (p.G + p.has_shared > kMaxGroups || clusters <= 0 || !p.cnt || !p.off)
        return cudaErrorInvalidValue;
    if (mxfp8 && p.has_shared) return cudaErrorInvalidValue;  // shared expert is bf16
    if (mode == GEMM_SWIGLU)
        return mxfp8 ? launch_pair_mode<GEMM_SWIGLU, true>(p, clusters, s)
                     : launch_pair_mode<GEMM_SWIGLU, false>(p, clusters, s);
    if (mode == GEMM_DOWN)
        return mxfp8 ? launch_pair_mode<GEMM_DOWN, true>(p, clusters, s)
                     : launch_pair_mode<GEMM_DOWN, false>(p, clusters, s);
    return cudaErrorInvalidValue;
}

}  // namespace moe
