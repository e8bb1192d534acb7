// gemm_bs.cu -- the expert GEMMs with both operands narrow, on the block-scaled
// tensor-core MMA, which multiplies the narrow values and applies their block
// scales itself: nothing is converted and the tensor pipe runs at its 8-bit or
// 4-bit rate.  Two formats, both from the Composer 2 Technical Report, §6.1
// "Training infrastructure", Kernels paragraph (block-scaled tensor-core matmul):
//   * MXFP8 (E4M3 weights and token rows, one E8M0 scale per 32 along K):
//     tcgen05.mma.kind::mxf8f6f4.block_scale.scale_vec::1X, K = 32 per MMA;
//   * NVFP4 (E2M1 weights and token rows, two per byte, one E4M3 scale per 16
//     along K, plus an fp32 scale per token and per weight matrix that the
//     epilogue applies): tcgen05.mma.kind::mxf4nvf4.block_scale.scale_vec::4X,
//     K = 64 per MMA.
//
// Shape: SM pairs (tcgen05 cta_group::2), M = 256 weight rows (128 per CTA),
// N = up to 224 (MXFP8) or 192 (NVFP4) tokens (each CTA loads half), K in
// blocks of 128 bytes per row (one 128-byte-swizzled row of the operand tile,
// four MMAs).  Each output element is one pair's fixed-order K loop into one
// TMEM accumulator; no split-K, no atomics; the MMA width N only selects how
// many independent token columns one instruction produces.  The MoE backward
// runs its dH and dXp GEMMs here too (MXFP8 down mode): fp32 output rows
// (out_f32) and the shared expert as one more group (has_shared) whose weights
// follow the routed experts' in the same tensors.
//
// Roles in each CTA (352 threads): warp 0 TMA producer of the weight tiles (and
// of the scale tiles); warp 10 TMA producer of the token tiles; warp 1 TMEM
// owner and, in the pair's leader, the MMA issuer; warps 2..5 epilogue; warps
// 6..9 write each K block's scales into TMEM (one warp per TMEM lane
// quadrant), where the MMA reads them.
#include <cuda_bf16.h>

#include "moe_internal.h"
#include "ptx.cuh"
#include "tile_walk.cuh"

namespace moe {
namespace {

constexpr int kK8 = 128;                   // bytes per stage and row (K block)
constexpr uint32_t kA8 = 128 * kK8;        // weight tile of a CTA: 16 KB
constexpr uint32_t kBox8 = 32 * kK8;       // one 32-row token box
constexpr int kThreads8 = 352;
constexpr int kXPad8 = 33;
constexpr uint32_t kXBytes8 = 2 * 32 * kXPad8 * 4;   // gate/up: up values handed to the gate warps
constexpr int kMaxGroups8 = 1024;
constexpr uint32_t kTmemCols8 = 512;

// Per format:
//   kTile     tokens per tile (MMA N at most); kStages operand stages;
//   kBigBox   token rows of the one-copy box of a CTA's rows (3 or 4 32-row boxes);
//   kScRow    scale bytes per row and K block; kScKb K blocks per scale slot;
//   kScAhead  scale groups loaded ahead of the weights when the launch asks
//             for it (sc_ahead: large batches; MXFP8 2 of 4 slots, gate/up 2 %
//             faster; NVFP4 1 of 3, 1.3 % faster, while 2 stalled the weight
//             loads on the ring; a decode batch ran 4 % slower with 1);
//   kSfKb     TMEM columns of one K block's scales.  MXFP8: one word per row
//             serves the block's four K steps (a byte each): 4 columns of
//             weight-row scales, then 8 of token scales.  NVFP4: a word per row
//             and K step: K step w's weight-row scales at columns 4w .. 4w + 3,
//             its token scales at 16 + 8w .. 16 + 8w + 7;
//   kSfSets   sets of those columns in flight.  MXFP8: one per stage, reused
//             once the stage's MMAs complete; NVFP4: two, each freed by its
//             own commit (the accumulators leave room for no more).
template <int FMT>
struct BsCfg;
template <>
struct BsCfg<BS_MXFP8> {
    static constexpr int kTile = 224, kBigBox = 128, kScRow = 4, kScKb = 4, kScSlots = 4;
    static constexpr int kScAhead = 2;
    static constexpr int kStages = 5;
    static constexpr uint32_t kSfKb = 12;
    static constexpr int kSfSets = kStages;
};
template <>
struct BsCfg<BS_NVFP4> {
    static constexpr int kTile = 192, kBigBox = 96, kScRow = 16, kScKb = 2, kScSlots = 3;
    static constexpr int kScAhead = 1;
    static constexpr int kStages = 5;
    static constexpr uint32_t kSfKb = 48;
    static constexpr int kSfSets = 2;
};

template <int FMT>
struct BsLayout {
    using C = BsCfg<FMT>;
    // token tile of a CTA: its rows at most, 1024-aligned for the swizzle
    static constexpr uint32_t kB = static_cast<uint32_t>(C::kTile / 2 + 31) / 32 * kBox8;
    static constexpr uint32_t kStage = kA8 + kB;
    // Scale ring: a slot holds the scales of kScKb consecutive K blocks of one
    // tile: the CTA's 128 weight rows, then the tile's tokens of both CTAs
    // (CTA 0's half at rows 0..127, CTA 1's at 128..255).
    static constexpr uint32_t kScRowBytes = C::kScRow * C::kScKb;  // one TMA box wide
    static constexpr uint32_t kScA = 128 * kScRowBytes;
    static constexpr uint32_t kScSlot = kScA + 256 * kScRowBytes;
    // TMEM: two accumulator slots of kTile columns, then the scale column sets
    static constexpr uint32_t kAcc = C::kTile;
    static constexpr uint32_t kSfCol = 2 * kAcc;
    static constexpr int kBarriers = 2 * C::kStages + 2 * C::kScSlots + C::kSfSets + 2 + 2 + 4 + 1;
    static_assert(kSfCol + C::kSfSets * C::kSfKb <= kTmemCols8, "TMEM columns");
    static_assert(kStage % 1024 == 0, "stages keep the 128-byte swizzle's alignment");
};

struct Tile8 {
    int m, g, n_valid, brow, arow;
    int half;  // MMA N / 2
};

// The tile at list position (g, m, nt): its token rows and the CTA's weight rows.
template <int MODE, int FMT>
__device__ __forceinline__ Tile8 make_tile8(const TilePos& pos, uint32_t rank, const GemmParams& p,
                                            const int* gcnt, const int* goff) {
    constexpr int kTile8 = BsCfg<FMT>::kTile;
    Tile8 tl;
    tl.g = pos.g;
    tl.m = pos.m;
    tl.n_valid = min(kTile8, gcnt[tl.g] - pos.nt * kTile8);
    tl.half = min(kTile8, max(64, (tl.n_valid + 31) & ~31)) >> 1;
    tl.brow = goff[tl.g] + pos.nt * kTile8;
    tl.arow = tl.g * p.M + tl.m * 2 * gemm_rows(MODE) + static_cast<int>(rank) * gemm_rows(MODE);
    return tl;
}

__device__ __forceinline__ int b_rows8(const Tile8& tl, uint32_t rank) {
    return min(max(tl.n_valid - static_cast<int>(rank) * tl.half, 0), tl.half);
}

__device__ __forceinline__ void raise_timeout8(const GemmParams& p, volatile int* abort, int where) {
    atomicOr(p.status, STATUS_TIMEOUT);
    atomicMax(p.status + 1, where);
    *abort = 1;
}

// bf16 row pairs of one token per 4-byte store (as in the other SM-pair
// epilogues): lanes 2i, 2i + 1 hold rows r, r + 1 for the same tokens.
template <int N>
__device__ __forceinline__ void store_pairs8(const float (&h)[N], int lane, __nv_bfloat16* at,
                                             int64_t ld, int n_left, bool row_ok) {
    const int odd = lane & 1;
    uint32_t pk[N / 2];
#pragma unroll
    for (int jj = 0; jj < N / 2; ++jj) {
        const float other = __shfl_xor_sync(0xffffffffu, odd ? h[2 * jj] : h[2 * jj + 1], 1);
        const float mine = odd ? h[2 * jj + 1] : h[2 * jj];
        const __nv_bfloat162 b = __floats2bfloat162_rn(odd ? other : mine, odd ? mine : other);
        pk[jj] = *reinterpret_cast<const uint32_t*>(&b);
    }
    uint32_t* y = reinterpret_cast<uint32_t*>(at + odd * ld);
#pragma unroll
    for (int jj = 0; jj < N / 2; ++jj)
        if (row_ok && 2 * jj + odd < n_left) y[jj * ld] = pk[jj];
}

template <int MODE, int FMT>
__global__ void __launch_bounds__(kThreads8, 1) bs_pair_kernel(const __grid_constant__ GemmParams p) {
    using C = BsCfg<FMT>;
    using L = BsLayout<FMT>;
    constexpr bool kNv = FMT == BS_NVFP4;
    constexpr bool kPair = MODE == GEMM_SWIGLU;  // 64 gate + 64 up weight rows per CTA
    constexpr int kRowsCta = gemm_rows(MODE);
    constexpr int kTile = C::kTile;
    constexpr int kScKb = C::kScKb;
    constexpr int kScSlots = C::kScSlots;
    constexpr int kStages = C::kStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    uint8_t* scring = smem + kStages * L::kStage;
    float* xbuf = reinterpret_cast<float*>(scring + kScSlots * L::kScSlot);
    uint64_t* full = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(xbuf) + kXBytes8);
    uint64_t* empty = full + kStages;
    uint64_t* scfull = empty + kStages;
    uint64_t* scempty = scfull + kScSlots;
    uint64_t* sffree = scempty + kScSlots;  // NVFP4: a TMEM scale set's MMAs completed
    uint64_t* tfull = sffree + C::kSfSets;
    uint64_t* tempty = tfull + 2;
    uint64_t* xfull = tempty + 2;
    uint64_t* xempty = xfull + 2;
    uint64_t* drain = xempty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(full + L::kBarriers);
    volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);
    // the shared expert (has_shared) is group G: its weights are group G of
    // the same tensors, its token rows shared_rows rows from shared_b_off
    const int GG = p.G + (p.has_shared ? 1 : 0);
    int* hs = reinterpret_cast<int*>(tmem_slot + 4);
    int* cs = hs + GG + 1;
    int* gcnt = cs + GG + 1;
    int* goff = gcnt + GG;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;

    if (warp == 0) {
        // per group: token tiles if hot (several), 1 in the cold count if cold
        const int per = (GG + 31) / 32;
        const int g0 = lane * per;
        int local_h = 0, local_c = 0;
        for (int g = g0; g < min(g0 + per, GG); ++g) {
            const int c = g < p.G ? p.cnt[g] : p.shared_rows;
            gcnt[g] = c;
            goff[g] = g < p.G ? p.off[g] : p.shared_b_off;
            const int ntg = (c + kTile - 1) / kTile;
            if (ntg > 1) local_h += ntg; else local_c += ntg;
        }
        int incl_h = local_h, incl_c = local_c;
#pragma unroll
        for (int s = 1; s < 32; s <<= 1) {
            const int vh = __shfl_up_sync(0xffffffffu, incl_h, s);
            const int vc = __shfl_up_sync(0xffffffffu, incl_c, s);
            if (lane >= s) {
                incl_h += vh;
                incl_c += vc;
            }
        }
        int run_h = incl_h - local_h, run_c = incl_c - local_c;
        for (int g = g0; g < min(g0 + per, GG); ++g) {
            hs[g] = run_h;
            cs[g] = run_c;
            const int ntg = (gcnt[g] + kTile - 1) / kTile;
            if (ntg > 1) run_h += ntg; else run_c += ntg;
        }
        if (lane == 31) {
            hs[GG] = incl_h;
            cs[GG] = incl_c;
        }
    } else if (warp == 1) {
        tmem_alloc_pair(tmem_slot, kTmemCols8);
        tmem_relinquish_pair();
    } else if (threadIdx.x == 64) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1 + 2 * 4);  // producer + the scale writers of both CTAs
            mbar_init(&empty[s], 1);
        }
        for (int s = 0; s < kScSlots; ++s) {
            mbar_init(&scfull[s], 1);
            mbar_init(&scempty[s], 4);  // the 4 scale writers, after the slot's last K block
        }
        for (int s = 0; s < C::kSfSets; ++s) mbar_init(&sffree[s], 1);
        for (int a = 0; a < 2; ++a) {
            mbar_init(&tfull[a], 1);
            mbar_init(&tempty[a], 8);  // 4 epilogue warps in each CTA
            mbar_init(&xfull[a], 1);
            mbar_init(&xempty[a], 1);
        }
        mbar_init(drain, 1);
        *abort = 0;
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // the static tile order (tile_walk.cuh); this pair takes positions cid,
    // cid + ncl, ...
    const TileOrder order{hs, cs, GG, p.MT, static_cast<uint32_t>(hs[GG] * p.MT),
                          static_cast<uint32_t>((hs[GG] + cs[GG]) * p.MT)};
    const uint64_t tmo = p.timeout_ns;
    const int cid = static_cast<int>(cluster_id_x());
    const int ncl = static_cast<int>(nclusters_x());
    // a CTA's token rows: one kBigBox-row box when they need three or more
    // 32-row boxes (fewer copies), else 32-row boxes
    auto token_boxes = [](int rows) {
        const int n = (rows + 31) >> 5;
        return n >= 3 ? C::kBigBox / 32 : n;
    };

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer (both CTAs) ----------------
            tma_prefetch_desc(&p.a0);
            tma_prefetch_desc(&p.b32);
            // weights: normal eviction, so that the next token tile of the
            // same weight tile, usually running at the same time on another
            // pair, still finds them in L2
            const uint64_t pol_w = l2_policy_evict_normal();
            const uint64_t pol_x = l2_policy_evict_last();
            int stage = 0, ss = 0;
            uint32_t phase = 0, sph = 0;
            uint32_t issued = 0, last_par = 0, s_issued = 0, s_par = 0;
            bool ok = p.stall_test == 0;
            // the scales of K blocks kb .. kb + kScKb - 1 of tile t: weight rows,
            // then both halves of the tile's tokens
            auto load_scales = [&](const Tile8& t, int kb) -> bool {
                if (!mbar_wait(&scempty[ss], sph ^ 1u, abort, tmo)) {
                    if (!*abort) raise_timeout8(p, abort, 40);
                    return false;
                }
                uint8_t* sc = scring + ss * L::kScSlot;
                mbar_arrive_expect_tx(&scfull[ss], L::kScA + 2 * 128 * L::kScRowBytes);
                const int x = kb * C::kScRow;
                if constexpr (kPair) {
                    tma_load_2d(sc, &p.sa0, &scfull[ss], x, t.arow, pol_w);
                    tma_load_2d(sc + L::kScA / 2, &p.sa1, &scfull[ss], x, t.arow, pol_w);
                } else {
                    tma_load_2d(sc, &p.sa0, &scfull[ss], x, t.arow, pol_w);
                }
                tma_load_2d(sc + L::kScA, &p.sb_scale, &scfull[ss], x, t.brow, pol_x);
                tma_load_2d(sc + L::kScA + 128 * L::kScRowBytes, &p.sb_scale, &scfull[ss], x,
                            t.brow + t.half, pol_x);
                s_issued |= 1u << ss;
                s_par = (s_par & ~(1u << ss)) | (sph << ss);
                if (++ss == kScSlots) {
                    ss = 0;
                    sph ^= 1u;
                }
                return true;
            };
            // Large batches (p.sc_ahead): the scale groups run C::kScAhead groups
            // ahead of the weights, from a cursor of their own over the same
            // tiles, so that the scale writers find them landed; the cursor stays
            // within the kScSlots-slot ring.  Otherwise each group is loaded with
            // its first K block.
            static_assert(C::kScAhead < kScSlots, "the ring holds the groups ahead");
            const bool ahead = p.sc_ahead != 0;
            TileWalk sw = tile_walk_begin(cid, order);
            Tile8 stl{};
            int skb = 0;
            auto scale_cursor = [&]() -> bool {  // the cursor's next group, if any
                if (sw.t < 0) return true;
                if (skb == 0) stl = make_tile8<MODE, FMT>(tile_walk_pos(sw, order), rank, p, gcnt, goff);
                if (!load_scales(stl, skb)) return false;
                skb += kScKb;
                if (skb == p.KB) {
                    skb = 0;
                    tile_walk_next(sw, ncl, order);
                }
                return true;
            };
            if (ahead)
                for (int a = 0; a < C::kScAhead && ok; ++a) ok = scale_cursor();
            for (TileWalk w = tile_walk_begin(cid, order); ok && w.t >= 0; tile_walk_next(w, ncl, order)) {
                const Tile8 tl = make_tile8<MODE, FMT>(tile_walk_pos(w, order), rank, p, gcnt, goff);
                const uint32_t expect =
                    2 * kA8 + (token_boxes(b_rows8(tl, 0)) + token_boxes(b_rows8(tl, 1))) * kBox8;
                for (int kb = 0; kb < p.KB; ++kb) {
                    if (kb % kScKb == 0 && !(ahead ? scale_cursor() : load_scales(tl, kb))) {
                        ok = false;
                        break;
                    }
                    if (!mbar_wait(&empty[stage], phase ^ 1u, abort, tmo)) {
                        if (!*abort) raise_timeout8(p, abort, 41);
                        ok = false;
                        break;
                    }
                    uint8_t* st = smem + stage * L::kStage;
                    if (leader) mbar_arrive_expect_tx(&full[stage], expect);
                    const uint32_t bar = map_to_rank(&full[stage], 0);
                    if constexpr (kPair) {
                        tma_load_2d_pair(st, &p.a0, bar, kb * kK8, tl.arow, pol_w);
                        tma_load_2d_pair(st + kA8 / 2, &p.a1, bar, kb * kK8, tl.arow, pol_w);
                    } else {
                        tma_load_2d_pair(st, &p.a0, bar, kb * kK8, tl.arow, pol_w);
                    }
                    issued |= 1u << stage;
                    last_par = (last_par & ~(1u << stage)) | (phase << stage);
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (leader)
                for (int s = 0; s < kStages; ++s)
                    if (issued & (1u << s))
                        if (!mbar_wait(&full[s], (last_par >> s) & 1u, nullptr, tmo))
                            raise_timeout8(p, abort, 42);
            for (int s = 0; s < kScSlots; ++s)
                if (s_issued & (1u << s))
                    if (!mbar_wait(&scfull[s], (s_par >> s) & 1u, nullptr, tmo))
                        raise_timeout8(p, abort, 43);
        }
    } else if (warp == 1) {
        if (lane == 0 && leader) {
            // ---------------- MMA issuer (leader only) ----------------
            int stage = 0, acc = 0, sfs = 0;
            uint32_t phase = 0, acc_phase = 0;
            bool ok = true;
            for (TileWalk w = tile_walk_begin(cid, order); ok && w.t >= 0; tile_walk_next(w, ncl, order)) {
                if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, abort, tmo)) {
                    if (!*abort) raise_timeout8(p, abort, 44);
                    break;
                }
                tc_fence_after();
                const Tile8 tl = make_tile8<MODE, FMT>(tile_walk_pos(w, order), rank, p, gcnt, goff);
                const uint32_t d0 = tmem_base + acc * L::kAcc;
                const uint32_t idesc = kNv ? idesc_nv4(2 * BM, 2 * tl.half) : idesc_mx8(2 * BM, 2 * tl.half);
                for (int kb = 0; kb < p.KB; ++kb) {
                    if (!mbar_wait(&full[stage], phase, abort, tmo)) {
                        if (!*abort) raise_timeout8(p, abort, 45);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = smem_addr(smem + stage * L::kStage);
                    const uint64_t da = sdesc_kmajor_sw128(sa);
                    const uint64_t db = sdesc_kmajor_sw128(sa + kA8);
                    if constexpr (kNv) {
                        const uint32_t sfa = tmem_base + L::kSfCol + sfs * C::kSfKb;
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            umma_nv4_pair(d0, da + 2 * k, db + 2 * k, idesc, sfa + 4 * k,
                                          sfa + 16 + 8 * k, (kb | k) != 0);
                        umma_commit_pair(&sffree[sfs], 0x3);
                        if (++sfs == C::kSfSets) sfs = 0;
                    } else {
                        const uint32_t sfa = tmem_base + L::kSfCol + stage * C::kSfKb;
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            umma_mx8_pair(d0, da + 2 * k, db + 2 * k, idesc_mx8_step(idesc, k), sfa,
                                          sfa + 4, (kb | k) != 0);
                    }
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
            if (!mbar_wait(drain, 0, nullptr, tmo)) raise_timeout8(p, abort, 46);
        }
    } else if (warp == 10) {
        if (lane == 0) {
            // ---------------- token TMA producer (both CTAs) ----------------
            // The token tiles come from a thread of their own: one thread
            // issuing every copy of a K block was the pipeline's limit.
            const uint64_t pol_x = l2_policy_evict_last();
            int stage = 0;
            uint32_t phase = 0;
            bool ok = p.stall_test == 0;
            for (TileWalk w = tile_walk_begin(cid, order); ok && w.t >= 0; tile_walk_next(w, ncl, order)) {
                const Tile8 tl = make_tile8<MODE, FMT>(tile_walk_pos(w, order), rank, p, gcnt, goff);
                const int nb = token_boxes(b_rows8(tl, rank));
                const int brow = tl.brow + static_cast<int>(rank) * tl.half;
                for (int kb = 0; kb < p.KB; ++kb) {
                    if (!mbar_wait(&empty[stage], phase ^ 1u, abort, tmo)) {
                        if (!*abort) raise_timeout8(p, abort, 52);
                        ok = false;
                        break;
                    }
                    uint8_t* st = smem + stage * L::kStage;
                    const uint32_t bar = map_to_rank(&full[stage], 0);
                    if (nb == C::kBigBox / 32) {
                        tma_load_2d_pair(st + kA8, &p.b, bar, kb * kK8, brow, pol_x);
                    } else {
                        for (int i = 0; i < nb; ++i)
                            tma_load_2d_pair(st + kA8 + i * kBox8, &p.b32, bar, kb * kK8, brow + 32 * i,
                                             pol_x);
                    }
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            // its copies complete on the leader's full barriers, which the
            // weight producer waits out before the block exits
        }
    } else if (warp >= 6) {
        // ---------------- scale writers (warps 6..9, both CTAs) ----------------
        // Warp of lane quadrant q writes, for each K block, the weight-row scales
        // of rows 32q .. 32q + 31 (lane r, column r / 32) and the scales of all
        // N token columns (lane 32q + n % 32, column 4 + n / 32) into a set of
        // TMEM scale columns, once the MMAs that last read that set completed.
        const int q = warp & 3;
        const uint32_t lane_base = static_cast<uint32_t>(32 * q) << 16;
        auto wait_all = [&](uint64_t* bar, uint32_t par, int where) {
            if (__all_sync(0xffffffffu, mbar_wait(bar, par, abort, tmo))) return true;
            if (lane == 0 && !*abort) raise_timeout8(p, abort, where);
            return false;
        };
        int stage = 0;
        uint32_t phase = 0;
        int64_t i = 0;  // K blocks done, over the pair's tile sequence
        bool ok = true;
        for (TileWalk w = tile_walk_begin(cid, order); ok && w.t >= 0; tile_walk_next(w, ncl, order)) {
            const Tile8 tl = make_tile8<MODE, FMT>(tile_walk_pos(w, order), rank, p, gcnt, goff);
            const int n_cols = 2 * tl.half;
            for (int kb = 0; kb < p.KB; ++kb, ++i) {
                const int ss = static_cast<int>((i / kScKb) % kScSlots);
                const uint32_t sph = static_cast<uint32_t>((i / kScKb / kScSlots) & 1);
                const int set = kNv ? static_cast<int>(i % C::kSfSets) : stage;
                const bool freed =
                    kNv ? wait_all(&sffree[set], static_cast<uint32_t>((i / C::kSfSets) & 1) ^ 1u, 53)
                        : wait_all(&empty[stage], phase ^ 1u, 48);
                if (!wait_all(&scfull[ss], sph, 47) || !freed) {
                    ok = false;
                    break;
                }
                const uint8_t* sc = scring + ss * L::kScSlot;
                const int kq = kb % kScKb;
                const uint32_t sf = tmem_base + lane_base + L::kSfCol + set * C::kSfKb;
                if constexpr (kNv) {
                    // a row's four K-step words are one 16-byte load; this
                    // quadrant's lanes of columns 4w .. 4w + 3 all get K step w's
                    // word (the MMA reads column 4w + q)
                    const uint4 a = *reinterpret_cast<const uint4*>(
                        sc + (32 * q + lane) * L::kScRowBytes + kq * 16);
                    const uint32_t aw[4] = {a.x, a.y, a.z, a.w};
                    uint32_t av[16];
#pragma unroll
                    for (int c = 0; c < 16; ++c) av[c] = aw[c >> 2];
                    uint32_t bv[32];
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        const int n = 32 * c + lane;  // token column of the MMA
                        const int r = n < tl.half ? n : 128 + n - tl.half;
                        uint4 b = make_uint4(0x38383838u, 0x38383838u, 0x38383838u, 0x38383838u);
                        if (n < n_cols)
                            b = *reinterpret_cast<const uint4*>(sc + L::kScA + r * L::kScRowBytes + kq * 16);
                        bv[c] = b.x;
                        bv[8 + c] = b.y;
                        bv[16 + c] = b.z;
                        bv[24 + c] = b.w;
                    }
                    tmem_st16(sf, av);
                    tmem_st32(sf + 16, bv);
                } else {
                    // one word per row: its 4 bytes are the block's 4 K steps
                    tmem_st1(sf + q, *reinterpret_cast<const uint32_t*>(
                                         sc + (32 * q + lane) * L::kScRowBytes + kq * C::kScRow));
                    uint32_t bw[8];
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        const int n = 32 * c + lane;  // token column of the MMA
                        const int r = n < tl.half ? n : 128 + n - tl.half;
                        bw[c] = n < n_cols ? *reinterpret_cast<const uint32_t*>(
                                                 sc + L::kScA + r * L::kScRowBytes + kq * C::kScRow)
                                           : 0x7F7F7F7Fu;  // 1.0
                    }
                    tmem_st8(sf + 4, bw);
                }
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    // CTA-scope release: the scales are read by the pair's MMA from
                    // this CTA's own TMEM, after the fence above
                    if (leader)
                        mbar_arrive(&full[stage]);
                    else
                        mbar_arrive_operand_ready(map_to_rank(&full[stage], 0));
                    if (kq == kScKb - 1) mbar_arrive(&scempty[ss]);
                }
                if (++stage == kStages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
    } else {
        // ---------------- epilogue (warps 2..5, both CTAs) ----------------
        // Warp q reads accumulator lanes [32q, 32q + 32).  gate/up: warps 0, 1
        // hold gate rows and warps 2, 3 the matching up rows, which they pass
        // on through xbuf.  NVFP4: each output is first multiplied by its
        // token's scale times the matrix's scale.
        const int q = warp & 3;
        const int pr = q & 1;
        const bool up_warp = q >= 2;
        int acc = 0;
        uint32_t acc_phase = 0, xph = 0;
        bool ok = true;
        for (TileWalk w = tile_walk_begin(cid, order); ok && w.t >= 0; tile_walk_next(w, ncl, order)) {
            const Tile8 tl = make_tile8<MODE, FMT>(tile_walk_pos(w, order), rank, p, gcnt, goff);
            if (!__all_sync(0xffffffffu, mbar_wait(&tfull[acc], acc_phase, abort, tmo))) {
                if (lane == 0 && !*abort) raise_timeout8(p, abort, 49);
                break;
            }
            tc_fence_after();
            const int row = tl.m * 2 * kRowsCta + static_cast<int>(rank) * kRowsCta +
                            (kPair ? pr : q) * 32 + lane;
            const bool row_ok = row < p.M;
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * L::kAcc;
            const float ws0 = kNv ? p.wscale0[tl.g] : 1.0f;
            const float ws1 = kNv && kPair ? p.wscale1[tl.g] : 1.0f;
            for (int c0 = 0; c0 < tl.n_valid && ok; c0 += 32) {
                float v[32];
                tmem_ld32(taddr + c0, v);
                tmem_ld_wait();
                tmem_regs_ready(v);
                // NVFP4: lane j holds the scale of the chunk's token j
                const float tok_scale =
                    kNv && c0 + lane < tl.n_valid ? p.row_scale[tl.brow + c0 + lane] : 0.0f;
                if constexpr (kPair) {
                    float* xb = xbuf + pr * 32 * kXPad8 + lane * kXPad8;
                    if (up_warp) {
                        if (!__all_sync(0xffffffffu, mbar_wait(&xempty[pr], xph ^ 1u, abort, tmo))) {
                            if (lane == 0 && !*abort) raise_timeout8(p, abort, 50);
                            ok = false;
                            break;
                        }
#pragma unroll
                        for (int jj = 0; jj < 32; ++jj) xb[jj] = v[jj];
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&xfull[pr]);
                    } else {
                        if (!__all_sync(0xffffffffu, mbar_wait(&xfull[pr], xph, abort, tmo))) {
                            if (lane == 0 && !*abort) raise_timeout8(p, abort, 51);
                            ok = false;
                            break;
                        }
                        float h[32];
#pragma unroll
                        for (int jj = 0; jj < 32; ++jj) {
                            float g = v[jj], u = xb[jj];
                            if constexpr (kNv) {
                                const float st = __shfl_sync(0xffffffffu, tok_scale, jj);
                                g *= st * ws0;
                                u *= st * ws1;
                            }
                            h[jj] = swiglu(g, u);
                        }
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&xempty[pr]);
                        store_pairs8<32>(h, lane,
                                         static_cast<__nv_bfloat16*>(p.out) +
                                             static_cast<int64_t>(tl.brow + c0) * p.ldo + (row & ~1),
                                         p.ldo, tl.n_valid - c0, row_ok);
                    }
                    xph ^= 1u;
                } else {
                    if constexpr (kNv) {
#pragma unroll
                        for (int jj = 0; jj < 32; ++jj)
                            v[jj] *= __shfl_sync(0xffffffffu, tok_scale, jj) * ws0;
                    }
                    if (!kNv && p.out_f32) {
                        // fp32 rows: for each token the 32 lanes store 128 bytes
                        float* yf = static_cast<float*>(p.out) + static_cast<int64_t>(tl.brow + c0) * p.ldo + row;
#pragma unroll
                        for (int jj = 0; jj < 32; ++jj)
                            if (row_ok && c0 + jj < tl.n_valid) yf[static_cast<int64_t>(jj) * p.ldo] = v[jj];
                    } else {
                        store_pairs8<32>(v, lane,
                                         static_cast<__nv_bfloat16*>(p.out) +
                                             static_cast<int64_t>(tl.brow + c0) * p.ldo + (row & ~1),
                                         p.ldo, tl.n_valid - c0, row_ok);
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
    cluster_sync();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, kTmemCols8);
    }
}

template <int FMT>
size_t bs_smem_bytes(int GG) {
    using L = BsLayout<FMT>;
    return 1024 + BsCfg<FMT>::kStages * L::kStage + BsCfg<FMT>::kScSlots * L::kScSlot + kXBytes8 +
           L::kBarriers * 8 + 16 + static_cast<size_t>(4 * GG + 2) * 4;
}

template <int MODE, int FMT>
cudaError_t launch_bs_mode(const GemmParams& p, int clusters, cudaStream_t s) {
    const size_t smem = bs_smem_bytes<FMT>(p.G + (p.has_shared ? 1 : 0));
    cudaError_t e = cudaFuncSetAttribute(bs_pair_kernel<MODE, FMT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * clusters, 1, 1);
    cfg.blockDim = dim3(kThreads8, 1, 1);
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
    e = cudaOccupancyMaxActiveClusters(&resident, bs_pair_kernel<MODE, FMT>, &cfg);
    if (e != cudaSuccess) return e;
    if (resident <= 0) return cudaErrorInvalidConfiguration;
    if (clusters > resident) {
        clusters = resident;
        cfg.gridDim = dim3(2 * clusters, 1, 1);
    }
    return cudaLaunchKernelEx(&cfg, bs_pair_kernel<MODE, FMT>, p);
}

template <int FMT>
cudaError_t launch_bs_fmt(int mode, const GemmParams& p, int clusters, cudaStream_t s) {
    if (p.KB % BsCfg<FMT>::kScKb) return cudaErrorInvalidValue;  // scale slots never straddle tiles
    if (mode == GEMM_SWIGLU) return launch_bs_mode<GEMM_SWIGLU, FMT>(p, clusters, s);
    if (mode == GEMM_DOWN) return launch_bs_mode<GEMM_DOWN, FMT>(p, clusters, s);
    return cudaErrorInvalidValue;
}

}  // namespace

int bs_tile_tokens(int fmt) { return fmt == BS_NVFP4 ? BsCfg<BS_NVFP4>::kTile : BsCfg<BS_MXFP8>::kTile; }
int bs_big_box(int fmt) { return fmt == BS_NVFP4 ? BsCfg<BS_NVFP4>::kBigBox : BsCfg<BS_MXFP8>::kBigBox; }
int bs_scale_box(int fmt) {
    return fmt == BS_NVFP4 ? static_cast<int>(BsLayout<BS_NVFP4>::kScRowBytes)
                           : static_cast<int>(BsLayout<BS_MXFP8>::kScRowBytes);
}
int bs_scale_kb(int fmt) { return fmt == BS_NVFP4 ? BsCfg<BS_NVFP4>::kScKb : BsCfg<BS_MXFP8>::kScKb; }

cudaError_t launch_bs_gemm(int fmt, int mode, const GemmParams& p, int clusters, cudaStream_t s) {
    if (p.G + (p.has_shared ? 1 : 0) > kMaxGroups8 || clusters <= 0 || !p.cnt || !p.off)
        return cudaErrorInvalidValue;
    // fp32 rows: MXFP8 down projections only; the shared group: MXFP8 only
    if ((p.out_f32 && (fmt != BS_MXFP8 || mode != GEMM_DOWN)) || (p.has_shared && fmt != BS_MXFP8))
        return cudaErrorInvalidValue;
    if (fmt == BS_MXFP8) return launch_bs_fmt<BS_MXFP8>(mode, p, clusters, s);
    if (fmt == BS_NVFP4) {
        if (!p.row_scale || !p.wscale0 || (mode == GEMM_SWIGLU && !p.wscale1))
            return cudaErrorInvalidValue;
        return launch_bs_fmt<BS_NVFP4>(mode, p, clusters, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace moe
