// gemm_pair.cu -- the expert GEMMs (gate/up + SwiGLU, down) on pairs of SMs:
// tcgen05.mma.cta_group::2 with M = 256 weight rows (128 in each CTA of a
// 2-CTA cluster) and up to N = 256 tokens (each CTA loads and holds half).
// Each SM thus loads 16 KB of weights and up to 16 KB of tokens per 64-wide K
// step for 4.2 MFLOP of MMA work, a third less operand traffic than a one-SM
// 128 x 256 tile, and a 32 KB pipeline stage leaves room for six stages.
// A tile with fewer tokens (the last tile of a group, or an expert that few
// tokens chose) issues its MMAs with N = its token count rounded up to 64, so
// the tensor pipe does not spend a full-width tile's time on padding while
// the weights stream.
//
// These are the grouped expert GEMMs of the Composer 2 Technical Report,
// §6.1 "Training infrastructure" (Fig. 10).  The fixed accumulation order of
// the Training Data No. 94 write-up (section "浮点数不守规矩，MoE 火上浇油")
// holds as in the one-SM kernel: one CTA pair produces each output element
// from M = 256 MMAs over K = 16 steps in K order into one TMEM accumulator; no
// split-K, no atomics.  The MMA's N only selects how many independent output
// columns (tokens) one instruction produces; each column's dot product takes
// the same K steps whatever N is, so a token's result does not depend on how
// many other tokens share its tile.
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
#include "tile_walk.cuh"

namespace moe {
namespace {

constexpr uint32_t kABytes = BM * BK * 2;        // 128 weight rows x 64 along K
constexpr uint32_t kBox32Bytes = 32 * BK * 2;
constexpr int kSmallTileN = 64;  // tokens per tile of the small-batch variant
constexpr int kXPad = 33;
constexpr int kMaxGroups = 1024;

// MX: expert weights stored as MXFP8 (E4M3 bytes + one E8M0 scale per 32
// along K).  A dedicated producer warp streams the CTA's fp8 weight
// tiles into their own ring, far ahead, and a 16-byte scale box per row every
// 8 k-blocks into a small scale ring; eight converter warps, in four groups
// of two, convert whole k-blocks (group g takes k-blocks g, g+4, ...) into the
// operand ring's A buffer, so several k-blocks are converted at once and HBM
// latency never sits between a conversion and its MMA.
// SMALL (MXFP8 weights, batches of at most 128 tokens): weight streaming
// with few tokens per expert.  Tiles of 64 tokens leave a 4 KB token slot per
// stage, so four operand stages take 80 KB and the weight ring gets 96 KB (the
// bytes in flight that streaming at an SM's share of HBM bandwidth needs), and
// sixteen converter warps keep up with it.
template <int MODE, int FMT, bool SMALL>
struct PCfg {
    static constexpr bool kConv = FMT != WFMT_BF16;   // weights converted in-kernel
    static constexpr bool kSmall = SMALL;
    static constexpr int kTileN = SMALL ? kSmallTileN : BN_EXPERT;  // tokens per MMA sub-tile
    static constexpr int kHalfN = kTileN / 2;                      // token rows per CTA
    // SUPER (the converting variants on regular batches): a tile is one weight
    // tile and up to kSuperN tokens of its group, in two MMA sub-tiles (the
    // first of up to kTileN tokens, the second of up to kSuperN - kTileN), so
    // that each weight k-block is converted once for all of them.  Its two
    // accumulators take both TMEM slots; other tiles take one slot each and
    // alternate between the two.
    static constexpr bool kSuper = FMT != WFMT_BF16 && !SMALL;
    static constexpr int kSuperN = kSuper ? 448 : kTileN;          // tokens per tile
    static constexpr int kHalf1 = (kSuperN - kTileN) / 2;          // sub-tile 1 rows per CTA
    static constexpr uint32_t kBBytes = (kHalfN + kHalf1) * BK * 2;
    static constexpr int kAccCols = kTileN;                        // TMEM columns per accumulator
    static constexpr uint32_t kTmemCols = 2 * kAccCols;            // two slots
    static constexpr int kChunks = SMALL ? 1 : 2;                  // 32-column TMEM loads per wait
    static constexpr bool kPair = MODE == GEMM_SWIGLU;      // 64 gate + 64 up rows per CTA
    static constexpr int kRowsCta = gemm_rows(MODE);        // output weight rows per CTA
    static constexpr int kRowsTile = 2 * kRowsCta;          // per CTA pair
    // MX gate/up: the converters lay the CTA's 128 operand rows out as blocks
    // of 16 gate rows followed by the same 16 up rows, so each epilogue warp's
    // 32 accumulator lanes hold both halves of 16 rows and exchange them with
    // a shuffle.  bf16 gate/up: TMA loads 64 gate rows and then 64 up rows
    // (two large boxes; sixteen-row boxes cost more in TMA issue than the
    // exchange they save) and the up warps pass their values to the gate
    // warps through shared memory.
    static constexpr bool kInterleave = kPair && kConv;
    static constexpr uint32_t kXBytes = kPair && !kConv ? 2 * 32 * kXPad * 4 : 0;
    static constexpr uint32_t kStageBytes = kABytes + kBBytes;  // operand ring entry
    static constexpr int kStages = SMALL ? 4 : (kSuper ? 4 : (kConv ? 5 : 6));
    static constexpr uint32_t kF8RowBytes = BK;                 // weight bytes per row and k-block
    static constexpr uint32_t kF8Bytes = BM * kF8RowBytes;      // fp8 weight tile
    static constexpr int kF8Stages = SMALL ? 12 : (kSuper ? 4 : (kConv ? 5 : 0));
    static constexpr int kScPerKb = BK / 32;                    // scale bytes per row and k-block
    static constexpr uint32_t kScBytes = BM * 8 * kScPerKb;     // 8 k-blocks of scales
    static constexpr int kScStages = kConv ? 2 : 0;
    static constexpr uint32_t kRingBytes =
        kStages * kStageBytes + kF8Stages * kF8Bytes + kScStages * kScBytes;
    // tile queue: kQueue entries; arrivals releasing an entry on the leader:
    // its MMA thread and 4 epilogue warps, the peer's producer and 4 epilogue
    // warps, and with converters both CTAs' weight producers and converter warps
    // bf16 weights: tiles come from a queue fed by a global counter (the
    // token tiles of a weight tile start together and share it in L2).  The
    // converting variants are limited by their converters, not by operand
    // traffic, and run faster on the static round-robin order.
    static constexpr bool kDynamic = !kConv;
    static constexpr int kQueue = 8;
    static constexpr int kQueueAhead = 2;  // < kQueue
    static constexpr int kQueueReaders = 10 + (kConv ? 2 + 2 * 8 : 0);
    static constexpr int kBarriers = 2 * kStages + 2 * kF8Stages + 2 * kScStages + 9 + 2 * kQueue;
    static constexpr int kConvWarps = SMALL ? 16 : 8;
    static constexpr int kConvPerKb = SMALL ? 4 : 2;            // warps per k-block
    static constexpr int kConvGroups = kConvWarps / kConvPerKb;  // k-blocks in flight
    // Warps: 0 TMA producer, 1 MMA issuer, 2..5 epilogue, then the converters
    // and the fp8 producer.  A warp issues on scheduler warp % 4; with SUPER
    // the block has 16 warps and no converter shares scheduler 1 with the MMA
    // issuer (converters 6, 7, 8, 10, 11, 12, 14, 15; fp8 producer 9; 13 idle):
    // the converters' dense arithmetic otherwise takes the issue slots the MMA
    // thread needs to keep the tensor pipe fed (measured: gate/up 14 % faster).
    static constexpr bool kRemap = kSuper;
    static constexpr int kThreads = kRemap ? 512 : (kConv ? 192 + 32 * kConvWarps + 32 : 192);
    static constexpr int kFp8Warp = kRemap ? 9 : 6 + kConvWarps;
    static constexpr int kIdleWarp = kRemap ? 13 : -1;
};

struct Tile {
    int m, g, n_valid, brow, arow;
    int half;     // sub-tile 0: MMA N / 2, token rows each CTA holds (a multiple of 16)
    int n1;       // tokens of sub-tile 1 (the tile's tokens from kTileN on); 0: none
    int half1;    // sub-tile 1: MMA N / 2 (0 when n1 == 0)
    bool shared;
    bool reused;  // the expert has several token tiles: its weight tiles are read again
};

// The tile order.  Groups (experts, then the shared expert) with several token
// tiles ("hot": their weight tiles are compute-bound, each read by several
// clusters) and groups with one ("cold": each weight tile streams from HBM once
// for a few tokens) form two lists, each in group order, and within a hot
// group's weight tile its token tiles run back to back (on neighbouring
// clusters) so that they share it in L2.  The two lists are merged in
// proportion -- position t is hot iff floor((t + 1) H / N) > floor(t H / N),
// H hot tiles of N -- so every wave of clusters mixes tensor-bound and
// HBM-bound tiles instead of running the hot experts and the cold ones in
// separate phases.  The order decides only which cluster computes a tile and
// when, never how: each tile is still computed whole by one CTA pair.
struct Sched {
    const int* hs;    // [GG + 1] prefix of token tiles over hot groups
    const int* cs;    // [GG + 1] prefix of cold groups
    const int* gcnt;  // [GG] tokens per group
    const int* goff;  // [GG] first token row of each group
    int GG;
    int64_t H, N;     // hot tiles, all tiles
};

// Token tiles of a group of c tokens: ceil(c / TS) of them, of equal size
// (the last one taking the rest) when TS > TN (a tile then holds two MMA
// sub-tiles: its first TN tokens and the rest), of TN and a tail otherwise.
// A sub-tile's MMA width N is its token count rounded up to 32 (at least 64):
// a valid N for the M = 256 pair MMA, which takes multiples of 16.
template <int MODE, int TN, int TS>
__device__ __forceinline__ Tile make_tile(const TilePos& pos, uint32_t rank, const GemmParams& p,
                                          const Sched& sc) {
    Tile tl;
    tl.g = pos.g;
    tl.m = pos.m;
    tl.reused = pos.hot;
    const int nt = pos.nt;
    const int lo = tl.g;
    const int* gcnt = sc.gcnt;
    const int* goff = sc.goff;
    const int c = gcnt[lo];
    int sz = TS;
    if (TS > TN) {
        const int ntg = max(1, (c + TS - 1) / TS);
        sz = (c + ntg - 1) / ntg;
    }
    tl.n_valid = min(sz, c - nt * sz);
    const int n0 = min(TN, tl.n_valid);
    tl.half = min(TN, max(64, (n0 + 31) & ~31)) >> 1;
    tl.n1 = tl.n_valid - n0;
    tl.half1 = tl.n1 > 0 ? max(64, (tl.n1 + 31) & ~31) >> 1 : 0;
    tl.brow = goff[lo] + nt * sz;
    tl.shared = lo >= p.G;
    tl.arow = (tl.shared ? 0 : lo * p.M) + tl.m * 2 * gemm_rows(MODE) + rank * gemm_rows(MODE);
    return tl;
}

// Token rows CTA `rank` holds of a tile: [rank * half, rank * half + half) of
// the tile's tokens, of which this many exist; they are loaded in 32-row boxes
// (a CTA with none leaves its rows stale: they only feed columns never stored;
// rows a last box loads past them, from the next group or zero-filled past
// the tensor's end, likewise).
__device__ __forceinline__ int b_rows(const Tile& tl, uint32_t rank) {
    return min(max(tl.n_valid - static_cast<int>(rank) * tl.half, 0), tl.half);
}
__device__ __forceinline__ uint32_t b_bytes(const Tile& tl, uint32_t rank) {
    return ((b_rows(tl, rank) + 31) >> 5) * kBox32Bytes;
}
// The same for sub-tile 1 (tokens [TN, TN + n1) of the tile).
__device__ __forceinline__ int b_rows1(const Tile& tl, uint32_t rank) {
    return min(max(tl.n1 - static_cast<int>(rank) * tl.half1, 0), tl.half1);
}
__device__ __forceinline__ uint32_t b_bytes1(const Tile& tl, uint32_t rank) {
    return ((b_rows1(tl, rank) + 31) >> 5) * kBox32Bytes;
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
// words (element 0 in the low half of `lo`), exactly, by the float route above.
// Used for blocks the integer route below does not cover.
__device__ __forceinline__ void e4m3x4_to_bf16x4(uint32_t w, uint32_t s, uint32_t& lo,
                                                 uint32_t& hi) {
    const float scale = e8m0_scale(s);
    lo = e4m3x2_to_bf16x2(w & 0xFFFFu, scale);
    hi = e4m3x2_to_bf16x2(w >> 16, scale);
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, 0, %2;" : "=r"(d) : "r"(a), "r"(sel));
    return d;
}

// Four normal E4M3 bytes (none flagged by e4m3x16_special) with 7 <= s <= 246
// -> four bf16, exactly.  The bf16 of e4m3 * 2^(s-127) is the E4M3 pattern
// with its 7 exponent+mantissa bits moved to bf16 bits [10:4], the sign to bit
// 15 and the exponent re-biased by s - 7 (E4M3 bias 7, bf16 bias 127); the
// sum E + s - 7 stays within [1, 254], so it never carries into the sign.
// The byte permute places each byte in the low half of a 16-bit lane with its
// sign replicated through the high byte; the mask keeps the seven bits [6:0]
// and one copy of the sign (bit 11), and one multiply-add by 16 moves them to
// [10:4] and bit 15 and adds the re-bias (no bit crosses into the other lane).
__device__ __forceinline__ void e4m3x4_rebias(uint32_t w, uint32_t k, uint32_t& lo, uint32_t& hi) {
    lo = (prmt(w, 0x9180u) & 0x087F087Fu) * 16u + k;  // bytes 0, 1
    hi = (prmt(w, 0xB3A2u) & 0x087F087Fu) * 16u + k;  // bytes 2, 3
}

// Nonzero (bit 7 of some byte) iff one of the sixteen E4M3 bytes of q is zero
// or subnormal (low seven bits below 8) or NaN (low seven bits all ones): with
// t the low seven bits of each byte, bit 7 of t + 0x78 is clear iff t < 8 and
// bit 7 of t + 0x01 is set iff t == 0x7F; neither sum carries out of its byte.
__device__ __forceinline__ uint32_t e4m3x16_special(const uint4& q) {
    uint32_t acc = 0;
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t t = w[i] & 0x7F7F7F7Fu;
        acc |= ~(t + 0x78787878u) | (t + 0x01010101u);
    }
    return acc & 0x80808080u;
}

// Operand row of converted weight row r (0..127) of a CTA's tile: with the
// gate/up interleave, 16 gate rows then the same 16 up rows, four times (the
// low 3 bits, which pick the 128-byte swizzle, stay r's).
template <bool kInterleave>
__device__ __forceinline__ int mx_operand_row(int r) {
    return kInterleave ? ((r & 63) >> 4) * 2 * kSwigluBlock + (r >= 64 ? kSwigluBlock : 0) + (r & 15)
                       : r;
}

// One converter warp's share of an MXFP8 k-block: rows [row0, row0 + kRows)
// of the CTA's 128 (64 E4M3 bytes per row in f8, 16 scale bytes per row per 8
// k-blocks in sc, this k-block's pair at 2 * kb8), written as bf16 into the
// 128-byte-swizzled operand tile st.  Lane l takes the 16-value tasks
// (c2 = 2 (l % 4), rows row0 + l / 4 + 8 i): its rows advance by 8, so the
// swizzled 16-byte chunks it writes are the same in every row.  Four tasks'
// loads are issued before their arithmetic and stores; the exceptional bytes
// (zero, subnormal, NaN) and scales outside [7, 246] are only detected on the
// way, and a lane redoes just the tasks that met one by the exact float route
// after the fast pass (about one task in 800 for quantised N(0, 0.02) weights).
template <int kRows, bool kInterleave>
__device__ __forceinline__ void mx_convert_rows(const uint8_t* f8, const uint8_t* sc, int kb8,
                                                uint8_t* st, int row0, int lane) {
    constexpr int kIters = kRows * 4 / 32;
    constexpr int kBatch = kIters < 4 ? kIters : 4;
    static_assert(kIters % kBatch == 0, "whole batches");
    const int rl = row0 + (lane >> 2);
    const int c2 = (lane & 3) * 2;
    const uint32_t sw0 = static_cast<uint32_t>((c2 ^ (rl & 7)) << 4);
    const uint32_t sw1 = static_cast<uint32_t>(((c2 + 1) ^ (rl & 7)) << 4);
    const uint8_t* fp = f8 + rl * 64 + c2 * 8;
    const uint8_t* sp = sc + rl * 16 + kb8 * 2 + (c2 >> 2);
    uint32_t bad = 0;
#pragma unroll
    for (int b0 = 0; b0 < kIters; b0 += kBatch) {
        uint4 q[kBatch];
        uint32_t sb[kBatch];
#pragma unroll
        for (int j = 0; j < kBatch; ++j) {
            q[j] = *reinterpret_cast<const uint4*>(fp + (b0 + j) * 8 * 64);
            sb[j] = sp[(b0 + j) * 8 * 16];
        }
#pragma unroll
        for (int j = 0; j < kBatch; ++j) {
            // ((s - 7) << 7) in both 16-bit lanes
            const uint32_t kk = sb[j] * 0x00800080u - 0x03800380u;
            uint4 o0, o1;
            e4m3x4_rebias(q[j].x, kk, o0.x, o0.y);
            e4m3x4_rebias(q[j].y, kk, o0.z, o0.w);
            e4m3x4_rebias(q[j].z, kk, o1.x, o1.y);
            e4m3x4_rebias(q[j].w, kk, o1.z, o1.w);
            if (e4m3x16_special(q[j]) | ((sb[j] - 7u) > 239u)) bad |= 1u << (b0 + j);
            uint8_t* row = st + mx_operand_row<kInterleave>(rl + 8 * (b0 + j)) * 128;
            *reinterpret_cast<uint4*>(row + sw0) = o0;
            *reinterpret_cast<uint4*>(row + sw1) = o1;
        }
    }
    while (bad) {
        const int i = __ffs(bad) - 1;
        bad &= bad - 1;
        {
            const uint4 q = *reinterpret_cast<const uint4*>(fp + i * 8 * 64);
            const uint32_t sbyte = sp[i * 8 * 16];
            uint4 o0, o1;
            e4m3x4_to_bf16x4(q.x, sbyte, o0.x, o0.y);
            e4m3x4_to_bf16x4(q.y, sbyte, o0.z, o0.w);
            e4m3x4_to_bf16x4(q.z, sbyte, o1.x, o1.y);
            e4m3x4_to_bf16x4(q.w, sbyte, o1.z, o1.w);
            uint8_t* row = st + mx_operand_row<kInterleave>(rl + 8 * i) * 128;
            *reinterpret_cast<uint4*>(row + sw0) = o0;
            *reinterpret_cast<uint4*>(row + sw1) = o1;
        }
    }
}

// Epilogue store of bf16 outputs: lanes 2i and 2i + 1 hold the values of two
// adjacent output rows (r, r + 1; rows are the contiguous axis of the output)
// for the same N tokens; they swap half of them so that lane 2i stores the
// even tokens' and lane 2i + 1 the odd tokens' row pair as one bf16x2 word:
// one conversion and one store per two outputs, the exchanges first.  `at`
// is the output element (first token, row r & ~1), `ld` the row stride of a
// token in elements, n_left the valid tokens from the first on.
template <int N>
__device__ __forceinline__ void store_bf16_row_pairs(const float (&h)[N], int lane,
                                                     __nv_bfloat16* at, int64_t ld, int n_left,
                                                     bool row_ok) {
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
        if (row_ok && 2 * jj + odd < n_left) y[jj * ld] = pk[jj];  // token 2 jj + odd
}

template <int MODE, int FMT, bool SMALL>
__global__ void __launch_bounds__(PCfg<MODE, FMT, SMALL>::kThreads, 1)
    pair_gemm_kernel(const __grid_constant__ GemmParams p) {
    using C = PCfg<MODE, FMT, SMALL>;
    constexpr bool MX = C::kConv;  // converter warps feed the A operand
    constexpr int kStages = C::kStages;
    constexpr uint32_t kStageBytes = C::kStageBytes;
    extern __shared__ uint8_t smem_raw[];
    // Offsetting the shared array itself (never through an integer) keeps every
    // derived pointer in the shared address space, so that accesses through
    // them compile to shared-memory loads and stores, not generic ones.
    uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    uint8_t* f8ring = smem + kStages * kStageBytes;
    uint8_t* scring = f8ring + C::kF8Stages * C::kF8Bytes;
    float* xbuf = reinterpret_cast<float*>(smem + C::kRingBytes);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kRingBytes + C::kXBytes);
    uint64_t* empty = full + kStages;
    uint64_t* tfull = empty + kStages;
    uint64_t* tempty = tfull + 2;
    uint64_t* drain = tempty + 2;
    uint64_t* xfull = drain + 1;               // bf16 gate/up: up values in xbuf
    uint64_t* xempty = xfull + 2;
    uint64_t* f8full = xempty + 2;             // MX, local: fp8 tile landed
    uint64_t* f8empty = f8full + C::kF8Stages;  // MX, local: converters done with it
    uint64_t* scfull = f8empty + C::kF8Stages;
    uint64_t* scempty = scfull + C::kScStages;
    uint64_t* qfull = scempty + C::kScStages;  // tile queue entry written (local)
    uint64_t* qempty = qfull + C::kQueue;      // leader: entry read by every role
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(full + C::kBarriers);
    volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);
    volatile int* tq = reinterpret_cast<volatile int*>(tmem_slot + 4);  // [kQueue] tile indices
    const int GG = p.G + p.has_shared;
    int* hs = reinterpret_cast<int*>(tmem_slot + 4 + C::kQueue);
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
            const int ntg = (c + C::kSuperN - 1) / C::kSuperN;
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
            const int ntg = (gcnt[g] + C::kSuperN - 1) / C::kSuperN;
            if (ntg > 1) run_h += ntg; else run_c += ntg;
        }
        if (lane == 31) {
            hs[GG] = incl_h;
            cs[GG] = incl_c;
        }
    } else if (warp == 1) {
        tmem_alloc_pair(tmem_slot, C::kTmemCols);
        tmem_relinquish_pair();
    } else if (threadIdx.x == 64) {
        for (int s = 0; s < kStages; ++s) {
            // MX: the leader's full barrier also waits for the 4 converter
            // warps of each CTA.
            // MX: + the converter warps of one k-block in each CTA
            mbar_init(&full[s], MX ? 1 + 2 * C::kConvPerKb : 1);
            mbar_init(&empty[s], 1);
        }
        for (int s = 0; s < C::kF8Stages; ++s) {
            mbar_init(&f8full[s], 1);
            mbar_init(&f8empty[s], C::kConvPerKb);
        }
        for (int s = 0; s < C::kScStages; ++s) {
            mbar_init(&scfull[s], 1);
            mbar_init(&scempty[s], 8 * C::kConvPerKb);  // 8 k-blocks per scale box
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&tfull[a], 1);
            mbar_init(&xfull[a], 1);
            mbar_init(&xempty[a], 1);
            mbar_init(&tempty[a], 8);  // 4 epilogue warps in each of the two CTAs
        }
        for (int q = 0; q < C::kQueue; ++q) {
            mbar_init(&qfull[q], 1);
            mbar_init(&qempty[q], C::kQueueReaders);
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
    const Sched sched{hs, cs, gcnt, goff, GG, static_cast<int64_t>(hs[GG]) * p.MT,
                   static_cast<int64_t>(hs[GG] + cs[GG]) * p.MT};
    const int total = static_cast<int>(sched.N);
    const uint64_t tmo = p.timeout_ns;
    // the tile order (tile_walk.cuh), walked forward by each role as it reads
    // the tiles (static: every ncl-th; dynamic: the queue's increasing entries)
    const TileOrder order{hs, cs, GG, p.MT, static_cast<uint32_t>(sched.H),
                          static_cast<uint32_t>(sched.N)};
    TileWalk walk = tile_walk_begin(0, order);

    // ---- tile queue ----
    // The pair takes tiles in order from the global counter: the leader's
    // producer thread draws the next index, writes it into entry j % kQueue of
    // both CTAs' queues (-1 once the tiles are exhausted) and arrives on both
    // CTAs' "written" barriers (cluster-scope release for the peer); every
    // other role reads entries j = 0, 1, ... in order (cluster-scope acquire)
    // and releases each on the leader's "read" barrier.  Pairs that run ahead
    // take more tiles, and the token tiles of a weight tile start together on
    // whichever pairs are free, so they share it in L2.  An entry is rewritten
    // only after all its readers released it, so a reader is never more than
    // one phase behind.
    auto q_release = [&](int slot) {
        if (leader)
            mbar_arrive(&qempty[slot]);
        else
            mbar_arrive_cluster(map_to_rank(&qempty[slot], 0));
    };
    // single-thread reader: false when the wait ran out (abort raised)
    auto q_read = [&](int j, int& t, int where) -> bool {
        const int slot = j % C::kQueue;
        if (!mbar_wait_cluster(&qfull[slot], static_cast<uint32_t>(j / C::kQueue) & 1u, abort, tmo)) {
            if (!*abort) raise_timeout(p, abort, where);
            return false;
        }
        t = tq[slot];
        q_release(slot);
        return true;
    };
    // whole-warp reader
    auto q_read_warp = [&](int j, int& t, int where) -> bool {
        const int slot = j % C::kQueue;
        if (!__all_sync(0xffffffffu, mbar_wait_cluster(&qfull[slot],
                                                      static_cast<uint32_t>(j / C::kQueue) & 1u,
                                                      abort, tmo))) {
            if (lane == 0 && !*abort) raise_timeout(p, abort, where);
            return false;
        }
        t = tq[slot];
        __syncwarp();
        if (lane == 0) q_release(slot);
        return true;
    };
    // the leader's producer: draw and publish entry j
    auto q_publish = [&](int j, int& t) -> bool {
        const int slot = j % C::kQueue;
        if (!mbar_wait(&qempty[slot], (static_cast<uint32_t>(j / C::kQueue) & 1u) ^ 1u, abort, tmo)) {
            if (!*abort) raise_timeout(p, abort, 19);
            return false;
        }
        t = atomicAdd(p.tile_counter, 1);
        if (t >= total) t = -1;
        tq[slot] = t;
        st_shared_cluster_u32(map_to_rank(const_cast<int*>(&tq[slot]), 1), static_cast<uint32_t>(t));
        mbar_arrive(&qfull[slot]);
        mbar_arrive_cluster(map_to_rank(&qfull[slot], 1));
        return true;
    };
    // static order: the pair's j-th tile is cid + j * ncl (-1 past the end)
    const int cid = static_cast<int>(cluster_id_x());
    const int ncl = static_cast<int>(nclusters_x());
    auto tile_static = [&](int j) -> int {
        const int64_t t = cid + static_cast<int64_t>(j) * ncl;
        return t < total ? static_cast<int>(t) : -1;
    };
    // the j-th tile for a reader role (single thread or whole warp)
    auto next_tile = [&](int j, int& t, int where, bool whole_warp) -> bool {
        if constexpr (!C::kDynamic) {
            t = tile_static(j);
            return true;
        } else {
            return whole_warp ? q_read_warp(j, t, where) : q_read(j, t, where);
        }
    };

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer (both CTAs) ----------------
            tma_prefetch_desc(&p.a0);
            tma_prefetch_desc(&p.b);
            if (p.has_shared) tma_prefetch_desc(&p.as0);
            // Weight tiles read by one cluster only stream through L2; those of
            // an expert with several token tiles stay, like the token rows.
            const uint64_t pol_once = l2_policy_evict_first();
            const uint64_t pol_again = l2_policy_evict_last();
            const uint64_t pol_x = l2_policy_evict_last();
            int stage = 0;
            uint32_t phase = 0;
            uint32_t issued = 0, last_par = 0;
            bool ok = p.stall_test == 0;
            // the leader publishes entries kQueueAhead beyond the one it loads,
            // so that the weight producer of the converting variants learns
            // the next tile early enough to prefetch it
            int published = 0;
            bool ended = false;
            for (int j = 0; ok; ++j) {
                int t;
                if (!C::kDynamic) {
                    t = tile_static(j);
                } else if (leader) {
                    while (!ended && published <= j + C::kQueueAhead) {
                        int drawn;
                        if (!q_publish(published, drawn)) {
                            ok = false;
                            break;
                        }
                        ++published;
                        ended = drawn < 0;
                    }
                    if (!ok) break;
                    t = tq[j % C::kQueue];  // written by this thread, not yet reusable
                } else if (!next_tile(j, t, 19, false)) {
                    break;
                }
                if (t < 0) break;
                tile_walk_to(walk, t, order);
                const Tile tl =
                    make_tile<MODE, C::kTileN, C::kSuperN>(tile_walk_pos(walk, order), rank, p, sched);
                const uint64_t pol_w = tl.reused ? pol_again : pol_once;
                const CUtensorMap* ma0 = tl.shared ? &p.as0 : &p.a0;
                const CUtensorMap* ma1 = tl.shared ? &p.as1 : &p.a1;
                const int nbox = (b_rows(tl, rank) + 31) >> 5;
                const bool whole = !C::kSmall && nbox == C::kHalfN / 32;
                const uint32_t expect = (MX ? 0 : 2 * kABytes) + b_bytes(tl, 0) + b_bytes(tl, 1) +
                                        b_bytes1(tl, 0) + b_bytes1(tl, 1);
                const int brow = tl.brow + static_cast<int>(rank) * tl.half;
                // sub-tile 1 (SUPER): its rows follow sub-tile 0's in the tile's
                // tokens, and sub-tile 0's kHalfN rows in shared memory
                const int nbox1 = (b_rows1(tl, rank) + 31) >> 5;
                const int brow1 = tl.brow + C::kTileN + static_cast<int>(rank) * tl.half1;
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
                        // the A operand comes from the converter warps
                    } else if constexpr (C::kPair) {
                        if (p.a_packed) {  // gate and up rows adjacent: one copy
                            tma_load_2d_pair(st, ma0, bar, kb * BK, 2 * tl.arow, pol_w);
                        } else {
                            tma_load_2d_pair(st, ma0, bar, kb * BK, tl.arow, pol_w);
                            tma_load_2d_pair(st + kABytes / 2, ma1, bar, kb * BK, tl.arow, pol_w);
                        }
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
                    if constexpr (C::kSuper) {
                        for (int i = 0; i < nbox1; ++i)
                            tma_load_2d_pair(sb + (C::kHalfN / 32 + i) * kBox32Bytes, &p.b32, bar,
                                             kb * BK, brow1 + 32 * i, pol_x);
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
        // bf16 and small-batch variants: the whole warp runs the issue loop and
        // one elected lane issues each MMA and commit, a shorter issue path than
        // a lone thread's (an N = 64 pair MMA every 67 cycles instead of 119;
        // decode-sized MXFP8 layer 3.95 -> 3.67 ms).  The super-tile variant
        // keeps one thread (its 16-warp block ran ~1.5 % slower the other way).
        if constexpr (!C::kSuper) {
          if (leader) {
            // ---------------- MMA issuer (leader only, whole warp) ----------------
            auto wait_w = [&](uint64_t* bar, uint32_t par, int where) {
                if (__all_sync(0xffffffffu, mbar_wait(bar, par, abort, tmo))) return true;
                if (lane == 0 && !*abort) raise_timeout(p, abort, where);
                return false;
            };
            int stage = 0;
            uint32_t phase = 0;
            int su = 0;  // TMEM slot uses so far (one per tile)
            bool ok = true;
            for (int j = 0; ok; ++j) {
                int t;
                if (!next_tile(j, t, 27, true) || t < 0) break;
                tile_walk_to(walk, t, order);
                const Tile tl =
                    make_tile<MODE, C::kTileN, C::kSuperN>(tile_walk_pos(walk, order), rank, p, sched);
                if (!wait_w(&tempty[su & 1], ((su >> 1) & 1) ^ 1u, 13)) break;
                tc_fence_after();
                const uint32_t d0 = tmem_base + (su & 1) * C::kAccCols;
                const uint32_t idesc = idesc_bf16_f32(2 * BM, 2 * tl.half);
                for (int kb = 0; kb < p.KB; ++kb) {
                    if (!wait_w(&full[stage], phase, 14)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    // descriptors of the stage's tiles (1024-byte aligned); a
                    // K step of 16 advances the start address by 32 bytes
                    const uint32_t sa = smem_addr(smem + stage * kStageBytes);
                    const uint64_t da = sdesc_kmajor_sw128(sa);
                    const uint64_t db = sdesc_kmajor_sw128(sa + kABytes);
#pragma unroll
                    for (int k = 0; k < BK / 16; ++k)
                        umma_bf16_pair_w(d0, da + 2 * k, db + 2 * k, idesc, (kb | k) != 0);
                    umma_commit_pair_w(&empty[stage], 0x3);
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                umma_commit_pair_w(&tfull[su & 1], 0x3);
                ++su;
            }
            __syncwarp();
            umma_commit_pair_w(drain, 0x1);
            if (!__all_sync(0xffffffffu, mbar_wait(drain, 0, nullptr, tmo)) && lane == 0)
                raise_timeout(p, abort, 15);
          }
        } else {
          if (lane == 0 && leader) {
              // ---------------- MMA issuer (leader only) ----------------
              int stage = 0;
              uint32_t phase = 0;
              // TMEM slot uses so far: use u takes slot u % 2 in phase (u / 2) % 2;
              // a tile takes one slot, or two (sub-tiles 0 and 1) with SUPER
              int su = 0;
              bool ok = true;
              for (int j = 0; ok; ++j) {
                  int t;
                  if (!next_tile(j, t, 27, false) || t < 0) break;
                  tile_walk_to(walk, t, order);
                  const Tile tl =
                      make_tile<MODE, C::kTileN, C::kSuperN>(tile_walk_pos(walk, order), rank, p, sched);
                  const int ns = tl.half1 ? 2 : 1;
                  for (int u = 0; u < ns && ok; ++u) {
                      const int v = su + u;
                      if (!mbar_wait(&tempty[v & 1], ((v >> 1) & 1) ^ 1u, abort, tmo)) {
                          if (!*abort) raise_timeout(p, abort, 13);
                          ok = false;
                      }
                  }
                  if (!ok) break;
                  tc_fence_after();
                  const uint32_t d0 = tmem_base + (su & 1) * C::kAccCols;
                  const uint32_t d1 = tmem_base + ((su + 1) & 1) * C::kAccCols;
                  const uint32_t idesc = idesc_bf16_f32(2 * BM, 2 * tl.half);
                  const uint32_t idesc1 = idesc_bf16_f32(2 * BM, 2 * (ns == 2 ? tl.half1 : 32));
                  for (int kb = 0; kb < p.KB; ++kb) {
                      if (!mbar_wait(&full[stage], phase, abort, tmo)) {
                          if (!*abort) raise_timeout(p, abort, 14);
                          ok = false;
                          break;
                      }
                      tc_fence_after();
                      // descriptors of the stage's tiles (1024-byte aligned); a
                      // K step of 16 advances the start address by 32 bytes
                      const uint32_t sa = smem_addr(smem + stage * kStageBytes);
                      const uint64_t da = sdesc_kmajor_sw128(sa);
                      const uint64_t db = sdesc_kmajor_sw128(sa + kABytes);
                      const uint64_t db1 = sdesc_kmajor_sw128(sa + kABytes + C::kHalfN * 128);
                      // the two sub-tiles' MMAs of each K step back to back: they
                      // multiply the same A (weights) with different B (tokens)
  #pragma unroll
                      for (int k = 0; k < BK / 16; ++k) {
                          umma_bf16_pair(d0, da + 2 * k, db + 2 * k, idesc, (kb | k) != 0);
                          if (C::kSuper && ns == 2)
                              umma_bf16_pair(d1, da + 2 * k, db1 + 2 * k, idesc1, (kb | k) != 0);
                      }
                      umma_commit_pair(&empty[stage], 0x3);
                      if (++stage == kStages) {
                          stage = 0;
                          phase ^= 1u;
                      }
                  }
                  if (!ok) break;
                  umma_commit_pair(&tfull[su & 1], 0x3);
                  if (ns == 2) umma_commit_pair(&tfull[(su + 1) & 1], 0x3);
                  su += ns;
              }
              umma_commit_pair(drain, 0x1);
              if (!mbar_wait(drain, 0, nullptr, tmo)) raise_timeout(p, abort, 15);
          }
        }
    } else if (warp == C::kFp8Warp) {
        if constexpr (MX) {
            if (lane == 0) {
                // ---------------- fp8 weight producer (both CTAs) ----------------
                const uint64_t pol_once = l2_policy_evict_first();
                const uint64_t pol_again = l2_policy_evict_last();
                int fs = 0, ss = 0;
                uint32_t fph = 0, sph = 0;
                uint32_t f_issued = 0, f_par = 0, s_issued = 0, s_par = 0;
                bool ok = p.stall_test == 0;
                for (int j = 0; ok; ++j) {
                    int t;
                    if (!next_tile(j, t, 28, false) || t < 0) break;
                    tile_walk_to(walk, t, order);
                    const Tile tl =
                        make_tile<MODE, C::kTileN, C::kSuperN>(tile_walk_pos(walk, order), rank, p, sched);
                    const uint64_t pol_w = tl.reused ? pol_again : pol_once;
                    for (int kb = 0; kb < p.KB; ++kb) {
                        if ((kb & 7) == 0) {  // scales of the next 8 k-blocks
                            if (!mbar_wait(&scempty[ss], sph ^ 1u, abort, tmo)) {
                                if (!*abort) raise_timeout(p, abort, 20);
                                ok = false;
                                break;
                            }
                            uint8_t* sc = scring + ss * C::kScBytes;
                            mbar_arrive_expect_tx(&scfull[ss], C::kScBytes);
                            if constexpr (C::kPair) {
                                tma_load_2d(sc, &p.sa0, &scfull[ss], kb * C::kScPerKb, tl.arow, pol_w);
                                tma_load_2d(sc + C::kScBytes / 2, &p.sa1, &scfull[ss], kb * C::kScPerKb,
                                            tl.arow, pol_w);
                            } else {
                                tma_load_2d(sc, &p.sa0, &scfull[ss], kb * C::kScPerKb, tl.arow, pol_w);
                            }
                            s_issued |= 1u << ss;
                            s_par = (s_par & ~(1u << ss)) | (sph << ss);
                            if (++ss == C::kScStages) {
                                ss = 0;
                                sph ^= 1u;
                            }
                        }
                        if (!mbar_wait(&f8empty[fs], fph ^ 1u, abort, tmo)) {
                            if (!*abort) raise_timeout(p, abort, 21);
                            ok = false;
                            break;
                        }
                        uint8_t* f8 = f8ring + fs * C::kF8Bytes;
                        mbar_arrive_expect_tx(&f8full[fs], C::kF8Bytes);
                        if constexpr (C::kPair) {
                            tma_load_2d(f8, &p.a0, &f8full[fs], kb * C::kF8RowBytes, tl.arow, pol_w);
                            tma_load_2d(f8 + C::kF8Bytes / 2, &p.a1, &f8full[fs], kb * C::kF8RowBytes,
                                        tl.arow, pol_w);
                        } else {
                            tma_load_2d(f8, &p.a0, &f8full[fs], kb * C::kF8RowBytes, tl.arow, pol_w);
                        }
                        f_issued |= 1u << fs;
                        f_par = (f_par & ~(1u << fs)) | (fph << fs);
                        if (++fs == C::kF8Stages) {
                            fs = 0;
                            fph ^= 1u;
                        }
                    }
                }
                for (int s2 = 0; s2 < C::kF8Stages; ++s2)
                    if (f_issued & (1u << s2))
                        if (!mbar_wait(&f8full[s2], (f_par >> s2) & 1u, nullptr, tmo))
                            raise_timeout(p, abort, 22);
                for (int s2 = 0; s2 < C::kScStages; ++s2)
                    if (s_issued & (1u << s2))
                        if (!mbar_wait(&scfull[s2], (s_par >> s2) & 1u, nullptr, tmo))
                            raise_timeout(p, abort, 23);
            }
        }
    } else if (warp == C::kIdleWarp) {
        // no role: keeps converter warps off the MMA issuer's scheduler
    } else if (warp >= 6) {
        if constexpr (MX) {
            // ---------------- converters (warps >= 6, both CTAs) ----------------
            // kConvGroups groups of kConvPerKb warps; group g converts this CTA's
            // k-blocks i = g, g + kConvGroups, ... of the tile sequence, warp j
            // of the group rows [j * 128 / kConvPerKb, ...).  A tile has KB
            // k-blocks with KB % 8 == 0, so scale groups never straddle tiles.
            // Phase safety of the parity waits below: a group's previous k-block
            // i - G (G = kConvGroups) needed MMA(i - G - kStages) and the loads of
            // k-block i - G and of its scale group; with G <= kStages,
            // G <= kF8Stages and G <= 8 this proves that every slot a wait of
            // k-block i looks at is at most one phase behind the awaited one.
            static_assert(C::kConvGroups <= C::kStages && C::kConvGroups <= C::kF8Stages &&
                              C::kConvGroups <= 8,
                          "converter groups must not outrun the rings");
            // 0 .. kConvWarps - 1, skipping the fp8 producer and idle warps
            const int cw = C::kRemap ? warp - 6 - (warp > C::kFp8Warp) - (warp > C::kIdleWarp)
                                     : warp - 6;
            const int grp_w = cw / C::kConvPerKb;
            const int sub = cw % C::kConvPerKb;
            constexpr int kRowsPerWarp = BM / C::kConvPerKb;
            auto wait_all = [&](uint64_t* bar, uint32_t par, int where) {
                if (__all_sync(0xffffffffu, mbar_wait(bar, par, abort, tmo))) return true;
                if (lane == 0 && !*abort) raise_timeout(p, abort, where);
                return false;
            };
            // k-block i of the pair's sequence belongs to queue entry i / KB;
            // KB is a multiple of the group count, so every group converts
            // KB / kConvGroups k-blocks of every tile and reads every entry, in
            // order, at its first k-block of that tile
            const int per_tile = p.KB / C::kConvGroups;
            int left = 0, j = 0;
            for (int64_t i = grp_w;; i += C::kConvGroups) {
                if (left == 0) {
                    int t;
                    if (!next_tile(j++, t, 29, true) || t < 0) break;
                    left = per_tile;
                }
                --left;
                const int os = static_cast<int>(i % kStages);
                const uint32_t oph = static_cast<uint32_t>((i / kStages) & 1);
                const int fs = static_cast<int>(i % C::kF8Stages);
                const uint32_t fph = static_cast<uint32_t>((i / C::kF8Stages) & 1);
                const int64_t grp = i >> 3;
                const int ss = static_cast<int>(grp % C::kScStages);
                const uint32_t sph = static_cast<uint32_t>((grp / C::kScStages) & 1);
                if (!wait_all(&scfull[ss], sph, 24) || !wait_all(&f8full[fs], fph, 25) ||
                    !wait_all(&empty[os], oph ^ 1u, 26))
                    break;
                uint8_t* st = smem + os * kStageBytes;
                const uint8_t* f8 = f8ring + fs * C::kF8Bytes;
                const uint8_t* sc = scring + ss * C::kScBytes;
                const int kb8 = static_cast<int>(i & 7);
                mx_convert_rows<kRowsPerWarp, C::kInterleave>(f8, sc, kb8, st, sub * kRowsPerWarp,
                                                              lane);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&f8empty[fs]);
                    mbar_arrive(&scempty[ss]);
                    if (leader)
                        mbar_arrive(&full[os]);
                    else
                        mbar_arrive_operand_ready(map_to_rank(&full[os], 0));
                }
            }
        }
    } else {
        // ---------------- epilogue (warps 2..5, both CTAs) ----------------
        // Warp q reads accumulator lanes [32q, 32q + 32).  MX gate/up: lanes
        // 0..15 of the warp hold gate rows f..f+15 and lanes 16..31 the same
        // rows of the up projection; each lane swaps half of its 32 columns
        // with the lane 16 away, then finishes 16 outputs of its row.  bf16
        // gate/up: warps 0, 1 hold gate rows and warps 2, 3 the matching up
        // rows, which they pass on through xbuf.
        const int q = warp & 3;
        const int pr = q & 1;
        const bool up_warp = q >= 2;
        const bool up_lane = lane >= kSwigluBlock;
        int su = 0;  // TMEM slot uses so far, as in the MMA issuer
        uint32_t xph = 0;
        bool ok = true;
        for (int j = 0; ok; ++j) {
            int t;
            if (!next_tile(j, t, 30, true) || t < 0) break;
            tile_walk_to(walk, t, order);
            const Tile tile =
                make_tile<MODE, C::kTileN, C::kSuperN>(tile_walk_pos(walk, order), rank, p, sched);
            const int ns = tile.half1 ? 2 : 1;
          for (int sub = 0; sub < ns && ok; ++sub) {
            // sub-tile `sub` of the tile: its tokens and its TMEM slot
            Tile tl = tile;
            if (sub == 1) {
                tl.brow += C::kTileN;
                tl.n_valid = tile.n1;
            } else {
                tl.n_valid = min(tile.n_valid, C::kTileN);
            }
            const int acc = (su + sub) & 1;
            const uint32_t acc_phase = static_cast<uint32_t>((su + sub) >> 1) & 1u;
            const bool ready = __all_sync(0xffffffffu, mbar_wait(&tfull[acc], acc_phase, abort, tmo));
            if (!ready) {
                if (lane == 0 && !*abort) raise_timeout(p, abort, 16);
                ok = false;
                break;
            }
            tc_fence_after();
            const int row = tl.m * C::kRowsTile + static_cast<int>(rank) * C::kRowsCta +
                            (C::kInterleave ? q * kSwigluBlock + (lane & (kSwigluBlock - 1))
                                            : (C::kPair ? pr : q) * 32 + lane);
            const bool row_ok = row < p.M;
            const uint32_t taddr =
                tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * C::kAccCols;
            // One chunk of 32 accumulator columns (tokens c0 .. c0 + 31);
            // false when a wait of the bf16 gate/up handoff ran out.
            auto chunk = [&](const float (&v)[32], int c0) -> bool {
                if constexpr (C::kInterleave) {
                    // all exchanges first, then 16 independent SwiGLUs, then the
                    // stores: no shuffle or store sits between two SwiGLUs, so
                    // they overlap
                    const int cb = c0 + (up_lane ? 16 : 0);
                    float other[16], h[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        other[j] = __shfl_xor_sync(0xffffffffu, up_lane ? v[j] : v[16 + j], 16);
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const float g = up_lane ? other[j] : v[j];
                        const float u = up_lane ? v[16 + j] : other[j];
                        h[j] = swiglu(g, u);
                    }
                    // rows pair up within M (a multiple of 64): both lanes of
                    // a pair agree on row_ok
                    store_bf16_row_pairs<16>(
                        h, lane,
                        static_cast<__nv_bfloat16*>(p.out) +
                            static_cast<int64_t>(tl.brow + p.out_row_off + cb) * p.ldo + (row & ~1),
                        p.ldo, tl.n_valid - cb, row_ok);
                } else if constexpr (C::kPair) {
                    float* xb = xbuf + pr * 32 * kXPad + lane * kXPad;
                    if (up_warp) {
                        if (!__all_sync(0xffffffffu, mbar_wait(&xempty[pr], xph ^ 1u, abort, tmo))) {
                            if (lane == 0 && !*abort) raise_timeout(p, abort, 17);
                            return false;
                        }
#pragma unroll
                        for (int j = 0; j < 32; ++j) xb[j] = v[j];
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&xfull[pr]);
                    } else {
                        if (!__all_sync(0xffffffffu, mbar_wait(&xfull[pr], xph, abort, tmo))) {
                            if (lane == 0 && !*abort) raise_timeout(p, abort, 18);
                            return false;
                        }
                        float u[32];
#pragma unroll
                        for (int j = 0; j < 32; ++j) u[j] = xb[j];
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&xempty[pr]);
                        float h[32];
#pragma unroll
                        for (int j = 0; j < 32; ++j) h[j] = swiglu(v[j], u[j]);
                        store_bf16_row_pairs<32>(
                            h, lane,
                            static_cast<__nv_bfloat16*>(p.out) +
                                static_cast<int64_t>(tl.brow + p.out_row_off + c0) * p.ldo + (row & ~1),
                            p.ldo, tl.n_valid - c0, row_ok);
                        if (p.save_a) {  // the backward keeps the pre-activations
#pragma unroll
                            for (int j = 0; j < 32; ++j) {
                                if (row_ok && c0 + j < tl.n_valid) {
                                    const int64_t at =
                                        static_cast<int64_t>(tl.brow + p.out_row_off + c0 + j) * p.ldo + row;
                                    p.save_a[at] = v[j];
                                    p.save_b[at] = u[j];
                                }
                            }
                        }
                    }
                    xph ^= 1u;
                } else {
                    if (tl.shared && p.out_shared) {
                        float* Ys = static_cast<float*>(p.out_shared);
                        const int tok0 = tl.brow - p.shared_b_off + c0;
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            if (row_ok && c0 + j < tl.n_valid)
                                Ys[static_cast<int64_t>(tok0 + j) * p.ldo + row] = v[j];
                    } else if (!C::kConv && p.out_f32) {
                        float* Yf = static_cast<float*>(p.out);
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            if (row_ok && c0 + j < tl.n_valid)
                                Yf[static_cast<int64_t>(tl.brow + c0 + j) * p.ldo + row] = v[j];
                    } else {
                        store_bf16_row_pairs<32>(
                            v, lane,
                            static_cast<__nv_bfloat16*>(p.out) +
                                static_cast<int64_t>(tl.brow + c0) * p.ldo + (row & ~1),
                            p.ldo, tl.n_valid - c0, row_ok);
                    }
                }
                return true;
            };
            // kChunks chunks per TMEM round trip
            for (int c0 = 0; c0 < tl.n_valid && ok; c0 += 32 * C::kChunks) {
                float va[32];
                tmem_ld32(taddr + c0, va);
                if constexpr (C::kChunks == 2) {
                    float vb[32];
                    tmem_ld32(taddr + c0 + 32, vb);
                    tmem_ld_wait();
                    tmem_regs_ready(va);
                    tmem_regs_ready(vb);
                    ok = chunk(va, c0) && (c0 + 32 >= tl.n_valid || chunk(vb, c0 + 32));
                } else {
                    tmem_ld_wait();
                    tmem_regs_ready(va);
                    ok = chunk(va, c0);
                }
            }
            if (!ok) break;
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(map_to_rank(&tempty[acc], 0));
          }
            su += ns;
        }
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync();  // neither CTA leaves while the pair may still touch its memory
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, C::kTmemCols);
    }
}

template <int MODE, int FMT, bool SMALL>
size_t pair_smem_bytes(int GG) {
    using C = PCfg<MODE, FMT, SMALL>;
    return 1024 + C::kRingBytes + C::kXBytes + C::kBarriers * 8 + 16 + C::kQueue * 4 +
           static_cast<size_t>(4 * GG + 2) * 4;
}

template <int MODE, int FMT, bool SMALL>
cudaError_t launch_pair_mode(const GemmParams& p, int clusters, cudaStream_t s) {
    const int GG = p.G + p.has_shared;
    const size_t smem = pair_smem_bytes<MODE, FMT, SMALL>(GG);
    cudaError_t e = cudaFuncSetAttribute(pair_gemm_kernel<MODE, FMT, SMALL>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * clusters, 1, 1);
    cfg.blockDim = dim3(PCfg<MODE, FMT, SMALL>::kThreads, 1, 1);
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
    e = cudaOccupancyMaxActiveClusters(&resident, pair_gemm_kernel<MODE, FMT, SMALL>, &cfg);
    if (e != cudaSuccess) return e;
    if (resident <= 0) return cudaErrorInvalidConfiguration;
    if (clusters > resident) {
        clusters = resident;
        cfg.gridDim = dim3(2 * clusters, 1, 1);
    }
    return cudaLaunchKernelEx(&cfg, pair_gemm_kernel<MODE, FMT, SMALL>, p);
}

}  // namespace

cudaError_t launch_pair_gemm(int mode, const GemmParams& p, int clusters, cudaStream_t s,
                             int wfmt, int small) {
    if (p.G + p.has_shared > kMaxGroups || clusters <= 0 || !p.cnt || !p.off || !p.tile_counter)
        return cudaErrorInvalidValue;
    if (wfmt != WFMT_BF16 && p.has_shared) return cudaErrorInvalidValue;  // shared expert is bf16
    if (wfmt != WFMT_BF16 && wfmt != WFMT_MXFP8) return cudaErrorInvalidValue;
    if (small && wfmt == WFMT_BF16) return cudaErrorInvalidValue;  // bf16 small batches: one-SM kernel
    if (mode == GEMM_SWIGLU) {
        if (wfmt == WFMT_MXFP8)
            return small ? launch_pair_mode<GEMM_SWIGLU, WFMT_MXFP8, true>(p, clusters, s)
                         : launch_pair_mode<GEMM_SWIGLU, WFMT_MXFP8, false>(p, clusters, s);
        return launch_pair_mode<GEMM_SWIGLU, WFMT_BF16, false>(p, clusters, s);
    }
    if (mode == GEMM_DOWN) {
        if (wfmt == WFMT_MXFP8)
            return small ? launch_pair_mode<GEMM_DOWN, WFMT_MXFP8, true>(p, clusters, s)
                         : launch_pair_mode<GEMM_DOWN, WFMT_MXFP8, false>(p, clusters, s);
        return launch_pair_mode<GEMM_DOWN, WFMT_BF16, false>(p, clusters, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace moe
