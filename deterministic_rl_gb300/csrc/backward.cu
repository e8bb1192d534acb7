// backward.cu -- the element-wise, quantising and data-movement kernels of the
// MoE layer backward (the grouped GEMMs are gemm_pair.cu and wgrad.cu).
//
// Composer 2 Technical Report, §6.1 "Training infrastructure" (Kernels): the
// MoE backward runs its grouped GEMMs in standard MXFP8 -- E4M3 values with
// one E8M0 scale per block of 32 elements.  MXFP8 is taken as the OCP
// Microscaling Formats (MX) v1.0 specification defines it: per block,
// X = floor(log2(max |v|)) - 8 (8 = the exponent of E4M3's largest normal),
// element = E4M3(v * 2^-X), nearest even, clamped to +-448.  Every operand of
// a grouped GEMM is quantised along that GEMM's contraction axis.  The operands
// of the dH and dXp GEMMs (the weight copies, dY and [dA | dB] along their
// rows) are written as E4M3 codes and E8M0 scale bytes (X + 127) for the
// block-scaled tensor-core MMA (gemm_bs.cu); the token-major operands of the
// weight-gradient GEMMs as the dequantised values e4m3 * 2^X in bf16, which
// holds them exactly (at most 4 significant bits, and the exponents the layer
// produces), so the bf16 tcgen05 MMAs there multiply exactly the MXFP8 values.
// The pages prefer a fast approximate division in the MXFP8 quantiser; the
// scaling by 2^-X here is a multiplication by a power of two, which is exact.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <cstdint>

#include "moe_internal.h"
#include "mx.cuh"

namespace moe {
namespace {

// ---- row sources ----------------------------------------------------------------

// 8 consecutive values of a row, as fp32.
struct SrcBf16 {
    static constexpr bool kUnitScale = true;  // every row's factor is 1
    const uint16_t* p;
    int64_t ld;
    // transposed quantiser: 8 bf16 of a row as stored, and the row's factor
    __device__ __forceinline__ uint4 raw8(int64_t row, int c, float& scale) const {
        scale = 1.0f;
        return *reinterpret_cast<const uint4*>(p + row * ld + c);
    }
};


// The gradient of an expert-input row: routed row r (dispatch order) is pair
// perm[r] = t*k + s and holds gate(t, s) * dout[t]; shared-expert row Tk + t
// holds dout[t]; both zero for a token whose replayed ids were rejected.
struct SrcDy {
    static constexpr bool kUnitScale = false;
    const uint16_t* dout;
    const float* gates;
    const int32_t* perm;
    const int32_t* valid;
    int k;
    int64_t Tk;
    int64_t ld;
    // the token t whose dout feeds row `row`, and the row's factor
    __device__ __forceinline__ void row_of(int64_t row, int64_t& t, float& scale) const {
        if (row < Tk) {
            const int32_t pair = perm[row];
            t = pair / k;
            scale = valid[t] ? gates[pair] : 0.0f;
        } else {
            t = row - Tk;
            scale = valid[t] ? 1.0f : 0.0f;
        }
    }
    // 8 bf16 of dout[t] as stored, from column c
    __device__ __forceinline__ uint4 load8(int64_t t, int c) const {
        return *reinterpret_cast<const uint4*>(dout + t * ld + c);
    }
    // transposed quantiser: 8 bf16 of the row's dout as stored, and its factor
    __device__ __forceinline__ uint4 raw8(int64_t row, int c, float& scale) const {
        int64_t t;
        row_of(row, t, scale);
        return load8(t, c);
    }
};

// ---- transposed quantisation (blocks of 32 along the rows) ----------------------------

// A tile covers 64 input rows (two MX blocks): its output columns, the input
// rows it reads and how many of them exist.
struct TqBlock {
    int64_t in_row0;
    int64_t out_col;  // element offset of the tile's column 0 in the output
    int nvalid;
};

struct TqArgs {
    int C;        // input columns = output rows
    int64_t ld;   // output row stride (elements)
    uint16_t* out;  // bf16 values (segment mode)
    // batch mode: E4M3 codes at the element offsets of `out`, and the E8M0
    // scale byte of each block of 32 at that offset / 32; sc_vec: every
    // group of kTqGroup tiles starts a 32-byte run of the scales (ld,
    // out_bstride and out_off multiples of 1024, scales 16-byte aligned)
    uint8_t* codes;
    uint8_t* scales;
    int sc_vec;
    // segment mode: groups of rows, each padded to a multiple of 64 output
    // columns starting at poff[g]; group g < E reads rows off[g] .. + cnt[g],
    // group E (the shared expert) rows shared_row0 .. + shared_rows
    const int32_t* cnt;
    const int32_t* off;
    const int32_t* poff;
    const int32_t* tile_g;  // group of each 64-row tile, -1 past the last
    int E, G;
    int64_t shared_row0;
    int shared_rows;
    // batch mode: nb matrices of R rows; matrix b's tile i -> output offset
    // b * out_bstride + out_off + 64 i
    int R;
    int64_t out_bstride, out_off;
    int64_t ntiles;  // 64-row tiles to visit
};

constexpr int kTqRows = 64;

template <bool SEG>
__device__ __forceinline__ bool tq_tile(const TqArgs& a, int64_t rt, TqBlock& blk) {
    if constexpr (SEG) {
        const int64_t p = rt * kTqRows;
        const int lo = a.tile_g[rt];  // poff[lo] <= p < poff[lo + 1]
        if (lo < 0) return false;
        const int local = static_cast<int>(p - a.poff[lo]);
        const int n = lo < a.E ? a.cnt[lo] : a.shared_rows;
        blk.in_row0 = (lo < a.E ? static_cast<int64_t>(a.off[lo]) : a.shared_row0) + local;
        blk.nvalid = min(max(n - local, 0), kTqRows);
        blk.out_col = p;
    } else {
        const int per = a.R / kTqRows;
        const int64_t b = rt / per;
        const int local = static_cast<int>(rt % per) * kTqRows;
        blk.in_row0 = b * a.R + local;
        blk.nvalid = kTqRows;
        blk.out_col = b * a.out_bstride + a.out_off + local;
    }
    return true;
}

// Two layouts of the CTA tile (64 input rows = two MX blocks, x 64 columns),
// both read down a column by the quantising threads without bank conflicts
// (the column index is XOR-swizzled by the row group) and written with 16-byte
// stores.  Quantising: thread t takes column t / 4 and rows 16 (t % 4) .. + 15;
// threads t and t ^ 1 hold the two halves of one 32-row block and share its
// maximum; the four threads of a column write its 64 output elements, one
// 128-byte line.

__device__ __forceinline__ void tq_store16(uint16_t* out, int64_t at, const float (&v)[16], int X) {
    float v0[8], v1[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        v0[i] = v[i];
        v1[i] = v[8 + i];
    }
    uint4* o = reinterpret_cast<uint4*>(out + at);
    o[0] = mx_qdq8(v0, X);
    o[1] = mx_qdq8(v1, X);
}

// 16 values of one block half as E4M3 codes of v * 2^-X (one 16-byte store),
// and the block's scale byte X + 127 from the thread holding its first half.
__device__ __forceinline__ uint4 mx_codes16(const float (&v)[16], int X) {
    const float inv = exp2i(-X);
    uint32_t w[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
        w[i] = __nv_cvt_float2_to_fp8x2(make_float2(v[2 * i] * inv, v[2 * i + 1] * inv),
                                        __NV_SATFINITE, __NV_E4M3);
    return make_uint4(w[0] | (w[1] << 16), w[2] | (w[3] << 16), w[4] | (w[5] << 16),
                      w[6] | (w[7] << 16));
}

__device__ __forceinline__ void mx_store_codes16(uint8_t* codes, uint8_t* scales, int64_t at,
                                                 const float (&v)[16], int X, bool first_half) {
    *reinterpret_cast<uint4*>(codes + at) = mx_codes16(v, X);
    if (first_half) scales[at / 32] = static_cast<uint8_t>(X + 127);
}

// bf16 rows as stored, times the row's factor where the source has one (the
// product is taken in fp32 before quantising): the tile holds the bf16 of
// rows 2R and 2R + 1 of a column in one 32-bit word, tp[R][column ^ sw(R)],
// sw(R) = 8 * ((R / 8) % 4).  Loading: thread t reads rows 2 (t / 8) and
// 2 (t / 8) + 1, columns 8 (t % 8) .. + 7 (two 16-byte loads).
// Rows 2R and 2R + 1 (R = t / 8), columns 8 (t % 8) .. + 7 into the tile.
__device__ __forceinline__ void tq_put_pair(uint32_t (*tp)[64], int tid, const uint4& lo,
                                            const uint4& hi) {
    const int R = tid >> 3, c8 = (tid & 7) * 8;
    const uint32_t l[4] = {lo.x, lo.y, lo.z, lo.w}, h[4] = {hi.x, hi.y, hi.z, hi.w};
    uint32_t w[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        w[2 * i] = __byte_perm(l[i], h[i], 0x5410);      // column 2i of both rows
        w[2 * i + 1] = __byte_perm(l[i], h[i], 0x7632);  // column 2i + 1
    }
    uint4* dst = reinterpret_cast<uint4*>(&tp[R][c8 ^ (((R >> 3) & 3) << 3)]);
    dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
    dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
}

template <class Src>
__device__ __forceinline__ void tq_load_tile(const Src& src, const TqBlock& blk, int cb, int tid,
                                             uint32_t (*tp)[64], float* rs) {
    const int R = tid >> 3, c8 = (tid & 7) * 8;
    uint4 lo = make_uint4(0, 0, 0, 0), hi = lo;
    float s0 = 0.0f, s1 = 0.0f;
    if (2 * R < blk.nvalid) lo = src.raw8(blk.in_row0 + 2 * R, cb + c8, s0);
    if (2 * R + 1 < blk.nvalid) hi = src.raw8(blk.in_row0 + 2 * R + 1, cb + c8, s1);
    if constexpr (!Src::kUnitScale) {
        if ((tid & 7) == 0) {
            rs[2 * R] = s0;
            rs[2 * R + 1] = s1;
        }
    }
    tq_put_pair(tp, tid, lo, hi);
}

// Column pass: thread t takes column c = t / 4, rows 16 (t % 4) .. + 15, times
// their factors; returns the block maximum shared with thread t ^ 1.
template <bool kUnitScale>
__device__ __forceinline__ float tq_column16(const uint32_t (*tp)[64], const float* rs, int tid,
                                             float (&v)[16]) {
    const int c = tid >> 2, part = tid & 3;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const uint32_t w = tp[part * 8 + j][c ^ (part << 3)];
        v[2 * j] = __uint_as_float(w << 16);
        v[2 * j + 1] = __uint_as_float(w & 0xFFFF0000u);
        if constexpr (!kUnitScale) {
            v[2 * j] *= rs[part * 16 + 2 * j];
            v[2 * j + 1] *= rs[part * 16 + 2 * j + 1];
        }
    }
    float m = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) m = fmaxf(m, fabsf(v[i]));
    return fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
}

template <class Src, bool SEG>
__global__ void __launch_bounds__(256, 8) tq16_kernel(Src src, TqArgs a) {
    __shared__ __align__(16) uint32_t tp[kTqRows / 2][64];
    __shared__ float rs[Src::kUnitScale ? 1 : kTqRows];
    const int tid = threadIdx.x;
    const int cchunks = a.C / 64;
    const int64_t items = a.ntiles * cchunks;
    for (int64_t it = blockIdx.x; it < items; it += gridDim.x) {
        const int64_t rt = it / cchunks;
        const int cb = static_cast<int>(it % cchunks) * 64;
        TqBlock blk;
        if (!tq_tile<SEG>(a, rt, blk)) continue;  // uniform across the CTA
        tq_load_tile(src, blk, cb, tid, tp, rs);
        __syncthreads();
        {
            const int c = tid >> 2, part = tid & 3;
            float v[16];
            const float m = tq_column16<Src::kUnitScale>(tp, rs, tid, v);
            tq_store16(a.out, static_cast<int64_t>(cb + c) * a.ld + blk.out_col + part * 16, v,
                       mx_block_exp(m));
        }
        __syncthreads();
    }
}

// The weight copies (batch mode) as E4M3 codes and scale bytes.  A tile gives
// each output row 2 scale bytes; a CTA item therefore takes one 64-column chunk
// of up to kTqGroup consecutive tiles of a matrix, collects their scale bytes
// in shared memory and stores each output row's 2 * kTqGroup = 32 bytes as one
// whole 32-byte sector (two 16-byte stores of neighbouring lanes) when the
// layout aligns them (a.sc_vec), bytewise otherwise.
constexpr int kTqGroup = 16;

__global__ void __launch_bounds__(256, 8) tq_codes_kernel(SrcBf16 src, TqArgs a) {
    __shared__ __align__(16) uint32_t tp[kTqRows / 2][64];
    __shared__ __align__(16) uint8_t sc[64][2 * kTqGroup];
    const int tid = threadIdx.x;
    const int cchunks = a.C / 64;
    const int per = a.R / kTqRows;                     // tiles per matrix
    const int gper = (per + kTqGroup - 1) / kTqGroup;  // tile groups per matrix
    const int64_t items = a.ntiles / per * gper * cchunks;
    const int c = tid >> 2, part = tid & 3;
    for (int64_t it = blockIdx.x; it < items; it += gridDim.x) {
        const int64_t grp = it / cchunks;
        const int cb = static_cast<int>(it % cchunks) * 64;
        const int64_t b = grp / gper;
        const int t0 = static_cast<int>(grp % gper) * kTqGroup;
        const int n = min(kTqGroup, per - t0);
        const int64_t col0 = b * a.out_bstride + a.out_off + static_cast<int64_t>(t0) * kTqRows;
        // this thread's input rows 2 (t / 8) and + 1 of the group's first tile,
        // and its 16 codes in output row cb + c; both advance by one tile
        const uint16_t* in =
            src.p + (b * a.R + t0 * kTqRows + 2 * (tid >> 3)) * src.ld + cb + (tid & 7) * 8;
        uint8_t* out = a.codes + static_cast<int64_t>(cb + c) * a.ld + col0 + part * 16;
        for (int j = 0; j < n; ++j) {
            tq_put_pair(tp, tid, *reinterpret_cast<const uint4*>(in),
                        *reinterpret_cast<const uint4*>(in + src.ld));
            in += kTqRows * src.ld;
            __syncthreads();
            float v[16];
            const int X = mx_block_exp(tq_column16<true>(tp, nullptr, tid, v));
            *reinterpret_cast<uint4*>(out) = mx_codes16(v, X);
            out += kTqRows;
            if ((part & 1) == 0) sc[c][2 * j + (part >> 1)] = static_cast<uint8_t>(X + 127);
            __syncthreads();
        }
        // row cb + r gets bytes [s0, s0 + 2n) of the scales; the next item's
        // first barrier orders these reads before sc is written again
        if (a.sc_vec && n == kTqGroup) {
            if (tid < 128) {
                const int r = tid >> 1, h = tid & 1;
                const int64_t s0 = (static_cast<int64_t>(cb + r) * a.ld + col0) / 32;
                *reinterpret_cast<uint4*>(a.scales + s0 + 16 * h) =
                    *reinterpret_cast<const uint4*>(&sc[r][16 * h]);
            }
        } else {
            for (int i = tid; i < 64 * 2 * n; i += blockDim.x) {
                const int r = i / (2 * n), q = i % (2 * n);
                a.scales[(static_cast<int64_t>(cb + r) * a.ld + col0) / 32 + q] = sc[r][q];
            }
        }
    }
}

// ---- fused row-wise and token-major quantisation ---------------------------------------

// A tile of 64 padded token rows x 64 columns whose values are computed once
// and quantised both ways: along the columns (blocks of 32 in a row; threads
// t and t ^ 1 hold one block) into the row-major operand of the dH or dXp GEMM,
// and along the rows (blocks of 32 tokens) into the token-major operand of the
// weight-gradient GEMM.  The tile is kept in shared memory as fp32,
// tf[r][column ^ sw(r)] with sw(r) = 8 * ((r / 16) % 4), so that the column
// pass reads without bank conflicts.
__device__ __forceinline__ int tf_sw(int r) { return ((r >> 4) & 3) << 3; }

__device__ __forceinline__ void tf_put16(float (*tf)[64], int r, int c16, const float (&v)[16]) {
    const int sw = tf_sw(r);
#pragma unroll
    for (int i = 0; i < 4; ++i)
        *reinterpret_cast<float4*>(&tf[r][(c16 + 4 * i) ^ sw]) =
            make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
}

// Row pass: the block maximum of threads t and t ^ 1 (every lane takes part in
// the shuffle); codes and scale byte (element offset `at` of a row-major
// operand) are written only for rows that exist.
__device__ __forceinline__ void row_q16(const float (&v)[16], bool store, uint8_t* codes,
                                        uint8_t* scales, int64_t at, bool first_half) {
    float m = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) m = fmaxf(m, fabsf(v[i]));
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
    if (store) mx_store_codes16(codes, scales, at, v, mx_block_exp(m), first_half);
}

// Column pass: thread (column c, part) takes rows 16 part .. + 15 of column c.
__device__ __forceinline__ void col_q16(const float (*tf)[64], int c, int part, uint16_t* dst) {
    float v[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = tf[part * 16 + i][c ^ (part << 3)];
    float m = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) m = fmaxf(m, fabsf(v[i]));
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
    tq_store16(dst, 0, v, mx_block_exp(m));
}

// Q_d(dY), dY = gate * dout, in token order: each token's dout row is read
// once and its k routed rows (gate(t, s) * dout[t], at dispatch position
// inv[t k + s]) and its shared-expert row (dout[t], at Tk + t) are quantised
// along d and stored as codes dyc [rows][d] and scale bytes dys [rows][d / 32];
// zero rows for a token whose replayed ids were rejected.  Thread i takes 8
// columns; four neighbouring threads hold one block of 32.  A token's scale
// bytes are gathered in shared memory and stored as whole 16-byte runs once its
// rows are done (byte stores from different warps would leave partial sectors).
constexpr int kDyMaxRows = 9;  // k slots + the shared expert
constexpr int kDyMaxD = 16384;

__global__ void __launch_bounds__(256) dy_rows_kernel(SrcDy src, const int32_t* __restrict__ inv,
                                                      int64_t T, int n_shared, int d,
                                                      uint8_t* __restrict__ dyc,
                                                      uint8_t* __restrict__ dys) {
    __shared__ int64_t dst[kDyMaxRows];
    __shared__ float sc[kDyMaxRows];
    __shared__ __align__(16) uint8_t sb[kDyMaxRows][kDyMaxD / 32];
    const int k = src.k;
    const int nd = k + (n_shared ? 1 : 0);
    for (int64_t t = blockIdx.x; t < T; t += gridDim.x) {
        if (threadIdx.x < nd) {
            const int j = threadIdx.x;
            const bool ok = src.valid[t] != 0;
            dst[j] = j < k ? static_cast<int64_t>(inv[t * k + j]) : src.Tk + t;
            sc[j] = !ok ? 0.0f : (j < k ? src.gates[t * k + j] : 1.0f);
        }
        __syncthreads();
        // d is a multiple of 256: a warp's 32 threads are all inside the row or
        // all past it
        for (int c = threadIdx.x * 8; c < d; c += blockDim.x * 8) {
            float x[8];
            unpack8(src.load8(t, c), x);
            for (int j = 0; j < nd; ++j) {
                const float w = sc[j];
                float v[8];
                float m = 0.0f;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    v[i] = w * x[i];
                    m = fmaxf(m, fabsf(v[i]));
                }
                m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
                m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
                const int X = mx_block_exp(m);
                const float rs = exp2i(-X);  // 2^-X
                uint32_t cw[4];
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    cw[i] = __nv_cvt_float2_to_fp8x2(make_float2(v[2 * i] * rs, v[2 * i + 1] * rs),
                                                     __NV_SATFINITE, __NV_E4M3);
                *reinterpret_cast<uint2*>(dyc + dst[j] * d + c) =
                    make_uint2(cw[0] | (cw[1] << 16), cw[2] | (cw[3] << 16));
                if ((threadIdx.x & 3) == 0) sb[j][c / 32] = static_cast<uint8_t>(X + 127);
            }
        }
        __syncthreads();
        // d / 32 scale bytes per row, a multiple of 16 (d % 512 == 0)
        const int runs = d / 512;
        for (int i = threadIdx.x; i < nd * runs; i += blockDim.x) {
            const int j = i / runs, q = i % runs;
            *reinterpret_cast<uint4*>(dys + dst[j] * (d / 32) + 16 * q) =
                *reinterpret_cast<const uint4*>(&sb[j][16 * q]);
        }
        __syncthreads();
    }
}

// SwiGLU backward (h = silu(a) * b, silu(a) = a * sigmoid(a)):
//   dA = dH * b * sigmoid(a) * (1 + a * (1 - sigmoid(a))),   dB = dH * silu(a),
// quantised into [Q_F(dA) | Q_F(dB)] rows [rows][2F] for the dXp GEMM (codes
// dabc, scale bytes dabs [rows][2F / 32]) and the token-major
// [Q_tok(dA) ; Q_tok(dB)] [2F][kpad] (bf16) for the dWg / dWu GEMM.
__global__ void __launch_bounds__(256, 4) swiglu_dual_kernel(
    const float* __restrict__ dh, const float* __restrict__ A, const float* __restrict__ Bv,
    TqArgs a, uint8_t* __restrict__ dabc, uint8_t* __restrict__ dabs, int F) {
    __shared__ __align__(16) float ta[kTqRows][64];
    __shared__ __align__(16) float tb[kTqRows][64];
    const int tid = threadIdx.x;
    const int cchunks = a.C / 64;
    const int64_t items = a.ntiles * cchunks;
    for (int64_t it = blockIdx.x; it < items; it += gridDim.x) {
        const int64_t rt = it / cchunks;
        const int cb = static_cast<int>(it % cchunks) * 64;
        TqBlock blk;
        if (!tq_tile<true>(a, rt, blk)) continue;  // uniform across the CTA
        {
            const int r = tid >> 2, c16 = (tid & 3) * 16;
            const bool ok = r < blk.nvalid;
            const int64_t row = blk.in_row0 + r;
            float da[16], db[16];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                float4 g = make_float4(0.f, 0.f, 0.f, 0.f), x = g, y = g;
                if (ok) {
                    g = *reinterpret_cast<const float4*>(dh + row * F + cb + c16 + 4 * q);
                    x = *reinterpret_cast<const float4*>(A + row * F + cb + c16 + 4 * q);
                    y = *reinterpret_cast<const float4*>(Bv + row * F + cb + c16 + 4 * q);
                }
                const float gg[4] = {g.x, g.y, g.z, g.w}, xa[4] = {x.x, x.y, x.z, x.w},
                            yb[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float sg = 1.0f / (1.0f + expf(-xa[j]));
                    da[4 * q + j] = gg[j] * yb[j] * (sg * (1.0f + xa[j] * (1.0f - sg)));
                    db[4 * q + j] = gg[j] * (xa[j] * sg);
                }
            }
            const int64_t at = row * 2 * F + cb + c16;
            const bool first = (tid & 1) == 0;
            row_q16(da, ok, dabc, dabs, at, first);
            row_q16(db, ok, dabc, dabs, at + F, first);
            tf_put16(ta, r, c16, da);
            tf_put16(tb, r, c16, db);
        }
        __syncthreads();
        {
            const int c = tid >> 2, part = tid & 3;
            const int64_t at = static_cast<int64_t>(cb + c) * a.ld + blk.out_col + part * 16;
            col_q16(ta, c, part, a.out + at);
            col_q16(tb, c, part, a.out + at + static_cast<int64_t>(F) * a.ld);
        }
        __syncthreads();
    }
}

// ---- padded segment offsets ----------------------------------------------------

// poff[g + 1] = poff[g] + round_up(n_g, 64), n_g = cnt[g] for g < E and
// shared_rows for the shared group; one warp.
__global__ void seg_offsets_kernel(const int32_t* __restrict__ cnt, int E, int G, int shared_rows,
                                   int32_t* __restrict__ poff) {
    const int lane = threadIdx.x;
    const int per = (G + 31) / 32;
    const int g0 = lane * per;
    int local = 0;
    for (int g = g0; g < min(g0 + per, G); ++g) local += ((g < E ? cnt[g] : shared_rows) + 63) & ~63;
    int incl = local;
#pragma unroll
    for (int s = 1; s < 32; s <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, s);
        if (lane >= s) incl += v;
    }
    int run = incl - local;
    for (int g = g0; g < min(g0 + per, G); ++g) {
        poff[g] = run;
        run += ((g < E ? cnt[g] : shared_rows) + 63) & ~63;
    }
    if (lane == 31) poff[G] = incl;
}

// tile_g[rt] = the group g with poff[g] <= 64 rt < poff[g + 1], or -1.
__global__ void seg_tiles_kernel(const int32_t* __restrict__ poff, int G, int64_t ntiles,
                                 int32_t* __restrict__ tile_g) {
    for (int64_t rt = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; rt < ntiles;
         rt += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t p = rt * kTqRows;
        int g = -1;
        if (p < poff[G]) {
            int lo = 0, hi = G;
            while (hi - lo > 1) {
                const int mid = (lo + hi) >> 1;
                if (poff[mid] <= p) lo = mid; else hi = mid;
            }
            g = lo;
        }
        tile_g[rt] = g;
    }
}

// ---- gate and router backward -------------------------------------------------------

constexpr int kGateWarps = 8;  // tokens in flight per CTA, one warp each
constexpr int kMaxSlots = 8;

// One warp per token t:
//   dg_s = dout[t] . Y[inv[t k + s]]                          (the gate gradient)
//   dl_s = w_s (dg_s - sum_s' w_s' dg_s')                    (softmax over the chosen)
//   dx[t] = sum_s dl_s Wr[ids[t, s]]   (the router's part of dx; s ascending)
// All sums in a fixed order: per lane over its columns ascending (lane l takes
// columns 8l .. 8l + 7 of every 256), then a butterfly over the lanes, which
// leaves every lane the same total (each step adds the same two values).
__global__ void __launch_bounds__(32 * kGateWarps) gate_bwd_kernel(
    const uint16_t* __restrict__ dout, const uint16_t* __restrict__ Y,
    const int32_t* __restrict__ inv, const int32_t* __restrict__ ids,
    const float* __restrict__ gates, const int32_t* __restrict__ valid,
    const uint16_t* __restrict__ wr, float* __restrict__ dg_out, float* __restrict__ dl_out,
    float* __restrict__ dx, int64_t T, int k, int d) {
    const int lane = threadIdx.x & 31;
    const int64_t nwarps = static_cast<int64_t>(gridDim.x) * kGateWarps;
    for (int64_t t = static_cast<int64_t>(blockIdx.x) * kGateWarps + (threadIdx.x >> 5); t < T;
         t += nwarps) {
        float acc[kMaxSlots];
        int32_t row[kMaxSlots];
#pragma unroll
        for (int s = 0; s < kMaxSlots; ++s) {
            acc[s] = 0.0f;
            row[s] = s < k ? inv[t * k + s] : 0;
        }
        for (int c = lane * 8; c < d; c += 256) {
            float g[8];
            unpack8(*reinterpret_cast<const uint4*>(dout + t * d + c), g);
#pragma unroll
            for (int s = 0; s < kMaxSlots; ++s) {
                if (s >= k) break;
                float y[8];
                unpack8(*reinterpret_cast<const uint4*>(Y + static_cast<int64_t>(row[s]) * d + c), y);
#pragma unroll
                for (int i = 0; i < 8; ++i) acc[s] = fmaf(g[i], y[i], acc[s]);
            }
        }
#pragma unroll
        for (int s = 0; s < kMaxSlots; ++s)
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) acc[s] += __shfl_xor_sync(0xffffffffu, acc[s], o);
        const bool ok = valid[t] != 0;
        float w[kMaxSlots], dl[kMaxSlots];
        float wdg = 0.0f;
#pragma unroll
        for (int s = 0; s < kMaxSlots; ++s) {
            w[s] = s < k ? gates[t * k + s] : 0.0f;
            if (s < k) wdg = fmaf(w[s], acc[s], wdg);
        }
#pragma unroll
        for (int s = 0; s < kMaxSlots; ++s) {
            dl[s] = s < k && ok ? w[s] * (acc[s] - wdg) : 0.0f;
            if (s < k && lane == s) {
                dg_out[t * k + s] = ok ? acc[s] : 0.0f;
                dl_out[t * k + s] = dl[s];
            }
        }
        int32_t id[kMaxSlots];
#pragma unroll
        for (int s = 0; s < kMaxSlots; ++s) id[s] = s < k ? ids[t * k + s] : 0;
        for (int c = lane * 8; c < d; c += 256) {
            float o[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) o[i] = 0.0f;
#pragma unroll
            for (int s = 0; s < kMaxSlots; ++s) {
                if (s >= k) break;
                float w8[8];
                unpack8(*reinterpret_cast<const uint4*>(wr + static_cast<int64_t>(id[s]) * d + c), w8);
#pragma unroll
                for (int i = 0; i < 8; ++i) o[i] = fmaf(dl[s], w8[i], o[i]);
            }
            float* dst = dx + t * d + c;
            *reinterpret_cast<float4*>(dst) = make_float4(o[0], o[1], o[2], o[3]);
            *reinterpret_cast<float4*>(dst + 4) = make_float4(o[4], o[5], o[6], o[7]);
        }
    }
}

// d_router[e] = sum over expert e's rows r (dispatch order) of dl[perm[r]] * Xp[r]:
// thread = 8 columns of one expert, rows in ascending order.
constexpr int kRouterWThreads = 128;
__global__ void __launch_bounds__(kRouterWThreads) router_wgrad_kernel(
    const uint16_t* __restrict__ xp, const int32_t* __restrict__ perm,
    const int32_t* __restrict__ cnt, const int32_t* __restrict__ off,
    const float* __restrict__ dl, float* __restrict__ d_router, int E, int d) {
    const int cpb = kRouterWThreads * 8;
    const int per_e = (d + cpb - 1) / cpb;
    for (int it = blockIdx.x; it < E * per_e; it += gridDim.x) {
        const int e = it / per_e;
        const int c = (it % per_e) * cpb + threadIdx.x * 8;
        if (c >= d) continue;
        float acc[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
        const int64_t r0 = off[e], r1 = r0 + cnt[e];
        // four rows' loads in flight; the products are added in row order
        constexpr int kAhead = 4;
        for (int64_t r = r0; r < r1; r += kAhead) {
            const int nr = static_cast<int>(r1 - r < kAhead ? r1 - r : kAhead);
            float l[kAhead];
            uint4 xr[kAhead];
#pragma unroll
            for (int u = 0; u < kAhead; ++u) {
                if (u < nr) {
                    l[u] = dl[perm[r + u]];
                    xr[u] = *reinterpret_cast<const uint4*>(xp + (r + u) * d + c);
                }
            }
#pragma unroll
            for (int u = 0; u < kAhead; ++u) {
                if (u < nr) {
                    float x[8];
                    unpack8(xr[u], x);
#pragma unroll
                    for (int i = 0; i < 8; ++i) acc[i] = fmaf(l[u], x[i], acc[i]);
                }
            }
        }
        float* dst = d_router + static_cast<int64_t>(e) * d + c;
        *reinterpret_cast<float4*>(dst) = make_float4(acc[0], acc[1], acc[2], acc[3]);
        *reinterpret_cast<float4*>(dst + 4) = make_float4(acc[4], acc[5], acc[6], acc[7]);
    }
}

// dx[t] = ((sum_s dXp[inv[t k + s]]) + dXp_shared[t]) + dx[t], the last term
// being the router's part written by gate_bwd_kernel; s ascending.
__global__ void __launch_bounds__(256) dx_assemble_kernel(
    const float* __restrict__ dxp, const int32_t* __restrict__ inv, float* __restrict__ dx,
    int64_t T, int k, int d, int has_shared) {
    const int q = d / 4;
    const int64_t Tk = T * k;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < T * q;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t t = i / q;
        const int c = static_cast<int>(i % q) * 4;
        float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        for (int s = 0; s < k; ++s) {
            const float4 v = *reinterpret_cast<const float4*>(dxp + static_cast<int64_t>(inv[t * k + s]) * d + c);
            acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
        }
        if (has_shared) {
            const float4 v = *reinterpret_cast<const float4*>(dxp + (Tk + t) * d + c);
            acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
        }
        float4* o = reinterpret_cast<float4*>(dx + t * d + c);
        const float4 r = *o;
        acc.x += r.x; acc.y += r.y; acc.z += r.z; acc.w += r.w;
        *o = acc;
    }
}

inline int grid_for(int64_t items, int per_block, int sms, int per_sm = 8) {
    int64_t b = (items + per_block - 1) / per_block;
    const int64_t cap = static_cast<int64_t>(sms) * per_sm;
    if (b > cap) b = cap;
    return static_cast<int>(b < 1 ? 1 : b);
}

}  // namespace

cudaError_t launch_seg_offsets(const int32_t* cnt, int E, int G, int shared_rows, int32_t* poff,
                               int64_t ntiles, cudaStream_t s) {
    seg_offsets_kernel<<<1, 32, 0, s>>>(cnt, E, G, shared_rows, poff);
    if (ntiles > 0)
        seg_tiles_kernel<<<static_cast<unsigned>((ntiles + 255) / 256), 256, 0, s>>>(poff, G, ntiles,
                                                                                   poff + G + 1);
    return cudaGetLastError();
}

namespace {
template <class Src, bool SEG>
cudaError_t tq_launch(const Src& src, const TqArgs& a, int sms, cudaStream_t s) {
    if (a.C % 64 || a.ld % 8) return cudaErrorInvalidValue;
    const int64_t items = a.ntiles * (a.C / 64);
    if (items == 0) return cudaSuccess;
    tq16_kernel<Src, SEG><<<grid_for(items, 1, sms, 8), 256, 0, s>>>(src, a);
    return cudaGetLastError();
}

}  // namespace

namespace {
TqArgs seg_args(int C, const int32_t* cnt, const int32_t* off, const int32_t* poff, int E, int G,
                int64_t shared_row0, int shared_rows, int64_t kpad, uint16_t* out) {
    TqArgs a{};
    a.C = C;
    a.ld = kpad;
    a.out = out;
    a.cnt = cnt;
    a.off = off;
    a.poff = poff;
    a.tile_g = poff + G + 1;
    a.E = E;
    a.G = G;
    a.shared_row0 = shared_row0;
    a.shared_rows = shared_rows;
    a.ntiles = kpad / kTqRows;
    return a;
}
}  // namespace

cudaError_t launch_tq_segments(const uint16_t* src, int64_t src_ld, int C, const int32_t* cnt,
                               const int32_t* off, const int32_t* poff, int E, int G,
                               int64_t shared_row0, int shared_rows, int64_t kpad, uint16_t* out,
                               int sms, cudaStream_t s) {
    if (kpad % kTqRows) return cudaErrorInvalidValue;
    return tq_launch<SrcBf16, true>(SrcBf16{src, src_ld},
                                    seg_args(C, cnt, off, poff, E, G, shared_row0, shared_rows,
                                             kpad, out),
                                    sms, s);
}

cudaError_t launch_dy_dual(const SegDyArgs& dy, int d, const int32_t* cnt, const int32_t* off,
                           const int32_t* poff, int E, int G, int shared_rows, int64_t kpad,
                           uint8_t* dyc, uint8_t* dys, uint16_t* dyt, int sms, cudaStream_t s) {
    if (kpad % kTqRows || d % 512 || d > kDyMaxD || dy.k + (dy.n_shared ? 1 : 0) > kDyMaxRows ||
        (reinterpret_cast<uintptr_t>(dys) & 15))
        return cudaErrorInvalidValue;
    const SrcDy src{dy.dout, dy.gates, dy.perm, dy.valid, dy.k, dy.Tk, d};
    if (dy.T > 0) {
        const int64_t cap = static_cast<int64_t>(sms) * 8;
        dy_rows_kernel<<<static_cast<unsigned>(dy.T < cap ? dy.T : cap), 256, 0, s>>>(
            src, dy.inv, dy.T, dy.n_shared, d, dyc, dys);
    }
    // Q_tok(dY): the same values, quantised along each expert's tokens
    return tq_launch<SrcDy, true>(src, seg_args(d, cnt, off, poff, E, G, dy.Tk, shared_rows, kpad,
                                                dyt),
                                  sms, s);
}

cudaError_t launch_swiglu_dual(const float* dh, const float* a_pre, const float* b_pre, int F,
                               const int32_t* cnt, const int32_t* off, const int32_t* poff, int E,
                               int G, int64_t shared_row0, int shared_rows, int64_t kpad,
                               uint8_t* dabc, uint8_t* dabs, uint16_t* dabt, int sms,
                               cudaStream_t s) {
    if (kpad % kTqRows || F % 64) return cudaErrorInvalidValue;
    const TqArgs a = seg_args(F, cnt, off, poff, E, G, shared_row0, shared_rows, kpad, dabt);
    const int64_t items = a.ntiles * (F / 64);
    if (items == 0) return cudaSuccess;
    swiglu_dual_kernel<<<grid_for(items, 1, sms, 4), 256, 0, s>>>(dh, a_pre, b_pre, a, dabc, dabs,
                                                                   F);
    return cudaGetLastError();
}

cudaError_t launch_tq_batch(const uint16_t* src, int nb, int R, int C, uint8_t* codes,
                            uint8_t* scales, int64_t out_bstride, int64_t out_ld, int64_t out_off,
                            int sms, cudaStream_t s) {
    if (R % kTqRows) return cudaErrorInvalidValue;
    TqArgs a{};
    a.C = C;
    a.ld = out_ld;
    a.codes = codes;
    a.scales = scales;
    a.R = R;
    a.out_bstride = out_bstride;
    a.out_off = out_off;
    a.ntiles = static_cast<int64_t>(nb) * (R / kTqRows);
    // every block of 32 starts on a multiple of 32 (one scale byte each)
    if (C % 64 || out_ld % 32 || out_off % 32 || out_bstride % 32) return cudaErrorInvalidValue;
    a.sc_vec = out_ld % 1024 == 0 && out_bstride % 1024 == 0 && out_off % 1024 == 0 &&
               (reinterpret_cast<uintptr_t>(scales) & 15) == 0;
    const int per = R / kTqRows, gper = (per + kTqGroup - 1) / kTqGroup;
    const int64_t items = static_cast<int64_t>(nb) * gper * (C / 64);
    if (items == 0) return cudaSuccess;
    tq_codes_kernel<<<grid_for(items, 1, sms, 8), 256, 0, s>>>(SrcBf16{src, C}, a);
    return cudaGetLastError();
}

cudaError_t launch_gate_bwd(const uint16_t* dout, const uint16_t* y, const int32_t* inv,
                            const int32_t* ids, const float* gates, const int32_t* valid,
                            const uint16_t* wr, float* dg, float* dl, float* dx, int64_t T, int k,
                            int d, int sms, cudaStream_t s) {
    if (k > kMaxSlots || d % 8) return cudaErrorInvalidValue;
    if (T == 0) return cudaSuccess;
    const int64_t cap = static_cast<int64_t>(sms) * 4;  // resident CTAs at 64 registers
    const int64_t blocks = (T + kGateWarps - 1) / kGateWarps;
    const int grid = static_cast<int>(blocks < cap ? blocks : cap);
    gate_bwd_kernel<<<grid, 32 * kGateWarps, 0, s>>>(dout, y, inv, ids, gates, valid, wr, dg, dl, dx,
                                                  T, k, d);
    return cudaGetLastError();
}

cudaError_t launch_router_wgrad(const uint16_t* xp, const int32_t* perm, const int32_t* cnt,
                                const int32_t* off, const float* dl, float* d_router, int E, int d,
                                int sms, cudaStream_t s) {
    if (d % 8) return cudaErrorInvalidValue;
    const int cpb = kRouterWThreads * 8;
    const int64_t items = static_cast<int64_t>(E) * ((d + cpb - 1) / cpb);
    router_wgrad_kernel<<<grid_for(items, 1, sms, 16), kRouterWThreads, 0, s>>>(xp, perm, cnt, off,
                                                                                dl, d_router, E, d);
    return cudaGetLastError();
}

cudaError_t launch_dx_assemble(const float* dxp, const int32_t* inv, float* dx, int64_t T, int k,
                               int d, int n_shared, int sms, cudaStream_t s) {
    if (d % 4) return cudaErrorInvalidValue;
    if (T == 0) return cudaSuccess;
    dx_assemble_kernel<<<grid_for(T * (d / 4), 256, sms), 256, 0, s>>>(dxp, inv, dx, T, k, d,
                                                                       n_shared);
    return cudaGetLastError();
}

}  // namespace moe
