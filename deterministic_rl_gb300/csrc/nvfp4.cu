// nvfp4.cu -- the NVFP4 activation quantiser of the MoE forward.
//
// The Composer 2 Technical Report, §6.1 "Training infrastructure" (Kernels):
// the MoE forward quantises BF16 values to FP4 E2M1 with one FP8 E4M3 scale
// per 16 consecutive values and one FP32 scale per token (not per tensor, so
// that a token's numbers do not depend on the rest of the batch), and the
// quantiser must use IEEE-compliant division.  Per row (token) of K values:
//   s   = amax(row) / (6 * 448)                          fp32, correctly rounded
//   S_b = E4M3(amax(block) / 6 / s)   nearest even, saturating at 448
//   q_i = E2M1(x_i / (S_b * s))       nearest, ties to the even code, +-6 at most
// (s = 0 for an all-zero row; a block whose S_b is 0 has all codes 0; zero is
// always +0).  The kernel writes the E2M1 codes (two per byte, element 2j in
// the low nibble), the E4M3 bytes S_b and s: the operands of the block-scaled
// FP4 expert GEMMs, which apply s in their epilogue.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <cstdint>

#include "moe_internal.h"

namespace moe {
namespace {

constexpr int kWarps = 8;

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ float absmax8(const uint4& a, float m) {
    const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) m = fmaxf(m, fmaxf(fabsf(bf16_lo(w[i])), fabsf(bf16_hi(w[i]))));
    return m;
}

// E2M1 magnitude index of |v| (0..7 for 0, .5, 1, 1.5, 2, 3, 4, 6): the
// nearest magnitude, a tie going to the even index, saturating above 6.
__device__ __forceinline__ int e2m1_index(float a) {
    return (a > 0.25f) + (a >= 0.75f) + (a > 1.25f) + (a >= 1.75f) + (a > 2.5f) + (a >= 3.5f) +
           (a > 5.0f);
}

// The E2M1 code (sign bit 8, magnitude index 0..7) of one value; zero is +0.
__device__ __forceinline__ uint32_t code_one(float v, float denom) {
    if (!(denom > 0.0f)) return 0u;
    const float t = __fdiv_rn(v, denom);
    const int m = e2m1_index(fabsf(t));
    return static_cast<uint32_t>(m) | (t < 0.0f && m != 0 ? 8u : 0u);
}

// Four bf16 pairs (8 values) -> 8 codes, element 0 in the lowest nibble.
__device__ __forceinline__ uint32_t codes8(const uint4& a, float denom) {
    const uint32_t w[4] = {a.x, a.y, a.z, a.w};
    uint32_t r = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i)
        r |= (code_one(bf16_lo(w[i]), denom) | (code_one(bf16_hi(w[i]), denom) << 4)) << (8 * i);
    return r;
}

// The block scale S_b of a 16-value block with largest magnitude bmax, as its
// E4M3 byte (0 when the row scale is 0).
__device__ __forceinline__ __nv_fp8_storage_t block_scale(float bmax, float s) {
    if (!(s > 0.0f)) return 0;
    return __nv_cvt_float_to_fp8(__fdiv_rn(__fdiv_rn(bmax, 6.0f), s), __NV_SATFINITE, __NV_E4M3);
}

__device__ __forceinline__ float e4m3_value(__nv_fp8_storage_t S) {
    return __half2float(__half(__nv_cvt_fp8_to_halfraw(S, __NV_E4M3)));
}

// W warps per row (1 for many rows, 4 for few), a lane per 16-value block:
// codes [R][K/2] bytes, bscale [R][K/16] E4M3 bytes, rscale [R] fp32.  The
// row's maximum is the maximum over its warps (exact, whatever the order).
// With inv (token rows of x): the same codes and scales also go to the k
// gathered rows inv[r * k + j] of codes_p, bscale_p, rscale_p (the gather,
// fused).
template <int kWarpsPerRow>
__global__ void __launch_bounds__(32 * kWarps) nvfp4_codes_kernel(
    const uint4* __restrict__ src, uint2* __restrict__ codes, uint8_t* __restrict__ bscale,
    float* __restrict__ rscale, int64_t R, int K, const int32_t* __restrict__ inv, int k,
    uint2* __restrict__ codes_p, uint8_t* __restrict__ bscale_p, float* __restrict__ rscale_p) {
    constexpr int kRowsPerBlock = kWarps / kWarpsPerRow;
    __shared__ float red[kWarps];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int wr = warp % kWarpsPerRow;  // this warp's share of its row
    const int slot = warp / kWarpsPerRow;
    const int nb = K / 16;
    const int vpr = K / 8;
    // the loop bound is the same for the whole block (it meets __syncthreads)
    for (int64_t r0 = static_cast<int64_t>(blockIdx.x) * kRowsPerBlock; r0 < R;
         r0 += static_cast<int64_t>(gridDim.x) * kRowsPerBlock) {
        const int64_t r = r0 + slot;
        const bool have = r < R;
        const uint4* row = src + (have ? r : 0) * vpr;
        float amax = 0.0f;
        if (have)
            for (int b = wr * 32 + lane; b < nb; b += 32 * kWarpsPerRow)
                amax = absmax8(row[2 * b + 1], absmax8(row[2 * b], amax));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        if constexpr (kWarpsPerRow > 1) {
            if (lane == 0) red[warp] = amax;
            __syncthreads();
#pragma unroll
            for (int w = 0; w < kWarpsPerRow; ++w) amax = fmaxf(amax, red[slot * kWarpsPerRow + w]);
            __syncthreads();
        }
        if (!have) continue;
        const float s = __fdiv_rn(amax, 2688.0f);  // 6 * 448
        if (wr == 0 && lane == 0) rscale[r] = s;
        // the row's gathered destinations, in every lane (k <= 8)
        int64_t dst[8];
        {
            const int dl = inv && lane < k ? inv[r * k + lane] : 0;
            if (inv && wr == 0 && lane < k) rscale_p[dl] = s;
#pragma unroll
            for (int j = 0; j < 8; ++j) dst[j] = __shfl_sync(0xffffffffu, dl, j);
        }
        for (int b = wr * 32 + lane; b < nb; b += 32 * kWarpsPerRow) {
            const uint4 a0 = row[2 * b], a1 = row[2 * b + 1];
            const __nv_fp8_storage_t S = block_scale(absmax8(a1, absmax8(a0, 0.0f)), s);
            const float denom = __fmul_rn(e4m3_value(S), s);
            const uint2 cw = make_uint2(codes8(a0, denom), codes8(a1, denom));
            codes[r * nb + b] = cw;
            bscale[r * nb + b] = S;
            if (inv) {
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    if (j < k) {
                        codes_p[dst[j] * nb + b] = cw;
                        bscale_p[dst[j] * nb + b] = S;
                    }
            }
        }
    }
}

}  // namespace

cudaError_t launch_nvfp4_codes(const uint16_t* src, uint8_t* codes, uint8_t* bscale, float* rscale,
                               int64_t R, int K, int sms, cudaStream_t s, const int32_t* inv, int k,
                               uint8_t* codes_p, uint8_t* bscale_p, float* rscale_p) {
    if (R == 0) return cudaSuccess;
    if (K % 16) return cudaErrorInvalidValue;
    if (inv && (k < 1 || k > 8 || !codes_p || !bscale_p || !rscale_p)) return cudaErrorInvalidValue;
    const int64_t cap = static_cast<int64_t>(sms) * 8;
    // few rows (a decode batch): four warps per row, else one
    if (R < cap * kWarps) {
        constexpr int kW = 4;
        int64_t blocks = (R + kWarps / kW - 1) / (kWarps / kW);
        if (blocks > cap) blocks = cap;
        nvfp4_codes_kernel<kW><<<static_cast<unsigned>(blocks), 32 * kWarps, 0, s>>>(
            reinterpret_cast<const uint4*>(src), reinterpret_cast<uint2*>(codes), bscale, rscale, R,
            K, inv, k, reinterpret_cast<uint2*>(codes_p), bscale_p, rscale_p);
    } else {
        int64_t blocks = (R + kWarps - 1) / kWarps;
        if (blocks > cap) blocks = cap;
        nvfp4_codes_kernel<1><<<static_cast<unsigned>(blocks), 32 * kWarps, 0, s>>>(
            reinterpret_cast<const uint4*>(src), reinterpret_cast<uint2*>(codes), bscale, rscale, R,
            K, inv, k, reinterpret_cast<uint2*>(codes_p), bscale_p, rscale_p);
    }
    return cudaGetLastError();
}

}  // namespace moe
