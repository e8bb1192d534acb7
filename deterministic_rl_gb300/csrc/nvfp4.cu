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
// always +0).  The kernel writes, per row, s and the bf16 values e2m1(q_i) *
// e4m3(S_b) -- exact in bf16 (at most 6 significant bits) -- which the expert
// GEMMs take as their token operand; s is applied in the GEMM epilogue.
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

__device__ __forceinline__ float e2m1_magnitude(int m) {
    // 0, 0.5, 1, 1.5, 2, 3, 4, 6
    return m < 4 ? 0.5f * m : (m == 7 ? 6.0f : static_cast<float>(m - 2));
}

// Quantise one value and return the bf16 bits of e2m1(q) * S (exact).
__device__ __forceinline__ uint32_t qdq_one(float v, float denom, float Sf) {
    if (!(denom > 0.0f)) return 0u;
    const float t = __fdiv_rn(v, denom);
    const int m = e2m1_index(fabsf(t));
    float val = e2m1_magnitude(m) * Sf;  // exact: <= 6 significant bits
    if (t < 0.0f && m != 0) val = -val;
    return static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(val)));
}

__device__ __forceinline__ uint32_t qdq_pair(uint32_t w, float denom, float Sf) {
    return qdq_one(bf16_lo(w), denom, Sf) | (qdq_one(bf16_hi(w), denom, Sf) << 16);
}

// src and dst may be the same rows (in place): a lane reads its blocks in full
// before it writes them, and no lane touches another lane's blocks.
__global__ void __launch_bounds__(32 * kWarps) nvfp4_qdq_kernel(
    const uint4* src, uint4* dst, uint8_t* __restrict__ bscale,
    float* __restrict__ rscale, int64_t R, int K) {
    const int lane = threadIdx.x & 31;
    const int nb = K / 16;        // 16-value blocks per row, 2 uint4 each
    const int vpr = K / 8;        // uint4 per row
    for (int64_t r = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5); r < R;
         r += static_cast<int64_t>(gridDim.x) * kWarps) {
        const uint4* row = src + r * vpr;
        float amax = 0.0f;
        for (int b = lane; b < nb; b += 32) amax = absmax8(row[2 * b + 1], absmax8(row[2 * b], amax));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        const float s = __fdiv_rn(amax, 2688.0f);  // 6 * 448
        if (lane == 0) rscale[r] = s;
        uint4* out = dst + r * vpr;
        for (int b = lane; b < nb; b += 32) {
            const uint4 a0 = row[2 * b], a1 = row[2 * b + 1];
            const float bmax = absmax8(a1, absmax8(a0, 0.0f));
            __nv_fp8_storage_t S = 0;
            if (s > 0.0f)
                S = __nv_cvt_float_to_fp8(__fdiv_rn(__fdiv_rn(bmax, 6.0f), s), __NV_SATFINITE,
                                          __NV_E4M3);
            const float Sf = __half2float(__half(__nv_cvt_fp8_to_halfraw(S, __NV_E4M3)));
            const float denom = __fmul_rn(Sf, s);
            uint4 o0, o1;
            o0.x = qdq_pair(a0.x, denom, Sf);
            o0.y = qdq_pair(a0.y, denom, Sf);
            o0.z = qdq_pair(a0.z, denom, Sf);
            o0.w = qdq_pair(a0.w, denom, Sf);
            o1.x = qdq_pair(a1.x, denom, Sf);
            o1.y = qdq_pair(a1.y, denom, Sf);
            o1.z = qdq_pair(a1.z, denom, Sf);
            o1.w = qdq_pair(a1.w, denom, Sf);
            out[2 * b] = o0;
            out[2 * b + 1] = o1;
            if (bscale) bscale[r * nb + b] = S;
        }
    }
}

}  // namespace

cudaError_t launch_nvfp4_qdq(const uint16_t* src, uint16_t* dst, uint8_t* bscale, float* rscale,
                             int64_t R, int K, int sms, cudaStream_t s) {
    if (R == 0) return cudaSuccess;
    if (K % 16) return cudaErrorInvalidValue;
    int64_t blocks = (R + kWarps - 1) / kWarps;
    const int64_t cap = static_cast<int64_t>(sms) * 8;
    if (blocks > cap) blocks = cap;
    nvfp4_qdq_kernel<<<static_cast<unsigned>(blocks), 32 * kWarps, 0, s>>>(
        reinterpret_cast<const uint4*>(src), reinterpret_cast<uint4*>(dst), bscale, rscale, R, K);
    return cudaGetLastError();
}

}  // namespace moe
