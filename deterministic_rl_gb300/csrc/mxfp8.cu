// mxfp8.cu -- MXFP8 activations of the forward with MXFP8 expert compute.
//
// Composer 2 Technical Report, §6.1 "Training infrastructure" (Kernels): the
// tokens are quantised to MXFP8 before dispatch, and the expert compute runs
// in MXFP8.  With MXFP8 weights, each token row of x is quantised along d and
// each row of the SwiGLU output h (stored in bf16) along F, in blocks of 32
// (mx.cuh), into E4M3 codes and E8M0 scale bytes; the expert GEMMs then
// multiply the MXFP8 values of both operands on the block-scaled tensor-core
// MMA (gemm_bs.cu).
#include <cuda_bf16.h>

#include <cstdint>

#include "moe_internal.h"
#include "mx.cuh"

namespace moe {
namespace {

__device__ __forceinline__ void unpack8_bf16(const uint4& u, float (&v)[8]) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        v[2 * i] = __uint_as_float(w[i] << 16);
        v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}

// One warp per (row, 256-column chunk): lane l holds columns 8l .. 8l + 7, so
// a block of 32 is held by lanes 4i .. 4i + 3.  Each lane writes its 8 E4M3
// codes, and the first lane of each block the block's E8M0 scale byte X + 127.
// With dst_of (the gather's inv, for token rows of x): the same codes and
// scales also go to the k gathered rows dst_of[r * k + j] of codes_p /
// scales_p (the gather, fused).
__global__ void __launch_bounds__(256) mx_rows_fp8_kernel(const uint4* src, uint2* codes,
                                                          uint8_t* scales, int64_t R, int K,
                                                          const int32_t* __restrict__ dst_of, int k,
                                                          uint2* codes_p, uint8_t* scales_p) {
    const int lane = threadIdx.x & 31;
    const int chunks = K / 256;
    const int64_t items = R * chunks;
    for (int64_t i = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; i < items;
         i += (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5) {
        const int64_t r = i / chunks;
        const int c = static_cast<int>(i % chunks);
        const int64_t at = (r * K + static_cast<int64_t>(c) * 256 + lane * 8) / 8;
        float v[8];
        unpack8_bf16(src[at], v);
        float m = 0.0f;
#pragma unroll
        for (int j = 0; j < 8; ++j) m = fmaxf(m, fabsf(v[j]));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
        const int X = mx_block_exp(m);
        const float inv = exp2i(-X);
        uint32_t w[4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
            w[j] = __nv_cvt_float2_to_fp8x2(make_float2(v[2 * j] * inv, v[2 * j + 1] * inv),
                                            __NV_SATFINITE, __NV_E4M3);
        const uint2 cw = make_uint2(w[0] | (w[1] << 16), w[2] | (w[3] << 16));
        const uint8_t sb = static_cast<uint8_t>(X + 127);
        codes[at] = cw;
        if ((lane & 3) == 0) scales[r * (K / 32) + c * 8 + (lane >> 2)] = sb;
        if (dst_of) {
            const int dl = lane < k ? dst_of[r * k + lane] : 0;
            for (int j = 0; j < k; ++j) {
                const int64_t dst = __shfl_sync(0xffffffffu, dl, j);
                codes_p[(dst * K + static_cast<int64_t>(c) * 256) / 8 + lane] = cw;
                if ((lane & 3) == 0) scales_p[dst * (K / 32) + c * 8 + (lane >> 2)] = sb;
            }
        }
    }
}

}  // namespace

cudaError_t launch_mx_rows_fp8(const uint16_t* src, uint8_t* codes, uint8_t* scales, int64_t R,
                               int K, int sms, cudaStream_t s, const int32_t* inv, int k,
                               uint8_t* codes_p, uint8_t* scales_p) {
    if (K % 256) return cudaErrorInvalidValue;
    if (inv && (k < 1 || k > 8 || !codes_p || !scales_p)) return cudaErrorInvalidValue;
    if (R == 0) return cudaSuccess;
    int64_t blocks = (R * (K / 256) + 7) / 8;  // 8 warps per block
    const int64_t cap = static_cast<int64_t>(sms) * 8;
    if (blocks > cap) blocks = cap;
    mx_rows_fp8_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(
        reinterpret_cast<const uint4*>(src), reinterpret_cast<uint2*>(codes), scales, R, K, inv, k,
        reinterpret_cast<uint2*>(codes_p), scales_p);
    return cudaGetLastError();
}

}  // namespace moe
