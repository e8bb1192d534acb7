// mx.cuh -- MXFP8 quantise-dequantise helpers shared by the kernels that
// quantise activations and backward operands.
//
// MXFP8 as the OCP Microscaling Formats (MX) v1.0 specification defines it
// (the format the Composer 2 Technical Report, §6.1 "Training infrastructure",
// names for the MoE backward and the expert compute): per block of 32 values,
// X = floor(log2(max |v|)) - 8 (8 = the exponent of E4M3's largest normal),
// element = E4M3(v * 2^-X), nearest even, clamped to +-448.  The helpers write
// the dequantised value e4m3 * 2^X as bf16, which holds it exactly (at most 4
// significant bits, and the exponents the layer produces), so a bf16 MMA on
// them multiplies the MXFP8 values themselves.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <cstdint>

namespace moe {
namespace {

// Shared exponent X of a block whose largest magnitude is amax (>= 0):
// floor(log2 amax) - 8 within [-127, 127]; -127 for zero or subnormal amax.
__device__ __forceinline__ int mx_block_exp(float amax) {
    const int ef = static_cast<int>((__float_as_uint(amax) >> 23) & 0xFFu);
    if (ef == 0) return -127;
    return max(ef - 127 - 8, -127);
}

// 2^n for n in [-127, 127] (2^-127 is an fp32 subnormal).
__device__ __forceinline__ float exp2i(int n) {
    return n >= -126 ? __uint_as_float(static_cast<uint32_t>(n + 127) << 23)
                     : __uint_as_float(0x00400000u);
}

// e4m3(v * 2^-X) * 2^X for two values, with inv = 2^-X and scale = 2^X,
// packed as bf16x2 (a in the low half): one paired conversion to E4M3 and one
// back to f16 (both exact per element), then the power-of-two rescale.
__device__ __forceinline__ uint32_t mx_qdq2(float a, float b, float inv, float scale) {
    const __nv_fp8x2_storage_t q =
        __nv_cvt_float2_to_fp8x2(make_float2(a * inv, b * inv), __NV_SATFINITE, __NV_E4M3);
    const float2 f = __half22float2(__half2(__nv_cvt_fp8x2_to_halfraw2(q, __NV_E4M3)));
    const __nv_bfloat162 r = __floats2bfloat162_rn(f.x * scale, f.y * scale);
    return static_cast<uint32_t>(__bfloat16_as_ushort(r.x)) |
           (static_cast<uint32_t>(__bfloat16_as_ushort(r.y)) << 16);
}

// Quantise 8 values with block exponent X and pack them as 8 bf16.
__device__ __forceinline__ uint4 mx_qdq8(const float (&v)[8], int X) {
    const float inv = exp2i(-X), sc = exp2i(X);
    return make_uint4(mx_qdq2(v[0], v[1], inv, sc), mx_qdq2(v[2], v[3], inv, sc),
                      mx_qdq2(v[4], v[5], inv, sc), mx_qdq2(v[6], v[7], inv, sc));
}

__device__ __forceinline__ void unpack8(const uint4& u, float (&v)[8]) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        v[2 * i] = __uint_as_float(w[i] << 16);
        v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}

}  // namespace
}  // namespace moe
