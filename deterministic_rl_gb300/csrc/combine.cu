// combine.cu -- fixed-order combine of each token's expert outputs.
//
// out[t] = sum_{s = 0..k-1} gate[t][s] * Y[inv[t*k + s]]  +  Ysh[t]
// accumulated in fp32 in ascending slot order, then the shared expert; the
// result is stored as fp32 or rounded once to bf16 (nearest even).  This is the
// combine step of the Composer 2 Technical Report, §6.1 "Training
// infrastructure" (combine kept in BF16 rather than a lower precision), done in
// the one fixed order the Training Data No. 94 write-up (section
// "浮点数不守规矩，MoE 火上浇油") asks of batch-invariant kernels: each output
// element is one thread's sequential sum, independent of every other token.
#include <cuda_bf16.h>

#include <cstdint>

#include "moe_internal.h"

namespace moe {
namespace {

constexpr int kMaxK = 8;
constexpr int kThreads = 128;

__device__ __forceinline__ void bf16x8_to_f32(const uint4& u, float (&f)[8]) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}

template <bool OUT_F32, bool SHARED>
__global__ void __launch_bounds__(kThreads) combine_kernel(
    const uint4* __restrict__ y, const float4* __restrict__ ysh, const int32_t* __restrict__ inv,
    const float* __restrict__ gates, const int32_t* __restrict__ valid, int k, int d, void* out) {
    // block (t, c): token t, 8-element vectors [c * kThreads, (c + 1) * kThreads)
    const int64_t t = blockIdx.x;
    const int vec = d / 8;
    int32_t rows[kMaxK];
    float g[kMaxK];
#pragma unroll
    for (int s = 0; s < kMaxK; ++s) {
        rows[s] = s < k ? inv[t * k + s] : 0;
        g[s] = s < k ? gates[t * k + s] : 0.0f;
    }
    const bool ok = valid[t] != 0;
    {
        const int v = blockIdx.y * kThreads + threadIdx.x;
        if (v >= vec) return;
        float acc[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
        if (ok) {
#pragma unroll
            for (int s = 0; s < kMaxK; ++s) {
                if (s >= k) break;
                float f[8];
                bf16x8_to_f32(y[static_cast<int64_t>(rows[s]) * vec + v], f);
#pragma unroll
                for (int i = 0; i < 8; ++i) acc[i] = fmaf(g[s], f[i], acc[i]);
            }
            if (SHARED) {
                const float4 a = ysh[(t * vec + v) * 2];
                const float4 b = ysh[(t * vec + v) * 2 + 1];
                acc[0] += a.x; acc[1] += a.y; acc[2] += a.z; acc[3] += a.w;
                acc[4] += b.x; acc[5] += b.y; acc[6] += b.z; acc[7] += b.w;
            }
        }
        if (OUT_F32) {
            float4* o = static_cast<float4*>(out) + (t * vec + v) * 2;
            o[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
            o[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
        } else {
            uint32_t w[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const __nv_bfloat162 h = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
                w[i] = *reinterpret_cast<const uint32_t*>(&h);
            }
            static_cast<uint4*>(out)[t * vec + v] = make_uint4(w[0], w[1], w[2], w[3]);
        }
    }
}

}  // namespace

cudaError_t launch_combine(const uint16_t* y, const float* ysh, const int32_t* inv,
                           const float* gates, const int32_t* valid, int64_t T, int k, int d,
                           int out_fp32, void* out, cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    if (k > kMaxK || d % 8) return cudaErrorInvalidValue;
    const auto* yv = reinterpret_cast<const uint4*>(y);
    const auto* sv = reinterpret_cast<const float4*>(ysh);
    const dim3 grid(static_cast<unsigned>(T), static_cast<unsigned>((d / 8 + kThreads - 1) / kThreads));
    if (out_fp32) {
        if (ysh) combine_kernel<true, true><<<grid, kThreads, 0, s>>>(yv, sv, inv, gates, valid, k, d, out);
        else combine_kernel<true, false><<<grid, kThreads, 0, s>>>(yv, sv, inv, gates, valid, k, d, out);
    } else {
        if (ysh) combine_kernel<false, true><<<grid, kThreads, 0, s>>>(yv, sv, inv, gates, valid, k, d, out);
        else combine_kernel<false, false><<<grid, kThreads, 0, s>>>(yv, sv, inv, gates, valid, k, d, out);
    }
    return cudaGetLastError();
}

}  // namespace moe
