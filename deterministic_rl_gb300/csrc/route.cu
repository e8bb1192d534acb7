// route.cu -- top-k selection by warp-shuffle arg-max, replay-id validation,
// and gate weights, one warp per token.
//
// Selection follows the gate of the Training Data No. 94 write-up (section
// "浮点数不守规矩，MoE 火上浇油": a gate picks 8 of 384 experts from the
// hidden state): the k largest logits in descending order, equal logits going
// to the lower expert id.  Replay follows the Composer 2 Technical Report,
// §6.2 "RL infrastructure": recorded ids replace the selection and the router
// still computes the gate scores over them.  Gate weights are the softmax of
// the k chosen logits (softmax over all E renormalised over the chosen set).
// Own mode and replay share one gate routine, so replaying the ids own mode
// chose gives bitwise the same weights.
#include <cfloat>
#include <climits>

#include "moe_internal.h"

namespace moe {
namespace {

constexpr int kMaxK = 8;
constexpr int kWarpsPerBlock = 8;
constexpr int kMaxSplit = 4;  // partial-logit buffers of the router's K split

// a ranks before b: larger value, or equal value and lower expert id.
__device__ __forceinline__ bool before(float va, int ea, float vb, int eb) {
    return va > vb || (va == vb && ea < eb);
}

// The k largest of the lane-distributed logits v (lane + 32 j), descending,
// equal logits to the lower expert id: warp-shuffle arg-max, k rounds.
template <int J>
__device__ __forceinline__ void warp_topk(const float (&v)[J], int E, int k, int lane,
                                          int (&sel)[kMaxK], float (&sl)[kMaxK]) {
    uint32_t taken = 0;
#pragma unroll
    for (int s = 0; s < kMaxK; ++s) {
        if (s >= k) break;
        float bv = -FLT_MAX;
        int be = INT_MAX;
#pragma unroll
        for (int j = 0; j < J; ++j) {
            const int e = lane + 32 * j;
            if (e < E && !(taken >> j & 1u) && before(v[j], e, bv, be)) {
                bv = v[j];
                be = e;
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int oe = __shfl_xor_sync(0xffffffffu, be, o);
            if (before(ov, oe, bv, be)) {
                bv = ov;
                be = oe;
            }
        }
        if (be == INT_MAX) be = 0;  // only if every remaining logit is NaN
        sel[s] = be;
        sl[s] = bv;
        if ((be & 31) == lane) taken |= 1u << (be >> 5);
    }
}

// Logits of a token either come finished (logits) or as nsplit partial sums
// over fixed K ranges (parts), added in order s = 0, 1, ... then + bias, and
// stored to logits_out.
template <int J>  // logits per lane: E <= 32 * J
__global__ void __launch_bounds__(32 * kWarpsPerBlock) topk_gates_kernel(
    const float* logits, const float* __restrict__ parts, int nsplit, int64_t stride,
    const float* __restrict__ bias, float* logits_out, int64_t T, int E, int k,
    const int32_t* __restrict__ ids_in, int32_t* __restrict__ ids_out,
    float* __restrict__ gates_out, int32_t* __restrict__ valid, int32_t* __restrict__ status,
    int filter, float log_tau) {
    const int lane = threadIdx.x & 31;
    const int64_t t = static_cast<int64_t>(blockIdx.x) * kWarpsPerBlock + (threadIdx.x >> 5);
    if (t >= T) return;
    float v[J];
    if (parts) {
        // all partial sums are loaded first (independent loads), then added
        // in the fixed order; the token's logits stay in registers
        float pv[kMaxSplit][J];
#pragma unroll
        for (int s = 0; s < kMaxSplit; ++s)
#pragma unroll
            for (int j = 0; j < J; ++j) {
                const int e = lane + 32 * j;
                pv[s][j] = s < nsplit && e < E ? parts[s * stride + t * E + e] : 0.0f;
            }
#pragma unroll
        for (int j = 0; j < J; ++j) {
            const int e = lane + 32 * j;
            float acc = pv[0][j];
#pragma unroll
            for (int s = 1; s < kMaxSplit; ++s)
                if (s < nsplit) acc += pv[s][j];
            if (bias && e < E) acc += bias[e];
            if (e < E) logits_out[t * E + e] = acc;
            v[j] = e < E ? acc : -FLT_MAX;
        }
        __syncwarp();
        logits = logits_out;
    }
    const float* l = logits + t * E;

    int sel[kMaxK];
    float sl[kMaxK];
    bool ok = true;
    if (!parts && (ids_in == nullptr || filter)) {
#pragma unroll
        for (int j = 0; j < J; ++j) {
            const int e = lane + 32 * j;
            v[j] = e < E ? l[e] : -FLT_MAX;
        }
    }
    if (ids_in == nullptr) {
        warp_topk<J>(v, E, k, lane, sel, sl);
    } else {
        int my = lane < k ? ids_in[t * k + lane] : 0;
        bool good = lane >= k || (my >= 0 && my < E);
#pragma unroll
        for (int s = 0; s < kMaxK; ++s) {
            if (s >= k) break;
            const int other = __shfl_sync(0xffffffffu, my, s);
            if (lane < k && s < lane && other == my) good = false;
        }
        ok = __all_sync(0xffffffffu, good);
        const float lv = (ok && lane < k) ? l[my] : 0.0f;
#pragma unroll
        for (int s = 0; s < kMaxK; ++s) {
            if (s >= k) break;
            sel[s] = ok ? __shfl_sync(0xffffffffu, my, s) : s;
            sl[s] = __shfl_sync(0xffffffffu, lv, s);
        }
        if (!ok && lane == 0) {
            atomicOr(status, STATUS_BAD_IDS);
            atomicAdd(status + 2, 1);
        }
        if (filter && ok) {
            // Replay plausibility filter (Composer 2 Technical Report, §6.2):
            // keep a replayed expert iff its logit is at least the router's own
            // k-th logit + ln(tau); refill dropped slots, in slot order, with the
            // router's own candidates not already present, in its own order.
            int own[kMaxK];
            float own_l[kMaxK];
            warp_topk<J>(v, E, k, lane, own, own_l);
            const float thr = own_l[k - 1] + log_tau;
            bool kept[kMaxK];
#pragma unroll
            for (int s = 0; s < kMaxK; ++s) kept[s] = s < k && sl[s] >= thr;
            int next = 0, replaced = 0;
#pragma unroll
            for (int s = 0; s < kMaxK; ++s) {
                if (s >= k || kept[s]) continue;
                for (;;) {
                    const int c = own[next];
                    const float cl = own_l[next];
                    ++next;
                    bool used = false;
#pragma unroll
                    for (int s2 = 0; s2 < kMaxK; ++s2)
                        if (s2 < k && (kept[s2] || s2 < s) && sel[s2] == c) used = true;
                    if (!used) {
                        sel[s] = c;
                        sl[s] = cl;
                        break;
                    }
                }
                ++replaced;
            }
            if (replaced && lane == 0) atomicAdd(status + 3, replaced);
        }
    }

    // Gate weights, identical arithmetic for own and replayed ids, fixed order.
    float m = sl[0];
#pragma unroll
    for (int s = 1; s < kMaxK; ++s)
        if (s < k) m = fmaxf(m, sl[s]);
    float ex[kMaxK];
    float den = 0.0f;
#pragma unroll
    for (int s = 0; s < kMaxK; ++s) {
        ex[s] = s < k ? expf(sl[s] - m) : 0.0f;
        den += ex[s];
    }
#pragma unroll
    for (int s = 0; s < kMaxK; ++s) {
        if (s < k && lane == s) {
            ids_out[t * k + s] = sel[s];
            gates_out[t * k + s] = ok ? ex[s] / den : 0.0f;
        }
    }
    if (lane == 0) valid[t] = ok ? 1 : 0;
}

struct TopkArgs {
    const float* logits;
    const float* parts;
    int nsplit;
    int64_t stride;
    const float* bias;
    float* logits_out;
    int64_t T;
    int E, k;
    const int32_t* ids_in;
    int32_t* ids_out;
    float* gates_out;
    int32_t* valid;
    int32_t* status;
    int filter;
    float log_tau;
};

template <int J>
cudaError_t launch_j(const TopkArgs& a, cudaStream_t s) {
    const int64_t blocks = (a.T + kWarpsPerBlock - 1) / kWarpsPerBlock;
    topk_gates_kernel<J><<<static_cast<unsigned>(blocks), 32 * kWarpsPerBlock, 0, s>>>(
        a.logits, a.parts, a.nsplit, a.stride, a.bias, a.logits_out, a.T, a.E, a.k, a.ids_in,
        a.ids_out, a.gates_out, a.valid, a.status, a.filter, a.log_tau);
    return cudaGetLastError();
}

cudaError_t launch_any(const TopkArgs& a, cudaStream_t s) {
    if (a.k < 1 || a.k > kMaxK || a.E < a.k || a.E > 512) return cudaErrorInvalidValue;
    if (a.T == 0) return cudaSuccess;
    if (a.E <= 64) return launch_j<2>(a, s);
    if (a.E <= 128) return launch_j<4>(a, s);
    if (a.E <= 256) return launch_j<8>(a, s);
    if (a.E <= 384) return launch_j<12>(a, s);
    return launch_j<16>(a, s);
}

}  // namespace

cudaError_t launch_topk_gates(const float* logits, int64_t T, int E, int k,
                              const int32_t* ids_in, int32_t* ids_out, float* gates_out,
                              int32_t* valid, int32_t* status, cudaStream_t s) {
    const TopkArgs a{logits, nullptr, 1, 0, nullptr, nullptr, T, E, k, ids_in, ids_out,
                     gates_out, valid, status, 0, 0.0f};
    return launch_any(a, s);
}

cudaError_t launch_topk_gates_split(const float* parts, int nsplit, int64_t stride,
                                    const float* bias, float* logits_out, int64_t T, int E,
                                    int k, const int32_t* ids_in, int32_t* ids_out,
                                    float* gates_out, int32_t* valid, int32_t* status,
                                    cudaStream_t s, int filter, float log_tau) {
    if (!logits_out || nsplit < 1 || nsplit > kMaxSplit || (nsplit > 1 && !parts))
        return cudaErrorInvalidValue;
    if (filter && !ids_in) return cudaErrorInvalidValue;
    const TopkArgs a{logits_out, nsplit > 1 ? parts : nullptr, nsplit, stride, bias, logits_out,
                     T, E, k, ids_in, ids_out, gates_out, valid, status, filter, log_tau};
    return launch_any(a, s);
}

}  // namespace moe
