// api.cu -- the C ABI of libmoedet (declared in include/moe_det.h): argument
// validation, workspace carving, TMA descriptor set-up and the launch sequence
//   router GEMM -> top-k/replay + gates -> counting sort -> gather
//   -> grouped gate/up GEMM + SwiGLU -> grouped down GEMM -> fixed-order combine
// of the MoE layer forward with router replay (Composer 2 Technical Report,
// §6.2 "RL infrastructure" for replay, §6.1 "Training infrastructure" for the
// grouped expert GEMMs and dispatch/combine).  Everything is enqueued on the
// caller's stream; nothing is allocated and nothing synchronises except
// moe_get_status.
#include <cudaTypedefs.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "moe_det.h"
#include "moe_internal.h"
#include "route_launch.h"

using namespace moe;

static_assert(moe::WFMT_BF16 == MOE_W_BF16 && moe::WFMT_MXFP8 == MOE_W_MXFP8 &&
                  moe::WFMT_NVFP4 == MOE_W_NVFP4,
              "weight format codes match the ABI");  // MOE_W_MXFP8_ACT runs the MXFP8 kernels

namespace {

constexpr uint64_t kWaitTimeoutNs = 1000000000ull;  // bounded device waits: 1 s
// The router GEMM splits K into this many fixed parts (when d/64 divides by it),
// summed in a fixed order by the top-k kernel: more CTAs stream the router
// weights at small T, and the split does not depend on T.
constexpr int kRouterSplit = 4;

inline size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

struct Layout {
    size_t status, logits, rpart, valid, cnt, off, perm, inv, scratch, xp, h, y, ysh;
    size_t xq, sx, sxp, sh;  // NVFP4; xq also MXFP8 activations (codes, scales)
    size_t hq;               // MXFP8 activations: codes and scales of h
    size_t total;
};


bool dims_ok(const moe_dims* d) {
    if (!d) return false;
    if (d->T < 0 || d->T > (int64_t(1) << 20)) return false;
    if (d->k != 8) return false;
    if (d->E < 8 || d->E > 512) return false;
    if (d->d < 64 || d->d > 16384 || d->d % 64) return false;
    if (d->F < 64 || d->F > 16384 || d->F % 64) return false;
    if (d->n_shared < 0 || d->n_shared > 1) return false;
    if (d->wfmt != MOE_W_BF16 && d->wfmt != MOE_W_MXFP8 && d->wfmt != MOE_W_NVFP4 &&
        d->wfmt != MOE_W_MXFP8_ACT)
        return false;
    // block-scaled weights: scale rows are loaded 8 k-blocks (512 along K) at a time
    if (d->wfmt != MOE_W_BF16 && (d->d % 512 || d->F % 512)) return false;
    if (d->out_fp32 != 0 && d->out_fp32 != 1) return false;
    return true;
}

Layout make_layout(const moe_dims* d) {
    Layout L{};
    const size_t T = static_cast<size_t>(d->T), k = d->k, E = d->E, S = d->n_shared;
    const size_t rows = T * k + T * S;
    size_t o = 0;
    auto take = [&](size_t bytes) { const size_t at = o; o = align256(o + bytes); return at; };
    L.status = take(32);  // int32 [0..3] status words, [4..5] SM-pair GEMM tile counters
    L.logits = take(T * E * 4);
    L.rpart = take(route_split(d) > 1 ? T * E * 4 * route_split(d) : 0);
    L.valid = take(T * 4);
    L.cnt = take(E * 4);
    L.off = take((E + 1) * 4);
    L.perm = take(T * k * 4);
    L.inv = take(T * k * 4);
    L.scratch = take(dispatch_scratch_bytes(static_cast<int64_t>(T * k), static_cast<int>(E)));
    L.xp = take(rows * d->d * 2);
    L.h = take(rows * d->F * 2);
    L.y = take(T * k * d->d * 2);
    L.ysh = take(S ? T * d->d * 4 : 0);
    const bool nv = d->wfmt == MOE_W_NVFP4;
    const bool mxa = d->wfmt == MOE_W_MXFP8_ACT;
    // Narrow activations, codes then block scales: MXFP8 E4M3 codes [T][d] and
    // E8M0 scales [T][d/32] of x; NVFP4 E2M1 codes [T][d/2] and E4M3 scales
    // [T][d/16] (the gathered rows' codes and scales in xp, those of h in hq)
    L.xq = take(nv ? T * d->d / 2 + T * d->d / 16 : (mxa ? T * d->d + T * d->d / 32 : 0));
    L.sx = take(nv ? T * 4 : 0);
    L.sxp = take(nv ? T * k * 4 : 0);
    L.sh = take(nv ? T * k * 4 : 0);
    L.hq = take(mxa ? T * k * d->F + T * k * d->F / 32
                    : (nv ? T * k * d->F / 2 + T * k * d->F / 16 : 0));
    L.total = o;
    return L;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// 2-D bf16 map over [rows][K] (K contiguous), box 64 x box_rows, 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* base, uint64_t K, uint64_t rows, uint32_t box_rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {K, rows};
    const cuuint64_t strides[1] = {K * 2};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(BK), box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D byte map over [rows][K] (K bytes contiguous), box box_k x box_rows, no
// swizzle (or the 128-byte swizzle, for 128-byte boxes that feed the MMA
// directly): MXFP8 weight tiles and their E8M0 scales (16-byte boxes).
bool make_map_u8(CUtensorMap* m, const void* base, uint64_t K, uint64_t rows, uint32_t box_k,
                 uint32_t box_rows, bool swizzle128 = false) {
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {K, rows};
    const cuuint64_t strides[1] = {K};
    const cuuint32_t box[2] = {box_k, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE,
              swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int num_sms() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return n;
}

inline bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

moe_status check_common(const moe_dims* d, const void* x, const moe_weights* w, void* ws,
                        size_t ws_bytes) {
    if (!d || !w) return MOE_ERR_ARG;
    if (!dims_ok(d)) return MOE_ERR_SHAPE;
    if (d->T == 0) return MOE_OK;
    if (!x || !ws || !w->w_router) return MOE_ERR_ARG;
    if (!al16(x) || !al16(ws) || !al16(w->w_router) || !al16(w->router_bias)) return MOE_ERR_ALIGN;
    if (ws_bytes < make_layout(d).total) return MOE_ERR_WORKSPACE;
    return MOE_OK;
}

moe_status check_experts(const moe_dims* d, const moe_weights* w) {
    if (!w->w_gate || !w->w_up || !w->w_down) return MOE_ERR_ARG;
    if (!al16(w->w_gate) || !al16(w->w_up) || !al16(w->w_down)) return MOE_ERR_ALIGN;
    if (d->wfmt != MOE_W_BF16) {
        if (!w->s_gate || !w->s_up || !w->s_down) return MOE_ERR_ARG;
        if (!al16(w->s_gate) || !al16(w->s_up) || !al16(w->s_down)) return MOE_ERR_ALIGN;
    }
    if (d->wfmt == MOE_W_NVFP4 && (!w->gs_gate || !w->gs_up || !w->gs_down)) return MOE_ERR_ARG;
    if (!al16(w->w_gate_up)) return MOE_ERR_ALIGN;
    if (w->w_gate_up && d->wfmt != MOE_W_BF16) return MOE_ERR_UNSUPPORTED;
    if (d->n_shared) {
        if (!w->ws_gate || !w->ws_up || !w->ws_down) return MOE_ERR_ARG;
        if (!al16(w->ws_gate) || !al16(w->ws_up) || !al16(w->ws_down)) return MOE_ERR_ALIGN;
    }
    return MOE_OK;
}

inline moe_status cu(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

// Per-host-thread stage timing events (moe_set_stage_events); null = off.
thread_local cudaEvent_t g_stage_events[2 * MOE_NUM_STAGES];
thread_local bool g_stage_timing = false;

inline moe_status mark(int stage, int edge, cudaStream_t s) {
    if (!g_stage_timing) return MOE_OK;
    return cu(cudaEventRecord(g_stage_events[2 * stage + edge], s));
}

thread_local cudaEvent_t g_bwd_events[2 * MOE_BWD_NUM_STAGES];
thread_local bool g_bwd_timing = false;

inline moe_status mark_b(int stage, int edge, cudaStream_t s) {
    if (!g_bwd_timing) return MOE_OK;
    return cu(cudaEventRecord(g_bwd_events[2 * stage + edge], s));
}

#define MOE_TRY(expr)                         \
    do {                                      \
        const moe_status st_ = (expr);        \
        if (st_ != MOE_OK) return st_;        \
    } while (0)

}  // namespace

namespace moe {

int route_split(const moe_dims* d) { return (d->d / BK) % kRouterSplit == 0 ? kRouterSplit : 1; }

// Router logits (fp32, + bias) and the routing decision for every token.
moe_status launch_route(const moe_dims* d, const void* x, const moe_weights* w,
                        const int32_t* ids_in, int32_t* ids_out, float* gates_out,
                        const RouteScratch& sc, cudaStream_t s, bool filter, float tau) {
    const int64_t T = d->T;
    MOE_TRY(cu(cudaMemsetAsync(sc.status, 0, 32, s)));
    GemmParams p;
    std::memset(&p, 0, sizeof p);
    if (!make_map(&p.a0, w->w_router, d->d, d->E, BM)) return MOE_ERR_CUDA;
    if (!make_map(&p.b, x, d->d, T, BN)) return MOE_ERR_CUDA;
    if (!make_map(&p.b32, x, d->d, T, 32)) return MOE_ERR_CUDA;
    p.partial_b = 1;
    const int split = route_split(d);
    p.ksplit = split;
    p.split_stride = T * d->E;
    p.G = 1;
    p.n_single = static_cast<int32_t>(T);
    p.M = d->E;
    p.MT = (d->E + BM - 1) / BM;
    p.KB = d->d / BK;
    p.out = split > 1 ? sc.parts : sc.logits;
    p.ldo = d->E;
    p.bias = split > 1 ? nullptr : w->router_bias;
    p.status = sc.status;
    p.timeout_ns = kWaitTimeoutNs;
    const int64_t tiles = int64_t(p.MT) * ((T + BN - 1) / BN) * split;
    const int sms = num_sms();
    if (sms <= 0) return MOE_ERR_CUDA;
    const int grid = static_cast<int>(tiles < sms ? tiles : sms);
    MOE_TRY(mark(MOE_STAGE_ROUTER_GEMM, 0, s));
    MOE_TRY(cu(launch_grouped_gemm(GEMM_ROUTER, p, grid, s)));
    MOE_TRY(mark(MOE_STAGE_ROUTER_GEMM, 1, s));
    MOE_TRY(mark(MOE_STAGE_TOPK, 0, s));
    const float log_tau = tau > 0.0f ? std::log(tau) : -INFINITY;
    if (split > 1 || filter)
        MOE_TRY(cu(launch_topk_gates_split(sc.parts, split, T * d->E,
                                           split > 1 ? w->router_bias : nullptr, sc.logits, T,
                                           d->E, d->k, ids_in, ids_out, gates_out, sc.valid,
                                           sc.status, s, filter ? 1 : 0, log_tau)));
    else
        MOE_TRY(cu(launch_topk_gates(sc.logits, T, d->E, d->k, ids_in, ids_out, gates_out,
                                     sc.valid, sc.status, s)));
    return mark(MOE_STAGE_TOPK, 1, s);
}

}  // namespace moe

namespace {

moe_status run_route(const moe_dims* d, const void* x, const moe_weights* w, const int32_t* ids_in,
                     int32_t* ids_out, float* gates_out, uint8_t* ws, const Layout& L,
                     cudaStream_t s, bool filter = false, float tau = 0.0f) {
    const RouteScratch sc{reinterpret_cast<int32_t*>(ws + L.status),
                          reinterpret_cast<float*>(ws + L.logits),
                          reinterpret_cast<float*>(ws + L.rpart),
                          reinterpret_cast<int32_t*>(ws + L.valid)};
    return launch_route(d, x, w, ids_in, ids_out, gates_out, sc, s, filter, tau);
}

// Kernel family of the expert GEMMs: the one-SM kernel for batches of at most
// kOneSmMaxTokens tokens (bf16 weights), SM pairs otherwise.  Both compute each
// output element with the same MMAs in the same K order.  MOE_EXPERT_KERNEL=
// one_sm | pair in the environment forces one family (bf16 weights only).
bool one_sm_experts(const moe_dims* d) {
    if (d->wfmt != MOE_W_BF16) return false;
    static const int forced = [] {
        const char* e = std::getenv("MOE_EXPERT_KERNEL");
        if (!e) return 0;
        if (std::strcmp(e, "one_sm") == 0) return 1;
        if (std::strcmp(e, "pair") == 0) return 2;
        return 0;
    }();
    if (forced) return forced == 1;
    return d->T <= kOneSmMaxTokens;
}

// Test hook for failure detection: MOE_TEST_STALL_CALLS=N makes the gate/up
// GEMM of the next N forward calls (process-wide) issue no loads, so its MMA
// wait runs out (bounded, 1 s) and the call reports MOE_ERR_TIMEOUT through
// moe_get_status.  Unset in normal use.
bool take_stall_test() {
    static std::atomic<int> left{[] {
        const char* e = std::getenv("MOE_TEST_STALL_CALLS");
        return e ? std::atoi(e) : 0;
    }()};
    int v = left.load();
    while (v > 0)
        if (left.compare_exchange_weak(v, v - 1)) return true;
    return false;
}

// Test hook for failure detection in the backward: MOE_TEST_STALL_BWD_CALLS=N
// makes the dWg/dWu weight-gradient GEMM of the next N backward calls
// (process-wide) issue no loads, so its MMA wait runs out (bounded, 1 s) and
// moe_get_status reports MOE_ERR_TIMEOUT.  Unset in normal use.
bool take_stall_test_bwd() {
    static std::atomic<int> left{[] {
        const char* e = std::getenv("MOE_TEST_STALL_BWD_CALLS");
        return e ? std::atoi(e) : 0;
    }()};
    int v = left.load();
    while (v > 0)
        if (left.compare_exchange_weak(v, v - 1)) return true;
    return false;
}

// A second stream (and its fork/join events) per device and host thread, for
// work that overlaps the caller's stream inside one call; created on first use
// and kept for the life of the process.  Work on it is ordered against the
// caller's stream by events only, so the call stays stream-ordered (and can be
// captured in a CUDA graph).
struct SideStream {
    cudaStream_t stream = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr;
};
constexpr int kMaxDevices = 64;
thread_local SideStream g_side[kMaxDevices];

moe_status side_stream(SideStream** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_CUDA;
    SideStream& sd = g_side[dev];
    if (!sd.stream) {
        // highest priority: its persistent CTAs are placed first and the
        // caller's memory-bound kernels fill the room they leave on each SM
        int least = 0, greatest = 0;
        MOE_TRY(cu(cudaDeviceGetStreamPriorityRange(&least, &greatest)));
        MOE_TRY(cu(cudaStreamCreateWithPriority(&sd.stream, cudaStreamNonBlocking, greatest)));
        MOE_TRY(cu(cudaEventCreateWithFlags(&sd.fork, cudaEventDisableTiming)));
        MOE_TRY(cu(cudaEventCreateWithFlags(&sd.join, cudaEventDisableTiming)));
    }
    *out = &sd;
    return MOE_OK;
}

// Both expert GEMMs on the block-scaled tensor-core MMA (gemm_bs.cu): every
// token row of x, and every row of the SwiGLU output h, is quantised along K
// (MXFP8 weights and activations: E4M3 codes with E8M0 scales per 32; NVFP4:
// E2M1 codes with E4M3 scales per 16 and an fp32 scale per row), gathered as
// codes and scales, and multiplied by the narrow weights.  Any batch size
// takes this one path, so the result of a token never depends on its batch.
moe_status run_experts_bs(const moe_dims* d, const void* x, const moe_weights* w, void* out,
                          const int32_t* ids, const float* gates, uint8_t* ws, const Layout& L,
                          cudaStream_t s) {
    const int64_t T = d->T;
    const int k = d->k, E = d->E;
    const int64_t rows = T * k;
    const int D = d->d, F = d->F;
    const bool nv = d->wfmt == MOE_W_NVFP4;
    const int fmt = nv ? BS_NVFP4 : BS_MXFP8;
    int32_t* status = reinterpret_cast<int32_t*>(ws + L.status);
    int32_t* cnt = reinterpret_cast<int32_t*>(ws + L.cnt);
    int32_t* off = reinterpret_cast<int32_t*>(ws + L.off);
    int32_t* perm = reinterpret_cast<int32_t*>(ws + L.perm);
    int32_t* inv = reinterpret_cast<int32_t*>(ws + L.inv);
    const int sms = num_sms();
    if (sms <= 0) return MOE_ERR_CUDA;
    if (d->n_shared) return MOE_ERR_UNSUPPORTED;
    // bytes per row of codes and of scales, along d and along F
    const int cd = nv ? D / 2 : D, sd = nv ? D / 16 : D / 32;
    const int cf = nv ? F / 2 : F, sf = nv ? F / 16 : F / 32;
    uint8_t* xc = ws + L.xq;                     // [T][cd] codes, then [T][sd] scales
    uint8_t* xs = xc + T * cd;
    uint8_t* xpc = ws + L.xp;                    // gathered: [rows][cd], then [rows][sd]
    uint8_t* xps = xpc + rows * cd;
    uint8_t* hc = ws + L.hq;                     // [rows][cf] codes, then [rows][sf] scales
    uint8_t* hsc = hc + rows * cf;
    float* sx = reinterpret_cast<float*>(ws + L.sx);    // NVFP4 row scales
    float* sxp = reinterpret_cast<float*>(ws + L.sxp);
    float* sh = reinterpret_cast<float*>(ws + L.sh);
    const uint64_t EF = uint64_t(E) * F, ED = uint64_t(E) * D;
    const int units = sms / 2;

    MOE_TRY(mark(MOE_STAGE_DISPATCH, 0, s));
    MOE_TRY(cu(launch_dispatch(ids, T, k, E, cnt, off, perm, inv,
                               reinterpret_cast<int32_t*>(ws + L.scratch), s)));
    MOE_TRY(mark(MOE_STAGE_DISPATCH, 1, s));
    MOE_TRY(mark(MOE_STAGE_GATHER, 0, s));
    // each token row quantised once and written to its own row and to its k
    // gathered rows (codes, block scales; NVFP4 also the row scale)
    if (nv)
        MOE_TRY(cu(launch_nvfp4_codes(static_cast<const uint16_t*>(x), xc, xs, sx, T, D, sms, s, inv,
                                      k, xpc, xps, sxp)));
    else
        MOE_TRY(cu(launch_mx_rows_fp8(static_cast<const uint16_t*>(x), xc, xs, T, D, sms, s, inv, k,
                                      xpc, xps)));
    MOE_TRY(mark(MOE_STAGE_GATHER, 1, s));

    const int tn = bs_tile_tokens(fmt), kk = 128, big = bs_big_box(fmt), sbox = bs_scale_box(fmt);
    const int64_t ntiles = (rows + tn - 1) / tn + E;
    auto common = [&](GemmParams& p) {
        p.cnt = cnt;
        p.off = off;
        p.G = E;
        p.status = status;
        p.timeout_ns = kWaitTimeoutNs;
        // scales ahead of the weights once the experts average a full tile
        p.sc_ahead = rows >= static_cast<int64_t>(E) * tn ? 1 : 0;
    };
    const uint32_t rg = gemm_rows(GEMM_SWIGLU);
    GemmParams p1;
    std::memset(&p1, 0, sizeof p1);
    common(p1);
    if (!make_map_u8(&p1.a0, w->w_gate, cd, EF, kk, rg, true)) return MOE_ERR_CUDA;
    if (!make_map_u8(&p1.a1, w->w_up, cd, EF, kk, rg, true)) return MOE_ERR_CUDA;
    if (!make_map_u8(&p1.sa0, w->s_gate, sd, EF, sbox, rg)) return MOE_ERR_CUDA;
    if (!make_map_u8(&p1.sa1, w->s_up, sd, EF, sbox, rg)) return MOE_ERR_CUDA;
    if (!make_map_u8(&p1.b, xpc, cd, rows, kk, big, true)) return MOE_ERR_CUDA;
    if (!make_map_u8(&p1.b32, xpc, cd, rows, kk, 32, true)) return MOE_ERR_CUDA;
    if (!make_map_u8(&p1.sb_scale, xps, sd, rows, sbox, 128)) return MOE_ERR_CUDA;
    if (nv) {
        p1.row_scale = sxp;
        p1.wscale0 = w->gs_gate;
        p1.wscale1 = w->gs_up;
    }
    p1.M = F;
    p1.MT = F / (2 * static_cast<int>(rg));
    p1.KB = cd / kk;
    p1.out = ws + L.h;
    p1.ldo = F;
    p1.stall_test = take_stall_test() ? 1 : 0;
    int64_t tb = ntiles * p1.MT;
    MOE_TRY(mark(MOE_STAGE_GATE_UP, 0, s));
    MOE_TRY(cu(launch_bs_gemm(fmt, GEMM_SWIGLU, p1, static_cast<int>(tb < units ? tb : units), s)));
    MOE_TRY(mark(MOE_STAGE_GATE_UP, 1, s));

    GemmParams p2;
    std::memset(&p2, 0, sizeof p2);
    common(p2);
    if (!make_map_u8(&p2.a0, w->w_down, cf, ED, kk, BM, true)) return MOE_ERR_CUDA;
    if (!make_map_u8(&p2.sa0, w->s_down, sf, ED, sbox, BM)) return MOE_ERR_CUDA;
    if (!make_map_u8(&p2.b, hc, cf, rows, kk, big, true)) return MOE_ERR_CUDA;
    if (!make_map_u8(&p2.b32, hc, cf, rows, kk, 32, true)) return MOE_ERR_CUDA;
    if (!make_map_u8(&p2.sb_scale, hsc, sf, rows, sbox, 128)) return MOE_ERR_CUDA;
    if (nv) {
        p2.row_scale = sh;
        p2.wscale0 = w->gs_down;
    }
    p2.M = D;
    p2.MT = D / (2 * BM);
    p2.KB = cf / kk;
    p2.out = ws + L.y;
    p2.ldo = D;
    tb = ntiles * p2.MT;
    MOE_TRY(mark(MOE_STAGE_DOWN, 0, s));
    const uint16_t* h = reinterpret_cast<const uint16_t*>(ws + L.h);
    if (nv)
        MOE_TRY(cu(launch_nvfp4_codes(h, hc, hsc, sh, rows, F, sms, s)));
    else
        MOE_TRY(cu(launch_mx_rows_fp8(h, hc, hsc, rows, F, sms, s)));
    MOE_TRY(cu(launch_bs_gemm(fmt, GEMM_DOWN, p2, static_cast<int>(tb < units ? tb : units), s)));
    MOE_TRY(mark(MOE_STAGE_DOWN, 1, s));

    MOE_TRY(mark(MOE_STAGE_COMBINE, 0, s));
    MOE_TRY(cu(launch_combine(reinterpret_cast<const uint16_t*>(ws + L.y), nullptr, inv, gates,
                              reinterpret_cast<const int32_t*>(ws + L.valid), T, k, D,
                              d->out_fp32, out, s)));
    return mark(MOE_STAGE_COMBINE, 1, s);
}

// Dispatch, expert FFNs and combine, given ids/gates of every token.
moe_status run_experts(const moe_dims* d, const void* x, const moe_weights* w, void* out,
                       const int32_t* ids, const float* gates, uint8_t* ws, const Layout& L,
                       cudaStream_t s) {
    if (d->wfmt == MOE_W_MXFP8_ACT || d->wfmt == MOE_W_NVFP4)
        return run_experts_bs(d, x, w, out, ids, gates, ws, L, s);
    const int64_t T = d->T;
    const int k = d->k, E = d->E, S = d->n_shared;
    const int64_t rows = T * k + T * S;
    int32_t* status = reinterpret_cast<int32_t*>(ws + L.status);
    int32_t* cnt = reinterpret_cast<int32_t*>(ws + L.cnt);
    int32_t* off = reinterpret_cast<int32_t*>(ws + L.off);
    int32_t* perm = reinterpret_cast<int32_t*>(ws + L.perm);
    int32_t* inv = reinterpret_cast<int32_t*>(ws + L.inv);
    const int sms = num_sms();
    if (sms <= 0) return MOE_ERR_CUDA;
    const bool mx = d->wfmt == MOE_W_MXFP8;
    const int kfmt = mx ? WFMT_MXFP8 : WFMT_BF16;  // the GEMM kernels' weight format
    const bool one = one_sm_experts(d);
    // MXFP8 weights with few tokens: the SM-pair weight-streaming variant
    const int small = !one && mx && T <= kOneSmMaxTokens;
    const int bn = one ? BN : (small ? 64 : BN_EXPERT);           // tokens per tile
    const uint32_t box_b = one ? BN : BN_EXPERT / 2;              // token rows per CTA
    const uint32_t rg = one ? BM : gemm_rows(GEMM_SWIGLU);        // gate (= up) rows per CTA
    const int tile_g = one ? BM : 2 * gemm_rows(GEMM_SWIGLU);     // gate rows per tile
    const int tile_d = one ? BM : 2 * BM;                         // down rows per tile
    const int units = one ? sms : sms / 2;                        // CTAs or CTA pairs
    const uint64_t EF = uint64_t(E) * d->F, ED = uint64_t(E) * d->d;
    // SM pairs, bf16, shared expert: the shared expert's gate/up needs no
    // routing, so it runs on a second stream, reading x directly, while the
    // dispatch and the gather run here; its tiles and the routed ones come
    // from queues, so the two launches share the SMs however they overlap.
    const bool overlap = S && !one && d->wfmt == MOE_W_BF16;
    // packed gate/up weights (moe_pack_weights): routed experts, then the shared one
    const bool packed = w->w_gate_up && !one && d->wfmt == MOE_W_BF16;
    const uint8_t* pk = static_cast<const uint8_t*>(w->w_gate_up);
    const uint8_t* pk_shared = pk ? pk + uint64_t(E) * 2 * d->F * d->d * 2 : nullptr;
    SideStream* side = nullptr;
    if (overlap) {
        MOE_TRY(side_stream(&side));
        GemmParams ps;
        std::memset(&ps, 0, sizeof ps);
        ps.cnt = cnt;
        ps.off = off;
        ps.G = 0;
        ps.has_shared = 1;
        ps.shared_rows = static_cast<int32_t>(T);
        ps.shared_b_off = 0;
        ps.out_row_off = static_cast<int32_t>(T * k);
        ps.partial_b = 1;
        ps.status = status;
        ps.timeout_ns = kWaitTimeoutNs;
        if (packed) {
            if (!make_map(&ps.a0, pk_shared, d->d, 2 * d->F, 2 * rg)) return MOE_ERR_CUDA;
            ps.a1 = ps.a0;
            ps.a_packed = 1;
        } else {
            if (!make_map(&ps.a0, w->ws_gate, d->d, d->F, rg)) return MOE_ERR_CUDA;
            if (!make_map(&ps.a1, w->ws_up, d->d, d->F, rg)) return MOE_ERR_CUDA;
        }
        ps.as0 = ps.a0;
        ps.as1 = ps.a1;
        if (!make_map(&ps.b, x, d->d, T, box_b)) return MOE_ERR_CUDA;
        if (!make_map(&ps.b32, x, d->d, T, 32)) return MOE_ERR_CUDA;
        ps.M = d->F;
        ps.MT = (d->F + tile_g - 1) / tile_g;
        ps.KB = d->d / BK;
        ps.out = ws + L.h;
        ps.ldo = d->F;
        ps.tile_counter = status + 6;
        const int64_t tbs = (T + bn - 1) / bn * ps.MT;
        MOE_TRY(cu(cudaEventRecord(side->fork, s)));
        MOE_TRY(cu(cudaStreamWaitEvent(side->stream, side->fork, 0)));
        MOE_TRY(cu(launch_pair_gemm(GEMM_SWIGLU, ps, static_cast<int>(tbs < units ? tbs : units),
                                    side->stream, d->wfmt)));
        MOE_TRY(cu(cudaEventRecord(side->join, side->stream)));
    }
    const int Sg = overlap ? 0 : S;  // shared expert inside the routed gate/up launch
    MOE_TRY(mark(MOE_STAGE_DISPATCH, 0, s));
    MOE_TRY(cu(launch_dispatch(ids, T, k, E, cnt, off, perm, inv,
                               reinterpret_cast<int32_t*>(ws + L.scratch), s)));
    MOE_TRY(mark(MOE_STAGE_DISPATCH, 1, s));
    MOE_TRY(mark(MOE_STAGE_GATHER, 0, s));
    MOE_TRY(cu(launch_gather(static_cast<const uint16_t*>(x), inv, T, k, d->d, Sg,
                             reinterpret_cast<uint16_t*>(ws + L.xp), s)));
    MOE_TRY(mark(MOE_STAGE_GATHER, 1, s));

    const int64_t ntiles = (T * k + bn - 1) / bn + E + (S ? (T + bn - 1) / bn : 0);

    auto common = [&](GemmParams& p) {
        p.cnt = cnt;
        p.off = off;
        p.G = E;
        p.has_shared = S;
        p.shared_rows = static_cast<int32_t>(T);
        p.shared_b_off = static_cast<int32_t>(T * k);
        p.partial_b = 1;
        p.status = status;
        p.timeout_ns = kWaitTimeoutNs;
    };

    // gate/up projections with the SwiGLU epilogue -> H
    GemmParams p1;
    std::memset(&p1, 0, sizeof p1);
    common(p1);
    p1.has_shared = Sg;
    if (mx) {
        if (!make_map_u8(&p1.a0, w->w_gate, d->d, EF, BK, rg)) return MOE_ERR_CUDA;
        if (!make_map_u8(&p1.a1, w->w_up, d->d, EF, BK, rg)) return MOE_ERR_CUDA;
        if (!make_map_u8(&p1.sa0, w->s_gate, d->d / 32, EF, 16, rg)) return MOE_ERR_CUDA;
        if (!make_map_u8(&p1.sa1, w->s_up, d->d / 32, EF, 16, rg)) return MOE_ERR_CUDA;
    } else if (packed) {
        if (!make_map(&p1.a0, pk, d->d, 2 * EF, 2 * rg)) return MOE_ERR_CUDA;
        p1.a1 = p1.a0;
        p1.a_packed = 1;
    } else {
        if (!make_map(&p1.a0, w->w_gate, d->d, EF, rg)) return MOE_ERR_CUDA;
        if (!make_map(&p1.a1, w->w_up, d->d, EF, rg)) return MOE_ERR_CUDA;
    }
    if (Sg) {
        if (packed) {
            if (!make_map(&p1.as0, pk_shared, d->d, 2 * d->F, 2 * rg)) return MOE_ERR_CUDA;
            p1.as1 = p1.as0;
        } else {
            if (!make_map(&p1.as0, w->ws_gate, d->d, d->F, rg)) return MOE_ERR_CUDA;
            if (!make_map(&p1.as1, w->ws_up, d->d, d->F, rg)) return MOE_ERR_CUDA;
        }
    }
    if (!make_map(&p1.b, ws + L.xp, d->d, rows, box_b)) return MOE_ERR_CUDA;
    if (!make_map(&p1.b32, ws + L.xp, d->d, rows, 32)) return MOE_ERR_CUDA;
    p1.M = d->F;
    p1.MT = (d->F + tile_g - 1) / tile_g;
    p1.KB = d->d / BK;
    p1.out = ws + L.h;
    p1.ldo = d->F;
    p1.stall_test = take_stall_test() ? 1 : 0;
    p1.tile_counter = status + 4;
    int64_t tb = ntiles * p1.MT;
    const int g1 = static_cast<int>(tb < units ? tb : units);
    MOE_TRY(mark(MOE_STAGE_GATE_UP, 0, s));
    MOE_TRY(cu(one ? launch_grouped_gemm(GEMM_SWIGLU, p1, g1, s)
                   : launch_pair_gemm(GEMM_SWIGLU, p1, g1, s, kfmt, small)));
    MOE_TRY(mark(MOE_STAGE_GATE_UP, 1, s));

    // down projection -> Y (routed, bf16) and Ysh (shared, fp32)
    GemmParams p2;
    std::memset(&p2, 0, sizeof p2);
    common(p2);
    if (mx) {
        if (!make_map_u8(&p2.a0, w->w_down, d->F, ED, BK, BM)) return MOE_ERR_CUDA;
        if (!make_map_u8(&p2.sa0, w->s_down, d->F / 32, ED, 16, BM)) return MOE_ERR_CUDA;
    } else if (!make_map(&p2.a0, w->w_down, d->F, ED, BM)) {
        return MOE_ERR_CUDA;
    }
    if (S && !make_map(&p2.as0, w->ws_down, d->F, d->d, BM)) return MOE_ERR_CUDA;
    if (!make_map(&p2.b, ws + L.h, d->F, rows, box_b)) return MOE_ERR_CUDA;
    if (!make_map(&p2.b32, ws + L.h, d->F, rows, 32)) return MOE_ERR_CUDA;
    p2.M = d->d;
    p2.MT = (d->d + tile_d - 1) / tile_d;
    p2.KB = d->F / BK;
    p2.out = ws + L.y;
    p2.out_shared = S ? ws + L.ysh : nullptr;
    p2.ldo = d->d;
    p2.tile_counter = status + 5;
    tb = ntiles * p2.MT;
    const int g2 = static_cast<int>(tb < units ? tb : units);
    if (overlap) MOE_TRY(cu(cudaStreamWaitEvent(s, side->join, 0)));
    MOE_TRY(mark(MOE_STAGE_DOWN, 0, s));
    MOE_TRY(cu(one ? launch_grouped_gemm(GEMM_DOWN, p2, g2, s)
                   : launch_pair_gemm(GEMM_DOWN, p2, g2, s, kfmt, small)));
    MOE_TRY(mark(MOE_STAGE_DOWN, 1, s));

    MOE_TRY(mark(MOE_STAGE_COMBINE, 0, s));
    MOE_TRY(cu(launch_combine(reinterpret_cast<const uint16_t*>(ws + L.y),
                              S ? reinterpret_cast<const float*>(ws + L.ysh) : nullptr, inv, gates,
                              reinterpret_cast<const int32_t*>(ws + L.valid), T, k, d->d,
                              d->out_fp32, out, s)));
    return mark(MOE_STAGE_COMBINE, 1, s);
}

moe_status forward_impl(const moe_dims* d, const void* x, const moe_weights* w,
                        const int32_t* ids_in, bool replay, void* out, int32_t* ids_out,
                        float* gates_out, void* ws, size_t ws_bytes, moe_stream_t stream,
                        bool filter = false, float tau = 0.0f) {
    MOE_TRY(check_common(d, x, w, ws, ws_bytes));
    if (d->T == 0) return MOE_OK;
    MOE_TRY(check_experts(d, w));
    if (!out || !ids_out || !gates_out || (replay && !ids_in)) return MOE_ERR_ARG;
    if (!al16(out) || !al16(ids_out) || !al16(gates_out) || (replay && !al16(ids_in)))
        return MOE_ERR_ALIGN;
    // Block-scaled expert weights: the shared expert (bf16 by definition) is not served.
    if (d->wfmt != MOE_W_BF16 && d->n_shared) return MOE_ERR_UNSUPPORTED;
    const Layout L = make_layout(d);
    auto* s = reinterpret_cast<cudaStream_t>(stream);
    auto* wsb = static_cast<uint8_t*>(ws);
    MOE_TRY(run_route(d, x, w, replay ? ids_in : nullptr, ids_out, gates_out, wsb, L, s, filter,
                      tau));
    return run_experts(d, x, w, out, ids_out, gates_out, wsb, L, s);
}

// ---- backward ------------------------------------------------------------------

struct BwdLayout {
    Layout f;  // the forward's regions first (status word at offset 0)
    size_t ids, gates, poff, a, b, dg, dl, dyq, dh, dabq, dxp, xpt, dyt, ht, dabt;
    int64_t kpad;
    size_t total;
};

// The weight copies of the dH and dXp GEMMs: E4M3 codes, then E8M0 scale
// bytes, of the routed experts followed by the shared expert (group E).
struct BwdWeights {
    size_t wd, wds, w2, w2s, total;
};

// d and 2F are multiples of 512: the block-scaled GEMMs load scales for four
// 128-wide K blocks at a time
moe_status bwd_dims_status(const moe_dims* d) {
    if (!d) return MOE_ERR_ARG;
    if (!dims_ok(d)) return MOE_ERR_SHAPE;
    if (d->wfmt != MOE_W_BF16) return MOE_ERR_UNSUPPORTED;
    if (d->d % 512 || d->F % 256) return MOE_ERR_SHAPE;
    return MOE_OK;
}

BwdLayout make_bwd_layout(const moe_dims* d) {
    BwdLayout L{};
    L.f = make_layout(d);
    const size_t T = static_cast<size_t>(d->T), k = d->k, E = d->E, S = d->n_shared;
    const size_t D = d->d, F = d->F;
    const size_t rows = T * k + T * S;
    // every expert's token run is padded to a multiple of 64: at most
    // rows + 63 per group, rounded up
    L.kpad = static_cast<int64_t>((rows + 64 * (E + S) + 63) / 64 * 64);
    const size_t kp = static_cast<size_t>(L.kpad);
    size_t o = L.f.total;
    auto take = [&](size_t bytes) { const size_t at = o; o = align256(o + bytes); return at; };
    L.ids = take(T * k * 4);
    L.gates = take(T * k * 4);
    L.poff = take((E + S + 1) * 4 + kp / 64 * 4);  // + the tile -> group table
    L.a = take(rows * F * 4);
    L.b = take(rows * F * 4);
    L.dg = take(T * k * 4);
    L.dl = take(T * k * 4);
    L.dyq = take(rows * D + rows * D / 32);          // codes, then scale bytes
    L.dh = take(rows * F * 4);
    L.dabq = take(rows * 2 * F + rows * 2 * F / 32);  // codes, then scale bytes
    L.dxp = take(rows * D * 4);
    L.xpt = take(D * kp * 2);
    L.dyt = take(D * kp * 2);
    L.ht = take(F * kp * 2);
    L.dabt = take(2 * F * kp * 2);
    L.total = o;
    return L;
}

BwdWeights make_bwd_weights(const moe_dims* d) {
    BwdWeights W{};
    const size_t G = size_t(d->E) + d->n_shared, FD = size_t(d->F) * d->d;
    size_t o = 0;
    auto take = [&](size_t bytes) { const size_t at = o; o = align256(o + bytes); return at; };
    W.wd = take(G * FD);
    W.wds = take(G * FD / 32);
    W.w2 = take(G * FD * 2);
    W.w2s = take(G * FD * 2 / 32);
    W.total = o;
    return W;
}

// What one call of the training path does.
enum TrainMode {
    TRAIN_BACKWARD = 0,  // moe_backward: routing with the given ids, forward recompute, backward
    TRAIN_FORWARD = 1,   // moe_forward_train: the forward, keeping what the backward reads
    TRAIN_SAVED = 2      // moe_backward_saved: the backward from a moe_forward_train workspace
};

moe_status train_impl(TrainMode mode, const moe_dims* d, const void* x, const moe_weights* w,
                      const void* wt, const int32_t* ids, const void* dout, float* dx,
                      const moe_grads* g, void* out, int32_t* ids_out, float* gates_out, void* ws,
                      size_t ws_bytes, cudaStream_t s) {
    MOE_TRY(bwd_dims_status(d));
    if (!w) return MOE_ERR_ARG;
    const bool fwd = mode != TRAIN_SAVED;   // routing .. down GEMM
    const bool bwd = mode != TRAIN_FORWARD;  // gradients
    if (bwd && !g) return MOE_ERR_ARG;
    if (d->T == 0) return MOE_OK;
    const int64_t T = d->T;
    const int k = d->k, E = d->E, S = d->n_shared, D = d->d, F = d->F;
    if ((fwd && !x) || !w->w_router || !ws) return MOE_ERR_ARG;
    MOE_TRY(check_experts(d, w));
    if (!al16(x) || !al16(w->w_router) || !al16(w->router_bias) || !al16(ws)) return MOE_ERR_ALIGN;
    if (mode == TRAIN_BACKWARD && !ids) return MOE_ERR_ARG;
    if (mode == TRAIN_FORWARD && (!out || !ids_out || !gates_out)) return MOE_ERR_ARG;
    if (!al16(ids) || !al16(out) || !al16(ids_out) || !al16(gates_out)) return MOE_ERR_ALIGN;
    if (bwd) {
        if (!wt || !dout || !dx) return MOE_ERR_ARG;
        if (!g->d_router || !g->d_gate || !g->d_up || !g->d_down) return MOE_ERR_ARG;
        if (S && (!g->ds_gate || !g->ds_up || !g->ds_down)) return MOE_ERR_ARG;
        if (!al16(wt) || !al16(dout) || !al16(dx) || !al16(g->d_router) || !al16(g->d_gate) ||
            !al16(g->d_up) || !al16(g->d_down) || !al16(g->ds_gate) || !al16(g->ds_up) ||
            !al16(g->ds_down))
            return MOE_ERR_ALIGN;
    }
    const BwdLayout L = make_bwd_layout(d);
    if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;
    const BwdWeights WW = make_bwd_weights(d);
    const int sms = num_sms();
    if (sms <= 0) return MOE_ERR_CUDA;
    auto* wsb = static_cast<uint8_t*>(ws);
    auto* wtb = static_cast<const uint8_t*>(wt);
    int32_t* status = reinterpret_cast<int32_t*>(wsb + L.f.status);
    int32_t* cnt = reinterpret_cast<int32_t*>(wsb + L.f.cnt);
    int32_t* off = reinterpret_cast<int32_t*>(wsb + L.f.off);
    int32_t* perm = reinterpret_cast<int32_t*>(wsb + L.f.perm);
    int32_t* inv = reinterpret_cast<int32_t*>(wsb + L.f.inv);
    int32_t* valid = reinterpret_cast<int32_t*>(wsb + L.f.valid);
    int32_t* ids_used = reinterpret_cast<int32_t*>(wsb + L.ids);
    float* gates = reinterpret_cast<float*>(wsb + L.gates);
    int32_t* poff = reinterpret_cast<int32_t*>(wsb + L.poff);
    const int64_t Tk = T * k;
    const int64_t rows = Tk + T * S;
    const int G = E + S;

    // 1. routing (own, or with the given ids: checked, gate weights computed),
    //    dispatch, padded token offsets, gather (with the shared rows)
    if (fwd) {
    MOE_TRY(mark_b(MOE_BWD_STAGE_ROUTE, 0, s));
    MOE_TRY(run_route(d, x, w, ids, ids_used, gates, wsb, L.f, s));
    MOE_TRY(mark_b(MOE_BWD_STAGE_ROUTE, 1, s));
    MOE_TRY(mark_b(MOE_BWD_STAGE_DISPATCH, 0, s));
    MOE_TRY(cu(launch_dispatch(ids_used, T, k, E, cnt, off, perm, inv,
                               reinterpret_cast<int32_t*>(wsb + L.f.scratch), s)));
    MOE_TRY(cu(launch_seg_offsets(cnt, E, G, S ? static_cast<int>(T) : 0, poff, L.kpad / 64, s)));
    MOE_TRY(cu(launch_gather(static_cast<const uint16_t*>(x), inv, T, k, D, S,
                             reinterpret_cast<uint16_t*>(wsb + L.f.xp), s)));
    MOE_TRY(mark_b(MOE_BWD_STAGE_DISPATCH, 1, s));
    }

    const int units = sms / 2;  // CTA pairs
    const uint32_t box_b = BN_EXPERT / 2;
    const uint32_t rg = gemm_rows(GEMM_SWIGLU);
    const int64_t tok_tiles = (Tk + BN_EXPERT - 1) / BN_EXPERT + E;
    const int64_t sh_tiles = S ? (T + BN_EXPERT - 1) / BN_EXPERT : 0;
    auto common = [&](GemmParams& p, int has_shared, int32_t* counter) {
        std::memset(&p, 0, sizeof p);
        p.cnt = cnt;
        p.off = off;
        p.G = E;
        p.has_shared = has_shared;
        p.shared_rows = static_cast<int32_t>(T);
        p.shared_b_off = static_cast<int32_t>(Tk);
        p.partial_b = 1;
        p.status = status;
        p.timeout_ns = kWaitTimeoutNs;
        p.tile_counter = counter;
    };
    auto launch = [&](int mode, const GemmParams& p, int64_t ntiles) {
        const int64_t tb = ntiles * p.MT;
        return cu(launch_pair_gemm(mode, p, static_cast<int>(tb < units ? tb : units), s));
    };
    const uint64_t EF = uint64_t(E) * F, ED = uint64_t(E) * D;

    // 2. the forward's expert GEMMs: gate/up (H, and the fp32 pre-activations),
    //    down (routed Y; the shared rows too when the forward's output is formed)
    if (fwd) {
    {
        GemmParams p;
        common(p, S, status + 4);
        if (!make_map(&p.a0, w->w_gate, D, EF, rg) || !make_map(&p.a1, w->w_up, D, EF, rg))
            return MOE_ERR_CUDA;
        if (S && (!make_map(&p.as0, w->ws_gate, D, F, rg) || !make_map(&p.as1, w->ws_up, D, F, rg)))
            return MOE_ERR_CUDA;
        if (!make_map(&p.b, wsb + L.f.xp, D, rows, box_b) ||
            !make_map(&p.b32, wsb + L.f.xp, D, rows, 32))
            return MOE_ERR_CUDA;
        p.M = F;
        p.MT = (F + 2 * rg - 1) / (2 * rg);
        p.KB = D / BK;
        p.out = wsb + L.f.h;
        p.ldo = F;
        p.save_a = reinterpret_cast<float*>(wsb + L.a);
        p.save_b = reinterpret_cast<float*>(wsb + L.b);
        MOE_TRY(mark_b(MOE_BWD_STAGE_GATE_UP, 0, s));
        MOE_TRY(launch(GEMM_SWIGLU, p, tok_tiles + sh_tiles));
        MOE_TRY(mark_b(MOE_BWD_STAGE_GATE_UP, 1, s));
    }
    {
        const int sh = mode == TRAIN_FORWARD ? S : 0;
        GemmParams p;
        common(p, sh, status + 5);
        if (!make_map(&p.a0, w->w_down, F, ED, BM)) return MOE_ERR_CUDA;
        if (sh && !make_map(&p.as0, w->ws_down, F, D, BM)) return MOE_ERR_CUDA;
        if (!make_map(&p.b, wsb + L.f.h, F, rows, box_b) ||
            !make_map(&p.b32, wsb + L.f.h, F, rows, 32))
            return MOE_ERR_CUDA;
        p.M = D;
        p.MT = (D + 2 * BM - 1) / (2 * BM);
        p.KB = F / BK;
        p.out = wsb + L.f.y;
        p.out_shared = sh ? wsb + L.f.ysh : nullptr;
        p.ldo = D;
        MOE_TRY(mark_b(MOE_BWD_STAGE_DOWN, 0, s));
        MOE_TRY(launch(GEMM_DOWN, p, tok_tiles + (sh ? sh_tiles : 0)));
        MOE_TRY(mark_b(MOE_BWD_STAGE_DOWN, 1, s));
    }
    }
    if (mode == TRAIN_FORWARD) {
        // the layer output (fixed-order combine) and the routing the forward used
        MOE_TRY(mark(MOE_STAGE_COMBINE, 0, s));
        MOE_TRY(cu(launch_combine(reinterpret_cast<const uint16_t*>(wsb + L.f.y),
                                  S ? reinterpret_cast<const float*>(wsb + L.f.ysh) : nullptr, inv,
                                  gates, valid, T, k, D, d->out_fp32, out, s)));
        MOE_TRY(mark(MOE_STAGE_COMBINE, 1, s));
        MOE_TRY(cu(cudaMemcpyAsync(ids_out, ids_used, Tk * sizeof(int32_t),
                                   cudaMemcpyDeviceToDevice, s)));
        return cu(cudaMemcpyAsync(gates_out, gates, Tk * sizeof(float), cudaMemcpyDeviceToDevice,
                                  s));
    }

    // 3. gate and router gradients; dx starts as the router's part.  The tile
    //    counters of the two gradient GEMMs are cleared here (the backward may
    //    run more than once on one training forward's workspace).
    MOE_TRY(cu(cudaMemsetAsync(status + 6, 0, 2 * sizeof(int32_t), s)));
    MOE_TRY(mark_b(MOE_BWD_STAGE_GATE, 0, s));
    MOE_TRY(cu(launch_gate_bwd(static_cast<const uint16_t*>(dout),
                               reinterpret_cast<const uint16_t*>(wsb + L.f.y), inv, ids_used, gates,
                               valid, static_cast<const uint16_t*>(w->w_router),
                               reinterpret_cast<float*>(wsb + L.dg),
                               reinterpret_cast<float*>(wsb + L.dl), dx, T, k, D, sms, s)));
    MOE_TRY(cu(launch_router_wgrad(reinterpret_cast<const uint16_t*>(wsb + L.f.xp), perm, cnt, off,
                                   reinterpret_cast<const float*>(wsb + L.dl), g->d_router, E, D,
                                   sms, s)));
    MOE_TRY(mark_b(MOE_BWD_STAGE_GATE, 1, s));

    // 4. dH = Q_d(dY) Q_d(Wd)  (block-scaled MXFP8 SM-pair GEMM, fp32 rows)
    uint8_t* dyc = wsb + L.dyq;
    uint8_t* dys = dyc + rows * D;
    uint16_t* xpt = reinterpret_cast<uint16_t*>(wsb + L.xpt);
    uint16_t* dyt = reinterpret_cast<uint16_t*>(wsb + L.dyt);
    uint16_t* ht = reinterpret_cast<uint16_t*>(wsb + L.ht);
    uint16_t* dabt = reinterpret_cast<uint16_t*>(wsb + L.dabt);
    const int srows = S ? static_cast<int>(T) : 0;
    MOE_TRY(mark_b(MOE_BWD_STAGE_DY, 0, s));
    const SegDyArgs dya{static_cast<const uint16_t*>(dout), gates, perm, valid, k, Tk, inv, T, S};
    MOE_TRY(cu(launch_dy_dual(dya, D, cnt, off, poff, E, G, srows, L.kpad, dyc, dys, dyt, sms, s)));
    MOE_TRY(mark_b(MOE_BWD_STAGE_DY, 1, s));
    // The dH and dXp GEMMs on the block-scaled MMA: E4M3 codes of the weight
    // copies (groups 0..E-1, the shared expert as group E) and of the token
    // rows, 128-byte K blocks, scale bytes per 32 along K; fp32 rows out.
    const int tn8 = bs_tile_tokens(BS_MXFP8), big8 = bs_big_box(BS_MXFP8);
    const int sbox8 = bs_scale_box(BS_MXFP8), kk8 = 128;
    const uint64_t GF = uint64_t(G) * F, GD = uint64_t(G) * D;
    auto bs_down = [&](GemmParams& p, const uint8_t* wc, const uint8_t* wsc, const uint8_t* bc,
                       const uint8_t* bsc, int K, uint64_t wrows, int M, void* out) -> moe_status {
        std::memset(&p, 0, sizeof p);
        p.cnt = cnt;
        p.off = off;
        p.G = E;
        p.has_shared = S;
        p.shared_rows = static_cast<int32_t>(T);
        p.shared_b_off = static_cast<int32_t>(Tk);
        p.status = status;
        p.timeout_ns = kWaitTimeoutNs;
        if (!make_map_u8(&p.a0, wc, K, wrows, kk8, BM, true) ||
            !make_map_u8(&p.sa0, wsc, K / 32, wrows, sbox8, BM) ||
            !make_map_u8(&p.b, bc, K, rows, kk8, big8, true) ||
            !make_map_u8(&p.b32, bc, K, rows, kk8, 32, true) ||
            !make_map_u8(&p.sb_scale, bsc, K / 32, rows, sbox8, 128))
            return MOE_ERR_CUDA;
        p.M = M;
        p.MT = M / (2 * BM);
        p.KB = K / kk8;
        p.out = out;
        p.out_f32 = 1;
        p.ldo = M;
        p.sc_ahead = rows >= static_cast<int64_t>(G) * tn8 ? 1 : 0;
        const int64_t tb = ((rows + tn8 - 1) / tn8 + G) * p.MT;
        return cu(launch_bs_gemm(BS_MXFP8, GEMM_DOWN, p, static_cast<int>(tb < units ? tb : units), s));
    };
    {
        GemmParams p;
        MOE_TRY(mark_b(MOE_BWD_STAGE_DH, 0, s));
        MOE_TRY(bs_down(p, wtb + WW.wd, wtb + WW.wds, dyc, dys, D, GF, F, wsb + L.dh));
        MOE_TRY(mark_b(MOE_BWD_STAGE_DH, 1, s));
    }

    // 5. SwiGLU backward -> [dA | dB], quantised along F and along tokens
    uint8_t* dabc = wsb + L.dabq;
    uint8_t* dabs = dabc + rows * 2 * F;
    MOE_TRY(mark_b(MOE_BWD_STAGE_SWIGLU, 0, s));
    MOE_TRY(cu(launch_swiglu_dual(reinterpret_cast<const float*>(wsb + L.dh),
                                  reinterpret_cast<const float*>(wsb + L.a),
                                  reinterpret_cast<const float*>(wsb + L.b), F, cnt, off, poff, E, G,
                                  Tk, srows, L.kpad, dabc, dabs, dabt, sms, s)));
    MOE_TRY(mark_b(MOE_BWD_STAGE_SWIGLU, 1, s));

    // 6. dXp = Q_F(dA) Q_F(Wg) + Q_F(dB) Q_F(Wu)  (one K = 2F GEMM), then dx
    {
        GemmParams p;
        MOE_TRY(mark_b(MOE_BWD_STAGE_DXP, 0, s));
        MOE_TRY(bs_down(p, wtb + WW.w2, wtb + WW.w2s, dabc, dabs, 2 * F, GD, D, wsb + L.dxp));
        MOE_TRY(mark_b(MOE_BWD_STAGE_DXP, 1, s));
    }
    MOE_TRY(mark_b(MOE_BWD_STAGE_DX, 0, s));
    MOE_TRY(cu(launch_dx_assemble(reinterpret_cast<const float*>(wsb + L.dxp), inv, dx, T, k, D, S,
                                  sms, s)));
    MOE_TRY(mark_b(MOE_BWD_STAGE_DX, 1, s));

    // 7. token-major Xp and H, quantised along the tokens of each expert
    MOE_TRY(mark_b(MOE_BWD_STAGE_TRANSPOSE, 0, s));
    MOE_TRY(cu(launch_tq_segments(reinterpret_cast<const uint16_t*>(wsb + L.f.xp), D, D, cnt, off,
                                  poff, E, G, Tk, srows, L.kpad, xpt, sms, s)));
    MOE_TRY(cu(launch_tq_segments(reinterpret_cast<const uint16_t*>(wsb + L.f.h), F, F, cnt, off,
                                  poff, E, G, Tk, srows, L.kpad, ht, sms, s)));
    MOE_TRY(mark_b(MOE_BWD_STAGE_TRANSPOSE, 1, s));

    // 8. weight gradients (ragged-K grouped GEMMs)
    const int wm = wgrad_tile_m(), wn = wgrad_tile_n(), wbox = wgrad_box_rows();
    auto wlaunch = [&](WgradParams& p) {
        const int64_t tiles = int64_t(p.G) * p.MT * p.NT;
        return cu(launch_wgrad(p, static_cast<int>(tiles < units ? tiles : units), s));
    };
    {
        WgradParams p;
        std::memset(&p, 0, sizeof p);
        if (!make_map(&p.a, ht, L.kpad, F, wbox) || !make_map(&p.b, dyt, L.kpad, D, wbox))
            return MOE_ERR_CUDA;
        p.poff = poff;
        p.G = G;
        p.G_routed = E;
        p.M = F;
        p.N = D;
        p.MT = F / wm;
        p.NT = D / wn;
        p.n_split = D;
        p.out0 = g->d_down;
        p.sout0 = g->ds_down;
        p.gstride = int64_t(D) * F;
        p.status = status;
        p.timeout_ns = kWaitTimeoutNs;
        MOE_TRY(mark_b(MOE_BWD_STAGE_WGRAD_DOWN, 0, s));
        MOE_TRY(wlaunch(p));
        MOE_TRY(mark_b(MOE_BWD_STAGE_WGRAD_DOWN, 1, s));
    }
    {
        WgradParams p;
        std::memset(&p, 0, sizeof p);
        if (!make_map(&p.a, xpt, L.kpad, D, wbox) || !make_map(&p.b, dabt, L.kpad, 2 * F, wbox))
            return MOE_ERR_CUDA;
        p.poff = poff;
        p.G = G;
        p.G_routed = E;
        p.M = D;
        p.N = 2 * F;
        p.MT = D / wm;
        p.NT = 2 * F / wn;
        p.n_split = F;
        p.out0 = g->d_gate;
        p.out1 = g->d_up;
        p.sout0 = g->ds_gate;
        p.sout1 = g->ds_up;
        p.gstride = int64_t(F) * D;
        p.status = status;
        p.timeout_ns = kWaitTimeoutNs;
        p.stall_test = take_stall_test_bwd() ? 1 : 0;
        MOE_TRY(mark_b(MOE_BWD_STAGE_WGRAD_GATE_UP, 0, s));
        MOE_TRY(wlaunch(p));
        MOE_TRY(mark_b(MOE_BWD_STAGE_WGRAD_GATE_UP, 1, s));
    }
    return MOE_OK;
}

}  // namespace

extern "C" {

size_t moe_workspace_size(const moe_dims* dims) {
    if (!dims_ok(dims)) return 0;
    return make_layout(dims).total;
}

moe_status moe_workspace_layout(const moe_dims* dims, moe_ws_layout* out) {
    if (!dims || !out) return MOE_ERR_ARG;
    if (!dims_ok(dims)) return MOE_ERR_SHAPE;
    const Layout L = make_layout(dims);
    out->status = L.status;
    out->logits = L.logits;
    out->valid = L.valid;
    out->cnt = L.cnt;
    out->off = L.off;
    out->perm = L.perm;
    out->inv = L.inv;
    out->xp = L.xp;
    out->h = L.h;
    out->y = L.y;
    out->ysh = L.ysh;
    out->xq = L.xq;
    out->sx = L.sx;
    out->sxp = L.sxp;
    out->sh = L.sh;
    out->hq = L.hq;
    out->total = L.total;
    return MOE_OK;
}

size_t moe_packed_weights_size(const moe_dims* dims) {
    if (!dims_ok(dims) || dims->wfmt != MOE_W_BF16) return 0;
    return size_t(dims->E + dims->n_shared) * 2 * dims->F * dims->d * 2;
}

moe_status moe_pack_weights(const moe_dims* d, const moe_weights* w, void* packed,
                            size_t packed_bytes, moe_stream_t stream) {
    if (!d || !w) return MOE_ERR_ARG;
    if (!dims_ok(d)) return MOE_ERR_SHAPE;
    if (d->wfmt != MOE_W_BF16) return MOE_ERR_UNSUPPORTED;
    if (!packed || !w->w_gate || !w->w_up || (d->n_shared && (!w->ws_gate || !w->ws_up)))
        return MOE_ERR_ARG;
    if (!al16(packed) || !al16(w->w_gate) || !al16(w->w_up) || !al16(w->ws_gate) ||
        !al16(w->ws_up))
        return MOE_ERR_ALIGN;
    if (packed_bytes < moe_packed_weights_size(d)) return MOE_ERR_WORKSPACE;
    auto* s = reinterpret_cast<cudaStream_t>(stream);
    auto* out = static_cast<uint16_t*>(packed);
    MOE_TRY(cu(launch_pack_gate_up(static_cast<const uint16_t*>(w->w_gate),
                                   static_cast<const uint16_t*>(w->w_up), d->E, d->F, d->d, out, s)));
    if (d->n_shared)
        MOE_TRY(cu(launch_pack_gate_up(static_cast<const uint16_t*>(w->ws_gate),
                                       static_cast<const uint16_t*>(w->ws_up), 1, d->F, d->d,
                                       out + int64_t(d->E) * 2 * d->F * d->d, s)));
    return MOE_OK;
}

moe_status moe_route(const moe_dims* dims, const void* x, const moe_weights* w, int32_t* ids_out,
                     float* gates_out, void* ws, size_t ws_bytes, moe_stream_t stream) {
    MOE_TRY(check_common(dims, x, w, ws, ws_bytes));
    if (dims->T == 0) return MOE_OK;
    if (!ids_out || !gates_out) return MOE_ERR_ARG;
    if (!al16(ids_out) || !al16(gates_out)) return MOE_ERR_ALIGN;
    const Layout L = make_layout(dims);
    return run_route(dims, x, w, nullptr, ids_out, gates_out, static_cast<uint8_t*>(ws), L,
                     reinterpret_cast<cudaStream_t>(stream));
}

moe_status moe_forward(const moe_dims* dims, const void* x, const moe_weights* w, void* out,
                       int32_t* ids_out, float* gates_out, void* ws, size_t ws_bytes,
                       moe_stream_t stream) {
    return forward_impl(dims, x, w, nullptr, false, out, ids_out, gates_out, ws, ws_bytes, stream);
}

moe_status moe_forward_replay(const moe_dims* dims, const void* x, const moe_weights* w,
                              const int32_t* ids_in, void* out, int32_t* ids_out, float* gates_out,
                              void* ws, size_t ws_bytes, moe_stream_t stream) {
    return forward_impl(dims, x, w, ids_in, true, out, ids_out, gates_out, ws, ws_bytes, stream);
}

moe_status moe_forward_replay_filtered(const moe_dims* dims, const void* x, const moe_weights* w,
                                       const int32_t* ids_in, float tau, void* out,
                                       int32_t* ids_out, float* gates_out, void* ws,
                                       size_t ws_bytes, moe_stream_t stream) {
    if (!(tau >= 0.0f && tau <= 1.0f)) return MOE_ERR_ARG;  // also rejects NaN
    return forward_impl(dims, x, w, ids_in, true, out, ids_out, gates_out, ws, ws_bytes, stream,
                        true, tau);
}

moe_status moe_get_status(const void* ws, moe_stream_t stream) {
    if (!ws) return MOE_ERR_ARG;
    auto* s = reinterpret_cast<cudaStream_t>(stream);
    int32_t h[4] = {0, 0, 0, 0};
    if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaMemcpy(h, ws, sizeof h, cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
    if (h[0] & STATUS_TIMEOUT) return MOE_ERR_TIMEOUT;
    if (h[0] & STATUS_BAD_IDS) return MOE_ERR_BAD_IDS;
    return MOE_OK;
}

moe_status moe_set_stage_events(void* const* events) {
    if (!events) {
        g_stage_timing = false;
        return MOE_OK;
    }
    for (int i = 0; i < 2 * MOE_NUM_STAGES; ++i)
        g_stage_events[i] = static_cast<cudaEvent_t>(events[i]);
    g_stage_timing = true;
    return MOE_OK;
}

const char* moe_status_str(moe_status s) {
    switch (s) {
        case MOE_OK: return "MOE_OK";
        case MOE_ERR_ARG: return "MOE_ERR_ARG: null pointer or invalid enum value";
        case MOE_ERR_SHAPE: return "MOE_ERR_SHAPE: dimension outside the supported limits";
        case MOE_ERR_ALIGN: return "MOE_ERR_ALIGN: pointer not 16-byte aligned";
        case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE: workspace smaller than moe_workspace_size";
        case MOE_ERR_BAD_IDS: return "MOE_ERR_BAD_IDS: replayed expert id out of range or repeated";
        case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT: a bounded device wait ran out";
        case MOE_ERR_CUDA: return "MOE_ERR_CUDA: a CUDA call failed";
        case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED: not supported by this build";
    }
    return "unknown moe_status";
}

size_t moe_backward_weights_size(const moe_dims* dims) {
    if (bwd_dims_status(dims) != MOE_OK) return 0;
    return make_bwd_weights(dims).total;
}

moe_status moe_backward_prepare_weights(const moe_dims* d, const moe_weights* w, void* wt,
                                        size_t wt_bytes, moe_stream_t stream) {
    MOE_TRY(bwd_dims_status(d));
    if (!w || !wt) return MOE_ERR_ARG;
    MOE_TRY(check_experts(d, w));
    if (!al16(wt)) return MOE_ERR_ALIGN;
    const BwdWeights W = make_bwd_weights(d);
    if (wt_bytes < W.total) return MOE_ERR_WORKSPACE;
    const int sms = num_sms();
    if (sms <= 0) return MOE_ERR_CUDA;
    auto* s = reinterpret_cast<cudaStream_t>(stream);
    auto* o = static_cast<uint8_t*>(wt);
    const int E = d->E, D = d->d, F = d->F;
    const int64_t FD = int64_t(F) * D;
    uint8_t* wd = o + W.wd;
    uint8_t* wds = o + W.wds;
    uint8_t* w2 = o + W.w2;
    uint8_t* w2s = o + W.w2s;
    // Wd [d][F] -> [F][d] quantised along d; Wg, Wu [F][d] -> [d][2F] quantised
    // along F; codes, and scale bytes at the code offset / 32; the shared
    // expert is group E
    auto q = [&](const void* src, int nb, int R, int C, int64_t g0, int64_t per, int64_t ld,
                 int64_t col0, uint8_t* codes, uint8_t* scales) {
        return cu(launch_tq_batch(static_cast<const uint16_t*>(src), nb, R, C, codes + g0 * per,
                                  scales + g0 * per / 32, per, ld, col0, sms, s));
    };
    MOE_TRY(mark_b(MOE_BWD_STAGE_PREPARE, 0, s));
    MOE_TRY(q(w->w_down, E, D, F, 0, FD, D, 0, wd, wds));
    MOE_TRY(q(w->w_gate, E, F, D, 0, 2 * FD, 2 * F, 0, w2, w2s));
    MOE_TRY(q(w->w_up, E, F, D, 0, 2 * FD, 2 * F, F, w2, w2s));
    if (d->n_shared) {
        MOE_TRY(q(w->ws_down, 1, D, F, E, FD, D, 0, wd, wds));
        MOE_TRY(q(w->ws_gate, 1, F, D, E, 2 * FD, 2 * F, 0, w2, w2s));
        MOE_TRY(q(w->ws_up, 1, F, D, E, 2 * FD, 2 * F, F, w2, w2s));
    }
    return mark_b(MOE_BWD_STAGE_PREPARE, 1, s);
}

moe_status moe_set_backward_stage_events(void* const* events) {
    if (!events) {
        g_bwd_timing = false;
        return MOE_OK;
    }
    for (int i = 0; i < 2 * MOE_BWD_NUM_STAGES; ++i)
        g_bwd_events[i] = static_cast<cudaEvent_t>(events[i]);
    g_bwd_timing = true;
    return MOE_OK;
}

size_t moe_backward_workspace_size(const moe_dims* dims) {
    if (bwd_dims_status(dims) != MOE_OK) return 0;
    return make_bwd_layout(dims).total;
}

moe_status moe_backward_workspace_layout(const moe_dims* dims, moe_bwd_ws_layout* out) {
    if (!out) return MOE_ERR_ARG;
    MOE_TRY(bwd_dims_status(dims));
    const BwdLayout L = make_bwd_layout(dims);
    out->status = L.f.status;
    out->logits = L.f.logits;
    out->valid = L.f.valid;
    out->cnt = L.f.cnt;
    out->off = L.f.off;
    out->perm = L.f.perm;
    out->inv = L.f.inv;
    out->xp = L.f.xp;
    out->h = L.f.h;
    out->y = L.f.y;
    out->ids = L.ids;
    out->gates = L.gates;
    out->poff = L.poff;
    out->a = L.a;
    out->b = L.b;
    out->dg = L.dg;
    out->dl = L.dl;
    out->dyq = L.dyq;
    out->dh = L.dh;
    out->dabq = L.dabq;
    out->dxp = L.dxp;
    out->xpt = L.xpt;
    out->dyt = L.dyt;
    out->ht = L.ht;
    out->dabt = L.dabt;
    out->kpad = static_cast<size_t>(L.kpad);
    out->total = L.total;
    return MOE_OK;
}

moe_status moe_backward(const moe_dims* dims, const void* x, const moe_weights* w, const void* wt,
                        const int32_t* ids, const void* dout, float* dx, const moe_grads* grads,
                        void* ws, size_t ws_bytes, moe_stream_t stream) {
    return train_impl(TRAIN_BACKWARD, dims, x, w, wt, ids, dout, dx, grads, nullptr, nullptr,
                      nullptr, ws, ws_bytes, reinterpret_cast<cudaStream_t>(stream));
}

moe_status moe_forward_train(const moe_dims* dims, const void* x, const moe_weights* w,
                             const int32_t* ids_in, void* out, int32_t* ids_out, float* gates_out,
                             void* ws, size_t ws_bytes, moe_stream_t stream) {
    return train_impl(TRAIN_FORWARD, dims, x, w, nullptr, ids_in, nullptr, nullptr, nullptr, out,
                      ids_out, gates_out, ws, ws_bytes, reinterpret_cast<cudaStream_t>(stream));
}

moe_status moe_backward_saved(const moe_dims* dims, const moe_weights* w, const void* wt,
                              const void* dout, float* dx, const moe_grads* grads, void* ws,
                              size_t ws_bytes, moe_stream_t stream) {
    return train_impl(TRAIN_SAVED, dims, nullptr, w, wt, nullptr, dout, dx, grads, nullptr,
                      nullptr, nullptr, ws, ws_bytes, reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"
