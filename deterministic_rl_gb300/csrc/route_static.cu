// route_static.cu -- moe_route_static: the routing call (router GEMM, top-k,
// gate weights) with its scratch memory in a static device array instead of a
// caller-provided workspace, for callers that cannot allocate device memory.
//
// The scratch (status word, per-token flags, fp32 logits) lives in
// g_route_scratch below: kStaticScratchBytes bytes that every GPU which loads
// this library keeps until the process exits.  In host code the array's name
// is only a host-side stand-in, so its device address is looked up with
// cudaGetSymbolAddress once per device (the first call on that device, with
// that device current) and passed to the kernels.  All calls share the array:
// calls that overlap on the GPU (different streams, or different host
// threads on one device) race on it.
#include <cudaTypedefs.h>

#include <cstdint>
#include <cstring>
#include <mutex>

#include "moe_det.h"
#include "moe_internal.h"

using namespace moe;

namespace {

constexpr size_t kStaticScratchBytes = size_t(4) << 20;  // 4 MiB
constexpr int kMaxDevices = 64;
constexpr uint64_t kTimeoutNs = 1000000000ull;

static __device__ __align__(256) unsigned char g_route_scratch[kStaticScratchBytes];

std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

inline size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

// Device address of the static scratch on the current device (looked up once).
moe_status scratch_address(unsigned char** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_route_scratch) != cudaSuccess || !p) return MOE_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *out = static_cast<unsigned char*>(g_scratch_addr[dev]);
    return MOE_OK;
}

bool encode_map(CUtensorMap* m, const void* base, uint64_t K, uint64_t rows, uint32_t box_rows) {
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
    if (!fn) return false;
    const cuuint64_t dims[2] = {K, rows};
    const cuuint64_t strides[1] = {K * 2};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(BK), box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace

extern "C" moe_status moe_route_static(const moe_dims* dims, const void* x, const moe_weights* w,
                                       int32_t* ids_out, float* gates_out, moe_stream_t stream) {
    if (!dims || !w) return MOE_ERR_ARG;
    if (dims->T < 0 || dims->k != 8 || dims->E < 8 || dims->E > 512 || dims->d < 64 ||
        dims->d > 16384 || dims->d % 64)
        return MOE_ERR_SHAPE;
    if (dims->T == 0) return MOE_OK;
    if (!x || !w->w_router || !ids_out || !gates_out) return MOE_ERR_ARG;
    if (!aligned16(x) || !aligned16(w->w_router) || !aligned16(w->router_bias) ||
        !aligned16(ids_out) || !aligned16(gates_out))
        return MOE_ERR_ALIGN;
    const size_t T = static_cast<size_t>(dims->T), E = static_cast<size_t>(dims->E);
    const size_t off_valid = 256, off_logits = off_valid + round256(T * 4);
    if (T > (size_t(1) << 20) || off_logits + T * E * 4 > kStaticScratchBytes) return MOE_ERR_WORKSPACE;

    unsigned char* scratch = nullptr;
    const moe_status st = scratch_address(&scratch);
    if (st != MOE_OK) return st;
    auto s = reinterpret_cast<cudaStream_t>(stream);
    int32_t* status = reinterpret_cast<int32_t*>(scratch);
    if (cudaMemsetAsync(status, 0, 16, s) != cudaSuccess) return MOE_ERR_CUDA;

    GemmParams p;
    std::memset(&p, 0, sizeof p);
    if (!encode_map(&p.a0, w->w_router, dims->d, E, BM)) return MOE_ERR_CUDA;
    if (!encode_map(&p.b, x, dims->d, T, BN)) return MOE_ERR_CUDA;
    p.G = 1;
    p.n_single = static_cast<int32_t>(T);
    p.M = dims->E;
    p.MT = (dims->E + BM - 1) / BM;
    p.KB = dims->d / BK;
    p.out = scratch + off_logits;
    p.ldo = dims->E;
    p.bias = w->router_bias;
    p.status = status;
    p.timeout_ns = kTimeoutNs;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
        return MOE_ERR_CUDA;
    const int64_t tiles = int64_t(p.MT) * ((dims->T + BN - 1) / BN);
    if (launch_grouped_gemm(GEMM_ROUTER, p, static_cast<int>(tiles < sms ? tiles : sms), s) !=
        cudaSuccess)
        return MOE_ERR_CUDA;
    if (launch_topk_gates(reinterpret_cast<const float*>(scratch + off_logits), dims->T, dims->E,
                          dims->k, nullptr, ids_out, gates_out,
                          reinterpret_cast<int32_t*>(scratch + off_valid), status, s) != cudaSuccess)
        return MOE_ERR_CUDA;
    return MOE_OK;
}
