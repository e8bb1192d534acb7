// route_static.cu -- moe_route_static: the routing call (router GEMM, top-k,
// gate weights) with its scratch memory in a static device array instead of a
// caller-provided workspace, for callers that cannot allocate device memory.
// It runs the very launch sequence moe_route runs (launch_route: the same
// router GEMM with the same fixed K split, the same top-k and gate kernels),
// so its ids and gate weights equal moe_route's bit for bit.
//
// The scratch (status word, per-token flags, fp32 logits and the router's
// partial logits) lives in g_route_scratch below: kStaticScratchBytes bytes
// that every GPU which loads this library keeps until the process exits.
// In host code the array's name
// is only a host-side stand-in, so its device address is looked up with
// cudaGetSymbolAddress once per device (the first call on that device, with
// that device current) and passed to the kernels.  All calls share the array:
// calls that overlap on the GPU (different streams, or different host
// threads on one device) race on it.
#include <cstdint>
#include <cstring>
#include <mutex>

#include "moe_det.h"
#include "moe_internal.h"
#include "route_launch.h"

using namespace moe;

namespace {

constexpr size_t kStaticScratchBytes = size_t(4) << 20;  // 4 MiB
constexpr int kMaxDevices = 64;

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
    const size_t nparts = route_split(dims) > 1 ? static_cast<size_t>(route_split(dims)) : 0;
    const size_t off_valid = 256, off_logits = off_valid + round256(T * 4);
    const size_t off_parts = off_logits + round256(T * E * 4);
    if (T > (size_t(1) << 20) || off_parts + nparts * T * E * 4 > kStaticScratchBytes)
        return MOE_ERR_WORKSPACE;

    unsigned char* scratch = nullptr;
    const moe_status st = scratch_address(&scratch);
    if (st != MOE_OK) return st;
    const RouteScratch sc{reinterpret_cast<int32_t*>(scratch),
                          reinterpret_cast<float*>(scratch + off_logits),
                          reinterpret_cast<float*>(scratch + off_parts),
                          reinterpret_cast<int32_t*>(scratch + off_valid)};
    return launch_route(dims, x, w, nullptr, ids_out, gates_out, sc,
                        reinterpret_cast<cudaStream_t>(stream));
}
