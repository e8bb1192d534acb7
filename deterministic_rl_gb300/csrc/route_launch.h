// route_launch.h -- the routing launch sequence (router GEMM with its fixed K
// split, then top-k / replay and gate weights) on scratch memory the caller
// names by pointer.  moe_route, the forward calls and moe_route_static all
// run this one sequence, so they produce the same logits, ids and gate
// weights bit for bit.  Not part of the public interface.
#pragma once
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "moe_det.h"

namespace moe {

// Fixed parts the router GEMM splits K into for these dims (1 = no split).
// It depends on d only, never on T.
int route_split(const moe_dims* d);

// Scratch of one routing launch: status words (32 bytes, zeroed here, also
// holding the expert GEMMs' tile counters in the forward's workspace), fp32
// logits [T][E], route_split(d) partial logits [T][E] each when the split is
// on (else unused), per-token valid flags [T].  All device pointers.
struct RouteScratch {
    int32_t* status;
    float* logits;
    float* parts;
    int32_t* valid;
};

// Enqueue the routing of x [T][d] on stream s.  ids_in null: own selection;
// otherwise replay of ids_in (validated), with the plausibility filter of
// threshold tau when filter is set.
moe_status launch_route(const moe_dims* d, const void* x, const moe_weights* w,
                        const int32_t* ids_in, int32_t* ids_out, float* gates_out,
                        const RouteScratch& sc, cudaStream_t s, bool filter = false,
                        float tau = 0.0f);

}  // namespace moe
