// The router GEMM's launcher with error reporting (the plain launcher,
// launch_router_gemm, is declared with the other kernels).
#pragma once

#include "common.cuh"

namespace moe {

// As launch_router_gemm. A bounded wait of the tensor-core kernel that gives
// up writes NaN logits for its tile and MOE_ERR_TIMEOUT into *status (when
// status is not null).
moe_status launch_router_gemm_status(const uint16_t* x, const uint16_t* w, int T, int H, int E, float* logits,
                                     cudaStream_t s, bool pdl, int* status);

}  // namespace moe
