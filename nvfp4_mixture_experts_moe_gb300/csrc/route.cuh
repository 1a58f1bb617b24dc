// Warp-level router top-k shared by the routing kernels: "Serving Solar Open
// 2 on DGX Spark", "Solar Open 2 in brief" (top-k over the routed experts);
// "vLLM on the NVIDIA DGX Spark: A Complete Technical Guide", section 7.1
// ([Router] stage).
#pragma once

#include "common.cuh"

namespace moe {

// ---------------------------------------------------------------------------
// One warp per token. Lane l holds logits l, l+32, l+64, ... in registers.
// k rounds of a warp-wide argmax pick the experts by rank: a larger logit
// wins, equal logits go to the lower expert index. The weights are
// exp(l_j - l_max) / sum over the chosen j (fp32), i.e. the softmax
// probabilities renormalised over the top k.
template <int PER_LANE>
__device__ __forceinline__ void route_token(const float* __restrict__ logits, int token, int E, int k,
                                            int32_t* __restrict__ ids, float* __restrict__ w,
                                            int32_t* sids = nullptr, float* sw = nullptr) {
  const int lane = threadIdx.x & 31;
  const float* row = logits + (size_t)token * E;
  float v[PER_LANE];
  uint32_t taken = 0;
#pragma unroll
  for (int i = 0; i < PER_LANE; ++i) {
    const int e = lane + 32 * i;
    v[i] = e < E ? __ldg(row + e) : 0.0f;
    if (e >= E) taken |= 1u << i;
  }
  float my_val = 0.0f;
  int my_id = 0;
  for (int j = 0; j < k; ++j) {
    float bv = 0.0f;
    int bi = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < PER_LANE; ++i) {
      if (!(taken & (1u << i))) {
        // ascending index within a lane: strict '>' keeps the lower index on ties
        if (bi == 0x7fffffff || v[i] > bv) {
          bv = v[i];
          bi = lane + 32 * i;
        }
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
      const bool other_valid = oi != 0x7fffffff;
      const bool mine_valid = bi != 0x7fffffff;
      if (other_valid && (!mine_valid || ov > bv || (ov == bv && oi < bi))) {
        bv = ov;
        bi = oi;
      }
    }
    if (bi == 0x7fffffff) bi = 0;  // only reachable with NaN logits (outside the contract)
    if ((bi & 31) == lane && bi < E) taken |= 1u << (bi >> 5);
    if (lane == j) {
      my_val = bv;
      my_id = bi;
    }
  }
  const float vmax = __shfl_sync(0xffffffffu, my_val, 0);
  float ex = lane < k ? expf(my_val - vmax) : 0.0f;
  float sum = ex;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
  if (lane < k) {
    if (ids != nullptr) {
      ids[(size_t)token * k + lane] = my_id;
      w[(size_t)token * k + lane] = ex / sum;
    }
    if (sids != nullptr) {  // shared-memory copies for the fused kernels
      sids[token * k + lane] = my_id;
      sw[token * k + lane] = ex / sum;
    }
  }
}

}  // namespace moe
