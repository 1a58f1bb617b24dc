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
// wins, equal logits go to the lower expert index (-0 and +0 are equal).
// Each round takes every lane's best untaken logit, reduces the warp's
// maximum of an order-preserving integer image of the values, then the
// smallest index among the lanes holding that maximum. The weights are
// exp(l_j - l_max) / sum over the chosen j (fp32), i.e. the softmax
// probabilities renormalised over the top k.
__device__ __forceinline__ uint32_t order_key(float v) {
  const uint32_t u = __float_as_uint(v == 0.0f ? 0.0f : v);   // -0 -> +0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float key_value(uint32_t key) {
  return __uint_as_float((key & 0x80000000u) ? (key & 0x7fffffffu) : ~key);
}

template <int PER_LANE>
__device__ __forceinline__ void route_token(const float* __restrict__ logits, int token, int E, int k,
                                            int32_t* __restrict__ ids, float* __restrict__ w,
                                            int32_t* sids = nullptr, float* sw = nullptr) {
  const int lane = threadIdx.x & 31;
  const float* row = logits + (size_t)token * E;
  uint32_t key[PER_LANE];
  uint32_t taken = 0;
#pragma unroll
  for (int i = 0; i < PER_LANE; ++i) {
    const int e = lane + 32 * i;
    key[i] = e < E ? order_key(__ldg(row + e)) : 0u;
    if (e >= E) taken |= 1u << i;
  }
  float my_val = 0.0f;
  int my_id = 0;
  for (int j = 0; j < k; ++j) {
    uint32_t bk = 0;
    int bi = -1;
#pragma unroll
    for (int i = 0; i < PER_LANE; ++i) {
      // ascending index within a lane: strict '>' keeps the lower index on ties
      if (!(taken & (1u << i)) && (bi < 0 || key[i] > bk)) {
        bk = key[i];
        bi = lane + 32 * i;
      }
    }
    const uint32_t kmax = __reduce_max_sync(0xffffffffu, bi >= 0 ? bk : 0u);
    const uint32_t cand = (bi >= 0 && bk == kmax) ? (uint32_t)bi : 0xffffffffu;
    uint32_t win = __reduce_min_sync(0xffffffffu, cand);
    if (win >= (uint32_t)E) win = 0;  // only reachable when no lane has an untaken logit (k > E)
    if ((int)(win & 31) == lane) taken |= 1u << (win >> 5);
    if (lane == j) {
      my_val = key_value(kmax);
      my_id = (int)win;
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
