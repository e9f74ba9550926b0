// Router step shared by the routing kernels: top-k of one token's logits and the
// renormalised softmax weights of the selection (descending logit, ties to the lower id,
// w_j = exp(l_j - l_max) / sum over the selection).  Sparse expert activation per token is
// what the FreeToken pages build their MoE engine around ("为什么 MoE 模型适合做 CPU–GPU
// 协同").
#pragma once

#include <climits>

#include "common.cuh"

namespace ftmoe {

// One warp routes token row `row` (E logits); lane L holds experts L, L + 32, ... (EPL of
// them).  Writes ids[0..k) and w[0..k).
template <int EPL>
__device__ __forceinline__ void route_token(const float* __restrict__ row, int E, int k,
                                            int32_t* __restrict__ ids, float* __restrict__ w,
                                            int* status) {
  const int lane = threadIdx.x & 31;
  float v[EPL];
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int e = lane + 32 * i;
    v[i] = e < E ? row[e] : -INFINITY;
  }
  uint32_t taken = 0;
  float my_val = 0.f;
  int my_id = 0;
  for (int j = 0; j < k; ++j) {
    float bv = -INFINITY;
    int be = INT_MAX;
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      const int e = lane + 32 * i;
      if (e < E && !((taken >> i) & 1u)) {
        if (v[i] > bv || (v[i] == bv && e < be)) { bv = v[i]; be = e; }
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
      const int oe = __shfl_xor_sync(0xffffffffu, be, off);
      if (ov > bv || (ov == bv && oe < be)) { bv = ov; be = oe; }
    }
    if (be == INT_MAX) {  // only NaN logits left
      if (lane == 0) set_device_code(status, DEV_BAD_SHAPE);
      be = 0;
    }
    if ((be & 31) == lane) taken |= 1u << (be >> 5);
    if (lane == j) { my_val = bv; my_id = be; }
  }
  const float lmax = __shfl_sync(0xffffffffu, my_val, 0);
  const float ex = lane < k ? expf(my_val - lmax) : 0.f;
  float sum = ex;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
  if (lane < k) {
    ids[lane] = my_id;
    w[lane] = ex / sum;
  }
}

// Calls F.template operator()<EPL>() with EPL = the lanes' experts per lane for E experts.
template <class F>
__host__ __forceinline__ void with_epl(int E, F&& f) {
  const int epl = (E + 31) / 32;
  if (epl <= 1) f.template operator()<1>();
  else if (epl <= 2) f.template operator()<2>();
  else if (epl <= 4) f.template operator()<4>();
  else if (epl <= 8) f.template operator()<8>();
  else if (epl <= 16) f.template operator()<16>();
  else f.template operator()<32>();
}

}  // namespace ftmoe
