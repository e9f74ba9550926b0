// Router: top-k of each token's logits and the renormalised softmax weights of the
// selection.  Sparse expert activation per token is what the FreeToken pages build
// their MoE engine around ("为什么 MoE 模型适合做 CPU–GPU 协同"); the exact rule
// is: descending logit, ties to the lower id, w_j = exp(l_j - l_max) / sum_sel.
#include <climits>

#include "common.cuh"
#include "internal.h"

namespace ftmoe {

// One warp per token; lane L holds experts L, L + 32, ... (EPL of them).
template <int EPL>
__global__ void __launch_bounds__(256) route_kernel(const float* __restrict__ logits, int T, int E,
                                                    int k, int32_t* __restrict__ ids,
                                                    float* __restrict__ w, int* status) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= T) return;
  const float* row = logits + (size_t)t * E;
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
    ids[(size_t)t * k + lane] = my_id;
    w[(size_t)t * k + lane] = ex / sum;
  }
}

cudaError_t launch_route(const float* logits, int T, int E, int k, int32_t* ids, float* w,
                         cudaStream_t st) {
  const DeviceInfo* di = device_info();
  if (!di) return cudaErrorUnknown;
  const dim3 grid((T + 7) / 8), block(256);
  const int epl = (E + 31) / 32;
#define FTMOE_ROUTE(N) route_kernel<N><<<grid, block, 0, st>>>(logits, T, E, k, ids, w, di->status)
  if (epl <= 1) FTMOE_ROUTE(1);
  else if (epl <= 2) FTMOE_ROUTE(2);
  else if (epl <= 4) FTMOE_ROUTE(4);
  else if (epl <= 8) FTMOE_ROUTE(8);
  else if (epl <= 16) FTMOE_ROUTE(16);
  else FTMOE_ROUTE(32);
#undef FTMOE_ROUTE
  return cudaGetLastError();
}

}  // namespace ftmoe
