// Router: one warp per token (route.cuh).
#include "common.cuh"
#include "internal.h"
#include "route.cuh"

namespace ftmoe {

template <int EPL>
__global__ void __launch_bounds__(256) route_kernel(const float* __restrict__ logits, int T, int E,
                                                    int k, int32_t* __restrict__ ids,
                                                    float* __restrict__ w, int* status) {
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= T) return;
  route_token<EPL>(logits + (size_t)t * E, E, k, ids + (size_t)t * k, w + (size_t)t * k, status);
}

cudaError_t launch_route(const float* logits, int T, int E, int k, int32_t* ids, float* w,
                         cudaStream_t st) {
  const DeviceInfo* di = device_info();
  if (!di) return cudaErrorUnknown;
  const dim3 grid((T + 7) / 8), block(256);
  with_epl(E, [&]<int N>() { route_kernel<N><<<grid, block, 0, st>>>(logits, T, E, k, ids, w, di->status); });
  return cudaGetLastError();
}

}  // namespace ftmoe
