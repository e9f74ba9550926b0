// Weighted combine back to token order:
//   out[t] = sum_{j ascending} w[t][j] * y_perm[inv_pos[t*k + j]]  (+ shared_y[t])
// fp32 accumulation, bf16 store.  One thread per 8 outputs (16-byte loads/stores).
#include "common.cuh"
#include "internal.h"

namespace ftmoe {

constexpr int COMBINE_THREADS = 128;

__global__ void __launch_bounds__(COMBINE_THREADS) combine_kernel(
    const uint16_t* __restrict__ y_perm, const float* __restrict__ w,
    const int32_t* __restrict__ inv_pos, const uint16_t* __restrict__ shared_y, int T, int k, int H,
    uint16_t* __restrict__ out, int* status) {
  const int t = blockIdx.x;
  const int col = (blockIdx.y * COMBINE_THREADS + threadIdx.x) * 8;
  if (col >= H) return;
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.f;
  for (int j = 0; j < k; ++j) {
    const int r = inv_pos[(size_t)t * k + j];
    if (r < 0) continue;
#if FTMOE_CHECKS
    if (r >= T * k) {
      set_device_code(status, DEV_BAD_INDEX);
      continue;
    }
#endif
    const float wj = w[(size_t)t * k + j];
    const uint4 v = *reinterpret_cast<const uint4*>(y_perm + (size_t)r * H + col);
    const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      acc[2 * i] = fmaf(wj, bf16_bits_to_f32(u[i] & 0xFFFFu), acc[2 * i]);
      acc[2 * i + 1] = fmaf(wj, bf16_bits_to_f32(u[i] >> 16), acc[2 * i + 1]);
    }
  }
  if (shared_y) {
    const uint4 v = *reinterpret_cast<const uint4*>(shared_y + (size_t)t * H + col);
    const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      acc[2 * i] += bf16_bits_to_f32(u[i] & 0xFFFFu);
      acc[2 * i + 1] += bf16_bits_to_f32(u[i] >> 16);
    }
  }
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
    o[i] = (uint32_t)f32_to_bf16_bits(acc[2 * i]) | ((uint32_t)f32_to_bf16_bits(acc[2 * i + 1]) << 16);
  *reinterpret_cast<uint4*>(out + (size_t)t * H + col) = make_uint4(o[0], o[1], o[2], o[3]);
}

cudaError_t launch_combine(const uint16_t* y_perm, const float* w, const int32_t* inv_pos,
                           const uint16_t* shared_y, int T, int k, int H, uint16_t* out,
                           cudaStream_t st) {
  const dim3 grid(T, (H / 8 + COMBINE_THREADS - 1) / COMBINE_THREADS);
  const DeviceInfo* di = device_info();
  combine_kernel<<<grid, COMBINE_THREADS, 0, st>>>(y_perm, w, inv_pos, shared_y, T, k, H, out,
                                                    di ? di->status : nullptr);
  return cudaGetLastError();
}

}  // namespace ftmoe
