// Internal launcher declarations shared by the C-ABI layer and the kernel files.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "ftmoe.h"

namespace ftmoe {

// Per-device facts the launchers need (queried once per device).
struct DeviceInfo {
  int sm_count = 0;
  int* status = nullptr;  // device address of this device's status word
};
const DeviceInfo* device_info();  // for the current device; nullptr on failure

// Raises kernel K's dynamic shared-memory limit on the current device the first time it
// is needed; later calls with no larger size return at once (no driver call, so the
// launch paths stay cheap and can be recorded into CUDA graphs).
template <auto K>
cudaError_t set_smem_limit(size_t bytes) {
  static int done[64] = {0};  // bytes granted so far, per device
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (__atomic_load_n(&done[dev], __ATOMIC_ACQUIRE) >= (int)bytes) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(K, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e == cudaSuccess) __atomic_store_n(&done[dev], (int)bytes, __ATOMIC_RELEASE);
  return e;
}

cudaError_t launch_repack(int qtype, const void* canon, void* tiles, int E, int N, int K,
                          cudaStream_t st);
cudaError_t launch_dequant(int qtype, const void* tiles, int E, int N, int K, float* out,
                           cudaStream_t st);
cudaError_t launch_operand(int qtype, int which, const void* tiles, int E, int N, int K,
                           uint16_t* out, cudaStream_t st);

cudaError_t launch_route(const float* logits, int T, int E, int k, int32_t* ids, float* w,
                         cudaStream_t st);

size_t permute_ws_bytes(int T, int k, int E);
// Also zeroes zero_bytes (a multiple of 4) at zero_ptr when zero_ptr is not null.
cudaError_t launch_permute(const int32_t* ids, int T, int k, int E, int32_t* offsets,
                           int32_t* sorted_pair, int32_t* inv_pos, void* ws, int* status,
                           void* zero_ptr, size_t zero_bytes, cudaStream_t st);

// Routing and permutation of a small batch in one launch (T <= ROUTE_PERMUTE_MAX_T);
// cudaErrorNotSupported beyond that.
constexpr int ROUTE_PERMUTE_MAX_T = 64;
bool route_permute_fits(int T, int k);
cudaError_t launch_route_permute(const float* logits, int T, int E, int k, int32_t* ids, float* w,
                                 int32_t* offsets, int32_t* sorted_pair, int32_t* inv_pos, int* status,
                                 void* zero_ptr, size_t zero_bytes, cudaStream_t st);

cudaError_t launch_combine(const uint16_t* y_perm, const float* w, const int32_t* inv_pos,
                           const uint16_t* shared_y, int T, int k, int H, uint16_t* out,
                           cudaStream_t st);

// Weights of one projection for the FFN kernels: expert e's tiles start at
// base + e * stride, or at table[e] + table_offset when a table is used.
constexpr int MAX_TABLE_EXPERTS = 256;
struct ExpertTable {
  const uint8_t* p[MAX_TABLE_EXPERTS];
};

struct FfnProblem {
  int qtype, E, H, I, T, k;
  const uint16_t* x;          // bf16 [T][H]
  const int32_t* offsets;     // [E+1]
  const int32_t* sorted_pair; // [P] or nullptr (identity, k == 1)
  uint16_t* h_act;            // bf16 [P][I] scratch
  uint16_t* y_perm;           // bf16 [P][H] out
  const uint8_t* w13;         // tiles base (or nullptr with table)
  const uint8_t* w2;
  const ExpertTable* table;   // host table or nullptr
  size_t w13_bytes;           // bytes of one expert's w13 tiles (blob offset of w2)
  int P;                      // T * k
};

// ws: ffn_gemv_ws_bytes of scratch whose first ffn_gemv_zero_bytes must be zero on entry;
// ws_zeroed tells that the caller already cleared them (otherwise a kernel does).
cudaError_t launch_ffn_gemv(const FfnProblem& pb, void* ws, bool ws_zeroed, cudaStream_t st);
size_t ffn_gemv_ws_bytes(int T, int k, int E, int H, int I);
size_t ffn_gemv_zero_bytes(int T, int k, int E, int H, int I);
// Grouped GEMM on tcgen05; returns cudaErrorNotSupported when the shape is outside
// what the kernel handles (callers then use the GEMV path).
cudaError_t launch_ffn_gemm(const FfnProblem& pb, void* ws, size_t ws_bytes, cudaStream_t st);
// Grouped GEMM on tcgen05 with 32-token tiles and the decoded weights in tensor memory,
// for few rows per expert (decode); cudaErrorNotSupported outside its shapes.
cudaError_t launch_ffn_gemm_decode(const FfnProblem& pb, cudaStream_t st);
size_t ffn_gemm_ws_bytes(int T, int k, int E, int H, int I);

}  // namespace ftmoe
