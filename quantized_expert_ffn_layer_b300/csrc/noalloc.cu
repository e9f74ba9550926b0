// ftmoe_permute_noalloc: the permutation entry point for callers that cannot hand
// the library any scratch memory.
//
// Some callers cannot call cudaMalloc and have no workspace to pass: a host program
// that owns every byte of device memory through its own fixed pool and forbids side
// allocations, or a plugin interface that offers no workspace hook.  For them the
// scratch of the multi-CTA permutation (one int32 per chunk of 1024 pairs and per
// expert) lives in a fixed array compiled into this library.  Every device that
// loads the library holds that array until the process exits.
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace ftmoe {
namespace {

// Largest scratch the entry point can use: ceil(T * k / 1024) * E int32 entries.
constexpr size_t NOALLOC_PERMUTE_MAX_INTS = 262144;  // 1 MiB

// The fixed scratch.  In host code this name is only a host-side stand-in for the
// device array, never a device address: launches get the address that
// cudaGetSymbolAddress returns for the current device.
static __device__ __align__(256) int32_t g_permute_scratch[NOALLOC_PERMUTE_MAX_INTS];

constexpr int MAX_DEVICES_NOALLOC = 64;
std::once_flag g_scratch_once[MAX_DEVICES_NOALLOC];
void* g_scratch_ptr[MAX_DEVICES_NOALLOC];
cudaError_t g_scratch_err[MAX_DEVICES_NOALLOC];

// Runs once per device, with that device current.
void resolve_scratch(int dev) {
  void* p = nullptr;
  g_scratch_err[dev] = cudaGetSymbolAddress(&p, g_permute_scratch);
  g_scratch_ptr[dev] = g_scratch_err[dev] == cudaSuccess ? p : nullptr;
}

}  // namespace
}  // namespace ftmoe

using namespace ftmoe;

extern "C" {

ftmoe_status ftmoe_permute_noalloc(const int32_t* ids, int T, int k, int E, int32_t* offsets,
                                   int32_t* sorted_pair, int32_t* inv_pos, ftmoe_stream_t stream) {
  if (T < 0 || E < 1 || E > 1024 || k < 1 || k > E || k > 32 || (long long)T * k >= (1LL << 31) ||
      !offsets)
    return FTMOE_ERR_INVALID_ARG;
  // Same scratch size as the workspace form of the call; beyond the fixed array -> refuse.
  const size_t need = permute_ws_bytes(T, k, E);
  if (need > NOALLOC_PERMUTE_MAX_INTS * sizeof(int32_t)) return FTMOE_ERR_WORKSPACE;
  if (T > 0 && (!ids || !sorted_pair || !inv_pos)) return FTMOE_ERR_INVALID_ARG;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES_NOALLOC)
    return FTMOE_ERR_CUDA;
  std::call_once(g_scratch_once[dev], resolve_scratch, dev);
  if (g_scratch_err[dev] != cudaSuccess || !g_scratch_ptr[dev]) return FTMOE_ERR_CUDA;
  const DeviceInfo* di = device_info();
  if (!di) return FTMOE_ERR_CUDA;
  cudaStream_t st = (cudaStream_t)stream;
  if (T == 0)
    return cudaMemsetAsync(offsets, 0, (E + 1) * sizeof(int32_t), st) == cudaSuccess ? FTMOE_OK
                                                                                    : FTMOE_ERR_CUDA;
  // The count kernel writes every scratch entry the scan and scatter kernels read,
  // so nothing has to be cleared between calls.
  const cudaError_t e = launch_permute(ids, T, k, E, offsets, sorted_pair, inv_pos,
                                       need ? g_scratch_ptr[dev] : nullptr, di->status, nullptr, 0, st);
  return e == cudaSuccess ? FTMOE_OK : FTMOE_ERR_CUDA;
}

}  // extern "C"
