// Self-check of the bounded waits that every pipelined kernel of the library uses.
//
// One CTA initialises an mbarrier that nothing will ever arrive on and waits on it
// with the same bounded wait as the tensor-core kernels, under a caller-given limit.
// The wait gives up, records DEV_WAIT_TIMEOUT in the device status word and the
// kernel returns normally, so a caller can check on a live GPU that a stuck
// producer / consumer handshake ends in a status code instead of a hang or a trap.
#include "internal.h"
#include "pipeline.cuh"
#include "tcgen05.cuh"

namespace ftmoe {

__global__ void wait_timeout_kernel(uint64_t limit_ns, int* status, int* waited_ok) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
  }
  fence_barrier_init();
  __syncthreads();
  if (threadIdx.x == 0) {
    const bool ok = mbar_wait_or_abort(&bar, 0, &abort_flag, status, limit_ns);
    if (waited_ok) *waited_ok = ok ? 1 : 0;
  }
}

}  // namespace ftmoe

using namespace ftmoe;

extern "C" ftmoe_status ftmoe_check_wait_timeout(long long limit_ns, int* waited_ok,
                                                 ftmoe_stream_t stream) {
  if (limit_ns < 1000 || limit_ns > 1000000000LL) return FTMOE_ERR_INVALID_ARG;
  const DeviceInfo* di = device_info();
  if (!di) return FTMOE_ERR_CUDA;
  wait_timeout_kernel<<<1, 32, 0, (cudaStream_t)stream>>>((uint64_t)limit_ns, di->status, waited_ok);
  return cudaGetLastError() == cudaSuccess ? FTMOE_OK : FTMOE_ERR_CUDA;
}
