// Permutation of (token, expert) pairs into per-expert groups, stable in the pair
// index p = t * k + j: histogram, exclusive prefix sum, stable scatter.
//
// A CTA ranks a chunk of 1024 pairs at once: __match_any_sync gives each pair's
// rank among equal ids inside its warp, per-warp counts in shared memory give the
// rank across warps, and a per-chunk base gives the rank across chunks.  Small
// problems run in one CTA; large ones use three kernels and a scratch table of
// per-chunk counts.
#include "common.cuh"
#include "internal.h"
#include "route.cuh"

namespace ftmoe {

constexpr int PCHUNK = 1024;           // pairs per chunk == threads per CTA
constexpr int PSMALL_MAX = 16 * 1024;  // single-CTA path up to this many pairs

__device__ __forceinline__ int load_id(const int32_t* ids, long long p, int P, int E, int* status) {
  if (p >= P) return -1;
  const int e = ids[p];
  if (e < 0 || e >= E) {
    set_device_code(status, DEV_BAD_EXPERT_ID);
    return -1;
  }
  return e;
}

// Block-wide exclusive scan of v over 1024 threads; returns the exclusive prefix,
// *total gets the sum.  `tmp` holds 32 ints of shared memory.
__device__ __forceinline__ int block_exclusive_scan(int v, int* tmp, int* total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) tmp[wid] = x;
  __syncthreads();
  if (wid == 0) {
    int s = tmp[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    tmp[lane] = s;  // inclusive warp totals
  }
  __syncthreads();
  const int before = (wid > 0 ? tmp[wid - 1] : 0) + x - v;
  *total = tmp[31];
  __syncthreads();
  return before;
}

// Ranks the chunk's pairs: returns this thread's id e (-1 if none) and its rank among
// equal ids in the chunk; afterwards chunk_cnt[e] holds the chunk's count of e.
// wcnt: [32][E] ints of shared memory.
__device__ __forceinline__ int chunk_rank(int e, int E, int* wcnt, int* chunk_cnt, int* rank_out) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  for (int i = threadIdx.x; i < 32 * E; i += PCHUNK) wcnt[i] = 0;
  __syncthreads();
  const unsigned peers = __match_any_sync(0xffffffffu, e);
  const int rank_w = __popc(peers & ((1u << lane) - 1u));
  if (e >= 0 && rank_w == 0) wcnt[wid * E + e] = __popc(peers);
  __syncthreads();
  for (int x = threadIdx.x; x < E; x += PCHUNK) {
    int run = 0;
    for (int w = 0; w < 32; ++w) {
      const int c = wcnt[w * E + x];
      wcnt[w * E + x] = run;
      run += c;
    }
    chunk_cnt[x] = run;
  }
  __syncthreads();
  *rank_out = e >= 0 ? wcnt[wid * E + e] + rank_w : 0;
  return e;
}

// Whole permutation in one CTA (P <= PSMALL_MAX).  Dynamic smem: (32 + 3) * E + 32 ints.
// With EPL > 0 the CTA first routes the T = P / k tokens from `logits` (warp w takes
// tokens w, w + 32, ...), writing ids / w, and then permutes them: routing and
// permutation of a small batch in one launch.
template <int EPL>
__global__ void __launch_bounds__(PCHUNK) permute_small_kernel(const int32_t* __restrict__ ids, int P,
                                                              int E, int32_t* __restrict__ offsets,
                                                              int32_t* __restrict__ sorted_pair,
                                                              int32_t* __restrict__ inv_pos,
                                                              int* status, int* zero_ptr, int zero_n,
                                                              const float* __restrict__ logits, int k,
                                                              float* __restrict__ wout) {
  extern __shared__ int sm[];
  if (EPL > 0) {
    int32_t* ids_w = const_cast<int32_t*>(ids);
    for (int t = threadIdx.x >> 5; t < P / k; t += PCHUNK / 32)
      route_token<(EPL > 0 ? EPL : 1)>(logits + (size_t)t * E, E, k, ids_w + (size_t)t * k,
                                       wout + (size_t)t * k, status);
    __syncthreads();  // the CTA's own global writes are visible to it after the barrier
  }
  for (int i = threadIdx.x; i < zero_n; i += PCHUNK) zero_ptr[i] = 0;
  int* wcnt = sm;                 // [32][E]
  int* cnt = wcnt + 32 * E;       // [E]
  int* base = cnt + E;            // [E]
  int* ccnt = base + E;           // [E]
  int* tmp = ccnt + E;            // [32]
  for (int x = threadIdx.x; x < E; x += PCHUNK) cnt[x] = 0;
  __syncthreads();
  for (int p0 = 0; p0 < P; p0 += PCHUNK) {
    const int e = load_id(ids, p0 + threadIdx.x, P, E, status);
    if (e >= 0) atomicAdd(&cnt[e], 1);
  }
  __syncthreads();
  // exclusive scan of counts over experts, 1024 at a time
  int carry = 0;
  for (int x0 = 0; x0 < E; x0 += PCHUNK) {
    const int x = x0 + threadIdx.x;
    const int v = x < E ? cnt[x] : 0;
    int tot;
    const int ex = block_exclusive_scan(v, tmp, &tot);
    if (x < E) {
      base[x] = carry + ex;
      offsets[x] = carry + ex;
    }
    carry += tot;
  }
  if (threadIdx.x == 0) offsets[E] = carry;
  __syncthreads();
  for (int p0 = 0; p0 < P; p0 += PCHUNK) {
    const int p = p0 + threadIdx.x;
    int rank;
    const int e = chunk_rank(load_id(ids, p, P, E, nullptr), E, wcnt, ccnt, &rank);
    if (e >= 0) {
      const int pos = base[e] + rank;
      sorted_pair[pos] = p;
      inv_pos[p] = pos;
    } else if (p < P) {
      inv_pos[p] = -1;
    }
    __syncthreads();
    for (int x = threadIdx.x; x < E; x += PCHUNK) base[x] += ccnt[x];
    __syncthreads();
  }
}

// Large P, step 1: per-chunk histogram hist[c][E].
__global__ void __launch_bounds__(PCHUNK) permute_count_kernel(const int32_t* __restrict__ ids, int P,
                                                              int E, int32_t* __restrict__ hist,
                                                              int* status, int* zero_ptr, int zero_n) {
  extern __shared__ int cnt[];
  if (blockIdx.x == 0)
    for (int i = threadIdx.x; i < zero_n; i += PCHUNK) zero_ptr[i] = 0;
  for (int x = threadIdx.x; x < E; x += PCHUNK) cnt[x] = 0;
  __syncthreads();
  const int e = load_id(ids, (long long)blockIdx.x * PCHUNK + threadIdx.x, P, E, status);
  if (e >= 0) atomicAdd(&cnt[e], 1);
  __syncthreads();
  for (int x = threadIdx.x; x < E; x += PCHUNK) hist[(size_t)blockIdx.x * E + x] = cnt[x];
}

// Large P, step 2 (one CTA): offsets = exclusive scan of per-expert totals; hist[c][e]
// becomes the first position of chunk c's pairs of expert e.
__global__ void __launch_bounds__(PCHUNK) permute_scan_kernel(int32_t* __restrict__ hist, int nchunk,
                                                             int E, int32_t* __restrict__ offsets) {
  __shared__ int tmp[32];
  int carry = 0;
  for (int x0 = 0; x0 < E; x0 += PCHUNK) {
    const int x = x0 + threadIdx.x;
    int tot_x = 0;
    if (x < E)
      for (int c = 0; c < nchunk; ++c) tot_x += hist[(size_t)c * E + x];
    int tot;
    const int ex = block_exclusive_scan(tot_x, tmp, &tot);
    if (x < E) {
      int run = carry + ex;
      offsets[x] = run;
      for (int c = 0; c < nchunk; ++c) {
        const int h = hist[(size_t)c * E + x];
        hist[(size_t)c * E + x] = run;
        run += h;
      }
    }
    carry += tot;
  }
  if (threadIdx.x == 0) offsets[E] = carry;
}

// Large P, step 3: stable scatter of each chunk.  Dynamic smem: (32 + 1) * E ints.
__global__ void __launch_bounds__(PCHUNK) permute_scatter_kernel(const int32_t* __restrict__ ids, int P,
                                                                int E, const int32_t* __restrict__ base,
                                                                int32_t* __restrict__ sorted_pair,
                                                                int32_t* __restrict__ inv_pos) {
  extern __shared__ int sm[];
  int* wcnt = sm;
  int* ccnt = wcnt + 32 * E;
  const int p = blockIdx.x * PCHUNK + threadIdx.x;
  int rank;
  const int e = chunk_rank(load_id(ids, p, P, E, nullptr), E, wcnt, ccnt, &rank);
  if (e >= 0) {
    const int pos = base[(size_t)blockIdx.x * E + e] + rank;
    sorted_pair[pos] = p;
    inv_pos[p] = pos;
  } else if (p < P) {
    inv_pos[p] = -1;
  }
}

size_t permute_ws_bytes(int T, int k, int E) {
  const long long P = (long long)T * k;
  if (P <= PSMALL_MAX) return 0;
  const long long nchunk = (P + PCHUNK - 1) / PCHUNK;
  return (size_t)(nchunk * E * sizeof(int32_t));
}

cudaError_t launch_permute(const int32_t* ids, int T, int k, int E, int32_t* offsets,
                           int32_t* sorted_pair, int32_t* inv_pos, void* ws, int* status,
                           void* zero_ptr, size_t zero_bytes, cudaStream_t st) {
  const int P = T * k;
  const int zero_n = zero_ptr ? (int)(zero_bytes / 4) : 0;
  if (P <= PSMALL_MAX) {
    const size_t smem = (size_t)(35 * E + 32) * sizeof(int);
    cudaError_t err = set_smem_limit<permute_small_kernel<0>>(smem);
    if (err != cudaSuccess) return err;
    permute_small_kernel<0><<<1, PCHUNK, smem, st>>>(ids, P, E, offsets, sorted_pair, inv_pos, status,
                                                   (int*)zero_ptr, zero_n, nullptr, k, nullptr);
    return cudaGetLastError();
  }
  const int nchunk = (P + PCHUNK - 1) / PCHUNK;
  int32_t* hist = (int32_t*)ws;
  permute_count_kernel<<<nchunk, PCHUNK, E * sizeof(int), st>>>(ids, P, E, hist, status,
                                                               (int*)zero_ptr, zero_n);
  permute_scan_kernel<<<1, PCHUNK, 0, st>>>(hist, nchunk, E, offsets);
  const size_t smem = (size_t)33 * E * sizeof(int);
  cudaError_t err = set_smem_limit<permute_scatter_kernel>(smem);
  if (err != cudaSuccess) return err;
  permute_scatter_kernel<<<nchunk, PCHUNK, smem, st>>>(ids, P, E, hist, sorted_pair, inv_pos);
  return cudaGetLastError();
}

bool route_permute_fits(int T, int k) { return T <= ROUTE_PERMUTE_MAX_T && (long long)T * k <= PSMALL_MAX; }

cudaError_t launch_route_permute(const float* logits, int T, int E, int k, int32_t* ids, float* w,
                                 int32_t* offsets, int32_t* sorted_pair, int32_t* inv_pos, int* status,
                                 void* zero_ptr, size_t zero_bytes, cudaStream_t st) {
  if (!route_permute_fits(T, k)) return cudaErrorNotSupported;
  const int P = T * k;
  const int zero_n = zero_ptr ? (int)(zero_bytes / 4) : 0;
  const size_t smem = (size_t)(35 * E + 32) * sizeof(int);
  cudaError_t err = cudaSuccess;
  with_epl(E, [&]<int N>() {
    err = set_smem_limit<permute_small_kernel<N>>(smem);
    if (err == cudaSuccess)
      permute_small_kernel<N><<<1, PCHUNK, smem, st>>>(ids, P, E, offsets, sorted_pair, inv_pos, status,
                                                     (int*)zero_ptr, zero_n, logits, k, w);
  });
  if (err != cudaSuccess) return err;
  return cudaGetLastError();
}

}  // namespace ftmoe
