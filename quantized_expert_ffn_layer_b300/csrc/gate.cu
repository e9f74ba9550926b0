// Router gate: the expert scores the router selects from ([P3] "为什么 MoE 模型适合做
// CPU–GPU 协同": a few experts per token are picked by these scores), computed from the
// hidden state as logits[t][e] = sum over h of x[t][h] * Wg[e][h] (bf16 in, fp32 out).
//
// One CTA computes a 16-token x 32-expert tile with 16 warps.  The reduction over h is
// cut into 16-element steps; warp w takes steps w, w + 16, w + 32, ... (m16n8k16 MMAs
// on the tensor cores, fp32 accumulation) and the 16 warps' sums are added in warp order
// through shared memory.  The split depends only on H, so a token's logits do not
// depend on the other tokens of the batch.
#include "common.cuh"
#include "internal.h"

namespace ftmoe {

constexpr int GT_TOK = 16;
constexpr int GT_EXP = 32;
constexpr int GT_WARPS = 16;
constexpr int GT_U = 4;  // k-steps per load round

__device__ __forceinline__ uint32_t ld32_or0(const uint16_t* row, int h) {
  return row ? __ldg(reinterpret_cast<const uint32_t*>(row + h)) : 0u;
}

__global__ void __launch_bounds__(GT_WARPS * 32) gate_kernel(const uint16_t* __restrict__ x,
                                                             const uint16_t* __restrict__ wg, int T,
                                                             int H, int E, float* __restrict__ logits) {
  __shared__ float part[GT_WARPS][GT_TOK][GT_EXP];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int g = lane >> 2, c = lane & 3;
  const int t0 = blockIdx.x * GT_TOK, e0 = blockIdx.y * GT_EXP;
  // this lane's A rows (tokens g, g + 8 of the tile) and B rows (experts 8j + g)
  const uint16_t* xa = t0 + g < T ? x + (size_t)(t0 + g) * H : nullptr;
  const uint16_t* xb = t0 + g + 8 < T ? x + (size_t)(t0 + g + 8) * H : nullptr;
  const uint16_t* wr[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int e = e0 + 8 * j + g;
    wr[j] = e < E ? wg + (size_t)e * H : nullptr;
  }
  float acc[4][4] = {};
  // GT_U of the warp's k-steps per round: every load of the round is issued before the
  // first MMA, so a round costs one memory latency; the MMAs still run in k order.
  constexpr int STEP = 16 * GT_WARPS;
  for (int k0 = 16 * w; k0 < H; k0 += GT_U * STEP) {
    uint32_t a[GT_U][4], b[GT_U][4][2];
#pragma unroll
    for (int u = 0; u < GT_U; ++u) {
      const bool in = k0 + u * STEP < H;
      const int h0 = k0 + u * STEP + 2 * c, h1 = h0 + 8;
      a[u][0] = in ? ld32_or0(xa, h0) : 0u;
      a[u][1] = in ? ld32_or0(xb, h0) : 0u;
      a[u][2] = in ? ld32_or0(xa, h1) : 0u;
      a[u][3] = in ? ld32_or0(xb, h1) : 0u;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        b[u][j][0] = in ? ld32_or0(wr[j], h0) : 0u;
        b[u][j][1] = in ? ld32_or0(wr[j], h1) : 0u;
      }
    }
#pragma unroll
    for (int u = 0; u < GT_U; ++u)
      if (k0 + u * STEP < H)
#pragma unroll
        for (int j = 0; j < 4; ++j) mma_16816(acc[j], a[u], b[u][j][0], b[u][j][1]);
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    part[w][g][8 * j + 2 * c] = acc[j][0];
    part[w][g][8 * j + 2 * c + 1] = acc[j][1];
    part[w][g + 8][8 * j + 2 * c] = acc[j][2];
    part[w][g + 8][8 * j + 2 * c + 1] = acc[j][3];
  }
  __syncthreads();
  for (int o = threadIdx.x; o < GT_TOK * GT_EXP; o += GT_WARPS * 32) {
    const int r = o / GT_EXP, col = o % GT_EXP;
    float s = 0.f;
#pragma unroll
    for (int v = 0; v < GT_WARPS; ++v) s += part[v][r][col];
    if (t0 + r < T && e0 + col < E) logits[(size_t)(t0 + r) * E + e0 + col] = s;
  }
}

}  // namespace ftmoe

using namespace ftmoe;

extern "C" ftmoe_status ftmoe_gate(const uint16_t* x, const uint16_t* wg, int T, int H, int E,
                                   float* logits, ftmoe_stream_t stream) {
  if (T < 0 || E < 1 || E > 1024 || H < 32 || H > 16384 || H % 32) return FTMOE_ERR_INVALID_ARG;
  if (T == 0) return FTMOE_OK;
  if (!x || !wg || !logits) return FTMOE_ERR_INVALID_ARG;
  const dim3 grid((T + GT_TOK - 1) / GT_TOK, (E + GT_EXP - 1) / GT_EXP);
  gate_kernel<<<grid, GT_WARPS * 32, 0, (cudaStream_t)stream>>>(x, wg, T, H, E, logits);
  return cudaGetLastError() == cudaSuccess ? FTMOE_OK : FTMOE_ERR_CUDA;
}
