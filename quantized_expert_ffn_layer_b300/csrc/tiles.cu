// Canonical GGUF Q4_0 / MXFP4 blocks <-> the kernels' tiled record layout, and an
// exact fp32 decode of the tiles (the expert banks' formats of the FreeToken
// architecture walkthrough, §五; its GGUF dequant kernels, §六).
#include "common.cuh"
#include "internal.h"

namespace ftmoe {

// One thread per (record, lane): gathers the 32 codes of rows g, g+8 at slab positions
// 16j + 4c + r from the canonical blocks and writes the lane's 16 bytes; lanes with
// c == 0 also write the 4 scales of rows g, g+8 for both blocks of the slab.
template <int QT>
__global__ void repack_kernel(const uint8_t* __restrict__ canon, uint8_t* __restrict__ tiles, int E,
                              int N, int K) {
  constexpr int CB = canon_block_bytes(QT);
  constexpr int RB = rec_bytes(QT);
  const int S = slabs_of(K), NB = K / 32, RT = N / 16;
  const long long nrec = (long long)E * RT * S;
  const long long gid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (gid >= nrec * 32) return;
  const int lane = (int)(gid & 31);
  const long long rec = gid >> 5;
  const int s = (int)(rec % S);
  const long long er = rec / S;
  const int rt = (int)(er % RT);
  const int e = (int)(er / RT);
  const int g = lane >> 2, c = lane & 3;
  const int row0 = rt * 16 + g, row1 = row0 + 8;

  auto code_at = [&](int row, int j, int r) -> uint32_t {
    const int blk = 2 * s + (j >> 1);
    if (blk >= NB) return QT == FTMOE_Q4_0 ? 8u : 0u;  // padded half slab: zero weight
    const uint8_t* b = canon + (((long long)e * N + row) * NB + blk) * CB + (QT == FTMOE_Q4_0 ? 2 : 1);
    const int i = 4 * c + r;  // element i (j even) or 16 + i (j odd) of the block
    return (j & 1) ? (uint32_t)(b[i] >> 4) : (uint32_t)(b[i] & 15);
  };
  uint32_t words[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    uint32_t w = 0;
    w |= code_at(row0, j, 0) << 0;
    w |= code_at(row0, j, 1) << 16;
    w |= code_at(row1, j, 0) << 4;
    w |= code_at(row1, j, 1) << 20;
    w |= code_at(row0, j, 2) << 8;
    w |= code_at(row0, j, 3) << 24;
    w |= code_at(row1, j, 2) << 12;
    w |= code_at(row1, j, 3) << 28;
    words[j] = w;
  }
  uint8_t* rp = tiles + rec * RB;
  *reinterpret_cast<uint4*>(rp + lane * 16) = make_uint4(words[0], words[1], words[2], words[3]);
  if (c == 0) {
#pragma unroll
    for (int b = 0; b < 2; ++b) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int row = h ? row1 : row0;
        const int blk = 2 * s + b;
        const int idx = (g * 2 + b) * 2 + h;
        if (QT == FTMOE_Q4_0) {
          uint16_t d = 0;
          if (blk < NB) {
            const uint8_t* bp = canon + (((long long)e * N + row) * NB + blk) * CB;
            d = (uint16_t)(bp[0] | (bp[1] << 8));
          }
          reinterpret_cast<uint16_t*>(rp + REC_CODE_BYTES)[idx] = d;
        } else {
          uint8_t sc = 127;
          if (blk < NB) sc = canon[(((long long)e * N + row) * NB + blk) * CB];
          rp[REC_CODE_BYTES + idx] = sc;
        }
      }
    }
  }
}

// Exact decode: one thread per (record, lane), 32 weights each.  Uses the same
// in-register code -> bf16 conversion as the FFN kernels, then multiplies by the
// block scale in fp32 (both factors and the product are exact in fp32).
template <int QT>
__global__ void dequant_kernel(const uint8_t* __restrict__ tiles, float* __restrict__ out, int E,
                               int N, int K) {
  constexpr int RB = rec_bytes(QT);
  const int S = slabs_of(K), RT = N / 16;
  const long long nrec = (long long)E * RT * S;
  const long long gid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (gid >= nrec * 32) return;
  const int lane = (int)(gid & 31);
  const long long rec = gid >> 5;
  const int s = (int)(rec % S);
  const long long er = rec / S;
  const int rt = (int)(er % RT);
  const int e = (int)(er / RT);
  const int g = lane >> 2, c = lane & 3;
  const uint8_t* rp = tiles + rec * RB;
  const uint4 q = *reinterpret_cast<const uint4*>(rp + lane * 16);
  const uint32_t wj[4] = {q.x, q.y, q.z, q.w};
  float sc[2][2];  // [block][row half]
#pragma unroll
  for (int b = 0; b < 2; ++b)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int idx = (g * 2 + b) * 2 + h;
      sc[b][h] = QT == FTMOE_Q4_0
                     ? half_bits_to_f32(reinterpret_cast<const uint16_t*>(rp + REC_CODE_BYTES)[idx])
                     : e8m0_to_f32(rp[REC_CODE_BYTES + idx]);
    }
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    uint32_t a[4];
    if (QT == FTMOE_Q4_0) q4_word_to_bf16x2(wj[j], a); else e2m1_word_to_bf16x2(wj[j], a);
    const int b = j >> 1;
    const int kbase = s * 64 + 16 * j + 4 * c;
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      const int h = p & 1;             // p = 1, 3: row g+8
      const int rofs = (p >> 1) * 2;   // p = 2, 3: positions r = 2, 3
      const int row = rt * 16 + g + 8 * h;
      const float v0 = bf16_bits_to_f32(a[p] & 0xFFFF) * sc[b][h];
      const float v1 = bf16_bits_to_f32(a[p] >> 16) * sc[b][h];
      const int k0 = kbase + rofs;
      float* o = out + ((long long)e * N + row) * K;
      if (k0 < K) o[k0] = v0;
      if (k0 + 1 < K) o[k0 + 1] = v1;
    }
  }
}

cudaError_t launch_repack(int qtype, const void* canon, void* tiles, int E, int N, int K,
                          cudaStream_t st) {
  const long long threads = (long long)E * (N / 16) * slabs_of(K) * 32;
  const int bs = 256;
  const unsigned grid = (unsigned)((threads + bs - 1) / bs);
  if (qtype == FTMOE_Q4_0)
    repack_kernel<FTMOE_Q4_0><<<grid, bs, 0, st>>>((const uint8_t*)canon, (uint8_t*)tiles, E, N, K);
  else
    repack_kernel<FTMOE_MXFP4><<<grid, bs, 0, st>>>((const uint8_t*)canon, (uint8_t*)tiles, E, N, K);
  return cudaGetLastError();
}

cudaError_t launch_dequant(int qtype, const void* tiles, int E, int N, int K, float* out,
                           cudaStream_t st) {
  const long long threads = (long long)E * (N / 16) * slabs_of(K) * 32;
  const int bs = 256;
  const unsigned grid = (unsigned)((threads + bs - 1) / bs);
  if (qtype == FTMOE_Q4_0)
    dequant_kernel<FTMOE_Q4_0><<<grid, bs, 0, st>>>((const uint8_t*)tiles, out, E, N, K);
  else
    dequant_kernel<FTMOE_MXFP4><<<grid, bs, 0, st>>>((const uint8_t*)tiles, out, E, N, K);
  return cudaGetLastError();
}

}  // namespace ftmoe
