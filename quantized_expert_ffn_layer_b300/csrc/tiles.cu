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
  constexpr int BE = canon_block_elems(QT);    // weights per canonical block
  constexpr int SB = QT == FTMOE_Q4_0 ? 2 : 1;  // scale bytes at the start of a block
  constexpr int BPR = 64 / BE;                 // blocks per row in one record
  constexpr int RB = rec_bytes(QT);
  const int S = slabs_of(K), NB = K / BE, RT = N / 16;
  const size_t stride = tiles_bytes_per_expert(QT, N, K);
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

  // code of element 16j + 4c + r of the slab: block (64 s + ...) / BE, element i of the
  // block in the low nibble of code byte i (i < BE / 2) or the high nibble of byte i - BE / 2
  auto code_at = [&](int row, int j, int r) -> uint32_t {
    const int kk = s * 64 + 16 * j + 4 * c + r;
    const int blk = kk / BE, i = kk - blk * BE;
    if (blk >= NB) return QT == FTMOE_Q4_0 ? 8u : 0u;  // padded half slab: zero weight
    const uint8_t* b = canon + (((long long)e * N + row) * NB + blk) * CB + SB;
    return i < BE / 2 ? (uint32_t)(b[i] & 15) : (uint32_t)(b[i - BE / 2] >> 4);
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
  uint8_t* rp = tiles + (size_t)e * stride + (size_t)(rec - (long long)e * RT * S) * RB;
  *reinterpret_cast<uint4*>(rp + lane * 16) = make_uint4(words[0], words[1], words[2], words[3]);
  if (c == 0) {
#pragma unroll
    for (int b = 0; b < BPR; ++b) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int row = h ? row1 : row0;
        const int blk = BPR * s + b;
        const int idx = (g * BPR + b) * 2 + h;
        const uint8_t* bp = canon + (((long long)e * N + row) * NB + blk) * CB;
        if (QT == FTMOE_Q4_0) {
          reinterpret_cast<uint16_t*>(rp + REC_CODE_BYTES)[idx] =
              blk < NB ? (uint16_t)(bp[0] | (bp[1] << 8)) : (uint16_t)0;
        } else if (QT == FTMOE_MXFP4) {
          rp[REC_CODE_BYTES + idx] = blk < NB ? bp[0] : (uint8_t)127;
        } else {
          rp[REC_CODE_BYTES + idx] = blk < NB ? bp[0] : (uint8_t)0;
        }
      }
    }
  }
}

// MXFP8: one thread per (record, lane) gathers the E4M3 bytes of elements 16j + 4c .. +3
// of rows g (word 2j) and g + 8 (word 2j + 1) and writes the lane's 32 bytes; lanes with
// c == 0 also write the 4 E8M0 scales of rows g, g + 8 for both blocks of the slab.
__global__ void repack_fp8_kernel(const uint8_t* __restrict__ canon, uint8_t* __restrict__ tiles,
                                  int E, int N, int K) {
  constexpr int RB = rec_bytes(FTMOE_MXFP8);
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
  uint32_t words[8];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int row = rt * 16 + g + 8 * h;
      uint32_t w = 0;
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int kk = s * 64 + 16 * j + 4 * c + r;
        const int blk = kk >> 5;
        const uint32_t b = blk < NB ? canon[(((long long)e * N + row) * NB + blk) * 33 + 1 + (kk & 31)] : 0u;
        w |= b << (8 * r);
      }
      words[2 * j + h] = w;
    }
  }
  uint8_t* rp = tiles + (size_t)rec * RB;
  *reinterpret_cast<uint4*>(rp + lane * 32) = make_uint4(words[0], words[1], words[2], words[3]);
  *reinterpret_cast<uint4*>(rp + lane * 32 + 16) = make_uint4(words[4], words[5], words[6], words[7]);
  if (c == 0) {
#pragma unroll
    for (int b = 0; b < 2; ++b)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int row = rt * 16 + g + 8 * h, blk = 2 * s + b;
        rp[1024 + (g * 2 + b) * 2 + h] = blk < NB ? canon[(((long long)e * N + row) * NB + blk) * 33] : (uint8_t)127;
      }
  }
}

// MXFP8 exact decode: E4M3 x 2^(e - 127) in fp32 (exact down to fp32's subnormals; beyond
// its range +-inf; NaN codes and scale 255 give NaN).
__global__ void dequant_fp8_kernel(const uint8_t* __restrict__ tiles, float* __restrict__ out, int E,
                                   int N, int K) {
  constexpr int RB = rec_bytes(FTMOE_MXFP8);
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
  const uint8_t* rp = tiles + (size_t)rec * RB;
  const uint4 q0 = *reinterpret_cast<const uint4*>(rp + lane * 32);
  const uint4 q1 = *reinterpret_cast<const uint4*>(rp + lane * 32 + 16);
  const uint32_t w[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
  for (int j = 0; j < 4; ++j)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const float sc = e8m0_to_f32(rp[1024 + (g * 2 + (j >> 1)) * 2 + h]);
      float* o = out + ((long long)e * N + rt * 16 + g + 8 * h) * K;
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int k = s * 64 + 16 * j + 4 * c + r;
        if (k < K) o[k] = e4m3_to_f32((w[2 * j + h] >> (8 * r)) & 0xFFu) * sc;
      }
    }
}

// NVFP4: expert e's tensor scale (the canonical buffer's trailing fp32 array, read byte by
// byte: the array need not be 4-byte aligned) into the trailer after its records.
__global__ void nvfp4_trailer_kernel(const uint8_t* __restrict__ canon, uint8_t* __restrict__ tiles,
                                     int E, int N, int K) {
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= E) return;
  const uint8_t* p = canon + (size_t)E * N * (K / 16) * 9 + (size_t)e * 4;
  const uint32_t bits = (uint32_t)p[0] | ((uint32_t)p[1] << 8) | ((uint32_t)p[2] << 16) | ((uint32_t)p[3] << 24);
  uint8_t* t = tiles + (size_t)e * tiles_bytes_per_expert(FTMOE_NVFP4, N, K) +
               records_bytes_per_expert(FTMOE_NVFP4, N, K);
  *reinterpret_cast<uint4*>(t) = make_uint4(bits, 0u, 0u, 0u);
}

// Exact decode: one thread per (record, lane), 32 weights each.  Uses the same
// in-register code -> bf16 conversion as the FFN kernels, then multiplies by the
// block scale in fp32 (both factors and the product are exact in fp32); NVFP4 then
// multiplies by the tensor scale, the one rounding of the exact value.
template <int QT>
__global__ void dequant_kernel(const uint8_t* __restrict__ tiles, float* __restrict__ out, int E,
                               int N, int K) {
  constexpr int RB = rec_bytes(QT);
  const int S = slabs_of(K), RT = N / 16;
  const size_t stride = tiles_bytes_per_expert(QT, N, K);
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
  const uint8_t* ebase = tiles + (size_t)e * stride;
  const uint8_t* rp = ebase + (size_t)(rec - (long long)e * RT * S) * RB;
  const uint4 q = *reinterpret_cast<const uint4*>(rp + lane * 16);
  const uint32_t wj[4] = {q.x, q.y, q.z, q.w};
  const float ts = QT == FTMOE_NVFP4
                       ? *reinterpret_cast<const float*>(ebase + records_bytes_per_expert(QT, N, K))
                       : 1.0f;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    uint32_t a[4];
    if (QT == FTMOE_Q4_0) q4_word_to_bf16x2(wj[j], a); else e2m1_word_to_bf16x2(wj[j], a);
    const int kbase = s * 64 + 16 * j + 4 * c;
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      const int h = p & 1;             // p = 1, 3: row g+8
      const int rofs = (p >> 1) * 2;   // p = 2, 3: positions r = 2, 3
      const int row = rt * 16 + g + 8 * h;
      float sc;
      if (QT == FTMOE_Q4_0)
        sc = half_bits_to_f32(reinterpret_cast<const uint16_t*>(rp + REC_CODE_BYTES)[(g * 2 + (j >> 1)) * 2 + h]);
      else if (QT == FTMOE_MXFP4)
        sc = e8m0_to_f32(rp[REC_CODE_BYTES + (g * 2 + (j >> 1)) * 2 + h]);
      else
        sc = e4m3_to_f32(rp[REC_CODE_BYTES + (g * 4 + j) * 2 + h]);
      float v0 = bf16_bits_to_f32(a[p] & 0xFFFF) * sc;
      float v1 = bf16_bits_to_f32(a[p] >> 16) * sc;
      if (QT == FTMOE_NVFP4) {
        v0 *= ts;
        v1 *= ts;
      }
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
  const uint8_t* c = (const uint8_t*)canon;
  uint8_t* t = (uint8_t*)tiles;
  if (qtype == FTMOE_Q4_0) {
    repack_kernel<FTMOE_Q4_0><<<grid, bs, 0, st>>>(c, t, E, N, K);
  } else if (qtype == FTMOE_MXFP4) {
    repack_kernel<FTMOE_MXFP4><<<grid, bs, 0, st>>>(c, t, E, N, K);
  } else if (qtype == FTMOE_NVFP4) {
    repack_kernel<FTMOE_NVFP4><<<grid, bs, 0, st>>>(c, t, E, N, K);
    nvfp4_trailer_kernel<<<(E + 255) / 256, 256, 0, st>>>(c, t, E, N, K);
  } else {
    repack_fp8_kernel<<<grid, bs, 0, st>>>(c, t, E, N, K);
  }
  return cudaGetLastError();
}

cudaError_t launch_dequant(int qtype, const void* tiles, int E, int N, int K, float* out,
                           cudaStream_t st) {
  const long long threads = (long long)E * (N / 16) * slabs_of(K) * 32;
  const int bs = 256;
  const unsigned grid = (unsigned)((threads + bs - 1) / bs);
  const uint8_t* t = (const uint8_t*)tiles;
  if (qtype == FTMOE_Q4_0)
    dequant_kernel<FTMOE_Q4_0><<<grid, bs, 0, st>>>(t, out, E, N, K);
  else if (qtype == FTMOE_MXFP4)
    dequant_kernel<FTMOE_MXFP4><<<grid, bs, 0, st>>>(t, out, E, N, K);
  else if (qtype == FTMOE_NVFP4)
    dequant_kernel<FTMOE_NVFP4><<<grid, bs, 0, st>>>(t, out, E, N, K);
  else
    dequant_fp8_kernel<<<grid, bs, 0, st>>>(t, out, E, N, K);
  return cudaGetLastError();
}

}  // namespace ftmoe
