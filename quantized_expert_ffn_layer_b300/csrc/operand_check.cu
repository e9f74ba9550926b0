// Verification aid: the tensor-core operands the FFN kernels build from the tiled
// weight records (the GGUF dequant of the FreeToken architecture walkthrough §六),
// written out as bf16 [E][N][K] so that they can be compared with the exact decode of
// the canonical blocks.  Each kernel runs the same device functions as the kernel whose
// operand it reproduces (operand.cuh) and reads the result back through that kernel's
// layout.
#include "common.cuh"
#include "internal.h"
#include "operand.cuh"

namespace ftmoe {

constexpr int OC_ROWS = 128;  // A-tile rows of the prefill GEMM

// One CTA per (expert, 128-row tile, 64-element slab): the tile's (up to) 8 records are
// copied to shared memory, converted exactly as the prefill GEMM's converters do
// (FTMOE_GP_NSTEP = 4: warp w < 4 converts records 2w + {0, 1} whole; 2: warp w
// records 2 (w / 2) + {0, 1}, quantization block w % 2), and the swizzled A tile is
// read back row by row (tile row -> record row via sigma^-1).
template <int QT>
__global__ void __launch_bounds__(256) operand_prefill_kernel(const uint8_t* __restrict__ tiles,
                                                              uint16_t* __restrict__ out, int E,
                                                              int N, int K) {
  constexpr int RB = rec_bytes(QT);
  __shared__ __align__(1024) uint8_t tile[OC_ROWS * 128];
  __shared__ __align__(16) uint8_t raw[8 * RB];
  const int S = slabs_of(K), RG = N / 16, NT = (N + OC_ROWS - 1) / OC_ROWS;
  int bid = blockIdx.x;
  const int s = bid % S;
  bid /= S;
  const int rt = bid % NT;
  const int e = bid / NT;
  if (e >= E) return;
  const int tid = threadIdx.x;
  for (int i = tid; i < 8 * RB / 16; i += blockDim.x) {
    const int rg = i / (RB / 16), off = i - rg * (RB / 16);
    const int g16 = rt * 8 + rg;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (g16 < RG)
      v = reinterpret_cast<const uint4*>(tiles + (size_t)e * tiles_bytes_per_expert(QT, N, K) +
                                         ((size_t)g16 * S + s) * RB)[off];
    reinterpret_cast<uint4*>(raw)[i] = v;
  }
  __syncthreads();
  const int warp = tid >> 5, lane = tid & 31;
  const int g = (lane & 15) >> 1, m = lane & 1;
  const uint32_t tbase = smem_u32(tile);
  if (FTMOE_GP_NSTEP == 4) {
    const int ri = 2 * warp + (lane >> 4);
    if (warp < 4) convert_record_operand<QT, 4, 0>(smem_u32(raw) + ri * RB, tbase, ri, g, m);
  } else {
    const int ri = 2 * (warp >> 1) + (lane >> 4);
    const uint32_t rec = smem_u32(raw) + ri * RB;
    if (warp & 1) convert_record_operand<QT, 2, 2>(rec, tbase, ri, g, m);
    else convert_record_operand<QT, 2, 0>(rec, tbase, ri, g, m);
  }
  __syncthreads();
  // thread t: tile row t / 2, chunks 4 (t % 2) .. +3 (8 bf16 each)
  const int Tr = tid >> 1, h = tid & 1;
  const int row = rt * OC_ROWS + (Tr >> 4) * 16 + gm_sigma_inv(Tr & 15);
  if (row >= N) return;
  uint16_t* orow = out + ((size_t)e * N + row) * K;
#pragma unroll
  for (int cc = 0; cc < 4; ++cc) {
    const int c = 4 * h + cc;
    const int k0 = s * 64 + 8 * c;
    if (k0 >= K) break;
    const uint4 v = lds128(tbase + (Tr >> 3) * 1024 + (Tr & 7) * 128 + ((c ^ (Tr & 7)) * 16));
    *reinterpret_cast<uint4*>(orow + k0) = v;
  }
}

// One thread per (record, lane): the decode GEMM converter's decode_plain of the lane's
// 16 bytes, placed where its 16x256b tensor-memory store puts them (register 4j + m of
// lane 4g + c -> row g + 8 (m >> 1), 32-bit column 8j + 2c + (m & 1) = elements
// 16j + 4c + 2 (m & 1) + {0, 1}).
template <int QT>
__global__ void operand_codes_kernel(const uint8_t* __restrict__ tiles, uint16_t* __restrict__ out,
                                     int E, int N, int K) {
  constexpr int RB = rec_bytes(QT);
  const int S = slabs_of(K), RG = N / 16;
  const long long nrec = (long long)E * RG * S;
  const long long gid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (gid >= nrec * 32) return;
  const int lane = (int)(gid & 31);
  const long long rec = gid >> 5;
  const int s = (int)(rec % S);
  const long long er = rec / S;
  const int rg = (int)(er % RG);
  const int e = (int)(er / RG);
  const int g = lane >> 2, c = lane & 3;
  const uint8_t* rp = tiles + (size_t)e * tiles_bytes_per_expert(QT, N, K) +
                      (size_t)(rec - (long long)e * RG * S) * RB;
  if (QT == FTMOE_MXFP8) {
    // the grouped GEMV's A operand: each E4M3 element as exact bf16, unscaled
    const uint4 q0 = *reinterpret_cast<const uint4*>(rp + lane * 32);
    const uint4 q1 = *reinterpret_cast<const uint4*>(rp + lane * 32 + 16);
    const uint32_t w8[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int row = rg * 16 + g + 8 * h;
        const int k = s * 64 + 16 * j + 4 * c;
        if (k >= K) continue;
        uint32_t* o = reinterpret_cast<uint32_t*>(out + ((size_t)e * N + row) * K + k);
        o[0] = e4m3x2_to_bf16x2(prmt(w8[2 * j + h], 0u, 0x4140u));
        o[1] = e4m3x2_to_bf16x2(prmt(w8[2 * j + h], 0u, 0x4342u));
      }
    return;
  }
  const uint4 q = *reinterpret_cast<const uint4*>(rp + lane * 16);
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    uint32_t o[4];
    decode_plain<QT>(w[j] & 0x0F0F0F0Fu, o[0], o[1]);
    decode_plain<QT>((w[j] >> 4) & 0x0F0F0F0Fu, o[2], o[3]);
#pragma unroll
    for (int mm = 0; mm < 4; ++mm) {
      const int row = rg * 16 + g + 8 * (mm >> 1);
      const int k = s * 64 + 16 * j + 4 * c + 2 * (mm & 1);
      if (k >= K) continue;
      *reinterpret_cast<uint32_t*>(out + ((size_t)e * N + row) * K + k) = o[mm];
    }
  }
}

cudaError_t launch_operand(int qtype, int which, const void* tiles, int E, int N, int K,
                           uint16_t* out, cudaStream_t st) {
  const uint8_t* t = (const uint8_t*)tiles;
  if (which == FTMOE_OPERAND_PREFILL) {
    const long long blocks = (long long)E * ((N + OC_ROWS - 1) / OC_ROWS) * slabs_of(K);
    if (blocks > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
    if (qtype == FTMOE_Q4_0)
      operand_prefill_kernel<FTMOE_Q4_0><<<(unsigned)blocks, 256, 0, st>>>(t, out, E, N, K);
    else if (qtype == FTMOE_MXFP4)
      operand_prefill_kernel<FTMOE_MXFP4><<<(unsigned)blocks, 256, 0, st>>>(t, out, E, N, K);
    else if (qtype == FTMOE_NVFP4)
      operand_prefill_kernel<FTMOE_NVFP4><<<(unsigned)blocks, 256, 0, st>>>(t, out, E, N, K);
    else
      operand_prefill_kernel<FTMOE_MXFP8><<<(unsigned)blocks, 256, 0, st>>>(t, out, E, N, K);
  } else {
    const long long threads = (long long)E * (N / 16) * slabs_of(K) * 32;
    const unsigned grid = (unsigned)((threads + 255) / 256);
    if (qtype == FTMOE_Q4_0)
      operand_codes_kernel<FTMOE_Q4_0><<<grid, 256, 0, st>>>(t, out, E, N, K);
    else if (qtype == FTMOE_MXFP4)
      operand_codes_kernel<FTMOE_MXFP4><<<grid, 256, 0, st>>>(t, out, E, N, K);
    else if (qtype == FTMOE_NVFP4)  // NVFP4 codes are E2M1, decoded like MXFP4's
      operand_codes_kernel<FTMOE_NVFP4><<<grid, 256, 0, st>>>(t, out, E, N, K);
    else
      operand_codes_kernel<FTMOE_MXFP8><<<grid, 256, 0, st>>>(t, out, E, N, K);
  }
  return cudaGetLastError();
}

}  // namespace ftmoe
