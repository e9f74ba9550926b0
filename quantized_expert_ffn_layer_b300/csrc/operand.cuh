// Tensor-core operand decode of the tiled 4-bit weight records (the GGUF dequant of the
// FreeToken architecture walkthrough §六, for the Q4_0 / MXFP4 banks of §五).
//
// Two operand forms, each used by one tcgen05 kernel and reproduced element by element
// by the verification kernels in operand_check.cu (ftmoe_dequant_operand):
//   * the prefill grouped GEMM's A tile: every weight rounded once to bf16
//     (round-to-nearest-even of the exact decoded value; for NVFP4 the E2M1 code times
//     its E4M3 block scale, exact, with the tensor scale left to the GEMM's epilogue) in
//     the 128-byte-swizzled K-major layout (convert_record_swizzled);
//   * the decode GEMM's A operand: the unscaled code value (q - 8 for Q4_0, the E2M1
//     value for MXFP4), exact in bf16 (decode_plain).
// Record layout: see common.cuh.
#pragma once

#include "common.cuh"
#include "pipeline.cuh"

namespace ftmoe {

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

__device__ __forceinline__ uint32_t lds32(uint32_t saddr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(saddr) : "memory");
  return v;
}

__device__ __forceinline__ uint2 lds64(uint32_t saddr) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(saddr) : "memory");
  return v;
}

__device__ __forceinline__ uint4 lds128(uint32_t saddr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(saddr)
               : "memory");
  return v;
}

__device__ __forceinline__ void sts128(uint32_t saddr, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(saddr), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

// ---------------------------------------------------------------- prefill A tile
// Steps (of 16 elements) one converter thread of the prefill GEMM decodes per record
// and stage: 4 (a half-warp converts a whole record) or 2 (half a record).  The
// operand check (operand_check.cu) converts with the same span.
#ifndef FTMOE_GP_NSTEP
#define FTMOE_GP_NSTEP 4
#endif
// A-tile row order: weight row r of a 16-row record is stored at tile row sigma(r)
// (rows 0..3 -> 0,2,4,6, rows 4..7 -> 1,3,5,7, and the same +8 for rows 8..15), so
// that the converter stores of a quarter-warp fall on 8 different 16-byte bank groups.
__host__ __device__ constexpr int gm_sigma(int r) {
  return (r & 8) | ((r & 7) < 4 ? 2 * (r & 3) : 2 * (r & 3) + 1);
}
__host__ __device__ inline int gm_sigma_inv(int t) {
  const int u = t & 7;
  return (t & 8) | ((u & 1) ? 4 + (u >> 1) : (u >> 1));
}

// W holds 8 E2M1 codes of one row as nibble slots (0,4,2,6,1,5,3,7) = elements 0..7;
// slots p and p + 4 form the bf16x2 pair p.  Returns the 8 values times the block
// scale s_hi (2^(e - 127) as bf16x2) in element order: exact unless the product
// leaves the bf16 range.
__device__ __forceinline__ uint4 e2m1_scaled8(uint32_t W, uint32_t s_hi) {
  uint32_t r[4];
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    const uint32_t v = (W >> (4 * p)) & 0x000F000Fu;
    uint32_t t = ((v & 0x00070007u) << 6) | ((v & 0x00080008u) << 12);  // E2M1 * 2^-126
    const uint32_t TWO126 = 0x7E807E80u;
    __nv_bfloat162 w = __hmul2(*reinterpret_cast<__nv_bfloat162*>(&t),
                               *reinterpret_cast<const __nv_bfloat162*>(&TWO126));
    w = __hmul2(w, *reinterpret_cast<const __nv_bfloat162*>(&s_hi));
    r[p] = *reinterpret_cast<const uint32_t*>(&w);
  }
  return make_uint4(r[0], r[2], r[1], r[3]);
}

// Block scale of one row as (hi, lo) bf16x2 pairs with hi + lo == the scale exactly
// (Q4_0 fp16 d; lo = 0 when d is not finite, so that +-inf scales give +-inf weights and
// NaN only where the code is q = 8), or (2^(e-127), 0) for an MXFP4 E8M0 byte
// (e = 0 is the subnormal 2^-127, e = 255 NaN).
// NVFP4: the E4M3 scale as bf16 (exact: 4 significant bits, in range), lo = 0; the
// tensor scale is not part of the operand (the GEMM multiplies its accumulators by it).
template <int QT>
__device__ __forceinline__ void row_scale(uint32_t bits, uint32_t& hi2, uint32_t& lo2) {
  if (QT == FTMOE_Q4_0) {
    const float d = half_bits_to_f32(bits);
    const uint32_t hi = f32_to_bf16_bits(d);
    const uint32_t lo = (bits & 0x7C00u) == 0x7C00u ? 0u : f32_to_bf16_bits(d - bf16_bits_to_f32(hi));
    hi2 = hi | (hi << 16);
    lo2 = lo | (lo << 16);
  } else if (QT == FTMOE_NVFP4) {
    const uint32_t b = f32_to_bf16_bits(e4m3_to_f32(bits));
    hi2 = b | (b << 16);
    lo2 = 0;
  } else {
    const uint32_t b = bits == 0 ? 0x0040u : (bits == 255 ? 0x7FC0u : (bits << 7));
    hi2 = b | (b << 16);
    lo2 = 0;
  }
}

// Four bf16x2 (128 + q) pairs from nibble bytes: E1 holds elements 0..3 and E2 elements
// 4..7 of one row as byte-aligned nibbles in the order (e0, e2, e1, e3).
__device__ __forceinline__ void q4_pairs(uint32_t E1, uint32_t E2, uint32_t (&t)[4]) {
  const uint32_t K = 0x43434343u;  // high byte of bf16 128
  t[0] = prmt(E1, K, 0x4240u);
  t[1] = prmt(E1, K, 0x4341u);
  t[2] = prmt(E2, K, 0x4240u);
  t[3] = prmt(E2, K, 0x4341u);
}

// (128 + q) pairs -> RNE((q - 8) * d) with d = hi + lo split exactly (see row_scale):
// (q - 8) * lo is exact in bf16 (at most 4 + 4 significant bits), so the one rounding
// of the fused multiply-add is the rounding of the exact product.
__device__ __forceinline__ uint4 q4_scale(const uint32_t (&t)[4], uint32_t s_hi, uint32_t s_lo) {
  const __nv_bfloat162 off = __floats2bfloat162_rn(136.0f, 136.0f);
  uint32_t r[4];
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    const __nv_bfloat162 u = __hsub2(*reinterpret_cast<const __nv_bfloat162*>(&t[p]), off);
    const __nv_bfloat162 lo = __hmul2(u, *reinterpret_cast<const __nv_bfloat162*>(&s_lo));
    const __nv_bfloat162 w = __hfma2(u, *reinterpret_cast<const __nv_bfloat162*>(&s_hi), lo);
    r[p] = *reinterpret_cast<const uint32_t*>(&w);
  }
  return make_uint4(r[0], r[1], r[2], r[3]);
}

// One converter thread's share of a record in shared memory.  Record lanes 4g + 2m (A)
// and 4g + 2m + 1 (B) hold elements 8m..8m+7 of each 16-element step j of rows g and
// g + 8 (A: elements 8m..8m+3, B: 8m+4..8m+7).  The thread decodes NSTEP steps starting
// at J0 (NSTEP = 1, 2 or 4; a span of 2 or 4 starts on a quantization block) of both
// rows into the A tile at `tile` (128 rows of 64 bf16, 128-byte swizzle), record row
// group rg.  Lane pairs (m = 0, 1) share the scale conversions through one shuffle, so
// all 32 lanes of the warp must call it together.  The two 16-byte code loads are issued
// in an order that depends on (g >> 1) & 1 so that each quarter-warp reads 8 different
// bank groups.
template <int QT, int NSTEP, int J0>
__device__ __forceinline__ void convert_record_swizzled(uint32_t rec, uint32_t tile, int rg, int g,
                                                        int m) {
  static_assert(NSTEP == 1 || (NSTEP == 2 && J0 % 2 == 0) || (NSTEP == 4 && J0 == 0), "step span");
  // scales per thread: one per 32-element block (Q4_0, MXFP4: two steps share one), one
  // per step for NVFP4's 16-element blocks
  constexpr int NSC = QT == FTMOE_NVFP4 ? NSTEP : (NSTEP + 1) / 2;
  const int sw = (g >> 1) & 1;
  const uint4 l1 = lds128(rec + (4 * g + 2 * m + sw) * 16);
  const uint4 l2 = lds128(rec + (4 * g + 2 * m + 1 - sw) * 16);
  const uint4 ca = sw ? l2 : l1, cb = sw ? l1 : l2;
  const int T0 = rg * 16 + gm_sigma(g);  // tile row of record row g (row g + 8: T0 + 8)
  const uint32_t row0 = tile + (T0 >> 3) * 1024 + (T0 & 7) * 128;
  const uint32_t row1 = row0 + 1024;
  const uint32_t ph = (uint32_t)(T0 & 7);
  // scale of row g + 8 m (this lane) and of the other row (partner lane)
  uint32_t sh0[NSC], sl0[NSC], sh1[NSC], sl1[NSC];
#pragma unroll
  for (int u = 0; u < NSC; ++u) {
    const int idx = QT == FTMOE_NVFP4 ? (g * 4 + J0 + u) * 2 + m : (g * 2 + (J0 >> 1) + u) * 2 + m;
    const int byte = QT == FTMOE_Q4_0 ? idx * 2 : idx;
    const uint32_t w = lds32(rec + REC_CODE_BYTES + (byte & ~3));
    const uint32_t sbits = QT == FTMOE_Q4_0 ? (w >> (8 * (byte & 3))) & 0xFFFFu : (w >> (8 * (byte & 3))) & 0xFFu;
    uint32_t mh, ml;
    row_scale<QT>(sbits, mh, ml);
    const uint32_t oh = __shfl_xor_sync(0xffffffffu, mh, 1);
    const uint32_t ol = __shfl_xor_sync(0xffffffffu, ml, 1);
    sh0[u] = m ? oh : mh;
    sl0[u] = m ? ol : ml;
    sh1[u] = m ? mh : oh;
    sl1[u] = m ? ml : ol;
  }
  const uint32_t wa[4] = {ca.x, ca.y, ca.z, ca.w};
  const uint32_t wb[4] = {cb.x, cb.y, cb.z, cb.w};
#pragma unroll
  for (int s = 0; s < NSTEP; ++s) {
    const int j = J0 + s;
    const int u = QT == FTMOE_NVFP4 ? s : (j >> 1) - (J0 >> 1);
    const uint32_t A = wa[j], Bw = wb[j];
    const uint32_t off = (((uint32_t)(2 * j + m)) ^ ph) * 16;
    if (QT == FTMOE_Q4_0) {
      uint32_t t0[4], t1[4];
      q4_pairs(A & 0x0F0F0F0Fu, Bw & 0x0F0F0F0Fu, t0);                // row g
      q4_pairs((A >> 4) & 0x0F0F0F0Fu, (Bw >> 4) & 0x0F0F0F0Fu, t1);  // row g + 8
      sts128(row0 + off, q4_scale(t0, sh0[u], sl0[u]));
      sts128(row1 + off, q4_scale(t1, sh1[u], sl1[u]));
    } else {
      const uint32_t wg = (A & 0x0F0F0F0Fu) | ((Bw & 0x0F0F0F0Fu) << 4);
      const uint32_t wg8 = ((A >> 4) & 0x0F0F0F0Fu) | (Bw & 0xF0F0F0F0u);
      sts128(row0 + off, e2m1_scaled8(wg, sh0[u]));
      sts128(row1 + off, e2m1_scaled8(wg8, sh1[u]));
    }
  }
}

// MXFP8: the same thread roles on 1056-byte records.  Thread (g, m) writes elements
// 8m..8m+7 of steps J0..J0+NSTEP-1 of rows g and g + 8: record lane 4g + 2m holds
// elements 8m..8m+3 (row g in word 2j, row g + 8 in word 2j + 1) and lane 4g + 2m + 1
// elements 8m+4..8m+7.  Each E4M3 pair becomes exact bf16 and is scaled by 2^(e - 127)
// (one more bf16 multiply: exact unless the product leaves the bf16 range).
template <int NSTEP, int J0>
__device__ __forceinline__ void convert_record_swizzled_fp8(uint32_t rec, uint32_t tile, int rg, int g,
                                                            int m) {
  static_assert(NSTEP == 1 || (NSTEP == 2 && J0 % 2 == 0) || (NSTEP == 4 && J0 == 0), "step span");
  constexpr int NB = (NSTEP + 1) / 2;  // 32-element blocks spanned
  const uint32_t la = rec + (4 * g + 2 * m) * 32;
  const int T0 = rg * 16 + gm_sigma(g);
  const uint32_t row0 = tile + (T0 >> 3) * 1024 + (T0 & 7) * 128;
  const uint32_t row1 = row0 + 1024;
  const uint32_t ph = (uint32_t)(T0 & 7);
  // E8M0 scales [g][b][h]: rows g (h = 0) and g + 8 (h = 1) of each spanned block
  uint32_t s0hb[NB], s1hb[NB];
#pragma unroll
  for (int b = 0; b < NB; ++b) {
    const int byte = (g * 2 + (J0 >> 1) + b) * 2;
    const uint32_t sw = lds32(rec + 1024 + (byte & ~3));
    uint32_t l0, l1;
    row_scale<FTMOE_MXFP4>((sw >> (8 * (byte & 3))) & 0xFFu, s0hb[b], l0);        // row g
    row_scale<FTMOE_MXFP4>((sw >> (8 * ((byte & 3) + 1))) & 0xFFu, s1hb[b], l1);  // row g + 8
  }
#pragma unroll
  for (int s = 0; s < NSTEP; ++s) {
    const int j = J0 + s;
    const uint32_t s0h = s0hb[(j >> 1) - (J0 >> 1)], s1h = s1hb[(j >> 1) - (J0 >> 1)];
    const uint2 A = lds64(la + 8 * j);        // (row g, row g + 8) elements 8m..8m+3
    const uint2 B = lds64(la + 32 + 8 * j);   // elements 8m+4..8m+7
    const uint32_t off = (((uint32_t)(2 * j + m)) ^ ph) * 16;
    uint32_t r0[4], r1[4];
    r0[0] = e4m3x2_to_bf16x2(prmt(A.x, 0u, 0x4140u));
    r0[1] = e4m3x2_to_bf16x2(prmt(A.x, 0u, 0x4342u));
    r0[2] = e4m3x2_to_bf16x2(prmt(B.x, 0u, 0x4140u));
    r0[3] = e4m3x2_to_bf16x2(prmt(B.x, 0u, 0x4342u));
    r1[0] = e4m3x2_to_bf16x2(prmt(A.y, 0u, 0x4140u));
    r1[1] = e4m3x2_to_bf16x2(prmt(A.y, 0u, 0x4342u));
    r1[2] = e4m3x2_to_bf16x2(prmt(B.y, 0u, 0x4140u));
    r1[3] = e4m3x2_to_bf16x2(prmt(B.y, 0u, 0x4342u));
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      __nv_bfloat162 v0 = __hmul2(*reinterpret_cast<const __nv_bfloat162*>(&r0[p]),
                                  *reinterpret_cast<const __nv_bfloat162*>(&s0h));
      __nv_bfloat162 v1 = __hmul2(*reinterpret_cast<const __nv_bfloat162*>(&r1[p]),
                                  *reinterpret_cast<const __nv_bfloat162*>(&s1h));
      r0[p] = *reinterpret_cast<const uint32_t*>(&v0);
      r1[p] = *reinterpret_cast<const uint32_t*>(&v1);
    }
    sts128(row0 + off, make_uint4(r0[0], r0[1], r0[2], r0[3]));
    sts128(row1 + off, make_uint4(r1[0], r1[1], r1[2], r1[3]));
  }
}

// Dispatch of the prefill converter on the format.
template <int QT, int NSTEP, int J0>
__device__ __forceinline__ void convert_record_operand(uint32_t rec, uint32_t tile, int rg, int g, int m) {
  if (QT == FTMOE_MXFP8) convert_record_swizzled_fp8<NSTEP, J0>(rec, tile, rg, g, m);
  else convert_record_swizzled<QT, NSTEP, J0>(rec, tile, rg, g, m);
}

// ---------------------------------------------------------------- decode GEMM A operand
// bf16x2 codes of elements (0, 1) and (2, 3) of a 4-element group from a word whose
// bytes hold the group's 4-bit codes in the order (e0, e2, e1, e3), one per low nibble:
// q - 8 for Q4_0 (the byte 0x43 above a code byte is bf16 128 + q; one bf16x2 subtract
// of 136), the E2M1 value for MXFP4.  Both are exact in bf16.
template <int QT>
__device__ __forceinline__ void decode_plain(uint32_t E, uint32_t& o0, uint32_t& o1) {
  if (QT == FTMOE_Q4_0) {
    const uint32_t K = 0x43434343u;
    const __nv_bfloat162 off = __floats2bfloat162_rn(136.0f, 136.0f);
    uint32_t t0 = prmt(E, K, 0x4240u), t1 = prmt(E, K, 0x4341u);
    const __nv_bfloat162 u0 = __hsub2(*reinterpret_cast<const __nv_bfloat162*>(&t0), off);
    const __nv_bfloat162 u1 = __hsub2(*reinterpret_cast<const __nv_bfloat162*>(&t1), off);
    o0 = *reinterpret_cast<const uint32_t*>(&u0);
    o1 = *reinterpret_cast<const uint32_t*>(&u1);
  } else {
    const uint32_t TWO126 = 0x7E807E80u;
    const uint32_t v[2] = {prmt(E, 0u, 0x4240u), prmt(E, 0u, 0x4341u)};  // 0x000c000c pairs
    uint32_t r[2];
#pragma unroll
    for (int p = 0; p < 2; ++p) {
      // ((c & 7) << 6) | ((c & 8) << 12) read as bf16 is E2M1(c) * 2^-126 (the E2M1
      // subnormal lands on a bf16 subnormal); one bf16 multiply by 2^126 makes it exact
      uint32_t t = ((v[p] & 0x00070007u) << 6) | ((v[p] & 0x00080008u) << 12);
      const __nv_bfloat162 w = __hmul2(*reinterpret_cast<const __nv_bfloat162*>(&t),
                                       *reinterpret_cast<const __nv_bfloat162*>(&TWO126));
      r[p] = *reinterpret_cast<const uint32_t*>(&w);
    }
    o0 = r[0];
    o1 = r[1];
  }
}

}  // namespace ftmoe
