// Shared device helpers for libftmoe (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "ftmoe.h"

namespace ftmoe {

// Bounds-checking build (FTMOE_CHECKS=1, libftmoe_checks.so): the FFN and combine kernels
// check every index they take from offsets / sorted_pair / inv_pos and report a bad one.
#ifndef FTMOE_CHECKS
#define FTMOE_CHECKS 0
#endif

// Device status word: kernels OR a code in here instead of trapping.
enum DeviceCode : int {
  DEV_OK = 0,
  DEV_BAD_EXPERT_ID = 1,      // permute saw an id outside [0, E)
  DEV_WAIT_TIMEOUT = 2,       // a bounded mbarrier / flag wait ran out
  DEV_BAD_SHAPE = 4,          // a kernel saw sizes it cannot handle
  DEV_BAD_INDEX = 8,          // (checks build) an offsets / sorted_pair / inv_pos entry out of range
};

// Every kernel that can detect a problem gets a pointer to the per-device status word.
__device__ __forceinline__ void set_device_code(int* status, int code) {
  if (status) atomicOr(status, code);
}

// Rows [r0, r0 + n) of expert e in permuted order.  The checks build clamps the range to
// [0, P) (a decreasing or out-of-range offsets entry is reported and its rows dropped).
__device__ __forceinline__ void expert_rows(const int32_t* offsets, int e, int P, int* status, int& r0,
                                            int& n) {
  r0 = offsets[e];
  int r1 = offsets[e + 1];
#if FTMOE_CHECKS
  if (r0 < 0 || r1 < r0 || r1 > P) {
    set_device_code(status, DEV_BAD_INDEX);
    r0 = min(max(r0, 0), P);
    r1 = min(max(r1, r0), P);
  }
#endif
  n = r1 - r0;
}

// Token of permuted row r: sorted_pair[r] / k (row r itself without a pair table).  The
// checks build reports a pair outside [0, T k) and reads token 0 instead.
__device__ __forceinline__ int row_token(const int32_t* sorted_pair, int r, int k, int T, int* status) {
  if (!sorted_pair) return r;
  const int p = sorted_pair[r];
#if FTMOE_CHECKS
  if (p < 0 || p >= T * k) {
    set_device_code(status, DEV_BAD_INDEX);
    return 0;
  }
#endif
  return p / k;
}

// ---------------------------------------------------------------- tiled weight format
// One record = 16 rows x 64 reduction elements: 512 code bytes (32 lanes x 16 B)
// followed by the 32 block scales of its 16 rows x 2 blocks, ordered
// [g (0..7)][block b (0..1)][row half h (0..1)] (row = g + 8h).
//
// Lane L = 4g + c holds, in word j (0..3) of its 16 bytes, the codes of rows
// g and g+8 at slab positions 16j + 4c + r (r = 0..3), laid out so that the
// pair (nibble at bit 4p, nibble at bit 16 + 4p) is one bf16x2 operand:
//   p = 0: (row g,   r=0 | r=1)     p = 1: (row g+8, r=0 | r=1)
//   p = 2: (row g,   r=2 | r=3)     p = 3: (row g+8, r=2 | r=3)
// Words j = 0, 1 lie in block 0 of the slab and j = 2, 3 in block 1, so each
// 16-element k-step of an m16n8k16 MMA stays inside one quantization block.
//
// NVFP4 records use the MXFP4 code layout (E2M1 nibbles) with 64 scale bytes: one E4M3
// scale per 16-element block, ordered [g (0..7)][block b (0..3)][row half h (0..1)].
// An NVFP4 expert matrix's records are followed by a 16-byte trailer holding its fp32
// tensor scale (then 12 zero bytes).
//
// MXFP8 records hold 1024 element bytes: lane L = 4g + c owns 32 of them, in word 2j the
// E4M3 bytes of elements 16j + 4c .. +3 of row g and in word 2j + 1 those of row g + 8;
// then the 32 E8M0 scales ordered as for MXFP4.
constexpr int REC_CODE_BYTES = 512;
__host__ __device__ constexpr int rec_code_bytes(int qtype) { return qtype == FTMOE_MXFP8 ? 1024 : 512; }
__host__ __device__ constexpr int rec_bytes(int qtype) {
  // Q4_0: 64 B of fp16 scales; MXFP4: 32 E8M0 bytes; NVFP4: 64 E4M3 bytes; MXFP8: 32 E8M0
  return qtype == FTMOE_MXFP4 ? 544 : (qtype == FTMOE_MXFP8 ? 1056 : 576);
}
__host__ __device__ constexpr int canon_block_bytes(int qtype) {
  return qtype == FTMOE_Q4_0 ? 18 : (qtype == FTMOE_MXFP4 ? 17 : (qtype == FTMOE_NVFP4 ? 9 : 33));
}
__host__ __device__ constexpr int canon_block_elems(int qtype) { return qtype == FTMOE_NVFP4 ? 16 : 32; }
constexpr int NVFP4_TRAILER = 16;
__host__ __device__ inline int slabs_of(int K) { return (K + 63) / 64; }
__host__ __device__ inline size_t records_bytes_per_expert(int qtype, int N, int K) {
  return (size_t)(N / 16) * slabs_of(K) * rec_bytes(qtype);
}
__host__ __device__ inline size_t tiles_bytes_per_expert(int qtype, int N, int K) {
  return records_bytes_per_expert(qtype, N, K) + (qtype == FTMOE_NVFP4 ? NVFP4_TRAILER : 0);
}

// Q4_0 word -> four bf16x2 of (q - 8), exact.
__device__ __forceinline__ void q4_word_to_bf16x2(uint32_t w, uint32_t (&a)[4]) {
  const uint32_t MAGIC = 0x43004300u;  // bf16 128.0 | 128.0
  const __nv_bfloat162 off = __floats2bfloat162_rn(136.0f, 136.0f);
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    uint32_t t = ((w >> (4 * p)) & 0x000F000Fu) | MAGIC;  // 128 + q
    __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162*>(&t);
    v = __hsub2(v, off);
    a[p] = *reinterpret_cast<uint32_t*>(&v);
  }
}

// MXFP4 word -> four bf16x2 of the E2M1 values, exact.
// ((c & 7) << 6) | ((c & 8) << 12) read as bf16 is E2M1(c) * 2^-126 (code 1, the
// E2M1 subnormal, lands on the bf16 subnormal 2^-127); one bf16 multiply by
// 2^126 (bf16 arithmetic keeps subnormal inputs) makes it E2M1(c) exactly.
__device__ __forceinline__ void e2m1_word_to_bf16x2(uint32_t w, uint32_t (&a)[4]) {
  const uint32_t TWO126 = 0x7E807E80u;
  const __nv_bfloat162 s = *reinterpret_cast<const __nv_bfloat162*>(&TWO126);
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    uint32_t mag, sgn;
    const int sh_m = 6 - 4 * p, sh_s = 12 - 4 * p;
    mag = (sh_m >= 0 ? (w << sh_m) : (w >> (-sh_m))) & 0x01C001C0u;
    sgn = (w << sh_s) & 0x80008000u;
    uint32_t t = mag | sgn;
    __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162*>(&t);
    v = __hmul2(v, s);
    a[p] = *reinterpret_cast<uint32_t*>(&v);
  }
}

// E8M0 scale byte -> 2^(e - 127) as fp32 (e = 0 gives the subnormal 2^-127; 255 -> NaN).
__device__ __forceinline__ float e8m0_to_f32(uint32_t e) {
  if (e == 0) return __int_as_float(0x00400000);
  if (e == 255) return __int_as_float(0x7FC00000);
  return __int_as_float((int)(e << 23));
}

// E4M3 byte (sign, 4 exponent bits with bias 7, 3 mantissa bits; S.1111.111 is NaN) -> its
// value as fp32, exact: the 7 magnitude bits placed at fp32 bit 20 read as 2^-120 times
// the value (also for E4M3 subnormals, which land on fp32 subnormals), times 2^120.
__device__ __forceinline__ float e4m3_to_f32(uint32_t b) {
  const uint32_t m = b & 0x7Fu;
  if (m == 0x7Fu) return __int_as_float(0x7FC00000);
  const float v = __uint_as_float(m << 20) * 0x1p120f;
  return (b & 0x80u) ? -v : v;
}

// Two E4M3 bytes held in the low byte of each 16-bit half of p (p = b1 << 16 | b0) ->
// bf16x2 of their values (b0 in the low half): the 7 magnitude bits placed at bf16 bit 4
// read as 2^-120 times the value (E4M3 subnormals land on bf16 subnormals) and one bf16
// multiply by 2^120 makes it exact for every finite code.  The NaN code S.1111.111 is
// not special-cased here (it reads as +-480); weight banks hold finite codes.
__device__ __forceinline__ uint32_t e4m3x2_to_bf16x2(uint32_t p) {
  uint32_t t = ((p & 0x007F007Fu) << 4) | ((p & 0x00800080u) << 8);
  const uint32_t TWO120 = 0x7B807B80u;
  const __nv_bfloat162 v = __hmul2(*reinterpret_cast<const __nv_bfloat162*>(&t),
                                   *reinterpret_cast<const __nv_bfloat162*>(&TWO120));
  return *reinterpret_cast<const uint32_t*>(&v);
}

__device__ __forceinline__ float half_bits_to_f32(uint32_t h) {
  return __half2float(__ushort_as_half((unsigned short)h));
}

// Q4_0 word -> four bf16x2 of the biased code 128 + q (exact), one bit operation per pair:
// the nibble lands in the low mantissa bits of bf16 128.  A product sum over these
// equals the sum over (q - 8) plus 136 times the sum of the other operand, which the
// caller removes (see gemv.cu).
__device__ __forceinline__ void q4_word_to_biased_bf16x2(uint32_t w, uint32_t (&a)[4]) {
#pragma unroll
  for (int p = 0; p < 4; ++p) a[p] = ((w >> (4 * p)) & 0x000F000Fu) | 0x43004300u;
}

// acc0 += s * p0, acc1 += s * p1 as one packed fp32x2 fused multiply-add (sm_100+), each
// lane rounded once like fmaf.
__device__ __forceinline__ void ffma2(float& acc0, float& acc1, float s, float p0, float p1) {
  asm("{\n .reg .b64 a, b, c;\n mov.b64 a, {%0,%1};\n mov.b64 b, {%2,%2};\n mov.b64 c, {%3,%4};\n"
      " fma.rn.f32x2 a, b, c, a;\n mov.b64 {%0,%1}, a;\n}\n"
      : "+f"(acc0), "+f"(acc1)
      : "f"(s), "f"(p0), "f"(p1));
}

// ---------------------------------------------------------------- mma.sync helper
// D(16x8, fp32) += A(16x16 bf16, row) * B(16x8 bf16, col)
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                          uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// D = A * B + C with a separate accumulator input.
__device__ __forceinline__ void mma_16816_c(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                            uint32_t b1, const float (&c)[4]) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%10,%11,%12,%13};\n"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]), "f"(c[2]),
        "f"(c[3]));
}

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t b) { return __uint_as_float(b << 16); }

__device__ __forceinline__ uint16_t f32_to_bf16_bits(float f) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

__device__ __forceinline__ float silu_f32(float g) { return g / (1.0f + __expf(-g)); }

// Programmatic dependent launch: wait for the previous grid's memory / let the next start.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

}  // namespace ftmoe
