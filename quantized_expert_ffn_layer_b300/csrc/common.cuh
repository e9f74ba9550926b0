// Shared device helpers for libftmoe (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "ftmoe.h"

namespace ftmoe {

// Device status word: kernels OR a code in here instead of trapping.
enum DeviceCode : int {
  DEV_OK = 0,
  DEV_BAD_EXPERT_ID = 1,      // permute saw an id outside [0, E)
  DEV_WAIT_TIMEOUT = 2,       // a bounded mbarrier / flag wait ran out
  DEV_BAD_SHAPE = 4,          // a kernel saw sizes it cannot handle
};

// Every kernel that can detect a problem gets a pointer to the per-device status word.
__device__ __forceinline__ void set_device_code(int* status, int code) {
  if (status) atomicOr(status, code);
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
constexpr int REC_CODE_BYTES = 512;
__host__ __device__ constexpr int rec_bytes(int qtype) { return qtype == FTMOE_Q4_0 ? 576 : 544; }
__host__ __device__ constexpr int canon_block_bytes(int qtype) { return qtype == FTMOE_Q4_0 ? 18 : 17; }
__host__ __device__ inline int slabs_of(int K) { return (K + 63) / 64; }
__host__ __device__ inline size_t tiles_bytes_per_expert(int qtype, int N, int K) {
  return (size_t)(N / 16) * slabs_of(K) * rec_bytes(qtype);
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

__device__ __forceinline__ float half_bits_to_f32(uint32_t h) {
  return __half2float(__ushort_as_half((unsigned short)h));
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
