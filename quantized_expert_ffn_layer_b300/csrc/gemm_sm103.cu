// Grouped expert FFN on the 5th-generation tensor cores (tcgen05) for many rows per
// expert (prefill): the ExpertFFN of the FreeToken architecture walkthrough §五 on
// its GGUF Q4_0 / MXFP4 banks, with the block decode of §六 fused into the operand
// staging.
//
// One persistent CTA per SM.  A work item is (expert, 128 feature rows x 2 tiles,
// up to 256 of the expert's token rows): for gate/up the two tiles are the gate and
// the up rows of the same 128 features, for down two consecutive 128-row tiles of
// the output.  Per 64-element reduction block:
//   * 8 producer warps decode the 4-bit weight records straight from HBM into exact
//     bf16 (round-to-nearest-even of the decoded value) and gather the token rows,
//     writing both into the 128-byte-swizzled K-major shared-memory layout that
//     the MMA descriptors read (3-stage ring, mbarrier full/empty);
//   * one thread issues tcgen05.mma kind::f16 (M = 128 weight rows, N = the token
//     count rounded up to 16, K = 16) into two fp32 accumulators in tensor memory
//     (columns [0, 256) and [256, 512)) and commits each stage back to the
//     producers;
//   * 4 epilogue warps read the accumulators with tcgen05.ld and write
//     h = silu(gate) * up (gate/up) or y (down) as bf16.
// The weights are the A operand (M) and the tokens the B operand (N), so a small
// expert costs a narrow MMA rather than a mostly empty 128-row tile.  Items are
// ordered expert by expert with the token tile innermost, so CTAs that run at the
// same time share weight tiles through L2.
#include "common.cuh"
#include "internal.h"
#include "pipeline.cuh"
#include "tcgen05.cuh"

namespace ftmoe {

constexpr int GM_TOK = 256;         // token rows per item (largest MMA N)
constexpr int GM_ROWS = 128;        // weight rows per tile (MMA M)
constexpr int GM_NS = 3;            // pipeline stages
constexpr int GM_EPI_WARPS = 4;     // warps 0..3 (one per TMEM lane quarter)
constexpr int GM_MMA_WARP = 4;      // TMEM owner; lane 0 issues the MMAs
constexpr int GM_PROD0 = 5;         // first producer warp
constexpr int GM_PROD_WARPS = 8;
constexpr int GM_PROD_THREADS = GM_PROD_WARPS * 32;
constexpr int GM_THREADS = (GM_PROD0 + GM_PROD_WARPS) * 32;  // 416
constexpr uint32_t GM_TMEM_COLS = 512;
constexpr int GM_A_TILE = GM_ROWS * 128;           // 16 KB of bf16 (128 rows x 64)
constexpr int GM_B_TILE = GM_TOK * 128;            // 32 KB of bf16 (256 rows x 64)
constexpr int GM_STAGE = 2 * GM_A_TILE + GM_B_TILE;
constexpr int GM_MAX_E = 1024;

struct GemmTail {
  uint64_t full[GM_NS], empty[GM_NS];
  uint64_t acc_full, acc_empty, drain;
  uint32_t tmem_base;
  int abort_flag;
  int citem[GM_MAX_E + 1];  // exclusive prefix of items per expert
};
constexpr size_t GM_SMEM = 1024 + (size_t)GM_NS * GM_STAGE + sizeof(GemmTail);

struct GemmArgs {
  const int32_t* offsets;
  const int32_t* sorted_pair;  // gate/up: pair of each permuted row (nullptr: identity)
  int k, E;
  const uint16_t* act;  // gate/up: x [T][H]; down: h [P][I]
  int act_ld;
  uint16_t* out;        // gate/up: h [P][I]; down: y_perm [P][H]
  int out_ld;
  const uint8_t* wbase;  // tiles of this projection for expert 0
  long long wstride;     // bytes between experts
  long long table_off;   // offset of this projection inside a blob
  int S;                 // 64-element reduction blocks (records per 16-row group)
  int K;                 // reduction length
  int nrows;             // output rows of the projection's result: I or H
  int up_row0;           // gate/up: first up row of w13 (= I)
  int ft_per_expert;     // feature items per token tile
  int* status;
};

struct GmNoTable {
  __device__ __forceinline__ const uint8_t* get(int e, const GemmArgs& a) const {
    return a.wbase + (long long)e * a.wstride;
  }
};
struct GmWithTable {
  ExpertTable t;
  __device__ __forceinline__ const uint8_t* get(int e, const GemmArgs& a) const {
    return t.p[e] + a.table_off;
  }
};

struct GmItem {
  int e, r0, n, f0;
};

template <int MODE>
__device__ __forceinline__ GmItem gm_item(int i, const GemmArgs& a, const int* citem) {
  int lo = 0, hi = a.E;  // largest e with citem[e] <= i (that expert has items)
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (citem[mid] <= i) lo = mid; else hi = mid;
  }
  GmItem it;
  it.e = lo;
  const int local = i - citem[lo];
  const int beg = a.offsets[lo], ne = a.offsets[lo + 1] - beg;
  const int ntt = (ne + GM_TOK - 1) / GM_TOK;
  const int ft = local / ntt, tt = local - ft * ntt;
  it.r0 = beg + tt * GM_TOK;
  it.n = min(GM_TOK, ne - tt * GM_TOK);
  it.f0 = MODE == 0 ? ft * GM_ROWS : ft * 2 * GM_ROWS;
  return it;
}

// ---------------------------------------------------------------- weight decode
// W holds 8 four-bit codes of one row as nibble slots (0,4,2,6,1,5,3,7) = elements
// 0..7; slots p and p + 4 form the bf16x2 pair p.  Returns the 8 bf16 in element
// order.  Q4_0: (q - 8) * d rounded once to bf16, with d = dhi + dlo split so that
// (q - 8) * dlo is exact and the fused multiply-add rounds the exact product.
// MXFP4: E2M1 value times 2^(e - 127), exact unless it leaves the bf16 range.
template <int QT>
__device__ __forceinline__ uint4 decode8(uint32_t W, uint32_t s_hi, uint32_t s_lo) {
  uint32_t r[4];
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    const uint32_t v = (W >> (4 * p)) & 0x000F000Fu;
    if (QT == FTMOE_Q4_0) {
      uint32_t t = v | 0x43004300u;  // bf16 128 + q
      const __nv_bfloat162 off = __floats2bfloat162_rn(136.0f, 136.0f);
      const __nv_bfloat162 u = __hsub2(*reinterpret_cast<__nv_bfloat162*>(&t), off);  // q - 8
      const __nv_bfloat162 lo = __hmul2(u, *reinterpret_cast<const __nv_bfloat162*>(&s_lo));
      const __nv_bfloat162 w = __hfma2(u, *reinterpret_cast<const __nv_bfloat162*>(&s_hi), lo);
      r[p] = *reinterpret_cast<const uint32_t*>(&w);
    } else {
      uint32_t t = ((v & 0x00070007u) << 6) | ((v & 0x00080008u) << 12);  // E2M1 * 2^-126
      const uint32_t TWO126 = 0x7E807E80u;
      __nv_bfloat162 w = __hmul2(*reinterpret_cast<__nv_bfloat162*>(&t),
                                 *reinterpret_cast<const __nv_bfloat162*>(&TWO126));
      w = __hmul2(w, *reinterpret_cast<const __nv_bfloat162*>(&s_hi));
      r[p] = *reinterpret_cast<const uint32_t*>(&w);
    }
  }
  return make_uint4(r[0], r[2], r[1], r[3]);
}

// fp16 scale -> (hi, lo) bf16x2 pairs with hi + lo == d exactly.
__device__ __forceinline__ void split_scale(uint32_t h16, uint32_t& hi2, uint32_t& lo2) {
  const float d = half_bits_to_f32(h16);
  const uint32_t hi = f32_to_bf16_bits(d);
  const uint32_t lo = f32_to_bf16_bits(d - bf16_bits_to_f32(hi));
  hi2 = hi | (hi << 16);
  lo2 = lo | (lo << 16);
}

__device__ __forceinline__ uint32_t e8m0_bf16x2(uint32_t e) {
  const uint32_t b = e == 0 ? 0x0040u : (e == 255 ? 0x7FC0u : (e << 7));
  return b | (b << 16);
}

__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ void sts128(uint32_t saddr, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(saddr), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

// Permutes the four words so that w[s] becomes the old w[s ^ h] (h = 0..3).
__device__ __forceinline__ void xperm4(uint32_t (&w)[4], int h) {
  if (h & 1) {
    uint32_t t = w[0]; w[0] = w[1]; w[1] = t;
    t = w[2]; w[2] = w[3]; w[3] = t;
  }
  if (h & 2) {
    uint32_t t = w[0]; w[0] = w[2]; w[2] = t;
    t = w[1]; w[1] = w[3]; w[3] = t;
  }
}

// Per producer thread and stage: its share of one weight record (the 32 code bytes of
// lanes 4g + 2m and 4g + 2m + 1, i.e. 8 elements x 4 words of rows g and g + 8) plus
// the scales of those rows, and 8 token-row chunks of 16 bytes.
struct ProdData {
  uint4 ca, cb;
  uint2 sc;
  uint4 b[8];
  int rec_ok;      // the record lies inside the matrix
  uint32_t bmask;  // bit i: token chunk i exists
};

// Where the producer thread loads from for the stage (item, kb).
struct ProdCtx {
  int item, kb;
  int rec_ok;
  const uint8_t* rec0;  // this thread's record at kb = 0 (advance by kb * RB)
  int arow[8];          // act rows of this thread's 8 token chunks (-1: none)
};

template <int QT, int MODE, class Tab>
__device__ __forceinline__ void prod_ctx_item(ProdCtx& c, int item, const GemmArgs& a,
                                              const Tab& tab, const int* citem, int pt) {
  const GmItem it = gm_item<MODE>(item, a, citem);
  c.item = item;
  c.kb = 0;
  const int lane = pt & 31, pw = pt >> 5;
  const int ri = pw * 2 + (lane >> 4);  // record of the stage: tile ri / 8, row group ri % 8
  const int t = ri >> 3, rg = ri & 7;
  int row;  // first row of the 16-row group within the matrix
  if (MODE == 0) {
    row = it.f0 + rg * 16;
    c.rec_ok = row < a.nrows;
    if (t == 1) row += a.up_row0;
  } else {
    row = it.f0 + t * GM_ROWS + rg * 16;
    c.rec_ok = row < a.nrows;
  }
  constexpr int RB = rec_bytes(QT);
  c.rec0 = tab.get(it.e, a) + (long long)(row / 16) * a.S * RB;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int rr = (pt >> 3) + 32 * i;
    int ar = -1;
    if (rr < it.n) {
      if (MODE == 0) ar = a.sorted_pair ? a.sorted_pair[it.r0 + rr] / a.k : (it.r0 + rr);
      else ar = it.r0 + rr;
    }
    c.arow[i] = ar;
  }
}

template <int QT>
__device__ __forceinline__ void prod_load(const ProdCtx& c, const GemmArgs& a, int pt,
                                          ProdData& d) {
  constexpr int RB = rec_bytes(QT);
  const int lane = pt & 31;
  const int g = (lane & 15) >> 1, m = lane & 1;
  d.rec_ok = c.rec_ok;
  if (c.rec_ok) {
    const uint8_t* rec = c.rec0 + (long long)c.kb * RB;
    d.ca = ldg_stream(rec + (4 * g + 2 * m) * 16);
    d.cb = ldg_stream(rec + (4 * g + 2 * m + 1) * 16);
    if (QT == FTMOE_Q4_0) {
      d.sc = __ldg(reinterpret_cast<const uint2*>(rec + REC_CODE_BYTES + g * 8));
    } else {
      d.sc.x = __ldg(reinterpret_cast<const uint32_t*>(rec + REC_CODE_BYTES + g * 4));
      d.sc.y = 0;
    }
  }
  const int col = c.kb * 64 + 8 * (pt & 7);
  const bool kok = col < a.K;
  uint32_t mask = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    if (c.arow[i] >= 0) {
      mask |= 1u << i;
      const uint16_t* p = a.act + (long long)c.arow[i] * a.act_ld + col;
      d.b[i] = kok ? __ldg(reinterpret_cast<const uint4*>(p)) : make_uint4(0, 0, 0, 0);
    }
  }
  d.bmask = mask;
}

template <int QT>
__device__ __forceinline__ void prod_store(const ProdData& d, int pt, uint32_t stage_addr) {
  const int lane = pt & 31, pw = pt >> 5;
  if (d.rec_ok) {
    const int ri = pw * 2 + (lane >> 4);
    const int t = ri >> 3, rg = ri & 7;
    const int g = (lane & 15) >> 1, m = lane & 1;
    // scales of rows g (h = 0) and g + 8 (h = 1) for blocks b = 0, 1
    uint32_t shi[2][2], slo[2][2];
    if (QT == FTMOE_Q4_0) {
      split_scale(d.sc.x & 0xFFFFu, shi[0][0], slo[0][0]);
      split_scale(d.sc.x >> 16, shi[0][1], slo[0][1]);
      split_scale(d.sc.y & 0xFFFFu, shi[1][0], slo[1][0]);
      split_scale(d.sc.y >> 16, shi[1][1], slo[1][1]);
    } else {
#pragma unroll
      for (int b = 0; b < 2; ++b)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          shi[b][h] = e8m0_bf16x2((d.sc.x >> (8 * (2 * b + h))) & 0xFFu);
          slo[b][h] = 0;
        }
    }
    uint32_t wa[4] = {d.ca.x, d.ca.y, d.ca.z, d.ca.w};
    uint32_t wb[4] = {d.cb.x, d.cb.y, d.cb.z, d.cb.w};
    // step s handles word j = s ^ h(g): with the row swizzle (chunk ^ g) this puts the
    // 8 lanes of each quarter-warp on 8 different 16-byte bank groups
    const int hx = (((g >> 1) & 1) << 1) | ((g ^ (g >> 1)) & 1);
    xperm4(wa, hx);
    xperm4(wb, hx);
    const uint32_t tile = stage_addr + t * GM_A_TILE;
    const uint32_t row0 = tile + (2 * rg) * 1024 + g * 128;  // row rg*16 + g
    const uint32_t row1 = row0 + 1024;                       // row rg*16 + g + 8
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      const int j = s ^ hx;
      const int b = j >> 1;
      const uint32_t A = wa[s], B = wb[s];
      const uint32_t wg = (A & 0x0F0F0F0Fu) | ((B & 0x0F0F0F0Fu) << 4);
      const uint32_t wg8 = ((A >> 4) & 0x0F0F0F0Fu) | (B & 0xF0F0F0F0u);
      const uint32_t sh0 = b ? shi[1][0] : shi[0][0], sl0 = b ? slo[1][0] : slo[0][0];
      const uint32_t sh1 = b ? shi[1][1] : shi[0][1], sl1 = b ? slo[1][1] : slo[0][1];
      const uint32_t cp = 2 * j + m;
      const uint32_t off = ((cp ^ (uint32_t)g) * 16);
      sts128(row0 + off, decode8<QT>(wg, sh0, sl0));
      sts128(row1 + off, decode8<QT>(wg8, sh1, sl1));
    }
  }
  const uint32_t btile = stage_addr + 2 * GM_A_TILE;
  const int ch = pt & 7;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    if (d.bmask & (1u << i)) {
      const int rr = (pt >> 3) + 32 * i;
      sts128(btile + (rr >> 3) * 1024 + (rr & 7) * 128 + ((ch ^ (rr & 7)) * 16), d.b[i]);
    }
  }
}

template <int QT, int MODE, class Tab>
__global__ void __launch_bounds__(GM_THREADS, 1) gemm_ffn_kernel(const GemmArgs a,
                                                               const __grid_constant__ Tab tab) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t base_addr = (raw_addr + 1023u) & ~1023u;
  uint8_t* base = smem_raw + (base_addr - raw_addr);
  GemmTail& tl = *reinterpret_cast<GemmTail*>(base + (size_t)GM_NS * GM_STAGE);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  volatile int* abort_flag = &tl.abort_flag;

  if (tid == 0) {
    for (int s = 0; s < GM_NS; ++s) {
      mbar_init(&tl.full[s], GM_PROD_THREADS);
      mbar_init(&tl.empty[s], 1);
    }
    mbar_init(&tl.acc_full, 1);
    mbar_init(&tl.acc_empty, GM_EPI_WARPS * 32);
    mbar_init(&tl.drain, 1);
    tl.abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == GM_MMA_WARP) {
    tmem_alloc(&tl.tmem_base, GM_TMEM_COLS);
    tmem_relinquish();
  }
  // items per expert: ceil(n_e / 256) token tiles x feature items
  if (warp == 0) {
    int carry = 0;
    for (int e0 = 0; e0 < a.E; e0 += 32) {
      const int e = e0 + lane;
      int v = 0;
      if (e < a.E) v = ((a.offsets[e + 1] - a.offsets[e] + GM_TOK - 1) / GM_TOK) * a.ft_per_expert;
      int x = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      if (e < a.E) tl.citem[e] = carry + x - v;
      carry += __shfl_sync(0xffffffffu, x, 31);
    }
    if (lane == 0) tl.citem[a.E] = carry;
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = tl.tmem_base;
  const int nitems = tl.citem[a.E];
  const int G = gridDim.x;

  if (warp >= GM_PROD0) {
    // ------------------------------------------------------------ producers
    const int pt = tid - GM_PROD0 * 32;
    ProdCtx c;
    int slot = 0;
    uint32_t phase = 0;
    if (blockIdx.x < nitems) {
      prod_ctx_item<QT, MODE>(c, blockIdx.x, a, tab, tl.citem, pt);
      ProdData dc;
      prod_load<QT>(c, a, pt, dc);
      for (;;) {
        // advance to the next stage: next block of the item, or the CTA's next item
        bool have_next = true;
        if (c.kb + 1 < a.S) {
          ++c.kb;
        } else if (c.item + G < nitems) {
          prod_ctx_item<QT, MODE>(c, c.item + G, a, tab, tl.citem, pt);
        } else {
          have_next = false;
        }
        ProdData dn;
        if (have_next) prod_load<QT>(c, a, pt, dn);
        if (!mbar_wait_or_abort(&tl.empty[slot], phase ^ 1u, abort_flag, a.status)) break;
        prod_store<QT>(dc, pt, base_addr + slot * GM_STAGE);
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        mbar_arrive(&tl.full[slot]);
        if (++slot == GM_NS) { slot = 0; phase ^= 1u; }
        if (!have_next) break;
        dc = dn;
      }
    }
  } else if (warp == GM_MMA_WARP) {
    // ------------------------------------------------------------ MMA issue
    if (lane == 0) {
      int slot = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      for (int i = blockIdx.x; i < nitems && ok; i += G) {
        const GmItem it = gm_item<MODE>(i, a, tl.citem);
        const int N = max(16, (it.n + 15) & ~15);
        const uint32_t idesc = idesc_bf16_f32(GM_ROWS, N);
        if (!mbar_wait_or_abort(&tl.acc_empty, acc_phase ^ 1u, abort_flag, a.status)) break;
        tc_fence_after_sync();
        for (int kb = 0; kb < a.S; ++kb) {
          if (!mbar_wait_or_abort(&tl.full[slot], phase, abort_flag, a.status)) { ok = false; break; }
          tc_fence_after_sync();
          const uint32_t sa = base_addr + slot * GM_STAGE;
#pragma unroll
          for (int k16 = 0; k16 < 4; ++k16) {
            const uint64_t bd = sdesc_kmajor_sw128(sa + 2 * GM_A_TILE + 32 * k16);
            const uint32_t acc = (kb | k16) ? 1u : 0u;
            mma_bf16(tmem, sdesc_kmajor_sw128(sa + 32 * k16), bd, idesc, acc);
            mma_bf16(tmem + 256, sdesc_kmajor_sw128(sa + GM_A_TILE + 32 * k16), bd, idesc, acc);
          }
          mma_commit(&tl.empty[slot]);
          if (++slot == GM_NS) { slot = 0; phase ^= 1u; }
        }
        if (!ok) break;
        mma_commit(&tl.acc_full);
        acc_phase ^= 1u;
      }
      // every MMA issued above has finished once this arrives
      mma_commit(&tl.drain);
      mbar_wait_or_abort(&tl.drain, 0, abort_flag, a.status, 100000000ull);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue (warps 0..3)
    const int q = warp;  // TMEM lanes [32q, 32q + 32)
    const int m = 32 * q + lane;
    uint32_t acc_phase = 0;
    for (int i = blockIdx.x; i < nitems; i += G) {
      const GmItem it = gm_item<MODE>(i, a, tl.citem);
      if (!mbar_wait_or_abort(&tl.acc_full, acc_phase, abort_flag, a.status)) break;
      acc_phase ^= 1u;
      tc_fence_after_sync();
      const uint32_t lane_base = tmem + ((uint32_t)(32 * q) << 16);
      if (MODE == 0) {
        const int fi = it.f0 + m;
        const bool ok = fi < a.nrows;
        for (int c0 = 0; c0 < it.n; c0 += 32) {
          uint32_t gv[32], uv[32];
          tmem_ld32(lane_base + c0, gv);
          tmem_ld32(lane_base + 256 + c0, uv);
          tmem_wait_ld();
          if (ok) {
            uint16_t* o = a.out + (long long)(it.r0 + c0) * a.out_ld + fi;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              if (c0 + j < it.n) {
                const float g = __uint_as_float(gv[j]), u = __uint_as_float(uv[j]);
                o[(long long)j * a.out_ld] = f32_to_bf16_bits(silu_f32(g) * u);
              }
            }
          }
        }
      } else {
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          const int fi = it.f0 + t * GM_ROWS + m;
          const bool ok = fi < a.nrows;
          for (int c0 = 0; c0 < it.n; c0 += 32) {
            uint32_t yv[32];
            tmem_ld32(lane_base + 256 * t + c0, yv);
            tmem_wait_ld();
            if (ok) {
              uint16_t* o = a.out + (long long)(it.r0 + c0) * a.out_ld + fi;
#pragma unroll
              for (int j = 0; j < 32; ++j)
                if (c0 + j < it.n) o[(long long)j * a.out_ld] = f32_to_bf16_bits(__uint_as_float(yv[j]));
            }
          }
        }
      }
      tc_fence_before_sync();
      mbar_arrive(&tl.acc_empty);
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == GM_MMA_WARP) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, GM_TMEM_COLS);
  }
}

size_t ffn_gemm_ws_bytes(int, int, int, int, int) { return 0; }

template <int QT, int MODE, class Tab>
static cudaError_t gm_launch(const GemmArgs& a, const Tab& tab, cudaStream_t st) {
  const DeviceInfo* di = device_info();
  if (!di) return cudaErrorUnknown;
  auto kern = gemm_ffn_kernel<QT, MODE, Tab>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)GM_SMEM);
  if (err != cudaSuccess) return err;
  kern<<<di->sm_count, GM_THREADS, GM_SMEM, st>>>(a, tab);
  return cudaGetLastError();
}

template <int QT, class Tab>
static cudaError_t gm_launch_qt(const FfnProblem& pb, const Tab& tab, cudaStream_t st) {
  const DeviceInfo* di = device_info();
  if (!di) return cudaErrorUnknown;
  GemmArgs a{};
  a.offsets = pb.offsets;
  a.sorted_pair = pb.sorted_pair;
  a.k = pb.k;
  a.E = pb.E;
  a.status = di->status;
  a.act = pb.x;
  a.act_ld = pb.H;
  a.out = pb.h_act;
  a.out_ld = pb.I;
  a.wbase = pb.w13;
  a.wstride = (long long)pb.w13_bytes;
  a.table_off = 0;
  a.S = slabs_of(pb.H);
  a.K = pb.H;
  a.nrows = pb.I;
  a.up_row0 = pb.I;
  a.ft_per_expert = (pb.I + GM_ROWS - 1) / GM_ROWS;
  GemmArgs d = a;
  d.act = pb.h_act;
  d.act_ld = pb.I;
  d.out = pb.y_perm;
  d.out_ld = pb.H;
  d.wbase = pb.w2;
  d.wstride = (long long)tiles_bytes_per_expert(pb.qtype, pb.H, pb.I);
  d.table_off = (long long)pb.w13_bytes;
  d.S = slabs_of(pb.I);
  d.K = pb.I;
  d.nrows = pb.H;
  d.up_row0 = 0;
  d.ft_per_expert = (pb.H + 2 * GM_ROWS - 1) / (2 * GM_ROWS);
  cudaError_t err = gm_launch<QT, 0>(a, tab, st);
  if (err != cudaSuccess) return err;
  return gm_launch<QT, 1>(d, tab, st);
}

cudaError_t launch_ffn_gemm(const FfnProblem& pb, void*, size_t, cudaStream_t st) {
  if (pb.E > GM_MAX_E) return cudaErrorNotSupported;
  if (pb.table) {
    GmWithTable t;
    t.t = *pb.table;
    return pb.qtype == FTMOE_Q4_0 ? gm_launch_qt<FTMOE_Q4_0>(pb, t, st)
                                  : gm_launch_qt<FTMOE_MXFP4>(pb, t, st);
  }
  GmNoTable t;
  return pb.qtype == FTMOE_Q4_0 ? gm_launch_qt<FTMOE_Q4_0>(pb, t, st)
                                : gm_launch_qt<FTMOE_MXFP4>(pb, t, st);
}

}  // namespace ftmoe
