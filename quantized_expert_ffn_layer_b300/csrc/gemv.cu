// Grouped expert FFN for few rows per expert (decode): HBM-bound streaming of the
// 4-bit expert weights with in-register decode (the ExpertFFN of the FreeToken
// architecture walkthrough §五, on GGUF Q4_0 / MXFP4 banks, §六).
//
// Work item = (active expert, two 16-row tiles, a group of reduction parts): the
// gate and up tile of one group of 16 features (gate/up projection), or two tiles of
// 16 output rows (down projection).  Every warp owns its items outright: its lane 0
// streams the items' 16-row x 64-column weight records with 1-D bulk copies (TMA)
// into the warp's own ring of shared-memory stages, and the warp turns the codes
// into exact bf16 (q - 8, or the E2M1 value) as the A operand of m16n8k16 MMAs
// whose B operand (up to 8 token rows) is loaded into registers one stage ahead.
// After the two k-steps of a quantization block the partial sums are scaled by the
// block's scale in fp32, so the only roundings are the fp32 accumulation, the bf16
// h between the projections and the bf16 output.
//
// The reduction dimension is cut into fixed parts of 512 elements; each part is
// summed from zero and the parts are added in order.  For small batches the parts
// of one tile pair are spread over several warps, which write per-part sums to
// scratch; the last warp to arrive adds them in part order.  Either way the result
// is bit-identical, so a token's output does not depend on the batch it is in.
#include <cstddef>

#include "common.cuh"
#include "internal.h"
#include "operand.cuh"
#include "pipeline.cuh"

namespace ftmoe {

// Launch shape (overridable at build time for sweeps): warps per CTA, CTAs per SM,
// slabs (64 reduction elements) per stage, stages per warp.
#ifndef FTMOE_GW_WARPS
#define FTMOE_GW_WARPS 8
#endif
#ifndef FTMOE_GW_MINB
#define FTMOE_GW_MINB 2
#endif
#ifndef FTMOE_GW_SL
#define FTMOE_GW_SL 4
#endif
#ifndef FTMOE_GW_NS
#define FTMOE_GW_NS 2
#endif
// Q4_0 A operand: biased codes 128 + q with a shared correction MMA per block (1), or
// exact codes q - 8 through one bf16 subtract per pair (0).
#ifndef FTMOE_GW_BIASED
#define FTMOE_GW_BIASED 1
#endif
constexpr bool GW_BIASED = FTMOE_GW_BIASED != 0;
constexpr int GW_WARPS = FTMOE_GW_WARPS;
constexpr int GW_MINB = FTMOE_GW_MINB;
constexpr int GW_THREADS = GW_WARPS * 32;
constexpr int GW_SL = FTMOE_GW_SL;
constexpr int GW_NS = FTMOE_GW_NS;
// slabs per fixed reduction part (a multiple of the stage's slab count)
#ifndef FTMOE_GW_PS
#define FTMOE_GW_PS 8
#endif
constexpr int GW_PS = FTMOE_GW_PS;
static_assert(GW_PS % FTMOE_GW_SL == 0, "stages must not cross reduction parts");
constexpr int GW_KPMAX = 16;    // most warps sharing one tile pair

// Slabs per stage by format: MXFP8's records are twice as large, so its stages hold half
// as many and the per-warp rings stay the same size.
template <int QT>
__host__ __device__ constexpr int gw_sl() { return QT == FTMOE_MXFP8 ? (GW_SL > 1 ? GW_SL / 2 : 1) : GW_SL; }

template <int QT>
struct GwSmem {
  static constexpr int STAGE = 2 * gw_sl<QT>() * rec_bytes(QT);
  uint8_t stage[GW_WARPS][GW_NS][STAGE];
  uint64_t full[GW_WARPS][GW_NS];
  int16_t act[1024];
  int pref[1025];  // first item of each active expert (items = tile pairs x rounds x groups)
  int wsum[GW_WARPS];
  // split reductions (kp > 1): per warp group (GW_WARPS / kp of them) barriers "all parts
  // written" and "read", and each warp's per-part sums of its item (at most 2 parts),
  // last so that launches without a split leave that space to L1
  uint64_t gfull[GW_WARPS], gfree[GW_WARPS];
  float red[GW_WARPS][2][256];
};

struct GemvArgs {
  const int32_t* offsets;
  const int32_t* sorted_pair;  // nullptr: row r is token r (k == 1)
  int k, E, T, P;
  const uint16_t* act;  // gate/up: x [T][H]; down: h [P][I]
  int act_ld;
  uint16_t* out;        // gate/up: h [P][I]; down: y_perm [P][H]
  int out_ld;
  const uint8_t* wbase;  // tiles of this projection for expert 0
  long long wstride;     // bytes between experts
  long long table_off;   // offset of this projection inside a blob
  int S;                 // slabs per row
  int K;                 // reduction length
  int NP;                // fixed parts: ceil(S / GW_PS)
  int up_rt;             // gate/up: first row tile of the up half (I / 16)
  int units_per_expert;  // gate/up: I / 16; down: H / 32
  int kp;                // part groups (warps) per unit
  int qtype;
  long long rec_total;   // bytes of one expert's records of this projection (NVFP4 trailer offset)
  int* status;
};

struct NoTable {
  __device__ __forceinline__ const uint8_t* get(int e, const GemvArgs& a) const {
    return a.wbase + (long long)e * a.wstride;
  }
};
struct WithTable {
  ExpertTable t;
  __device__ __forceinline__ const uint8_t* get(int e, const GemvArgs& a) const {
    return t.p[e] + a.table_off;
  }
};

// Ordered list of experts with at least one row, built by every CTA from offsets, and the
// exclusive prefix of their work items: units_per_expert x rounds (of 8 rows) x kp groups
// each.  Returns the number of active experts; s_pref[nact] is the item total.
__device__ __forceinline__ int build_active_list(const int32_t* offsets, int E, int P, int* status,
                                                 int units_per_expert, int kp, int16_t* s_act,
                                                 int* s_pref, int* s_wsum) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  int nact = 0;
  for (int e0 = 0; e0 < E; e0 += GW_THREADS) {
    const int e = e0 + threadIdx.x;
    int r0 = 0, n = 0;
    if (e < E) expert_rows(offsets, e, P, status, r0, n);
    const bool f = n > 0;
    const unsigned b = __ballot_sync(0xffffffffu, f);
    if (lane == 0) s_wsum[wid] = __popc(b);
    __syncthreads();
    int before = nact, tot = 0;
#pragma unroll
    for (int w = 0; w < GW_WARPS; ++w) {
      if (w < wid) before += s_wsum[w];
      tot += s_wsum[w];
    }
    if (f) s_act[before + __popc(b & ((1u << lane) - 1u))] = (int16_t)e;
    nact += tot;
    __syncthreads();
  }
  if (wid == 0) {
    int carry = 0;
    for (int i0 = 0; i0 < nact; i0 += 32) {
      const int i = i0 + lane;
      int v = 0;
      if (i < nact) {
        int r0, n;
        expert_rows(offsets, s_act[i], P, nullptr, r0, n);
        v = units_per_expert * ((n + 7) / 8) * kp;
      }
      int x = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      if (i < nact) s_pref[i] = carry + x - v;
      carry += __shfl_sync(0xffffffffu, x, 31);
    }
    if (lane == 0) s_pref[nact] = carry;
  }
  __syncthreads();
  return nact;
}

// Scales of rows (g, g+8) for the blocks of a record: [b][h] as fp32 (two 32-element
// blocks for Q4_0 / MXFP4; four 16-element blocks for NVFP4).
template <int QT>
__device__ __forceinline__ void load_scales(const uint8_t* rec, int g, float (&sc)[4][2]) {
  if (QT == FTMOE_NVFP4) {
    const uint2 s = *reinterpret_cast<const uint2*>(rec + REC_CODE_BYTES + g * 8);
#pragma unroll
    for (int i = 0; i < 8; ++i) sc[i >> 1][i & 1] = e4m3_to_f32(((i < 4 ? s.x : s.y) >> (8 * (i & 3))) & 0xFFu);
  } else if (QT == FTMOE_Q4_0) {
    const uint2 s = *reinterpret_cast<const uint2*>(rec + REC_CODE_BYTES + g * 8);
    sc[0][0] = half_bits_to_f32(s.x & 0xFFFFu);
    sc[0][1] = half_bits_to_f32(s.x >> 16);
    sc[1][0] = half_bits_to_f32(s.y & 0xFFFFu);
    sc[1][1] = half_bits_to_f32(s.y >> 16);
  } else {  // MXFP4, MXFP8: E8M0 [g][b][h] after the code bytes
    const uint32_t s = *reinterpret_cast<const uint32_t*>(rec + rec_code_bytes(QT) + g * 4);
    sc[0][0] = e8m0_to_f32(s & 0xFFu);
    sc[0][1] = e8m0_to_f32((s >> 8) & 0xFFu);
    sc[1][0] = e8m0_to_f32((s >> 16) & 0xFFu);
    sc[1][1] = e8m0_to_f32(s >> 24);
  }
}

// A warp's position in its flattened sequence of stages: item -> stage.  An item is one
// (tile pair, round of 8 rows, group of reduction parts) of an active expert, numbered
// expert by expert with the group innermost, then the round, so that the rounds of one
// tile pair run side by side on neighbouring warps and share its weights through L2.
struct Cursor {
  int item;
  int r0, n_e, tile0, tile1;
  int s0, s1;          // slab range of the item's group of parts
  int r, sp;           // round (8 tokens), first slab of the stage
  const uint8_t* w0;   // records of tile0 / tile1
  const uint8_t* w1;
  const uint16_t* brow;  // this lane's token row (B operand) for the round
  float ts;              // NVFP4 tensor scale of the item's expert matrix (else 1)
};

template <int MODE>
__device__ __forceinline__ void cursor_row(Cursor& c, const GemvArgs& a, int g) {
  const int rr = min(8 * c.r + g, c.n_e - 1);  // padded lanes re-read a valid row
  long long row;
  if (MODE == 0) row = row_token(a.sorted_pair, c.r0 + rr, a.k, a.T, a.status);
  else row = c.r0 + rr;
  c.brow = a.act + row * a.act_ld;
}

template <int MODE, class Tab>
__device__ __forceinline__ void cursor_load(Cursor& c, const GemvArgs& a, const Tab& tab,
                                            const int16_t* s_act, const int* s_pref, int nact,
                                            int total, int g) {
  if (c.item >= total) return;
  int lo = 0, hi = nact;  // last active expert whose first item is <= item
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (s_pref[mid] <= c.item) lo = mid; else hi = mid;
  }
  const int ui = lo;
  const int e = s_act[ui];
  expert_rows(a.offsets, e, a.P, nullptr, c.r0, c.n_e);  // (reported once, by the active list)
  const int rounds = (c.n_e + 7) / 8;
  const int local = c.item - s_pref[ui];
  const int grp = local % a.kp;
  const int t = local / a.kp;
  c.r = t % rounds;
  const int sub = t / rounds;
  c.tile0 = MODE == 0 ? sub : 2 * sub;
  c.tile1 = MODE == 0 ? a.up_rt + sub : 2 * sub + 1;
  c.s0 = (grp * a.NP / a.kp) * GW_PS;
  c.s1 = min(((grp + 1) * a.NP / a.kp) * GW_PS, a.S);
  c.sp = c.s0;
  const uint8_t* wexp = tab.get(e, a);
  c.w0 = wexp;
  c.w1 = wexp;
  c.ts = a.qtype == FTMOE_NVFP4 ? __ldg(reinterpret_cast<const float*>(wexp + a.rec_total)) : 1.0f;
  cursor_row<MODE>(c, a, g);
}

// Next stage; returns true when the item just left is complete.
template <int MODE, int SL, class Tab>
__device__ __forceinline__ bool cursor_next(Cursor& c, const GemvArgs& a, const Tab& tab,
                                            const int16_t* s_act, const int* s_pref, int nact,
                                            int total, int nwarps, int g) {
  c.sp += SL;
  if (c.sp < c.s1) return false;
  c.item += nwarps;
  cursor_load<MODE>(c, a, tab, s_act, s_pref, nact, total, g);
  return true;
}

template <int QT, int MODE, class Tab>
__global__ void __launch_bounds__(GW_THREADS, GW_MINB) gemv_ffn_kernel(const GemvArgs a,
                                                              const __grid_constant__ Tab tab) {
  using SM = GwSmem<QT>;
  constexpr int RB = rec_bytes(QT);
  constexpr int SL = gw_sl<QT>();
  extern __shared__ __align__(128) uint8_t smem_raw[];
  SM& sm = *reinterpret_cast<SM*>(smem_raw);
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int g = lane >> 2, c4 = lane & 3;

  if (MODE == 0) pdl_wait();  // offsets come from the permutation kernel
  pdl_launch_dependents();

  if (lane == 0) {
    for (int i = 0; i < GW_NS; ++i) mbar_init(&sm.full[wid][i], 1);
    // group barriers, one per group of kp warps (initialised by the group's first warp)
    if (a.kp > 1 && wid % a.kp == 0) {
      mbar_init(&sm.gfull[wid], 32 * a.kp);
      mbar_init(&sm.gfree[wid], 32);
    }
  }
  fence_barrier_init();
  const int nact = build_active_list(a.offsets, a.E, a.P, a.status, a.units_per_expert, a.kp, sm.act,
                                     sm.pref, sm.wsum);  // __syncthreads inside
  const int total = sm.pref[nact];
  const int nwarps = gridDim.x * GW_WARPS;
  const int gw = blockIdx.x * GW_WARPS + wid;
  const bool ragged = (a.K & 63) != 0;
  uint8_t (*stage)[SM::STAGE] = sm.stage[wid];
  uint64_t* full = sm.full[wid];
  const long long tile_bytes = (long long)a.S * RB;

  // ---- producer side (lane 0 issues the copies, every lane keeps the cursor)
  Cursor pc;
  pc.item = gw;
  cursor_load<MODE>(pc, a, tab, sm.act, sm.pref, nact, total, g);
  uint32_t issued = 0;
  auto issue = [&]() {
    if (pc.item >= total) return;
    const int st = issued % GW_NS;
    if (lane == 0) {
      const int ns = min(SL, pc.s1 - pc.sp);
      const uint32_t bytes = (uint32_t)(ns * RB);
      mbar_arrive_expect_tx(&full[st], 2 * bytes);
      bulk_g2s(&stage[st][0], pc.w0 + pc.tile0 * tile_bytes + (long long)pc.sp * RB, bytes, &full[st]);
      bulk_g2s(&stage[st][SL * RB], pc.w1 + pc.tile1 * tile_bytes + (long long)pc.sp * RB, bytes,
               &full[st]);
    }
    ++issued;
    cursor_next<MODE, SL>(pc, a, tab, sm.act, sm.pref, nact, total, nwarps, g);
  };
  for (int i = 0; i < GW_NS; ++i) issue();

  if (MODE == 1) pdl_wait();  // h comes from the gate/up kernel

  // ---- consumer side
  Cursor cc;
  cc.item = gw;
  cursor_load<MODE>(cc, a, tab, sm.act, sm.pref, nact, total, g);
  // B operand (this lane's token row) of one slab: 4 k-steps x 2 registers
  auto load_slab = [&](const Cursor& c, int sl, uint2 (&bv)[4]) {
    if (c.item >= total) return;
    const int s = c.sp + sl;
    if (s >= c.s1) return;
    const bool half = ragged && s == a.S - 1;
    const uint2* src = reinterpret_cast<const uint2*>(c.brow + 4 * c4) + s * 16;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (j >= 2 && half) break;
      bv[j] = __ldg(src + 4 * j);  // (h of the down projection: written before pdl_wait returned)
    }
  };
  // Warms L1 with the token-row lines of a stage: lane 4g + c takes slab c of token row g
  // (one 128-byte line each), so the per-slab loads above hit L1.
  auto prefetch_stage_rows = [&](const Cursor& c) {
    if (c.item >= total) return;
    for (int sl = c4; sl < SL && c.sp + sl < c.s1; sl += 4)
      asm volatile("prefetch.global.L1 [%0];" ::"l"(c.brow + (long long)(c.sp + sl) * 64));
  };
  uint32_t consumed = 0;
  const int gbase = a.kp > 1 ? wid - wid % a.kp : wid;  // first warp of this warp's group
  uint32_t red_items = 0;                               // split reductions done so far
  float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};  // current part
  float tot[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};  // finished parts, in order
  // Two slab buffers: while one slab computes, the next slab's rows load into the other
  // (the next stage's first slab after a stage's last).  `flip` says which buffer holds
  // the first slab of the coming stage.
  uint2 bA[4], bB[4];
  bool flip = false;
  load_slab(cc, 0, bA);
  while (cc.item < total) {
    const Cursor cur = cc;
    const bool done = cursor_next<MODE, SL>(cc, a, tab, sm.act, sm.pref, nact, total, nwarps, g);
    prefetch_stage_rows(cc);

    const int st = consumed % GW_NS;
    if (!mbar_wait(&full[st], (consumed / GW_NS) & 1u, a.status)) return;
    const int ns = min(SL, cur.s1 - cur.sp);
    auto stage_body = [&](uint2 (&b0)[4], uint2 (&b1)[4]) {
#pragma unroll
      for (int sl = 0; sl < SL; ++sl) {
        if (sl >= ns) break;
        uint2 (&bv)[4] = (sl & 1) ? b1 : b0;
        uint2 (&bn)[4] = (sl & 1) ? b0 : b1;
        if (sl + 1 < ns) load_slab(cur, sl + 1, bn);
        else load_slab(cc, 0, bn);
        const int s = cur.sp + sl;
        const bool half = ragged && s == a.S - 1;
        // Q4_0: the MMAs take the biased codes 128 + q; the block's -136 * sum(x) per token
        // (the same for every weight row) comes from MMAs with a constant -136 A operand
        // and seeds both tiles' block sums
        float corr[2][4];
        if (QT == FTMOE_Q4_0 && GW_BIASED) {
          const uint32_t M136[4] = {0xC308C308u, 0xC308C308u, 0xC308C308u, 0xC308C308u};
#pragma unroll
          for (int b = 0; b < 2; ++b) {
            if (b == 1 && half) break;
            const float z[4] = {0.f, 0.f, 0.f, 0.f};
            mma_16816_c(corr[b], M136, bv[2 * b].x, bv[2 * b].y, z);
            mma_16816(corr[b], M136, bv[2 * b + 1].x, bv[2 * b + 1].y);
          }
        }
#pragma unroll
        for (int ti = 0; ti < 2; ++ti) {
          const uint8_t* rec = &stage[st][(ti * SL + sl) * RB];
          float sc[4][2];
          load_scales<QT>(rec, g, sc);
          if (QT == FTMOE_MXFP8) {
            // E4M3 bytes: word 2j row g, word 2j + 1 row g + 8 (elements 16j + 4c .. +3)
            const uint4 q0 = *reinterpret_cast<const uint4*>(rec + lane * 32);
            const uint4 q1 = *reinterpret_cast<const uint4*>(rec + lane * 32 + 16);
            const uint32_t w8[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
            for (int b = 0; b < 2; ++b) {
              if (b == 1 && half) break;
              float part[4];
              const float z[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
              for (int jj = 0; jj < 2; ++jj) {
                const int j = 2 * b + jj;
                const uint32_t av[4] = {e4m3x2_to_bf16x2(prmt(w8[2 * j], 0u, 0x4140u)),
                                        e4m3x2_to_bf16x2(prmt(w8[2 * j + 1], 0u, 0x4140u)),
                                        e4m3x2_to_bf16x2(prmt(w8[2 * j], 0u, 0x4342u)),
                                        e4m3x2_to_bf16x2(prmt(w8[2 * j + 1], 0u, 0x4342u))};
                if (jj == 0) mma_16816_c(part, av, bv[j].x, bv[j].y, z);
                else mma_16816(part, av, bv[j].x, bv[j].y);
              }
              ffma2(acc[ti][0], acc[ti][1], sc[b][0], part[0], part[1]);
              ffma2(acc[ti][2], acc[ti][3], sc[b][1], part[2], part[3]);
            }
            continue;
          }
          const uint4 q = *reinterpret_cast<const uint4*>(rec + lane * 16);
          const uint32_t wj[4] = {q.x, q.y, q.z, q.w};
          if (QT == FTMOE_NVFP4) {
            // one 16-element block per k-step: scale every MMA's sums
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              if (j >= 2 && half) break;
              float part[4];
              uint32_t av[4];
              const float z[4] = {0.f, 0.f, 0.f, 0.f};
              e2m1_word_to_bf16x2(wj[j], av);
              mma_16816_c(part, av, bv[j].x, bv[j].y, z);
              ffma2(acc[ti][0], acc[ti][1], sc[j][0], part[0], part[1]);
              ffma2(acc[ti][2], acc[ti][3], sc[j][1], part[2], part[3]);
            }
            continue;
          }
#pragma unroll
          for (int b = 0; b < 2; ++b) {
            if (b == 1 && half) break;
            float part[4];
            uint32_t av[4];
            if (QT == FTMOE_Q4_0 && GW_BIASED) {
              q4_word_to_biased_bf16x2(wj[2 * b], av);
              mma_16816_c(part, av, bv[2 * b].x, bv[2 * b].y, corr[b]);
              q4_word_to_biased_bf16x2(wj[2 * b + 1], av);
              mma_16816(part, av, bv[2 * b + 1].x, bv[2 * b + 1].y);
            } else {
              const float z[4] = {0.f, 0.f, 0.f, 0.f};
              if (QT == FTMOE_Q4_0) q4_word_to_bf16x2(wj[2 * b], av); else e2m1_word_to_bf16x2(wj[2 * b], av);
              mma_16816_c(part, av, bv[2 * b].x, bv[2 * b].y, z);
              if (QT == FTMOE_Q4_0) q4_word_to_bf16x2(wj[2 * b + 1], av); else e2m1_word_to_bf16x2(wj[2 * b + 1], av);
              mma_16816(part, av, bv[2 * b + 1].x, bv[2 * b + 1].y);
            }
            ffma2(acc[ti][0], acc[ti][1], sc[b][0], part[0], part[1]);
            ffma2(acc[ti][2], acc[ti][3], sc[b][1], part[2], part[3]);
          }
        }
      }
    };
    if (flip) stage_body(bB, bA); else stage_body(bA, bB);
    flip ^= (ns & 1) != 0;
    ++consumed;
    // the stage is free again: order this warp's reads before the next bulk write into it
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncwarp();
    issue();

    const int send = cur.sp + ns;
    if (send % GW_PS == 0 || send == cur.s1) {
      // ---- end of a fixed part
      if (a.kp == 1) {
#pragma unroll
        for (int ti = 0; ti < 2; ++ti)
#pragma unroll
          for (int qq = 0; qq < 4; ++qq) tot[ti][qq] += acc[ti][qq];
      } else {
        // this warp's j-th part of the item: wait until the group's previous reduction has
        // been read (its finalising warp released the buffers), then park the sums
        const int j = (send - 1) / GW_PS - cur.s0 / GW_PS;
        if (j == 0 && red_items > 0 &&
            !mbar_wait(&sm.gfree[gbase], (uint32_t)((red_items - 1) & 1), a.status))
          return;
#pragma unroll
        for (int ti = 0; ti < 2; ++ti)
#pragma unroll
          for (int qq = 0; qq < 4; ++qq) sm.red[wid][j][(ti * 4 + qq) * 32 + lane] = acc[ti][qq];
      }
#pragma unroll
      for (int ti = 0; ti < 2; ++ti)
#pragma unroll
        for (int qq = 0; qq < 4; ++qq) acc[ti][qq] = 0.f;
    }

    if (done) {
      // ---- end of (item, round)
      bool finalize = true;
      if (a.kp > 1) {
        // the group's warps (same unit, consecutive part ranges) meet in shared memory; the
        // group's first warp adds every part in order, as one warp does without a split
        mbar_arrive(&sm.gfull[gbase]);
        finalize = wid == gbase;
        if (finalize) {
          if (!mbar_wait(&sm.gfull[gbase], (uint32_t)(red_items & 1), a.status)) return;
#pragma unroll
          for (int ti = 0; ti < 2; ++ti)
#pragma unroll
            for (int qq = 0; qq < 4; ++qq) tot[ti][qq] = 0.f;
          for (int gg = 0; gg < a.kp; ++gg) {
            const int np = (gg + 1) * a.NP / a.kp - gg * a.NP / a.kp;
            for (int j = 0; j < np; ++j)
#pragma unroll
              for (int ti = 0; ti < 2; ++ti)
#pragma unroll
                for (int qq = 0; qq < 4; ++qq) tot[ti][qq] += sm.red[gbase + gg][j][(ti * 4 + qq) * 32 + lane];
          }
          mbar_arrive(&sm.gfree[gbase]);
        }
        ++red_items;
      }
      if (finalize) {
        const int tok0 = 8 * cur.r;
#pragma unroll
        for (int qq = 0; qq < 4; ++qq) {
          const int rr = tok0 + 2 * c4 + (qq & 1);
          if (rr >= cur.n_e) continue;
          const int rofs = g + 8 * (qq >> 1);
          uint16_t* orow = a.out + (long long)(cur.r0 + rr) * a.out_ld;
          const float t0 = QT == FTMOE_NVFP4 ? tot[0][qq] * cur.ts : tot[0][qq];
          const float t1 = QT == FTMOE_NVFP4 ? tot[1][qq] * cur.ts : tot[1][qq];
          if (MODE == 0) {
            orow[cur.tile0 * 16 + rofs] = f32_to_bf16_bits(silu_f32(t0) * t1);
          } else {
            orow[cur.tile0 * 16 + rofs] = f32_to_bf16_bits(t0);
            orow[cur.tile1 * 16 + rofs] = f32_to_bf16_bits(t1);
          }
        }
      }
#pragma unroll
      for (int ti = 0; ti < 2; ++ti)
#pragma unroll
        for (int qq = 0; qq < 4; ++qq) tot[ti][qq] = 0.f;
    }
  }
}

template <class K, class... Args>
static cudaError_t launch_pdl(K kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

static size_t al256(size_t x) { return (x + 255) & ~(size_t)255; }

// Split rule (overridable at build time for sweeps): largest batch whose tile pairs are
// split over several warps, and the work items per warp the split aims for.
#ifndef FTMOE_GW_KPT
#define FTMOE_GW_KPT 8
#endif
#ifndef FTMOE_GW_IPW
#define FTMOE_GW_IPW 2
#endif

// Part groups per unit: only for batches of at most FTMOE_GW_KPT tokens.  kp is a power
// of two up to GW_WARPS (so that a unit's groups are warps of one CTA) and large enough
// that no group holds more than 2 of the NP fixed parts; beyond that it grows while the
// GPU has fewer than about FTMOE_GW_IPW items per warp.  1 when no such kp exists.
static int pick_kp(int T, long long units, int NP, int sm_count) {
  if (T > FTMOE_GW_KPT || NP < 2) return 1;
  int kp = 1;
  while (kp < GW_WARPS && (NP + kp - 1) / kp > 2) kp *= 2;
  if ((NP + kp - 1) / kp > 2) return 1;
  const long long want = (long long)FTMOE_GW_IPW * sm_count * GW_MINB * GW_WARPS;
  while (2 * kp <= GW_WARPS && 2 * kp <= NP && units * kp < want) kp *= 2;
  return kp;
}

// The split reductions meet in shared memory: the grouped GEMV needs no scratch.
size_t ffn_gemv_ws_bytes(int, int, int, int, int) { return 0; }
size_t ffn_gemv_zero_bytes(int, int, int, int, int) { return 0; }

template <int QT, int MODE, class Tab>
static cudaError_t launch_mode(const GemvArgs& a, const Tab& tab, int max_active, cudaStream_t st) {
  const DeviceInfo* di = device_info();
  if (!di) return cudaErrorUnknown;
  auto kern = gemv_ffn_kernel<QT, MODE, Tab>;
  cudaError_t err = set_smem_limit<gemv_ffn_kernel<QT, MODE, Tab>>(sizeof(GwSmem<QT>));
  if (err != cudaSuccess) return err;
  const size_t smem = a.kp > 1 ? sizeof(GwSmem<QT>) : offsetof(GwSmem<QT>, red);
  // rounds of 8 rows over all active experts: at most P / 8 + (active experts)
  const long long rounds = (long long)a.P / 8 + max_active;
  const long long items = rounds * a.units_per_expert * a.kp;
  long long grid = (items + GW_WARPS - 1) / GW_WARPS;
  const long long cap = (long long)di->sm_count * GW_MINB;
  if (grid > cap) grid = cap;
  if (grid < 1) grid = 1;
  return launch_pdl(kern, dim3((unsigned)grid), dim3(GW_THREADS), smem, st, a, tab);
}

template <int QT, class Tab>
static cudaError_t launch_qt(const FfnProblem& pb, const Tab& tab, void* ws, bool ws_zeroed,
                             cudaStream_t st) {
  const DeviceInfo* di = device_info();
  if (!di) return cudaErrorUnknown;
  const int max_active = pb.P < pb.E ? pb.P : pb.E;

  GemvArgs a{};
  a.offsets = pb.offsets;
  a.sorted_pair = pb.sorted_pair;
  a.k = pb.k;
  a.E = pb.E;
  a.T = pb.T;
  a.P = pb.P;
  a.status = di->status;
  // gate/up + SwiGLU
  a.act = pb.x;
  a.act_ld = pb.H;
  a.out = pb.h_act;
  a.out_ld = pb.I;
  a.wbase = pb.w13;
  a.wstride = (long long)pb.w13_bytes;
  a.table_off = 0;
  a.S = slabs_of(pb.H);
  a.K = pb.H;
  a.NP = (a.S + GW_PS - 1) / GW_PS;
  a.up_rt = pb.I / 16;
  a.units_per_expert = pb.I / 16;
  a.qtype = pb.qtype;
  a.rec_total = (long long)records_bytes_per_expert(pb.qtype, 2 * pb.I, pb.H);
  a.kp = pick_kp(pb.T, (long long)max_active * a.units_per_expert, a.NP, di->sm_count);
  // down
  GemvArgs d = a;
  d.act = pb.h_act;
  d.act_ld = pb.I;
  d.out = pb.y_perm;
  d.out_ld = pb.H;
  d.wbase = pb.w2;
  d.wstride = (long long)tiles_bytes_per_expert(pb.qtype, pb.H, pb.I);
  d.table_off = (long long)pb.w13_bytes;
  d.S = slabs_of(pb.I);
  d.K = pb.I;
  d.NP = (d.S + GW_PS - 1) / GW_PS;
  d.up_rt = 0;
  d.units_per_expert = pb.H / 32;
  d.rec_total = (long long)records_bytes_per_expert(pb.qtype, pb.H, pb.I);
  d.kp = pick_kp(pb.T, (long long)max_active * d.units_per_expert, d.NP, di->sm_count);
  cudaError_t err = launch_mode<QT, 0>(a, tab, max_active, st);
  if (err != cudaSuccess) return err;
  return launch_mode<QT, 1>(d, tab, max_active, st);
}

cudaError_t launch_ffn_gemv(const FfnProblem& pb, void* ws, bool ws_zeroed, cudaStream_t st) {
  if (pb.table) {
    WithTable t;
    t.t = *pb.table;
    return pb.qtype == FTMOE_Q4_0    ? launch_qt<FTMOE_Q4_0>(pb, t, ws, ws_zeroed, st)
           : pb.qtype == FTMOE_MXFP4 ? launch_qt<FTMOE_MXFP4>(pb, t, ws, ws_zeroed, st)
           : pb.qtype == FTMOE_NVFP4 ? launch_qt<FTMOE_NVFP4>(pb, t, ws, ws_zeroed, st)
                                     : launch_qt<FTMOE_MXFP8>(pb, t, ws, ws_zeroed, st);
  }
  NoTable t;
  return pb.qtype == FTMOE_Q4_0    ? launch_qt<FTMOE_Q4_0>(pb, t, ws, ws_zeroed, st)
         : pb.qtype == FTMOE_MXFP4 ? launch_qt<FTMOE_MXFP4>(pb, t, ws, ws_zeroed, st)
         : pb.qtype == FTMOE_NVFP4 ? launch_qt<FTMOE_NVFP4>(pb, t, ws, ws_zeroed, st)
                                   : launch_qt<FTMOE_MXFP8>(pb, t, ws, ws_zeroed, st);
}

}  // namespace ftmoe
