// Grouped expert FFN on the 5th-generation tensor cores (tcgen05) for many rows per
// expert (prefill): the ExpertFFN of the FreeToken architecture walkthrough §五 on
// its GGUF Q4_0 / MXFP4 banks, with the block decode of §六 fused into the operand
// staging.
//
// One persistent CTA per SM.  A work item is (expert, a slice of weight rows, up to
// 256 of the expert's token rows).  For gate/up the slice is 128 features: a tile of
// their gate rows and a tile of their up rows, accumulated side by side in tensor
// memory (columns [0, 256) and [256, 512)) so that the epilogue sees g and u of a
// feature in one thread.  For down the slice is one 128-row tile, and two
// accumulator buffers alternate so that the epilogue of one item overlaps the MMAs of
// the next.  Per 64-element reduction block ("stage"):
//   * a raw-weight warp copies the stage's weight records (16 rows x 64 codes +
//     scales each) into a ring of shared-memory slots with 1-D bulk copies and warms
//     L2 with the next item's records;
//   * 8 converter warps decode the records into exact bf16 (round-to-nearest-even of
//     the decoded value) in the 128-byte-swizzled K-major A tiles, and for gate/up
//     also gather the item's token rows of x with cp.async into the B tile;
//   * for down a token warp loads the (contiguous) rows of h with one TMA box;
//   * one thread issues tcgen05.mma kind::f16 (M = 128 weight rows, N = the token
//     count rounded up to 16, K = 16) and commits each stage back to the ring;
//   * 4 epilogue warps read the accumulators with tcgen05.ld, compute
//     h = silu(gate) * up or take y, and store bf16 rows through a small staging
//     tile as 16-byte vectors.
// The weights are the A operand (M) and the tokens the B operand (N), so a small
// expert costs a narrow MMA rather than a mostly empty 128-row tile.  Items are
// ordered expert by expert with the token tile innermost, so CTAs that run at the
// same time share weight tiles through L2.
//
// A-tile row order: weight row r of a 16-row record is stored at tile row sigma(r)
// (operand.cuh), so that the converter stores of a quarter-warp fall on 8 different
// 16-byte bank groups of the swizzled rows; the epilogue maps TMEM lanes back.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>
#include <type_traits>

#include "common.cuh"
#include "internal.h"
#include "pipeline.cuh"
#include "operand.cuh"
#include "tcgen05.cuh"

namespace ftmoe {

constexpr int GM_TOK = 256;         // token rows per item (largest MMA N)
constexpr int GM_ROWS = 128;        // weight rows per tile (MMA M)
constexpr int GM_EPI_WARPS = 4;     // warps 0..3 (one per TMEM lane quarter)
constexpr int GM_MMA_WARP = 4;      // TMEM owner; lane 0 issues the MMAs
constexpr int GM_RAW_WARP = 5;      // bulk copies of the raw weight records
constexpr int GM_TOK_WARP = 6;      // token rows of the down projection (TMA); warp 7 idles
constexpr int GM_CONV0 = 8;         // first converter warp
constexpr int GM_CONV_WARPS = 16;
constexpr int GM_CONV_THREADS = GM_CONV_WARPS * 32;
constexpr int GM_THREADS = (GM_CONV0 + GM_CONV_WARPS) * 32;  // 768
constexpr uint32_t GM_TMEM_COLS = 512;
constexpr int GM_A_TILE = GM_ROWS * 128;  // 16 KB of bf16 (128 rows x 64)
constexpr int GM_B_TILE = GM_TOK * 128;   // 32 KB of bf16 (256 rows x 64)
constexpr int GM_ECOL = 16;               // accumulator columns (tokens) per epilogue step
constexpr int GM_STG = GM_ECOL * 64;      // epilogue staging per warp: 16 rows x 32 bf16
constexpr int GM_MAX_E = 1024;

// Per-projection layout: gate/up stages hold two A tiles, down stages one.  MXFP8's raw
// records are twice as large, so it trades one operand stage for deeper raw rings.
// Ring depths (overridable at build time for sweeps): operand stages and raw-record
// stages of the gate/up (0) and down (1) projections, for the 4-bit formats.
#ifndef FTMOE_GM_NS0
#define FTMOE_GM_NS0 3
#endif
#ifndef FTMOE_GM_NR0
#define FTMOE_GM_NR0 2
#endif
#ifndef FTMOE_GM_NS1
#define FTMOE_GM_NS1 4
#endif
#ifndef FTMOE_GM_NR1
#define FTMOE_GM_NR1 4
#endif
constexpr int GM_MAX_STAGES = 12;
template <int QT, int MODE>
struct GmCfg {
  static constexpr bool FP8 = QT == FTMOE_MXFP8;
  static constexpr int NT = MODE == 0 ? 2 : 1;           // A tiles (MMAs per k-step)
  static constexpr int NACC = MODE == 0 ? 1 : 2;         // accumulator buffers
  static constexpr int NS = MODE == 0 ? (FP8 ? 2 : FTMOE_GM_NS0) : (FP8 ? 3 : FTMOE_GM_NS1);  // operand stages
  static constexpr int NR = MODE == 0 ? (FP8 ? 3 : FTMOE_GM_NR0) : (FP8 ? 4 : FTMOE_GM_NR1);  // raw stages
  static_assert(NS <= GM_MAX_STAGES && NR <= GM_MAX_STAGES, "ring depth");
  static constexpr int NREC = 8 * NT;                    // records per stage
  static constexpr int STAGE = NT * GM_A_TILE + GM_B_TILE;
  static constexpr int RAW_STAGE = NREC * rec_bytes(QT);
};

struct GemmTail {
  uint64_t a_full[GM_MAX_STAGES], b_full[GM_MAX_STAGES], empty[GM_MAX_STAGES];
  uint64_t raw_full[GM_MAX_STAGES], raw_empty[GM_MAX_STAGES];
  uint64_t acc_full[2], acc_empty[2], drain;
  uint32_t tmem_base;
  int abort_flag;
  int citem[GM_MAX_E + 1];  // exclusive prefix of items per expert
};
template <int QT, int MODE>
constexpr size_t gm_smem_bytes() {
  return 1024 + (size_t)GmCfg<QT, MODE>::NS * GmCfg<QT, MODE>::STAGE +
         (size_t)GmCfg<QT, MODE>::NR * GmCfg<QT, MODE>::RAW_STAGE + (size_t)GM_EPI_WARPS * GM_STG +
         sizeof(GemmTail);
}
static_assert(gm_smem_bytes<FTMOE_Q4_0, 0>() <= 227 * 1024 && gm_smem_bytes<FTMOE_Q4_0, 1>() <= 227 * 1024 &&
                  gm_smem_bytes<FTMOE_MXFP8, 0>() <= 227 * 1024 && gm_smem_bytes<FTMOE_MXFP8, 1>() <= 227 * 1024,
              "shared memory per CTA");

struct GemmArgs {
  const int32_t* offsets;
  const int32_t* sorted_pair;  // gate/up: pair of each permuted row (nullptr: identity)
  int k, E, T, P;
  const uint16_t* act;  // gate/up: x [T][H] (rows gathered); down: h [P][I] (via act_map)
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
  int ft_per_expert;     // weight-row slices per token tile
  int f_step;            // weight rows (features) per slice
  long long rec_total;   // bytes of one expert's records of this projection (NVFP4 trailer offset)
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
  int beg, ne;
  expert_rows(a.offsets, lo, a.P, nullptr, beg, ne);  // (reported by the item count)
  const int ntt = (ne + GM_TOK - 1) / GM_TOK;
  const int ft = local / ntt, tt = local - ft * ntt;
  it.r0 = beg + tt * GM_TOK;
  it.n = min(GM_TOK, ne - tt * GM_TOK);
  it.f0 = ft * a.f_step;
  return it;
}

// First matrix row of record ri (tile ri / 8, 16-row group ri % 8) of an item, and
// whether that row group lies inside the projection's result rows.
template <int MODE>
__device__ __forceinline__ int gm_record_row(const GmItem& it, int ri, const GemmArgs& a,
                                             bool& ok) {
  const int row = it.f0 + (ri & 7) * 16;
  ok = row < a.nrows;
  return (MODE == 0 && (ri >> 3)) ? row + a.up_row0 : row;
}

// 16-byte global -> shared copy (LDGSTS); src_bytes = 0 writes zeros.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Brings [p, p + bytes) into L2 ahead of use (bytes % 16 == 0, p 16-byte aligned).
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// 2-D TMA tile load (box from the tensor map) into shared memory, completion counted
// on `bar`.  c0 is the inner (element) coordinate, c1 the row.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, "
      "{%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
      : "memory");
}

// Token rows of gate/up: gathered one stage ahead of their conversion (1), or at the
// start of the same stage (0: the converters then wait on the MMAs of three stages back
// instead of two).
#ifndef FTMOE_GM_GATHER_AHEAD
#define FTMOE_GM_GATHER_AHEAD 1
#endif

// Waits of each role: a suspending try_wait (bit clear) or a polling one (bit set) for
// the raw-record warp (1), converters (2), MMA thread (4), epilogue (8), token warp (16).
#ifndef FTMOE_GM_SPIN
#define FTMOE_GM_SPIN 0
#endif
template <int ROLE>
__device__ __forceinline__ bool gm_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                        int* status) {
  if (FTMOE_GM_SPIN & ROLE) return mbar_wait_spin_or_abort(bar, parity, abort_flag, status);
  return mbar_wait_or_abort(bar, parity, abort_flag, status);
}
constexpr int GM_R_RAW = 1, GM_R_CONV = 2, GM_R_MMA = 4, GM_R_EPI = 8, GM_R_TOK = 16;

template <int QT, int MODE, class Tab>
__global__ void __launch_bounds__(GM_THREADS, 1)
    gemm_ffn_kernel(const GemmArgs a, const __grid_constant__ Tab tab,
                    const __grid_constant__ CUtensorMap act_map) {
  using C = GmCfg<QT, MODE>;
  constexpr int RB = rec_bytes(QT);
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t base_addr = (raw_addr + 1023u) & ~1023u;
  uint8_t* base = smem_raw + (base_addr - raw_addr);
  const uint32_t rawring = base_addr + C::NS * C::STAGE;
  const uint32_t staging = rawring + C::NR * C::RAW_STAGE;
  GemmTail& tl = *reinterpret_cast<GemmTail*>(base + (size_t)C::NS * C::STAGE +
                                              (size_t)C::NR * C::RAW_STAGE + GM_EPI_WARPS * GM_STG);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  volatile int* abort_flag = &tl.abort_flag;

  if (tid == 0) {
    for (int s = 0; s < C::NS; ++s) {
      mbar_init(&tl.a_full[s], GM_CONV_WARPS);
      mbar_init(&tl.b_full[s], 1);
      mbar_init(&tl.empty[s], 1);
    }
    for (int s = 0; s < C::NR; ++s) {
      mbar_init(&tl.raw_full[s], 1);
      mbar_init(&tl.raw_empty[s], GM_CONV_WARPS);
    }
    for (int b = 0; b < C::NACC; ++b) {
      mbar_init(&tl.acc_full[b], 1);
      mbar_init(&tl.acc_empty[b], GM_EPI_WARPS * 32);
    }
    mbar_init(&tl.drain, 1);
    tl.abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == GM_MMA_WARP) {
    tmem_alloc(&tl.tmem_base, GM_TMEM_COLS);
    tmem_relinquish();
  }
  // items per expert: ceil(n_e / 256) token tiles x weight-row slices
  if (warp == 0) {
    int carry = 0;
    for (int e0 = 0; e0 < a.E; e0 += 32) {
      const int e = e0 + lane;
      int v = 0;
      if (e < a.E) {
        int r0, n;
        expert_rows(a.offsets, e, a.P, a.status, r0, n);
        v = ((n + GM_TOK - 1) / GM_TOK) * a.ft_per_expert;
      }
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

  if (warp == GM_RAW_WARP) {
    // ------------------------------------------------------------ raw weight records
    int rslot = 0;
    uint32_t rphase = 0;
    for (int i = blockIdx.x; i < nitems; i += G) {
      const GmItem it = gm_item<MODE>(i, a, tl.citem);
      // lane r < NREC: record r of every stage (tile r / 8, row group r % 8)
      bool rok = false;
      const uint8_t* rec0 = nullptr;
      if (lane < C::NREC)
        rec0 = tab.get(it.e, a) + (long long)(gm_record_row<MODE>(it, lane, a, rok) / 16) * a.S * RB;
      const int nrec = __popc(__ballot_sync(0xffffffffu, lane < C::NREC && rok));
      // warm L2 with the CTA's next item's records while this one streams
      if (i + G < nitems && lane < C::NREC) {
        const GmItem nx = gm_item<MODE>(i + G, a, tl.citem);
        bool nok;
        const int nrow = gm_record_row<MODE>(nx, lane, a, nok);
        if (nok) prefetch_l2(tab.get(nx.e, a) + (long long)(nrow / 16) * a.S * RB, (uint32_t)(a.S * RB));
      }
      for (int kb = 0; kb < a.S; ++kb) {
        if (!gm_wait<GM_R_RAW>(&tl.raw_empty[rslot], rphase ^ 1u, abort_flag, a.status)) break;
        if (lane == 0) mbar_arrive_expect_tx(&tl.raw_full[rslot], (uint32_t)(nrec * RB));
        __syncwarp();
        if (lane < C::NREC && rok)
          bulk_g2s(base + C::NS * C::STAGE + rslot * C::RAW_STAGE + lane * RB,
                   rec0 + (long long)kb * RB, RB, &tl.raw_full[rslot]);
        if (++rslot == C::NR) { rslot = 0; rphase ^= 1u; }
      }
      if (*abort_flag) break;
    }
  } else if (warp == GM_TOK_WARP) {
    // ------------------------------------------------------------ token rows, down projection
    // (h rows of an item are contiguous: one 64 x 256 TMA box per stage)
    if (MODE == 1) {
      int slot = 0;
      uint32_t phase = 0;
      for (int i = blockIdx.x; i < nitems; i += G) {
        const GmItem it = gm_item<MODE>(i, a, tl.citem);
        for (int kb = 0; kb < a.S; ++kb) {
          if (!gm_wait<GM_R_TOK>(&tl.empty[slot], phase ^ 1u, abort_flag, a.status)) break;
          if (lane == 0) {
            mbar_arrive_expect_tx(&tl.b_full[slot], (uint32_t)GM_B_TILE);
            tma_load_2d(base_addr + slot * C::STAGE + C::NT * GM_A_TILE, &act_map, kb * 64, it.r0,
                        &tl.b_full[slot]);
          }
          if (++slot == C::NS) { slot = 0; phase ^= 1u; }
        }
        if (*abort_flag) break;
      }
    }
  } else if (warp >= GM_CONV0) {
    // ------------------------------------------------------------ converters
    const int ct = tid - GM_CONV0 * 32;
    const int cw = ct >> 5;  // converter warp
    // each warp converts the same steps of two records (lanes 0..15 and 16..31):
    // gate/up: records 2 (cw / 2) + {0, 1}, quantization block cw % 2;
    // down:    records 2 (cw % 4) + {0, 1}, 16-element step cw / 4
    const int ri = (MODE == 0 ? 2 * (cw >> 1) : 2 * (cw & 3)) + (lane >> 4);
    const int jsel = MODE == 0 ? (cw & 1) : (cw >> 2);
    const int g = (lane & 15) >> 1, m = lane & 1;
    int slot = 0, rslot = 0;
    uint32_t phase = 0, rphase = 0;
    // gate/up token rows: this thread copies 16-byte chunk (ct & 7) of rows (ct >> 3) + 64 r,
    // one stage ahead of the conversion so that the copies land while it decodes
    constexpr int RPT = GM_TOK * 8 / GM_CONV_THREADS;  // rows per thread
    const int ch = ct & 7;
    int bi = blockIdx.x, bkb = 0, bslot = 0;
    uint32_t bphase = 0;
    const uint16_t* rowp[RPT];
    auto load_rows = [&](int item) {
      const GmItem it = gm_item<MODE>(item, a, tl.citem);
#pragma unroll
      for (int r = 0; r < RPT; ++r) {
        const int rr = (ct >> 3) + (GM_CONV_THREADS / 8) * r;
        rowp[r] = nullptr;
        if (rr < it.n) {
          const long long ar = row_token(a.sorted_pair, it.r0 + rr, a.k, a.T, a.status);
          rowp[r] = a.act + ar * a.act_ld + ch * 8;
        }
      }
    };
    auto issue_rows = [&]() -> bool {  // copies of stage (bi, bkb); false when none / aborted
      if (bi >= nitems) return false;
      if (!gm_wait<GM_R_CONV>(&tl.empty[bslot], bphase ^ 1u, abort_flag, a.status)) return false;
      const uint32_t bt = base_addr + bslot * C::STAGE + C::NT * GM_A_TILE;
      const bool kok = bkb * 64 + ch * 8 < a.K;  // beyond K: zeros
#pragma unroll
      for (int r = 0; r < RPT; ++r) {
        if (rowp[r]) {
          const int rr = (ct >> 3) + (GM_CONV_THREADS / 8) * r;
          cp_async16(bt + (rr >> 3) * 1024 + (rr & 7) * 128 + ((ch ^ (rr & 7)) * 16),
                     kok ? rowp[r] + bkb * 64 : rowp[r], kok ? 16u : 0u);
        }
      }
      cp_async_commit();
      if (++bslot == C::NS) { bslot = 0; bphase ^= 1u; }
      if (++bkb == a.S) {
        bkb = 0;
        bi += G;
        if (bi < nitems) load_rows(bi);
      }
      return true;
    };
    if (MODE == 0 && bi < nitems) {
      load_rows(bi);
      if (FTMOE_GM_GATHER_AHEAD) issue_rows();
    }
    for (int i = blockIdx.x; i < nitems; i += G) {
      const GmItem it = gm_item<MODE>(i, a, tl.citem);
      bool rok;
      gm_record_row<MODE>(it, ri, a, rok);
      for (int kb = 0; kb < a.S; ++kb) {
        const bool ahead = MODE == 0 && issue_rows() && FTMOE_GM_GATHER_AHEAD;
        if (!gm_wait<GM_R_CONV>(&tl.raw_full[rslot], rphase, abort_flag, a.status)) break;
        if (!gm_wait<GM_R_CONV>(&tl.empty[slot], phase ^ 1u, abort_flag, a.status)) break;
        if (rok) {
          const uint32_t rec = rawring + rslot * C::RAW_STAGE + ri * RB;
          const uint32_t tile = base_addr + slot * C::STAGE + (ri >> 3) * GM_A_TILE;
          if (MODE == 0) {
            if (jsel) convert_record_operand<QT, 2, 2>(rec, tile, ri & 7, g, m);
            else convert_record_operand<QT, 2, 0>(rec, tile, ri & 7, g, m);
          } else {
            switch (jsel) {
              case 0: convert_record_operand<QT, 1, 0>(rec, tile, ri & 7, g, m); break;
              case 1: convert_record_operand<QT, 1, 1>(rec, tile, ri & 7, g, m); break;
              case 2: convert_record_operand<QT, 1, 2>(rec, tile, ri & 7, g, m); break;
              default: convert_record_operand<QT, 1, 3>(rec, tile, ri & 7, g, m); break;
            }
          }
        }
        if (MODE == 0) {
          if (ahead) cp_async_wait<1>(); else cp_async_wait<0>();  // this stage's rows have landed
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&tl.raw_empty[rslot]);
          mbar_arrive(&tl.a_full[slot]);
        }
        if (++rslot == C::NR) { rslot = 0; rphase ^= 1u; }
        if (++slot == C::NS) { slot = 0; phase ^= 1u; }
      }
      if (*abort_flag) break;
    }
    if (MODE == 0) cp_async_wait<0>();
  } else if (warp == GM_MMA_WARP) {
    // ------------------------------------------------------------ MMA issue
    if (lane == 0) {
      int slot = 0, buf = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      // Operand descriptors of slot 0, computed once: a slot's descriptors are these plus
      // its byte offset / 16 in the start-address field (shared-memory addresses stay
      // below 2^18, so the sum never leaves that 14-bit field).  The issue loop below is
      // then a straight run of MMAs; scalar work between them costs issue rate.
      uint64_t ad0[4], ad1[4], bdk[4];
#pragma unroll
      for (int k16 = 0; k16 < 4; ++k16) {
        ad0[k16] = sdesc_kmajor_sw128(base_addr + 32 * k16);
        ad1[k16] = sdesc_kmajor_sw128(base_addr + GM_A_TILE + 32 * k16);
        bdk[k16] = sdesc_kmajor_sw128(base_addr + C::NT * GM_A_TILE + 32 * k16);
      }
      for (int i = blockIdx.x; i < nitems && ok; i += G) {
        const GmItem it = gm_item<MODE>(i, a, tl.citem);
        const int N = max(16, (it.n + 15) & ~15);
        const uint32_t idesc = idesc_bf16_f32(GM_ROWS, N);
        if (!gm_wait<GM_R_MMA>(&tl.acc_empty[buf], acc_phase ^ 1u, abort_flag, a.status)) break;
        tc_fence_after_sync();
        const uint32_t d0 = tmem + buf * 256;
        for (int kb = 0; kb < a.S; ++kb) {
          if (!gm_wait<GM_R_MMA>(&tl.a_full[slot], phase, abort_flag, a.status) ||
              (MODE == 1 && !gm_wait<GM_R_MMA>(&tl.b_full[slot], phase, abort_flag, a.status))) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint64_t so = (uint64_t)(slot * (C::STAGE >> 4));
          const uint32_t acc0 = kb != 0 ? 1u : 0u;  // the item's first k-step overwrites
#pragma unroll
          for (int k16 = 0; k16 < 4; ++k16) {
            const uint32_t acc = k16 ? 1u : acc0;
            mma_bf16(d0, ad0[k16] + so, bdk[k16] + so, idesc, acc);
            if (C::NT == 2) mma_bf16(d0 + 256, ad1[k16] + so, bdk[k16] + so, idesc, acc);
          }
          mma_commit(&tl.empty[slot]);
          if (++slot == C::NS) { slot = 0; phase ^= 1u; }
        }
        if (!ok) break;
        mma_commit(&tl.acc_full[buf]);
        if (++buf == C::NACC) { buf = 0; acc_phase ^= 1u; }
      }
      // every MMA issued above has finished once this arrives
      mma_commit(&tl.drain);
      mbar_wait_or_abort(&tl.drain, 0, abort_flag, a.status, 100000000ull);
    }
    __syncwarp();
  } else if (warp < GM_EPI_WARPS) {
    // ------------------------------------------------------------ epilogue (warps 0..3)
    const int q = warp;  // TMEM lanes [32q, 32q + 32)
    // TMEM lane 32q + lane holds feature 32q + fl of the item (tile row order -> features)
    const int fl = (lane & 16) + gm_sigma_inv(lane & 15);
    // lanes l and l ^ 2 hold adjacent features fl and fl ^ 1
    const int odd = fl & 1;
    const uint32_t stg = staging + q * GM_STG;
    int buf = 0;
    uint32_t acc_phase = 0;
    for (int i = blockIdx.x; i < nitems; i += G) {
      const GmItem it = gm_item<MODE>(i, a, tl.citem);
      // NVFP4: the operand held E2M1 x block scale; the tensor scale multiplies the sums
      const float ts = QT == FTMOE_NVFP4 ? __ldg(reinterpret_cast<const float*>(tab.get(it.e, a) + a.rec_total))
                                         : 1.0f;
      if (!gm_wait<GM_R_EPI>(&tl.acc_full[buf], acc_phase, abort_flag, a.status)) break;
      tc_fence_after_sync();
      const uint32_t lane_base = tmem + ((uint32_t)(32 * q) << 16) + buf * 256;
      // Each 32 x 16 block (this warp's 32 features x 16 tokens) goes through the warp's
      // staging tile [token][feature] so that the global stores are 16-byte vectors.
      const int fw = it.f0 + 32 * q;  // first feature of this warp
      const bool ok = fw < a.nrows;
      uint16_t* obase = a.out + (long long)it.r0 * a.out_ld + fw + 8 * (lane & 3);
      for (int c0 = 0; c0 < it.n; c0 += GM_ECOL) {
        float v[GM_ECOL];
        if (MODE == 0) {
          uint32_t gv[GM_ECOL], uv[GM_ECOL];
          tmem_ld16(lane_base + c0, gv);
          tmem_ld16(lane_base + 256 + c0, uv);
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < GM_ECOL; ++j) {
            const float gg = QT == FTMOE_NVFP4 ? __uint_as_float(gv[j]) * ts : __uint_as_float(gv[j]);
            const float uu = QT == FTMOE_NVFP4 ? __uint_as_float(uv[j]) * ts : __uint_as_float(uv[j]);
            v[j] = __fdividef(gg, 1.0f + __expf(-gg)) * uu;
          }
        } else {
          uint32_t yv[GM_ECOL];
          tmem_ld16(lane_base + c0, yv);
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < GM_ECOL; ++j)
            v[j] = QT == FTMOE_NVFP4 ? __uint_as_float(yv[j]) * ts : __uint_as_float(yv[j]);
        }
#pragma unroll
        for (int p = 0; p < GM_ECOL / 2; ++p) {
          const float send = odd ? v[2 * p] : v[2 * p + 1];
          const float recv = __shfl_xor_sync(0xffffffffu, send, 2);
          const float lo = odd ? recv : v[2 * p];
          const float hi = odd ? v[2 * p + 1] : recv;
          const uint32_t w = (uint32_t)f32_to_bf16_bits(lo) | ((uint32_t)f32_to_bf16_bits(hi) << 16);
          asm volatile("st.shared.u32 [%0], %1;" ::"r"(stg + (2 * p + odd) * 64 + (fl & ~1) * 2), "r"(w)
                       : "memory");
        }
        __syncwarp();
#pragma unroll
        for (int r4 = 0; r4 < GM_ECOL / 8; ++r4) {
          const int row = 8 * r4 + (lane >> 2);
          const uint4 d = lds128(stg + row * 64 + (lane & 3) * 16);
          if (ok && c0 + row < it.n)
            *reinterpret_cast<uint4*>(obase + (long long)(c0 + row) * a.out_ld) = d;
        }
        __syncwarp();
      }
      tc_fence_before_sync();
      mbar_arrive(&tl.acc_empty[buf]);
      if (++buf == C::NACC) { buf = 0; acc_phase ^= 1u; }
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == GM_MMA_WARP) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, GM_TMEM_COLS);
  }
}


// ================================================================ CTA-pair kernel
// The same grouped FFN on pairs of CTAs (a cluster of 2 on neighbouring SMs) issuing
// tcgen05.mma.cta_group::2: one M = 256 MMA covers 256 weight rows, 128 held and
// decoded by each CTA, against the item's up to 256 token rows, whose first half sits in
// the first CTA's shared memory and the second half in the second's.  Every CTA's tensor
// memory receives its 128 rows x all token columns.  Per SM this halves the token-row
// traffic and the operand bytes the tensor core reads for a given amount of work, which
// is what bounds the single-CTA kernel above (its stages are limited by shared-memory
// bandwidth, not by the tensor core).
//   gate/up item: (expert, 128 features, <= 256 tokens); CTA r decodes gate and up rows
//     of features f0 + 64 r .. + 63, interleaved per TMEM lane quarter q: lanes 32q + t
//     (t < 16) hold the gate row and 32q + 16 + t the up row of the same feature, so one
//     shuffle brings g and u together in the epilogue;
//   down item: (expert, 256 rows of H, <= 256 tokens); CTA r decodes rows f0 + 128 r ...
// Roles per CTA as in the single-CTA kernel, except that the gate/up token rows come, like
// h for down, as TMA boxes from x_perm, the x rows written once in the permuted order by
// gather_rows_kernel: a gather of 128-byte rows through cp.async from every stage of
// every feature slice is limited by the L1's outstanding misses, and the TMA's row-gather
// form by its copy rate.  The first CTA (rank 0) issues every MMA.
// Its "operands ready" barrier counts the converter warps of both CTAs (and, for down,
// both token warps, after their TMA box has landed); each MMA stage's commit arrives on
// the stage's "free" barrier in both CTAs, and the accumulator barriers likewise.
constexpr int GP_TOKH = GM_TOK / 2;           // token rows per CTA
constexpr int GP_B_TILE = GP_TOKH * 128;      // 16 KB of bf16 (128 rows x 64)
constexpr int GP_STAGE = GM_A_TILE + GP_B_TILE;
#ifndef FTMOE_GP_NS
#define FTMOE_GP_NS 5
#endif
// Converter warps of the pair kernel: GP_GROUPS groups of 8 that take every GP_GROUPS-th
// stage, so that the latency chains of consecutive stages' decodes overlap.  They share
// the operand ring safely while GP_GROUPS <= NS: a group reaching stage t has seen the
// MMAs of stage t - GP_GROUPS - NS complete, hence those of t - 2 NS, so the slot's
// barrier is at most one phase behind the one it waits for.
// A group converts a stage's 8 records with 8 warps (each thread 2 of a record's 4
// steps) or, with FTMOE_GP_NSTEP = 4, with 4 warps (each half-warp a whole record).
constexpr int GP_GROUP_WARPS = FTMOE_GP_NSTEP == 4 ? 4 : 8;
#ifndef FTMOE_GP_GROUPS
#define FTMOE_GP_GROUPS (16 / GP_GROUP_WARPS)
#endif
constexpr int GP_GROUPS = FTMOE_GP_GROUPS;
constexpr int GP_CONV_WARPS = GP_GROUPS * GP_GROUP_WARPS;
constexpr int GP_THREADS = (GM_CONV0 + GP_CONV_WARPS) * 32;
// Arrivals on the first CTA's operand barrier per stage, from each CTA: the converting
// group and warp 7 once the stage's token rows have landed.  The second CTA's arrive
// remotely.
constexpr int GP_SHARE = GP_GROUP_WARPS + 1;
template <int QT>
struct GpCfg {
  static constexpr int NS = FTMOE_GP_NS;  // operand stages
  // Raw-record stages: a private ring of RPG slots per converter group, which the group
  // consumes strictly in order.  (With one ring shared by groups that take stages in
  // turn, a group could wait on a slot two phases ahead of the slot's barrier, and a
  // parity wait cannot tell that phase from the one completed two uses earlier.)
  // MXFP8's records are twice as large.
  static constexpr int RPG = QT == FTMOE_MXFP8 ? (GP_GROUPS > 2 ? 1 : 2) : (GP_GROUPS > 2 ? 2 : 4);
  static constexpr int NR = GP_GROUPS * RPG;
  static_assert(NS <= GM_MAX_STAGES && NR <= GM_MAX_STAGES && GP_GROUPS <= NS, "ring depth");
  static constexpr int NREC = 8;          // records per stage (128 rows)
  static constexpr int RAW_STAGE = NREC * rec_bytes(QT);
};
template <int QT>
constexpr size_t gp_smem_bytes() {
  return 1024 + (size_t)GpCfg<QT>::NS * GP_STAGE + (size_t)GpCfg<QT>::NR * GpCfg<QT>::RAW_STAGE +
         (size_t)GM_EPI_WARPS * GM_STG + sizeof(GemmTail);
}
static_assert(gp_smem_bytes<FTMOE_Q4_0>() <= 227 * 1024 && gp_smem_bytes<FTMOE_MXFP8>() <= 227 * 1024,
              "shared memory per CTA");
// Raw-record slot and phase parity of stage t (the j-th stage of group t % GP_GROUPS).
template <int QT>
__device__ __forceinline__ void gp_raw_slot(int t, int& slot, uint32_t& parity) {
  const int g = t % GP_GROUPS, j = t / GP_GROUPS;
  slot = g * GpCfg<QT>::RPG + j % GpCfg<QT>::RPG;
  parity = (uint32_t)(j / GpCfg<QT>::RPG) & 1u;
}

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Address of the same shared-memory object in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t cluster_addr(const void* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
  return r;
}
// Arrival on a barrier of either CTA of the pair (default semantics: release at CTA
// scope, the form used for cross-CTA pipeline barriers; a cluster-scope release also
// waits for this thread's outstanding copies, which costs the converters a stage).
__device__ __forceinline__ void mbar_arrive_remote(uint32_t caddr) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(caddr) : "memory");
}
// A role's share of stage `slot` is ready: arrive on the first CTA's operand barrier.
__device__ __forceinline__ void gp_arrive_ready(uint64_t* a_full, int slot, uint32_t rank) {
  if (rank == 0) mbar_arrive(&a_full[slot]);
  else mbar_arrive_remote(cluster_addr(&a_full[slot], 0));
}
// Bounded wait on a local barrier that also receives arrivals from the other CTA.
__device__ __forceinline__ bool gp_wait_cluster(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                                int* status, uint64_t limit_ns = 2000000000ull) {
  auto try_once = [&](uint32_t hint) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(hint)
        : "memory");
    return ok != 0;
  };
  if (try_once(0u)) return true;
  const uint64_t t0 = global_timer_ns();
  for (;;) {
    if (try_once(FTMOE_WAIT_HINT_NS)) return true;
    if (*abort_flag) return false;
    if (global_timer_ns() - t0 > limit_ns) {
      *abort_flag = 1;
      set_device_code(status, DEV_WAIT_TIMEOUT);
      return false;
    }
  }
}
__device__ __forceinline__ void tmem_alloc2(uint32_t* smem_dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(smem_dst)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish2() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc2(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void mma2_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive once on `bar` in every CTA of `mask` when the pair's MMAs issued so far complete.
__device__ __forceinline__ void mma2_commit(uint64_t* bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_u32(bar)),
      "h"(mask)
      : "memory");
}

// First matrix row of record ri (0..7) of CTA `rank`'s half of an item, and whether it
// lies inside the projection's result rows.
template <int MODE>
__device__ __forceinline__ int gp_record_row(const GmItem& it, int ri, uint32_t rank, const GemmArgs& a,
                                             bool& ok) {
  if (MODE == 0) {
    const int f = it.f0 + 64 * (int)rank + 16 * (ri >> 1);  // first feature of the record
    ok = f < a.nrows;
    return (ri & 1) ? f + a.up_row0 : f;
  }
  const int row = it.f0 + 128 * (int)rank + 16 * ri;
  ok = row < a.nrows;
  return row;
}

template <int QT, int MODE, class Tab>
__global__ void __launch_bounds__(GP_THREADS, 1)
    gemm_pair_kernel(const GemmArgs a, const __grid_constant__ Tab tab,
                     const __grid_constant__ CUtensorMap act_map) {
  using C = GpCfg<QT>;
  constexpr int RB = rec_bytes(QT);
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t base_addr = (raw_addr + 1023u) & ~1023u;
  uint8_t* base = smem_raw + (base_addr - raw_addr);
  const uint32_t rawring = base_addr + C::NS * GP_STAGE;
  const uint32_t staging = rawring + C::NR * C::RAW_STAGE;
  GemmTail& tl = *reinterpret_cast<GemmTail*>(base + (size_t)C::NS * GP_STAGE +
                                              (size_t)C::NR * C::RAW_STAGE + GM_EPI_WARPS * GM_STG);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  volatile int* abort_flag = &tl.abort_flag;
  const uint32_t rank = cluster_ctarank();
  const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;

  if (tid == 0) {
    for (int s = 0; s < C::NS; ++s) {
      mbar_init(&tl.a_full[s], 2 * GP_SHARE);
      mbar_init(&tl.b_full[s], 1);
      mbar_init(&tl.empty[s], 1);
    }
    for (int s = 0; s < C::NR; ++s) {
      mbar_init(&tl.raw_full[s], 1);
      mbar_init(&tl.raw_empty[s], GP_GROUP_WARPS);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tl.acc_full[b], 1);
      mbar_init(&tl.acc_empty[b], 2 * GM_EPI_WARPS);
    }
    mbar_init(&tl.drain, 1);
    tl.abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == GM_MMA_WARP) {
    // collective over the pair: both CTAs allocate, and both receive the same columns
    tmem_alloc2(&tl.tmem_base, GM_TMEM_COLS);
    tmem_relinquish2();
  }
  if (warp == 0) {
    int carry = 0;
    for (int e0 = 0; e0 < a.E; e0 += 32) {
      const int e = e0 + lane;
      int v = 0;
      if (e < a.E) {
        int r0, n;
        expert_rows(a.offsets, e, a.P, a.status, r0, n);
        v = ((n + GM_TOK - 1) / GM_TOK) * a.ft_per_expert;
      }
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
  cluster_sync();  // both CTAs' barriers exist before any remote arrival
  tc_fence_after_sync();
  const uint32_t tmem = tl.tmem_base;
  const int nitems = tl.citem[a.E];

  if (warp == GM_RAW_WARP) {
    // ------------------------------------------------------------ raw weight records
    int t = 0;  // stage number in this pair's sequence
    for (int i = pair; i < nitems; i += npairs) {
      const GmItem it = gm_item<MODE>(i, a, tl.citem);
      bool rok = false;
      const uint8_t* rec0 = nullptr;
      if (lane < C::NREC) rec0 = tab.get(it.e, a) + (long long)(gp_record_row<MODE>(it, lane, rank, a, rok) / 16) * a.S * RB;
      const int nrec = __popc(__ballot_sync(0xffffffffu, lane < C::NREC && rok));
      if (i + npairs < nitems && lane < C::NREC) {
        const GmItem nx = gm_item<MODE>(i + npairs, a, tl.citem);
        bool nok;
        const int nrow = gp_record_row<MODE>(nx, lane, rank, a, nok);
        if (nok) prefetch_l2(tab.get(nx.e, a) + (long long)(nrow / 16) * a.S * RB, (uint32_t)(a.S * RB));
      }
      for (int kb = 0; kb < a.S; ++kb, ++t) {
        int rslot;
        uint32_t rphase;
        gp_raw_slot<QT>(t, rslot, rphase);
        if (!gm_wait<GM_R_RAW>(&tl.raw_empty[rslot], rphase ^ 1u, abort_flag, a.status)) break;
        if (lane == 0) mbar_arrive_expect_tx(&tl.raw_full[rslot], (uint32_t)(nrec * RB));
        __syncwarp();
        if (lane < C::NREC && rok)
          bulk_g2s(base + C::NS * GP_STAGE + rslot * C::RAW_STAGE + lane * RB, rec0 + (long long)kb * RB, RB,
                   &tl.raw_full[rslot]);
      }
      if (*abort_flag) break;
    }
  } else if (warp == GM_TOK_WARP || warp == GM_TOK_WARP + 1) {
    // ------------------------------------------------------------ token rows
    // this CTA's half of the item's rows of x_perm (gate/up) or h (down), contiguous in
    // the permuted order: one 64 x 128 TMA box per stage, issued by warp 6 as soon as the
    // stage is free; warp 7 reports each landed box to the first CTA's operand barrier,
    // so that several boxes stay in flight
    {
      const bool issuer = warp == GM_TOK_WARP;
      int slot = 0;
      uint32_t phase = 0;
      for (int i = pair; i < nitems; i += npairs) {
        const GmItem it = gm_item<MODE>(i, a, tl.citem);
        const int half = max(16, (it.n + 15) & ~15) / 2;
        for (int kb = 0; kb < a.S; ++kb) {
          if (issuer) {
            if (!gm_wait<GM_R_TOK>(&tl.empty[slot], phase ^ 1u, abort_flag, a.status)) break;
            if (lane == 0) {
              mbar_arrive_expect_tx(&tl.b_full[slot], (uint32_t)GP_B_TILE);
              tma_load_2d(base_addr + slot * GP_STAGE + GM_A_TILE, &act_map, kb * 64, it.r0 + (int)rank * half,
                          &tl.b_full[slot]);
            }
          } else {
            if (!gm_wait<GM_R_TOK>(&tl.b_full[slot], phase, abort_flag, a.status)) break;
            if (lane == 0) gp_arrive_ready(tl.a_full, slot, rank);
          }
          if (++slot == C::NS) { slot = 0; phase ^= 1u; }
        }
        if (*abort_flag) break;
      }
    }
  } else if (warp >= GM_CONV0) {
    // ------------------------------------------------------------ converters
    // group cw / GP_GROUP_WARPS converts stages t with t % GP_GROUPS == group; in a stage,
    // warp w = cw % GP_GROUP_WARPS converts records 2 (w % 4) + {0, 1} (half-warps), whole
    // (4 warps a group) or quantization block w / 4 (8 warps a group)
    const int ct = tid - GM_CONV0 * 32;
    const int cw = ct >> 5;
    const int grp = cw / GP_GROUP_WARPS;
    const int ri = 2 * (cw & 3) + (lane >> 4);
    const int jsel = ((cw % GP_GROUP_WARPS) >> 2) & 1;
    const int g = (lane & 15) >> 1, m = lane & 1;
    int t = 0;  // stage number in this pair's sequence
    for (int i = pair; i < nitems; i += npairs) {
      const GmItem it = gm_item<MODE>(i, a, tl.citem);
      bool rok;
      gp_record_row<MODE>(it, ri, rank, a, rok);
      for (int kb = 0; kb < a.S; ++kb, ++t) {
        if (t % GP_GROUPS != grp) continue;
        const int slot = t % C::NS;
        const uint32_t phase = (uint32_t)(t / C::NS) & 1u;
        int rslot;
        uint32_t rphase;
        gp_raw_slot<QT>(t, rslot, rphase);
        if (!gm_wait<GM_R_CONV>(&tl.empty[slot], phase ^ 1u, abort_flag, a.status)) break;
        if (!gm_wait<GM_R_CONV>(&tl.raw_full[rslot], rphase, abort_flag, a.status)) break;
        if (rok) {
          const uint32_t rec = rawring + rslot * C::RAW_STAGE + ri * RB;
          const uint32_t st_base = base_addr + slot * GP_STAGE;
          if (FTMOE_GP_NSTEP == 4) convert_record_operand<QT, 4, 0>(rec, st_base, ri, g, m);
          else if (jsel) convert_record_operand<QT, 2, 2>(rec, st_base, ri, g, m);
          else convert_record_operand<QT, 2, 0>(rec, st_base, ri, g, m);
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&tl.raw_empty[rslot]);
          gp_arrive_ready(tl.a_full, slot, rank);
        }
      }
      if (*abort_flag) break;
    }
  } else if (warp == GM_MMA_WARP) {
    // ------------------------------------------------------------ MMA issue (first CTA)
    if (rank == 0 && lane == 0) {
      int slot = 0, buf = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      uint64_t adk[4], bdk[4];
#pragma unroll
      for (int k16 = 0; k16 < 4; ++k16) {
        adk[k16] = sdesc_kmajor_sw128(base_addr + 32 * k16);
        bdk[k16] = sdesc_kmajor_sw128(base_addr + GM_A_TILE + 32 * k16);
      }
      for (int i = pair; i < nitems && ok; i += npairs) {
        const GmItem it = gm_item<MODE>(i, a, tl.citem);
        const int N = max(16, (it.n + 15) & ~15);
        const uint32_t idesc = idesc_bf16_f32(2 * GM_ROWS, N);
        if (!gp_wait_cluster(&tl.acc_empty[buf], acc_phase ^ 1u, abort_flag, a.status)) break;
        tc_fence_after_sync();
        const uint32_t d0 = tmem + buf * 256;
        for (int kb = 0; kb < a.S; ++kb) {
          if (!gp_wait_cluster(&tl.a_full[slot], phase, abort_flag, a.status)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint64_t so = (uint64_t)(slot * (GP_STAGE >> 4));
          const uint32_t acc0 = kb != 0 ? 1u : 0u;
#pragma unroll
          for (int k16 = 0; k16 < 4; ++k16) mma2_bf16(d0, adk[k16] + so, bdk[k16] + so, idesc, k16 ? 1u : acc0);
          mma2_commit(&tl.empty[slot], 3);
          if (++slot == C::NS) { slot = 0; phase ^= 1u; }
        }
        if (!ok) break;
        mma2_commit(&tl.acc_full[buf], 3);
        if (++buf == 2) { buf = 0; acc_phase ^= 1u; }
      }
      mma2_commit(&tl.drain, 1);
      mbar_wait_or_abort(&tl.drain, 0, abort_flag, a.status, 100000000ull);
    }
    __syncwarp();
  } else if (warp < GM_EPI_WARPS) {
    // ------------------------------------------------------------ epilogue (warps 0..3)
    const int q = warp;
    const uint32_t stg = staging + q * GM_STG;
    const uint32_t lead_accempty = cluster_addr(&tl.acc_empty[0], 0);
    int buf = 0;
    uint32_t acc_phase = 0;
    for (int i = pair; i < nitems; i += npairs) {
      const GmItem it = gm_item<MODE>(i, a, tl.citem);
      const float ts = QT == FTMOE_NVFP4 ? __ldg(reinterpret_cast<const float*>(tab.get(it.e, a) + a.rec_total))
                                         : 1.0f;
      if (!gm_wait<GM_R_EPI>(&tl.acc_full[buf], acc_phase, abort_flag, a.status)) break;
      tc_fence_after_sync();
      const uint32_t lane_base = tmem + ((uint32_t)(32 * q) << 16) + buf * 256;
      if (MODE == 0) {
        // lanes t and t + 16 hold the gate and up sums of feature fw + sigma^-1(t); after
        // one exchange lane t computes tokens c0..c0+7 and lane t + 16 tokens c0+8..c0+15
        const int fw = it.f0 + 64 * (int)rank + 16 * q;
        const int fl = gm_sigma_inv(lane & 15);
        const int hi = lane >> 4;
        const bool ok = fw < a.nrows;
        for (int c0 = 0; c0 < it.n; c0 += GM_ECOL) {
          uint32_t v[GM_ECOL];
          tmem_ld16(lane_base + c0, v);
          tmem_wait_ld();
          float h[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            // lane t sends its column 8 + j (needed by t + 16), lane t + 16 its column j
            const uint32_t send = hi ? v[j] : v[8 + j];
            const uint32_t recv = __shfl_xor_sync(0xffffffffu, send, 16);
            const float gg = __uint_as_float(hi ? recv : v[j]) * ts;
            const float uu = __uint_as_float(hi ? v[8 + j] : recv) * ts;
            h[j] = __fdividef(gg, 1.0f + __expf(-gg)) * uu;
          }
#pragma unroll
          for (int j = 0; j < 8; ++j)
            asm volatile("st.shared.u16 [%0], %1;" ::"r"(stg + (8 * hi + j) * 32 + fl * 2),
                         "h"(f32_to_bf16_bits(h[j]))
                         : "memory");
          __syncwarp();
          const int row = lane >> 1;
          const uint4 d = lds128(stg + row * 32 + (lane & 1) * 16);
          if (ok && c0 + row < it.n)
            *reinterpret_cast<uint4*>(a.out + (long long)(it.r0 + c0 + row) * a.out_ld + fw + 8 * (lane & 1)) = d;
          __syncwarp();
        }
      } else {
        // lanes hold rows fw + fl of H; lanes l and l ^ 2 hold adjacent rows fl and fl ^ 1
        const int fl = (lane & 16) + gm_sigma_inv(lane & 15);
        const int odd = fl & 1;
        const int fw = it.f0 + 128 * (int)rank + 32 * q;
        const bool ok = fw < a.nrows;
        uint16_t* obase = a.out + (long long)it.r0 * a.out_ld + fw + 8 * (lane & 3);
        for (int c0 = 0; c0 < it.n; c0 += GM_ECOL) {
          uint32_t yv[GM_ECOL];
          tmem_ld16(lane_base + c0, yv);
          tmem_wait_ld();
          float v[GM_ECOL];
#pragma unroll
          for (int j = 0; j < GM_ECOL; ++j) v[j] = __uint_as_float(yv[j]) * ts;
#pragma unroll
          for (int p = 0; p < GM_ECOL / 2; ++p) {
            const float send = odd ? v[2 * p] : v[2 * p + 1];
            const float recv = __shfl_xor_sync(0xffffffffu, send, 2);
            const float lo = odd ? recv : v[2 * p];
            const float hv = odd ? v[2 * p + 1] : recv;
            const uint32_t w = (uint32_t)f32_to_bf16_bits(lo) | ((uint32_t)f32_to_bf16_bits(hv) << 16);
            asm volatile("st.shared.u32 [%0], %1;" ::"r"(stg + (2 * p + odd) * 64 + (fl & ~1) * 2), "r"(w)
                         : "memory");
          }
          __syncwarp();
#pragma unroll
          for (int r4 = 0; r4 < GM_ECOL / 8; ++r4) {
            const int row = 8 * r4 + (lane >> 2);
            const uint4 d = lds128(stg + row * 64 + (lane & 3) * 16);
            if (ok && c0 + row < it.n) *reinterpret_cast<uint4*>(obase + (long long)(c0 + row) * a.out_ld) = d;
          }
          __syncwarp();
        }
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive_remote(lead_accempty + 8u * buf);
      if (++buf == 2) { buf = 0; acc_phase ^= 1u; }
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  cluster_sync();  // no CTA leaves while the pair's MMAs or remote arrivals may touch it
  if (warp == GM_MMA_WARP) {
    tc_fence_after_sync();
    tmem_dealloc2(tmem, GM_TMEM_COLS);
  }
  cluster_sync();
}

// x rows in the permuted order: xp[r][:] = x[token of permuted row r][:], one warp per
// row, 16-byte vectors (H is a multiple of 32).
__global__ void __launch_bounds__(256) gather_rows_kernel(const uint16_t* __restrict__ x, int H,
                                                          const int32_t* __restrict__ sorted_pair, int k, int T,
                                                          int P, uint16_t* __restrict__ xp, int* status) {
  const int lane = threadIdx.x & 31;
  const int nwarps = gridDim.x * 8;
  const int vecs = H / 8;
  for (int r = (int)(blockIdx.x * 8 + (threadIdx.x >> 5)); r < P; r += nwarps) {
    const long long t = row_token(sorted_pair, r, k, T, status);
    const uint4* src = reinterpret_cast<const uint4*>(x + t * H);
    uint4* dst = reinterpret_cast<uint4*>(xp + (long long)r * H);
    for (int v = lane; v < vecs; v += 32) dst[v] = __ldg(src + v);
  }
}

// Scratch of the grouped GEMM: x_perm, bf16 [T * k][H].
size_t ffn_gemm_ws_bytes(int T, int k, int, int H, int) { return (size_t)T * k * H * 2; }

// ---------------------------------------------------------------- host side
namespace {
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;
void resolve_encode() {
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
          cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    g_encode = (PFN_cuTensorMapEncodeTiled_v12000)fn;
}

// bf16 matrix [rows][cols] (row-major), box = 64 columns x box_rows rows, 128-byte swizzle.
bool make_act_map(CUtensorMap* map, const void* ptr, long long rows, int cols, int box_rows) {
  std::call_once(g_encode_once, resolve_encode);
  if (!g_encode) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  const cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
}  // namespace

template <int QT, int MODE, class Tab>
static cudaError_t gm_launch(const GemmArgs& a, const Tab& tab, const CUtensorMap& map,
                             cudaStream_t st) {
  const DeviceInfo* di = device_info();
  if (!di) return cudaErrorUnknown;
  auto kern = gemm_ffn_kernel<QT, MODE, Tab>;
  constexpr size_t smem = gm_smem_bytes<QT, MODE>();
  static_assert(smem <= 232448, "shared memory per CTA");
  cudaError_t err = set_smem_limit<gemm_ffn_kernel<QT, MODE, Tab>>(smem);
  if (err != cudaSuccess) return err;
  kern<<<di->sm_count, GM_THREADS, smem, st>>>(a, tab, map);
  return cudaGetLastError();
}

// CTA-pair launch: clusters of 2, as many as can be resident at once (persistent).
// Returns cudaErrorNotSupported when no cluster of 2 fits, so that the caller can fall
// back to the single-CTA kernel.
template <int QT, int MODE, class Tab>
static cudaError_t gp_launch(const GemmArgs& a, const Tab& tab, const CUtensorMap& map, cudaStream_t st) {
  const DeviceInfo* di = device_info();
  if (!di) return cudaErrorUnknown;
  auto kern = gemm_pair_kernel<QT, MODE, Tab>;
  constexpr size_t smem = gp_smem_bytes<QT>();
  cudaError_t err = set_smem_limit<gemm_pair_kernel<QT, MODE, Tab>>(smem);
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(di->sm_count & ~1));
  cfg.blockDim = dim3(GP_THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  static int max_clusters[2][2][5] = {};  // per (table, mode, format): resident clusters
  int& mc = max_clusters[std::is_same<Tab, GmWithTable>::value][MODE][QT];
  if (mc == 0) {
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n < 1) {
      (void)cudaGetLastError();
      return cudaErrorNotSupported;
    }
    mc = n;
  }
  cfg.gridDim = dim3((unsigned)(2 * std::min(mc, di->sm_count / 2)));
  return cudaLaunchKernelEx(&cfg, kern, a, tab, map);
}

// Which kernel runs the prefill FFN: CTA pairs (1) or single CTAs (0).
#ifndef FTMOE_GM_PAIR
#define FTMOE_GM_PAIR 1
#endif

template <int QT, class Tab>
static cudaError_t gm_launch_qt(const FfnProblem& pb, const Tab& tab, void* ws, size_t ws_bytes,
                                cudaStream_t st) {
  const DeviceInfo* di = device_info();
  if (!di) return cudaErrorUnknown;
  uint16_t* xperm = static_cast<uint16_t*>(ws);
  const bool pair = FTMOE_GM_PAIR != 0 && xperm && ws_bytes >= (size_t)pb.P * pb.H * 2;
  CUtensorMap xmap, hmap, xpmap;
  if (!make_act_map(&xmap, pb.x, pb.T, pb.H, 1) ||
      !make_act_map(&hmap, pb.h_act, (long long)pb.P, pb.I, pair ? GP_TOKH : GM_TOK) ||
      (pair && !make_act_map(&xpmap, xperm, (long long)pb.P, pb.H, GP_TOKH)))
    return cudaErrorNotSupported;
  GemmArgs a{};
  a.offsets = pb.offsets;
  a.sorted_pair = pb.sorted_pair;
  a.k = pb.k;
  a.E = pb.E;
  a.T = pb.T;
  a.P = pb.P;
  a.status = di->status;
  a.act = pb.x;
  a.act_ld = pb.H;
  a.K = pb.H;
  a.out = pb.h_act;
  a.out_ld = pb.I;
  a.wbase = pb.w13;
  a.wstride = (long long)pb.w13_bytes;
  a.table_off = 0;
  a.S = slabs_of(pb.H);
  a.nrows = pb.I;
  a.up_row0 = pb.I;
  a.f_step = GM_ROWS;
  a.ft_per_expert = (pb.I + GM_ROWS - 1) / GM_ROWS;
  a.rec_total = (long long)records_bytes_per_expert(pb.qtype, 2 * pb.I, pb.H);
  GemmArgs d = a;
  d.sorted_pair = nullptr;
  d.act = pb.h_act;
  d.act_ld = pb.I;
  d.K = pb.I;
  d.out = pb.y_perm;
  d.out_ld = pb.H;
  d.wbase = pb.w2;
  d.wstride = (long long)tiles_bytes_per_expert(pb.qtype, pb.H, pb.I);
  d.table_off = (long long)pb.w13_bytes;
  d.S = slabs_of(pb.I);
  d.nrows = pb.H;
  d.up_row0 = 0;
  d.f_step = pair ? 2 * GM_ROWS : GM_ROWS;
  d.ft_per_expert = (pb.H + d.f_step - 1) / d.f_step;
  d.rec_total = (long long)records_bytes_per_expert(pb.qtype, pb.H, pb.I);
  if (pair) {
    const int gblocks = std::max(1, std::min((pb.P + 7) / 8, di->sm_count * 8));
    gather_rows_kernel<<<gblocks, 256, 0, st>>>(pb.x, pb.H, pb.sorted_pair, pb.k, pb.T, pb.P, xperm, di->status);
    cudaError_t err = cudaGetLastError();
    if (err == cudaSuccess) err = gp_launch<QT, 0>(a, tab, xpmap, st);
    if (err == cudaSuccess) err = gp_launch<QT, 1>(d, tab, hmap, st);
    if (err != cudaErrorNotSupported) return err;
    // no pair fits: the single-CTA kernel with its own tensor map and slices
    if (!make_act_map(&hmap, pb.h_act, (long long)pb.P, pb.I, GM_TOK)) return cudaErrorNotSupported;
    d.f_step = GM_ROWS;
    d.ft_per_expert = (pb.H + GM_ROWS - 1) / GM_ROWS;
  }
  cudaError_t err = gm_launch<QT, 0>(a, tab, xmap, st);
  if (err != cudaSuccess) return err;
  return gm_launch<QT, 1>(d, tab, hmap, st);
}

cudaError_t launch_ffn_gemm(const FfnProblem& pb, void* ws, size_t ws_bytes, cudaStream_t st) {
  if (pb.E > GM_MAX_E) return cudaErrorNotSupported;
  if (pb.table) {
    GmWithTable t;
    t.t = *pb.table;
    return pb.qtype == FTMOE_Q4_0    ? gm_launch_qt<FTMOE_Q4_0>(pb, t, ws, ws_bytes, st)
           : pb.qtype == FTMOE_MXFP4 ? gm_launch_qt<FTMOE_MXFP4>(pb, t, ws, ws_bytes, st)
           : pb.qtype == FTMOE_NVFP4 ? gm_launch_qt<FTMOE_NVFP4>(pb, t, ws, ws_bytes, st)
                                     : gm_launch_qt<FTMOE_MXFP8>(pb, t, ws, ws_bytes, st);
  }
  GmNoTable t;
  return pb.qtype == FTMOE_Q4_0    ? gm_launch_qt<FTMOE_Q4_0>(pb, t, ws, ws_bytes, st)
         : pb.qtype == FTMOE_MXFP4 ? gm_launch_qt<FTMOE_MXFP4>(pb, t, ws, ws_bytes, st)
         : pb.qtype == FTMOE_NVFP4 ? gm_launch_qt<FTMOE_NVFP4>(pb, t, ws, ws_bytes, st)
                                   : gm_launch_qt<FTMOE_MXFP8>(pb, t, ws, ws_bytes, st);
}

}  // namespace ftmoe
