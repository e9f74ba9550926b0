// Grouped expert FFN on the 5th-generation tensor cores for few rows per expert
// (decode): the ExpertFFN of the FreeToken architecture walkthrough §五 on its GGUF
// Q4_0 / MXFP4 banks, with the block decode of §六 done by the SM into tensor memory.
//
// Decode reads every selected expert's weights once for a handful of tokens, so the
// layer is bound by streaming the 4-bit weights from HBM, and what limits a kernel is
// the number of instructions it spends per weight.  One persistent CTA per SM works
// through items (expert, 2 x 128 weight rows, up to 16 of the expert's token rows): for
// gate/up the gate and the up rows of 128 features, for down 256 output rows (two A
// tiles either way).  Per 64-element reduction slab ("stage"):
//   * a raw-weight warp keeps a deep ring of shared-memory slots filled with the
//     stage's 4-bit weight records (one 1-D bulk copy per record row group and four
//     stages) and warms L2 with the CTA's next item;
//   * 8 converter warps turn each 16-row record into exact, unscaled bf16 codes: q - 8
//     for Q4_0 (an integer in [-8, 7]), the E2M1 value for MXFP4.  Lane
//     4g + c of a record holds elements 4c..4c+3 of every 16-element step for rows g
//     and g + 8, which is exactly the thread layout of the 16x256b tensor-memory store,
//     so every lane decodes its own 16 bytes and stores them without any exchange;
//     they also gather the item's token rows (x through the permutation for gate/up, h
//     for down) with cp.async into the 128-byte-swizzled K-major B tile;
//   * one thread issues tcgen05.mma kind::f16 (A from tensor memory, B from shared
//     memory, M = 128, N = 16, K = 16) into one fresh partial-sum accumulator per
//     tile and 32-element quantization block;
//   * 4 epilogue warps read the partial sums with tcgen05.ld and add block scale x
//     partial sum into fp32 registers (one weight row per thread), then store
//     h = silu(g) * u or y as bf16.  The converters copy each stage's block scales
//     into a small ring of their own, so the raw ring is recycled as soon as the codes
//     are decoded, and the token-row tiles have a deeper ring than the A stages, so
//     neither waits on the latency of the MMAs.
// So the only roundings are the fp32 sums, the bf16 h between the projections and the
// bf16 output, as in the grouped GEMV.  The order of every sum is fixed and each output
// depends only on its own weight row and token row, so a token's result does not depend
// on the other tokens of the batch.
//
// Measured limit: each M = 128, N = 16, K = 16 tcgen05.mma costs its issuing thread
// about 70-80 cycles whatever N is, so the 8 MMAs of a 9.2 KB slab bound this design
// near 0.6 of HBM bandwidth.  Below about 8 token rows per expert the mma.sync grouped
// GEMV is faster and the library uses that instead.
#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "pipeline.cuh"
#include "operand.cuh"
#include "tcgen05.cuh"

namespace ftmoe {
namespace dec {

#define GD_WAIT mbar_wait_spin_or_abort
constexpr int GD_TOK = 16;          // token rows per item (MMA N)
constexpr int GD_ROWS = 128;        // weight rows per tile (MMA M, TMEM lanes)
constexpr int GD_EPI_WARPS = 4;     // warps 0..3 (one per TMEM lane quarter)
constexpr int GD_MMA_WARP = 4;      // TMEM owner; lane 0 issues the MMAs
constexpr int GD_RAW_WARP = 5;      // bulk copies of the raw weight records; warps 6, 7 idle
constexpr int GD_CONV0 = 8;         // first converter warp (a multiple of 4)
constexpr int GD_CONV_WARPS = 8;
constexpr int GD_THREADS = (GD_CONV0 + GD_CONV_WARPS) * 32;  // 512
constexpr uint32_t GD_TMEM_COLS = 512;
constexpr int GD_B_TILE = GD_TOK * 128;   // 2 KB of bf16 (16 token rows x 64)
constexpr int GD_STG = GD_TOK * 64;       // epilogue staging per warp: 16 rows x 32 bf16
constexpr int GD_MAX_E = 1024;
constexpr int GD_MAX_NR = 8;
constexpr int GD_MAX_NS = 8;
constexpr int GD_SC_REC = 64;             // scale bytes of one record (16 rows x 2 blocks)

// Per-projection layout.  Tensor-memory columns: NPS partial-sum stages (per A tile
// and quantization block, GD_TOK fp32 columns), then NS stages of A tiles (NT x 32
// columns: 64 bf16 per lane).  The raw weight ring (shared memory) holds super-stages
// of NKB consecutive slabs, filled with one bulk copy per record row group (the records
// of a row group are contiguous along the reduction dimension).
template <int MODE>
struct GdCfg {
  static constexpr int NT = 2;                            // A tiles (MMAs per k-step)
  static constexpr int NS = 4;                            // A stages (tensor memory)
  static constexpr int NPS = 3;                           // partial-sum stages
  static constexpr int NSB = 8;                           // B stages (shared memory)
  static constexpr int LA = NSB - NS;                     // token-row copy stages in flight
  static constexpr int NSS = 8;                           // block-scale stages (shared memory)
  static constexpr int NKB = 4;                           // slabs per raw super-stage
  static constexpr int NR = 4;                            // raw weight super-stages
  static constexpr int NREC = 8 * NT;                     // weight records per stage
  static constexpr int RAW_STAGE = NREC * NKB * 576;      // [record][slab][576]
  static constexpr int PS_STAGE_COLS = NT * 2 * GD_TOK;   // [tile][block][token]
  static constexpr int A_COL0 = NPS * PS_STAGE_COLS;
  static constexpr int A_STAGE_COLS = NT * 32;
  static_assert(A_COL0 + NS * A_STAGE_COLS <= (int)GD_TMEM_COLS, "tensor memory columns");
  static_assert(NS <= GD_MAX_NS && NPS <= GD_MAX_NS && NSB <= GD_MAX_NS && NSS <= GD_MAX_NS &&
                    NR <= GD_MAX_NR && LA >= 1 && LA < NSB, "ring sizes");
  // One MMA commit per stage (on empty[s % NS]) serves every consumer:
  //  * converters wait for the MMAs of stage s - NS before writing A slot s % NS, and
  //    then copy the token rows of stage s + LA into B slot (s + LA) % NSB, whose last
  //    user was stage s + LA - NSB = s - NS;
  //  * the epilogue waits for the MMAs of stage s itself on the same barrier; the MMAs
  //    of stage s + NS cannot complete before the epilogue is done with stage
  //    s + NS - NPS > s (partial-sum ring), so the barrier is never two phases ahead;
  //  * a converter overwrites scale slot s % NSS only after the MMAs of stage s - NS
  //    completed, which needed the epilogue done with stage s - NS - NPS, so the slot's
  //    previous stage (s - NSS) has been read.
  static_assert(NPS < NS, "partial-sum ring shorter than the A ring");
  static_assert(NSS > NS + NPS, "scale ring must outlast the A and partial-sum rings");
};

struct GdTail {
  uint64_t raw_full[GD_MAX_NR], raw_empty[GD_MAX_NR];
  uint64_t a_full[GD_MAX_NS], empty[GD_MAX_NS], sc_full[GD_MAX_NS], ps_empty[GD_MAX_NS], drain;
  uint32_t tmem_base;
  int abort_flag;
  int citem[GD_MAX_E + 1];  // exclusive prefix of items per expert
};
template <int MODE>
constexpr size_t gd_smem_bytes() {
  return 1024 + (size_t)GdCfg<MODE>::NSB * GD_B_TILE + (size_t)GdCfg<MODE>::NR * GdCfg<MODE>::RAW_STAGE +
         (size_t)GdCfg<MODE>::NSS * GdCfg<MODE>::NREC * GD_SC_REC + (size_t)GD_EPI_WARPS * GD_STG +
         sizeof(GdTail);
}


struct GemmArgs {
  const int32_t* offsets;
  const int32_t* sorted_pair;  // gate/up: pair of each permuted row (nullptr: identity)
  int k, E, T, P;
  const uint16_t* act;  // gate/up: x [T][H] (rows gathered); down: h [P][I] (contiguous rows)
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
  const int ntt = (ne + GD_TOK - 1) / GD_TOK;
  const int ft = local / ntt, tt = local - ft * ntt;
  it.r0 = beg + tt * GD_TOK;
  it.n = min(GD_TOK, ne - tt * GD_TOK);
  it.f0 = ft * (MODE == 0 ? GD_ROWS : 2 * GD_ROWS);
  return it;
}

// First matrix row of record ri (tile ri / 8, 16-row group ri % 8) of an item, and
// whether that row group lies inside the projection's result rows.  Gate/up: tile 0
// holds the gate rows and tile 1 the up rows of the same features; down: tile 1 holds
// the 128 rows after tile 0's.
template <int MODE>
__device__ __forceinline__ int gm_record_row(const GmItem& it, int ri, const GemmArgs& a,
                                             bool& ok) {
  const int row = it.f0 + (MODE == 1 ? (ri >> 3) * GD_ROWS : 0) + (ri & 7) * 16;
  ok = row < a.nrows;
  return (MODE == 0 && (ri >> 3)) ? row + a.up_row0 : row;
}

// ---------------------------------------------------------------- weight decode
// One converter warp decodes a 16-row x 64-element record into its 16 tensor-memory
// lanes (the A tile rows of the record) at `taddr`.  Lane L = 4g + c reads its own 16
// bytes: word j holds elements 16j + 4c + (0..3) of row g in the low nibbles (bytes in
// the order e0, e2, e1, e3) and of row g + 8 in the high nibbles.  In the 16x256b store
// shape register 4j + m of lane 4g + c goes to row g + 8 (m >> 1), column
// 8j + 2c + (m & 1) (two bf16 per 32-bit column), which is where those elements belong.
template <int QT>
__device__ __forceinline__ void convert_record(uint32_t rec, uint32_t taddr, int lane) {
  const uint4 q = lds128(rec + lane * 16);
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
  uint32_t out[16];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    decode_plain<QT>(w[j] & 0x0F0F0F0Fu, out[4 * j + 0], out[4 * j + 1]);
    decode_plain<QT>((w[j] >> 4) & 0x0F0F0F0Fu, out[4 * j + 2], out[4 * j + 3]);
  }
  tmem_st_16x256b_x4(taddr, out);
}

// Block scale of weight row g + 8 h for quantization block b, as fp32, from a copy of
// a record's scale bytes at `sc` (per row group g: (g, b0), (g + 8, b0), (g, b1),
// (g + 8, b1), fp16 for Q4_0, E8M0 for MXFP4).
template <int QT>
__device__ __forceinline__ float block_scale(uint32_t sc, int g, int h, int b) {
  if (QT == FTMOE_Q4_0) {
    const uint32_t wd = lds32(sc + g * 8 + b * 4);
    return half_bits_to_f32(h ? (wd >> 16) : (wd & 0xFFFFu));
  } else {
    const uint32_t wd = lds32(sc + g * 4);
    return e8m0_to_f32((wd >> (8 * (2 * b + h))) & 0xFFu);
  }
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

template <int QT, int MODE, class Tab>
__global__ void __launch_bounds__(GD_THREADS, 1)
    gemm_decode_kernel(const GemmArgs a, const __grid_constant__ Tab tab) {
  using C = GdCfg<MODE>;
  constexpr int RB = rec_bytes(QT);
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t base_addr = (raw_addr + 1023u) & ~1023u;  // B stages (128-byte swizzle)
  uint8_t* base = smem_raw + (base_addr - raw_addr);
  const uint32_t rawring = base_addr + C::NSB * GD_B_TILE;
  const uint32_t scring = rawring + C::NR * C::RAW_STAGE;  // [NSS][NREC][64] block scales
  const uint32_t staging = scring + C::NSS * C::NREC * GD_SC_REC;
  GdTail& tl = *reinterpret_cast<GdTail*>(base + (size_t)C::NSB * GD_B_TILE + (size_t)C::NR * C::RAW_STAGE +
                                          (size_t)C::NSS * C::NREC * GD_SC_REC + GD_EPI_WARPS * GD_STG);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  volatile int* abort_flag = &tl.abort_flag;

  if (MODE == 0) pdl_wait();  // offsets come from the permutation kernel
  if (tid == 0) {
    for (int s = 0; s < C::NR; ++s) {
      mbar_init(&tl.raw_full[s], 1);
      mbar_init(&tl.raw_empty[s], GD_CONV_WARPS);
    }
    for (int s = 0; s < C::NS; ++s) {
      mbar_init(&tl.a_full[s], GD_CONV_WARPS);
      mbar_init(&tl.empty[s], 1);
    }
    for (int s = 0; s < C::NSS; ++s) mbar_init(&tl.sc_full[s], GD_CONV_WARPS);
    for (int s = 0; s < C::NPS; ++s) mbar_init(&tl.ps_empty[s], GD_EPI_WARPS);
    mbar_init(&tl.drain, 1);
    tl.abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == GD_MMA_WARP) {
    tmem_alloc(&tl.tmem_base, GD_TMEM_COLS);
    tmem_relinquish();
  }
  // items per expert: ceil(n_e / GD_TOK) token tiles x weight-row slices
  if (warp == 0) {
    int carry = 0;
    for (int e0 = 0; e0 < a.E; e0 += 32) {
      const int e = e0 + lane;
      int v = 0;
      if (e < a.E) {
        int r0, n;
        expert_rows(a.offsets, e, a.P, a.status, r0, n);
        v = ((n + GD_TOK - 1) / GD_TOK) * a.ft_per_expert;
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
  pdl_launch_dependents();
  const int nitems = tl.citem[a.E];
  const int G = gridDim.x;

  if (warp == GD_RAW_WARP) {
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
      for (int kb0 = 0; kb0 < a.S; kb0 += C::NKB) {
        const int nkb = min(C::NKB, a.S - kb0);
        if (!GD_WAIT(&tl.raw_empty[rslot], rphase ^ 1u, abort_flag, a.status)) break;
        if (lane == 0) mbar_arrive_expect_tx(&tl.raw_full[rslot], (uint32_t)(nrec * nkb * RB));
        __syncwarp();
        if (lane < C::NREC && rok)
          bulk_g2s(base + C::NSB * GD_B_TILE + rslot * C::RAW_STAGE + lane * (C::NKB * RB),
                   rec0 + (long long)kb0 * RB, (uint32_t)(nkb * RB), &tl.raw_full[rslot]);
        if (++rslot == C::NR) { rslot = 0; rphase ^= 1u; }
      }
      if (*abort_flag) break;
    }
  } else if (warp >= GD_CONV0) {
    // ------------------------------------------------------------ converters
    const int ct = tid - GD_CONV0 * 32;
    const int cw = ct >> 5;          // converter warp; its TMEM lane quarter = cw % 4
    const int grp = 2 * (cw & 3) + (cw >> 2);  // record row group: TMEM lanes 16 grp ..
    const uint32_t tlane = tmem + ((uint32_t)(16 * grp) << 16) + C::A_COL0;
    int slot = 0, rslot = 0, sslot = 0;
    uint32_t phase = 0, rphase = 0;
    constexpr int SCB = QT == FTMOE_Q4_0 ? 64 : 32;  // scale bytes per record
    // token rows: threads ct < GD_TOK * 8 copy 16-byte chunk (ct & 7) of row ct >> 3, LA
    // stages ahead of the conversion so that the copies' latency hides behind the decode.
    // Every call commits one cp.async group (empty past the last stage), so that waiting
    // for all but the newest LA groups always means "this stage's rows have landed".
    const int brow = ct >> 3, ch = ct & 7;
    int bi = blockIdx.x, bkb = 0, bslot = 0;
    const uint16_t* rowp = nullptr;
    auto load_rows = [&](int item) {
      const GmItem it = gm_item<MODE>(item, a, tl.citem);
      rowp = nullptr;
      if (brow < it.n) {
        const long long ar = row_token(a.sorted_pair, it.r0 + brow, a.k, a.T, a.status);
        rowp = a.act + ar * a.act_ld + ch * 8;
      }
    };
    auto issue_rows = [&]() {  // copies of stage (bi, bkb); its B slot is free (see GdCfg)
      if (bi >= nitems) {
        cp_async_commit();
        return;
      }
      if (rowp) {
        const bool kok = bkb * 64 + ch * 8 < a.K;  // beyond K: zeros
        cp_async16(base_addr + bslot * GD_B_TILE + (brow >> 3) * 1024 + (brow & 7) * 128 +
                       ((ch ^ (brow & 7)) * 16),
                   kok ? rowp + bkb * 64 : rowp, kok ? 16u : 0u);
      }
      cp_async_commit();
      if (++bslot == C::NSB) bslot = 0;
      if (++bkb == a.S) {
        bkb = 0;
        bi += G;
        if (bi < nitems) load_rows(bi);
      }
    };
    if (MODE == 1) pdl_wait();  // h comes from the gate/up kernel
    if (bi < nitems) load_rows(bi);
    for (int s = 0; s < C::LA; ++s) issue_rows();
    for (int i = blockIdx.x; i < nitems; i += G) {
      const GmItem it = gm_item<MODE>(i, a, tl.citem);
      bool rok[C::NT];
#pragma unroll
      for (int t = 0; t < C::NT; ++t) gm_record_row<MODE>(it, t * 8 + grp, a, rok[t]);
      for (int kb = 0; kb < a.S; ++kb) {
        const int jkb = kb % C::NKB;  // slab within the raw super-stage
        const bool last_of_super = jkb == C::NKB - 1 || kb == a.S - 1;
        if (!GD_WAIT(&tl.empty[slot], phase ^ 1u, abort_flag, a.status)) break;
        issue_rows();
        if (!GD_WAIT(&tl.raw_full[rslot], rphase, abort_flag, a.status)) break;
        tc_fence_after_sync();
#pragma unroll
        for (int t = 0; t < C::NT; ++t) {  // (records outside the result rows are left as they are)
          const uint32_t rec = rawring + rslot * C::RAW_STAGE + ((t * 8 + grp) * C::NKB + jkb) * RB;
          if (rok[t]) {
            convert_record<QT>(rec, tlane + slot * C::A_STAGE_COLS + t * 32, lane);
            // the record's block scales go to the scale ring for the epilogue
            if (lane < SCB / 4)
              asm volatile("st.shared.u32 [%0], %1;" ::"r"(scring + (sslot * C::NREC + t * 8 + grp) * GD_SC_REC +
                                                          lane * 4),
                           "r"(lds32(rec + REC_CODE_BYTES + lane * 4))
                           : "memory");
          }
        }
        tmem_wait_st();
        cp_async_wait<C::LA>();  // this stage's rows have landed
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) {
          if (last_of_super) mbar_arrive(&tl.raw_empty[rslot]);
          mbar_arrive(&tl.sc_full[sslot]);
          mbar_arrive(&tl.a_full[slot]);
        }
        if (last_of_super && ++rslot == C::NR) { rslot = 0; rphase ^= 1u; }
        if (++slot == C::NS) { slot = 0; phase ^= 1u; }
        if (++sslot == C::NSS) sslot = 0;
      }
      if (*abort_flag) break;
    }
    cp_async_wait<0>();
  } else if (warp == GD_MMA_WARP) {
    // ------------------------------------------------------------ MMA issue
    if (lane == 0) {
      int slot = 0, ps = 0, bslot = 0;
      uint32_t phase = 0, pphase = 0;
      const uint32_t idesc = idesc_bf16_f32(GD_ROWS, GD_TOK);
      bool ok = true;
      for (int i = blockIdx.x; i < nitems && ok; i += G) {
        for (int kb = 0; kb < a.S; ++kb) {
          if (!GD_WAIT(&tl.a_full[slot], phase, abort_flag, a.status) ||
              !GD_WAIT(&tl.ps_empty[ps], pphase ^ 1u, abort_flag, a.status)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint32_t bs = base_addr + bslot * GD_B_TILE;
          const uint32_t as = tmem + C::A_COL0 + slot * C::A_STAGE_COLS;
          const uint32_t pd = tmem + ps * C::PS_STAGE_COLS;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {  // k16 step; block kk / 2 starts from zero
            const uint64_t bd = sdesc_kmajor_sw128(bs + 32 * kk);
#pragma unroll
            for (int t = 0; t < C::NT; ++t) {
              const uint32_t d = pd + (t * 2 + (kk >> 1)) * GD_TOK;
              mma_bf16_tmem_a(d, as + t * 32 + 8 * kk, bd, idesc, (uint32_t)(kk & 1));
            }
          }
          mma_commit(&tl.empty[slot]);
          if (++slot == C::NS) { slot = 0; phase ^= 1u; }
          if (++bslot == C::NSB) bslot = 0;
          if (++ps == C::NPS) { ps = 0; pphase ^= 1u; }
        }
      }
      // every MMA issued above has finished once this arrives
      mma_commit(&tl.drain);
      mbar_wait_or_abort(&tl.drain, 0, abort_flag, a.status, 100000000ull);
    }
    __syncwarp();
  } else if (warp < GD_EPI_WARPS) {
    // ------------------------------------------------------------ epilogue (warps 0..3)
    const int q = warp;                 // TMEM lanes [32q, 32q + 32): weight rows of the tile
    const int r = 32 * q + lane;
    const int grp = r >> 4, g = r & 7, h = (r >> 3) & 1;
    const uint32_t lane_base = tmem + ((uint32_t)(32 * q) << 16);
    // lanes l and l ^ 1 hold adjacent features: they swap values to store bf16 pairs
    const int odd = lane & 1;
    const uint32_t stg = staging + q * GD_STG;
    int ps = 0, sslot = 0, eslot = 0;
    uint32_t sphase = 0, ephase = 0;
    for (int i = blockIdx.x; i < nitems; i += G) {
      const GmItem it = gm_item<MODE>(i, a, tl.citem);
      const int nch = (it.n + 3) >> 2;  // 4-token chunks with real tokens
      float acc[C::NT][GD_TOK];
#pragma unroll
      for (int t = 0; t < C::NT; ++t)
#pragma unroll
        for (int j = 0; j < GD_TOK; ++j) acc[t][j] = 0.f;
      bool ok = true;
      for (int kb = 0; kb < a.S; ++kb) {
        if (!GD_WAIT(&tl.sc_full[sslot], sphase, abort_flag, a.status) ||
            !GD_WAIT(&tl.empty[eslot], ephase, abort_flag, a.status)) {  // this stage's MMAs
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const bool b1 = kb * 64 + 32 < a.K;  // the slab's second block lies inside K
#pragma unroll
        for (int t = 0; t < C::NT; ++t) {
          const uint32_t sc = scring + (sslot * C::NREC + t * 8 + grp) * GD_SC_REC;
          const float d0 = block_scale<QT>(sc, g, h, 0);
          const float d1 = b1 ? block_scale<QT>(sc, g, h, 1) : 0.f;
          uint32_t p0[GD_TOK], p1[GD_TOK];
          const uint32_t pc = lane_base + ps * C::PS_STAGE_COLS + t * 2 * GD_TOK;
          tmem_ld16(pc, p0);
          tmem_ld16(pc + GD_TOK, p1);
          tmem_wait_ld();
#pragma unroll
          for (int c = 0; c < GD_TOK / 4; ++c) {
            if (c < nch) {
#pragma unroll
              for (int j = 4 * c; j < 4 * c + 4; ++j) {
                acc[t][j] = fmaf(d0, __uint_as_float(p0[j]), acc[t][j]);
                if (b1) acc[t][j] = fmaf(d1, __uint_as_float(p1[j]), acc[t][j]);
              }
            }
          }
        }
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tl.ps_empty[ps]);
        if (++sslot == C::NSS) { sslot = 0; sphase ^= 1u; }
        if (++eslot == C::NS) { eslot = 0; ephase ^= 1u; }
        if (++ps == C::NPS) ps = 0;
      }
      if (!ok) break;
      // ---- item result: h = silu(gate) * up (one output tile), or y (two); row r of each
      // output tile for tokens 0..n-1.  The warp's 32 features x 16 tokens go through its
      // staging tile [token][feature] so that the global stores are 16-byte vectors.
#pragma unroll
      for (int ot = 0; ot < (MODE == 0 ? 1 : C::NT); ++ot) {
        float v[GD_TOK];
#pragma unroll
        for (int j = 0; j < GD_TOK; ++j) {
          if (MODE == 0) {
            const float gg = acc[0][j];
            v[j] = __fdividef(gg, 1.0f + __expf(-gg)) * acc[1][j];
          } else {
            v[j] = acc[ot][j];
          }
        }
        const int fw = it.f0 + ot * GD_ROWS + 32 * q;  // first feature of this warp
        const bool fok = fw < a.nrows;
        uint16_t* obase = a.out + (long long)it.r0 * a.out_ld + fw + 8 * (lane & 3);
#pragma unroll
        for (int p = 0; p < GD_TOK / 2; ++p) {
          const float send = odd ? v[2 * p] : v[2 * p + 1];
          const float recv = __shfl_xor_sync(0xffffffffu, send, 1);
          const float lo = odd ? recv : v[2 * p];
          const float hi = odd ? v[2 * p + 1] : recv;
          const uint32_t w = (uint32_t)f32_to_bf16_bits(lo) | ((uint32_t)f32_to_bf16_bits(hi) << 16);
          asm volatile("st.shared.u32 [%0], %1;" ::"r"(stg + (2 * p + odd) * 64 + (lane & ~1) * 2), "r"(w)
                       : "memory");
        }
        __syncwarp();
#pragma unroll
        for (int r4 = 0; r4 < GD_TOK / 8; ++r4) {
          const int row = 8 * r4 + (lane >> 2);
          const uint4 d = lds128(stg + row * 64 + (lane & 3) * 16);
          if (fok && row < it.n) *reinterpret_cast<uint4*>(obase + (long long)row * a.out_ld) = d;
        }
        __syncwarp();
      }
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == GD_MMA_WARP) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, GD_TMEM_COLS);
  }
}

template <int QT, int MODE, class Tab>
static cudaError_t gd_launch(const GemmArgs& a, const Tab& tab, cudaStream_t st) {
  const DeviceInfo* di = device_info();
  if (!di) return cudaErrorUnknown;
  constexpr size_t smem = gd_smem_bytes<MODE>();
  static_assert(smem <= 232448, "shared memory per CTA");
  cudaError_t err = set_smem_limit<gemm_decode_kernel<QT, MODE, Tab>>(smem);
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(di->sm_count);
  cfg.blockDim = dim3(GD_THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gemm_decode_kernel<QT, MODE, Tab>, a, tab);
}

template <int QT, class Tab>
static cudaError_t gd_launch_qt(const FfnProblem& pb, const Tab& tab, cudaStream_t st) {
  const DeviceInfo* di = device_info();
  if (!di) return cudaErrorUnknown;
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
  a.ft_per_expert = (pb.I + GD_ROWS - 1) / GD_ROWS;
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
  d.ft_per_expert = (pb.H + 2 * GD_ROWS - 1) / (2 * GD_ROWS);
  cudaError_t err = gd_launch<QT, 0>(a, tab, st);
  if (err != cudaSuccess) return err;
  return gd_launch<QT, 1>(d, tab, st);
}

}  // namespace dec

cudaError_t launch_ffn_gemm_decode(const FfnProblem& pb, cudaStream_t st) {
  // NVFP4's 16-element blocks would need twice the partial-sum stages and MXFP8's records
  // another converter; the library runs those formats through the grouped GEMV at these
  // batch sizes instead
  if (pb.qtype == FTMOE_NVFP4 || pb.qtype == FTMOE_MXFP8) return cudaErrorNotSupported;
  if (pb.E > dec::GD_MAX_E) return cudaErrorNotSupported;
  if (pb.table) {
    dec::GmWithTable t;
    t.t = *pb.table;
    return pb.qtype == FTMOE_Q4_0 ? dec::gd_launch_qt<FTMOE_Q4_0>(pb, t, st)
                                  : dec::gd_launch_qt<FTMOE_MXFP4>(pb, t, st);
  }
  dec::GmNoTable t;
  return pb.qtype == FTMOE_Q4_0 ? dec::gd_launch_qt<FTMOE_Q4_0>(pb, t, st)
                                : dec::gd_launch_qt<FTMOE_MXFP4>(pb, t, st);
}

}  // namespace ftmoe
