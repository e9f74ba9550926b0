// Grouped expert FFN for few rows per expert (decode): HBM-bound streaming of the
// 4-bit expert weights with in-register decode (the ExpertFFN of the FreeToken
// architecture walkthrough §五, on GGUF Q4_0 / MXFP4 banks, §六).
//
// Persistent CTAs: one producer warp streams 16-row x 64-column weight records with
// 1-D bulk copies (TMA) into a ring of shared-memory stages; eight consumer warps
// turn the codes into exact bf16 (q - 8, or the E2M1 value) and feed them as the A
// operand of m16n8k16 MMAs whose B operand is up to 8 token rows; after the two
// k-steps of a quantization block the partial sums are scaled by that block's scale
// in fp32.  So the only roundings are the fp32 accumulation, the bf16 h between the
// projections and the bf16 output.
//
// Unit of work = (active expert, two 16-row tiles): gate and up tile of one group of
// 16 features (gate/up), or two tiles of 16 output rows (down).  A unit's records
// arrive in chunks of up to 16 slabs (64 reduction elements each); consumer warp w
// works on slab w of every chunk for both tiles, with its token fragment (up to 8
// token rows) loaded into registers one chunk ahead, and the 16 partial sums of a
// tile are added in shared memory at the end of the unit.
#include "common.cuh"
#include "internal.h"
#include "pipeline.cuh"

namespace ftmoe {

constexpr int GV_CONS_WARPS = 16;
constexpr int GV_THREADS = (GV_CONS_WARPS + 1) * 32;
constexpr int GV_CH = 16;      // slabs per chunk (one per consumer warp)
constexpr int GV_NSTAGE = 8;   // 8 x 18 KB of weights in flight per SM

template <int QT>
struct GvSmem {
  static constexpr int STAGE = 2 * GV_CH * rec_bytes(QT);
  uint8_t stage[GV_NSTAGE][STAGE];
  float red[2][GV_CONS_WARPS][2][4][32];  // [parity][warp][tile][C fragment][lane]
  uint64_t full[GV_NSTAGE];
  uint64_t empty[GV_NSTAGE];
  uint64_t ebar;  // all consumer warps meet here once per unit epilogue
  int act[1024];
  int wsum[GV_THREADS / 32];
};

struct GemvArgs {
  const int32_t* offsets;
  const int32_t* sorted_pair;  // nullptr: row r is token r (k == 1)
  int k, E;
  const uint16_t* act;  // gate/up: x [T][H]; down: h [P][I]
  int act_ld;
  uint16_t* out;        // gate/up: h [P][I]; down: y_perm [P][H]
  int out_ld;
  const uint8_t* wbase;  // tiles of this projection for expert 0
  long long wstride;     // bytes between experts
  long long table_off;   // offset of this projection inside a blob
  int S;                 // slabs per row
  int K;                 // reduction length
  int up_rt;             // gate/up: first row tile of the up half (I / 16)
  int units_per_expert;  // gate/up: I / 16; down: H / 32
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

// Ordered list of experts with at least one row, built by every CTA from offsets.
__device__ __forceinline__ int build_active_list(const int32_t* offsets, int E, int* s_act,
                                                 int* s_wsum) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  constexpr int NW = GV_THREADS / 32;
  int nact = 0;
  for (int e0 = 0; e0 < E; e0 += GV_THREADS) {
    const int e = e0 + threadIdx.x;
    const bool f = e < E && offsets[e + 1] > offsets[e];
    const unsigned b = __ballot_sync(0xffffffffu, f);
    if (lane == 0) s_wsum[wid] = __popc(b);
    __syncthreads();
    int before = nact, tot = 0;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      if (w < wid) before += s_wsum[w];
      tot += s_wsum[w];
    }
    if (f) s_act[before + __popc(b & ((1u << lane) - 1u))] = e;
    nact += tot;
    __syncthreads();
  }
  return nact;
}

template <int QT>
__device__ __forceinline__ void decode_word(uint32_t w, uint32_t (&a)[4]) {
  if (QT == FTMOE_Q4_0) q4_word_to_bf16x2(w, a); else e2m1_word_to_bf16x2(w, a);
}

// Scales of rows (g, g+8) for both blocks of a record: [b][h] as fp32.
template <int QT>
__device__ __forceinline__ void load_scales(const uint8_t* rec, int g, float (&sc)[2][2]) {
  if (QT == FTMOE_Q4_0) {
    const uint2 s = *reinterpret_cast<const uint2*>(rec + REC_CODE_BYTES + g * 8);
    sc[0][0] = half_bits_to_f32(s.x & 0xFFFFu);
    sc[0][1] = half_bits_to_f32(s.x >> 16);
    sc[1][0] = half_bits_to_f32(s.y & 0xFFFFu);
    sc[1][1] = half_bits_to_f32(s.y >> 16);
  } else {
    const uint32_t s = *reinterpret_cast<const uint32_t*>(rec + REC_CODE_BYTES + g * 4);
    sc[0][0] = e8m0_to_f32(s & 0xFFu);
    sc[0][1] = e8m0_to_f32((s >> 8) & 0xFFu);
    sc[1][0] = e8m0_to_f32((s >> 16) & 0xFFu);
    sc[1][1] = e8m0_to_f32(s >> 24);
  }
}

struct UnitInfo {
  int e, r0, n_e, tile0, tile1;
};

template <int MODE>
__device__ __forceinline__ UnitInfo unit_info(const GemvArgs& a, const int* s_act, int unit) {
  UnitInfo u;
  const int ui = unit / a.units_per_expert;
  const int sub = unit - ui * a.units_per_expert;
  u.e = s_act[ui];
  u.r0 = a.offsets[u.e];
  u.n_e = a.offsets[u.e + 1] - u.r0;
  if (MODE == 0) {
    u.tile0 = sub;
    u.tile1 = a.up_rt + sub;
  } else {
    u.tile0 = 2 * sub;
    u.tile1 = 2 * sub + 1;
  }
  return u;
}

template <int QT, int MODE, class Tab>
__global__ void __launch_bounds__(GV_THREADS, 1) gemv_ffn_kernel(const GemvArgs a,
                                                                 const __grid_constant__ Tab tab) {
  using SM = GvSmem<QT>;
  constexpr int RB = rec_bytes(QT);
  extern __shared__ __align__(128) uint8_t smem_raw[];
  SM& sm = *reinterpret_cast<SM*>(smem_raw);
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;

  if (MODE == 0) pdl_wait();  // offsets come from the permutation kernel
  pdl_launch_dependents();

  if (threadIdx.x == 0) {
    for (int i = 0; i < GV_NSTAGE; ++i) {
      mbar_init(&sm.full[i], 1);
      mbar_init(&sm.empty[i], GV_CONS_WARPS);
    }
    mbar_init(&sm.ebar, GV_CONS_WARPS);
    fence_barrier_init();
  }
  const int nact = build_active_list(a.offsets, a.E, sm.act, sm.wsum);  // contains __syncthreads
  const int total = nact * a.units_per_expert;
  // contiguous share of the units per CTA
  const int u_begin = (int)((long long)total * blockIdx.x / gridDim.x);
  const int u_end = (int)((long long)total * (blockIdx.x + 1) / gridDim.x);
  const int nchunk = (a.S + GV_CH - 1) / GV_CH;
  const bool ragged = (a.K & 63) != 0;

  if (wid == GV_CONS_WARPS) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol = l2_evict_first_policy();
      uint32_t it = 0;
      bool ok = true;
      for (int unit = u_begin; unit < u_end && ok; ++unit) {
        const UnitInfo u = unit_info<MODE>(a, sm.act, unit);
        const uint8_t* wexp = tab.get(u.e, a);
        const uint8_t* b0 = wexp + (long long)u.tile0 * a.S * RB;
        const uint8_t* b1 = wexp + (long long)u.tile1 * a.S * RB;
        const int rounds = (u.n_e + 7) / 8;
        for (int r = 0; r < rounds && ok; ++r) {
          for (int c = 0; c < nchunk; ++c, ++it) {
            const int st = it % GV_NSTAGE;
            const uint32_t ph = (it / GV_NSTAGE) & 1u;
            if (!mbar_wait(&sm.empty[st], ph ^ 1u, a.status)) { ok = false; break; }
            const int ns = min(GV_CH, a.S - c * GV_CH);
            const uint32_t wbytes = (uint32_t)(ns * RB);
            mbar_arrive_expect_tx(&sm.full[st], 2 * wbytes);
            bulk_g2s_stream(&sm.stage[st][0], b0 + (long long)c * GV_CH * RB, wbytes, &sm.full[st], pol);
            bulk_g2s_stream(&sm.stage[st][GV_CH * RB], b1 + (long long)c * GV_CH * RB, wbytes, &sm.full[st], pol);
          }
        }
      }
      // drain: do not leave the CTA with copies in flight
      for (uint32_t j = (it > GV_NSTAGE ? it - GV_NSTAGE : 0); j < it; ++j)
        mbar_wait(&sm.full[j % GV_NSTAGE], (j / GV_NSTAGE) & 1u, a.status);
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  if (MODE == 1) pdl_wait();  // h comes from the gate/up kernel
  const int g = lane >> 2, c4 = lane & 3;
  // flat walk over (unit, round, chunk); the token fragment of the next step is loaded
  // into registers before waiting for the current step's weights
  int unit = u_begin, r = 0, c = 0;
  UnitInfo u;
  if (unit < u_end) u = unit_info<MODE>(a, sm.act, unit);
  auto load_b = [&](const UnitInfo& uu, int rr_, int cc, uint2 (&bv)[4]) {
    const int s = cc * GV_CH + wid;
    if (s >= a.S) return;
    const int rr = min(8 * rr_ + g, uu.n_e - 1);  // padded lanes re-read a valid row
    long long row;
    if (MODE == 0) row = a.sorted_pair ? a.sorted_pair[uu.r0 + rr] / a.k : (uu.r0 + rr);
    else row = uu.r0 + rr;
    const uint2* src = reinterpret_cast<const uint2*>(a.act + row * a.act_ld + s * 64 + 4 * c4);
    const bool half = ragged && s == a.S - 1;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (j >= 2 && half) break;
      bv[j] = MODE == 0 ? __ldg(src + 4 * j) : __ldcg(src + 4 * j);
    }
  };
  uint2 bnext[4] = {};
  if (unit < u_end) load_b(u, 0, 0, bnext);
  uint32_t it = 0;
  int ep = 0;  // epilogue count (red buffer parity)
  float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
  while (unit < u_end) {
    const uint2 bv[4] = {bnext[0], bnext[1], bnext[2], bnext[3]};
    // next position
    int nunit = unit, nr = r, nc = c + 1;
    const int rounds = (u.n_e + 7) / 8;
    if (nc == nchunk) {
      nc = 0;
      if (++nr == rounds) { nr = 0; ++nunit; }
    }
    UnitInfo nu = u;
    if (nunit != unit && nunit < u_end) nu = unit_info<MODE>(a, sm.act, nunit);
    if (nunit < u_end) load_b(nu, nr, nc, bnext);

    const int st = it % GV_NSTAGE;
    const uint32_t ph = (it / GV_NSTAGE) & 1u;
    if (!mbar_wait(&sm.full[st], ph, a.status)) return;
    const int ns = min(GV_CH, a.S - c * GV_CH);
    if (wid < ns) {
      const int s = c * GV_CH + wid;
      const bool half = ragged && s == a.S - 1;
#pragma unroll
      for (int ti = 0; ti < 2; ++ti) {
        const uint8_t* rec = &sm.stage[st][(ti * GV_CH + wid) * RB];
        const uint4 q = *reinterpret_cast<const uint4*>(rec + lane * 16);
        float sc[2][2];
        load_scales<QT>(rec, g, sc);
        const uint32_t wj[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int b = 0; b < 2; ++b) {
          if (b == 1 && half) break;
          float part[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int jj = 0; jj < 2; ++jj) {
            uint32_t av[4];
            decode_word<QT>(wj[2 * b + jj], av);
            mma_16816(part, av, bv[2 * b + jj].x, bv[2 * b + jj].y);
          }
          acc[ti][0] = fmaf(sc[b][0], part[0], acc[ti][0]);
          acc[ti][1] = fmaf(sc[b][0], part[1], acc[ti][1]);
          acc[ti][2] = fmaf(sc[b][1], part[2], acc[ti][2]);
          acc[ti][3] = fmaf(sc[b][1], part[3], acc[ti][3]);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.empty[st]);
    ++it;

    if (nc == 0) {
      // ---- end of (unit, round): add the 16 slab partial sums of each tile
      const int tok0 = 8 * r;
      float (*red)[2][4][32] = sm.red[ep & 1];
#pragma unroll
      for (int ti = 0; ti < 2; ++ti)
#pragma unroll
        for (int qq = 0; qq < 4; ++qq) {
          red[wid][ti][qq][lane] = acc[ti][qq];
          acc[ti][qq] = 0.f;
        }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.ebar);
      if (!mbar_wait(&sm.ebar, ep & 1, a.status)) return;
      if (wid < 4) {
        const int qq = wid;
        float v0 = 0.f, v1 = 0.f;
#pragma unroll
        for (int w2 = 0; w2 < GV_CONS_WARPS; ++w2) {
          v0 += red[w2][0][qq][lane];
          v1 += red[w2][1][qq][lane];
        }
        const int rr = tok0 + 2 * c4 + (qq & 1);
        if (rr < u.n_e) {
          const int rofs = g + 8 * (qq >> 1);
          uint16_t* orow = a.out + (long long)(u.r0 + rr) * a.out_ld;
          if (MODE == 0) {
            orow[u.tile0 * 16 + rofs] = f32_to_bf16_bits(silu_f32(v0) * v1);
          } else {
            orow[u.tile0 * 16 + rofs] = f32_to_bf16_bits(v0);
            orow[u.tile1 * 16 + rofs] = f32_to_bf16_bits(v1);
          }
        }
      }
      ++ep;
    }
    unit = nunit;
    r = nr;
    c = nc;
    u = nu;
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

template <int QT, int MODE, class Tab>
static cudaError_t launch_mode(const GemvArgs& a, const Tab& tab, int max_active, cudaStream_t st) {
  const DeviceInfo* di = device_info();
  if (!di) return cudaErrorUnknown;
  auto kern = gemv_ffn_kernel<QT, MODE, Tab>;
  const size_t smem = sizeof(GvSmem<QT>);
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  int grid = di->sm_count;
  const int upper = max_active * a.units_per_expert;
  if (upper < grid) grid = upper;
  if (grid < 1) grid = 1;
  return launch_pdl(kern, dim3(grid), dim3(GV_THREADS), smem, st, a, tab);
}

template <int QT, class Tab>
static cudaError_t launch_qt(const FfnProblem& pb, const Tab& tab, cudaStream_t st) {
  const DeviceInfo* di = device_info();
  if (!di) return cudaErrorUnknown;
  const int max_active = pb.P < pb.E ? pb.P : pb.E;
  GemvArgs a{};
  a.offsets = pb.offsets;
  a.sorted_pair = pb.sorted_pair;
  a.k = pb.k;
  a.E = pb.E;
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
  a.up_rt = pb.I / 16;
  a.units_per_expert = pb.I / 16;
  cudaError_t err = launch_mode<QT, 0>(a, tab, max_active, st);
  if (err != cudaSuccess) return err;
  // down
  a.act = pb.h_act;
  a.act_ld = pb.I;
  a.out = pb.y_perm;
  a.out_ld = pb.H;
  a.wbase = pb.w2;
  a.wstride = (long long)tiles_bytes_per_expert(pb.qtype, pb.H, pb.I);
  a.table_off = (long long)pb.w13_bytes;
  a.S = slabs_of(pb.I);
  a.K = pb.I;
  a.up_rt = 0;
  a.units_per_expert = pb.H / 32;
  return launch_mode<QT, 1>(a, tab, max_active, st);
}

cudaError_t launch_ffn_gemv(const FfnProblem& pb, cudaStream_t st) {
  if (pb.table) {
    WithTable t;
    t.t = *pb.table;
    return pb.qtype == FTMOE_Q4_0 ? launch_qt<FTMOE_Q4_0>(pb, t, st) : launch_qt<FTMOE_MXFP4>(pb, t, st);
  }
  NoTable t;
  return pb.qtype == FTMOE_Q4_0 ? launch_qt<FTMOE_Q4_0>(pb, t, st) : launch_qt<FTMOE_MXFP4>(pb, t, st);
}

}  // namespace ftmoe
