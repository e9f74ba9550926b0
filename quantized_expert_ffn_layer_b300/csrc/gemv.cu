// Grouped expert FFN for few rows per expert (decode): HBM-bound streaming of the
// 4-bit expert weights with in-register decode (the ExpertFFN of the FreeToken
// architecture walkthrough §五, on GGUF Q4_0 / MXFP4 banks, §六).
//
// Work item = (active expert, a few 16-row tiles).  Each warp streams tile records
// with one 16-byte load per lane, turns the codes into exact bf16 (q - 8 or the
// E2M1 value) and feeds them as the A operand of m16n8k16 MMAs whose B operand is
// up to 8 token rows; after the two k-steps of a quantization block the partial
// sums are scaled by that block's scale in fp32.  So the only roundings are the
// fp32 accumulation, the bf16 h between the projections and the bf16 output.
// The reduction dimension is split over KS warps and summed in shared memory.
#include "common.cuh"
#include "internal.h"

namespace ftmoe {

constexpr int GEMV_THREADS = 256;  // 8 warps
constexpr int GEMV_TG = 2;         // token groups of 8 per pass

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
  int tiles_total;       // gate/up: feature tiles (I / 16); down: row tiles (H / 16)
  int items_per_expert;  // ceil(tiles_total / RT)
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
  int nact = 0;
  for (int e0 = 0; e0 < E; e0 += GEMV_THREADS) {
    const int e = e0 + threadIdx.x;
    const bool f = e < E && offsets[e + 1] > offsets[e];
    const unsigned b = __ballot_sync(0xffffffffu, f);
    if (lane == 0) s_wsum[wid] = __popc(b);
    __syncthreads();
    int before = nact, tot = 0;
#pragma unroll
    for (int w = 0; w < GEMV_THREADS / 32; ++w) {
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
struct RecRegs {
  uint4 q;
  uint32_t s0, s1;  // Q4_0: 4 fp16 scales; MXFP4: s0 holds 4 E8M0 bytes
};

template <int QT>
__device__ __forceinline__ RecRegs<QT> load_rec(const uint8_t* rec, int lane) {
  RecRegs<QT> r;
  r.q = __ldg(reinterpret_cast<const uint4*>(rec + lane * 16));
  const int g = lane >> 2;
  if (QT == FTMOE_Q4_0) {
    const uint2 s = __ldg(reinterpret_cast<const uint2*>(rec + REC_CODE_BYTES + g * 8));
    r.s0 = s.x;
    r.s1 = s.y;
  } else {
    r.s0 = __ldg(reinterpret_cast<const uint32_t*>(rec + REC_CODE_BYTES + g * 4));
    r.s1 = 0;
  }
  return r;
}

// scale of (block b, row half h) from the lane's scale registers
template <int QT>
__device__ __forceinline__ float rec_scale(const RecRegs<QT>& r, int b, int h) {
  if (QT == FTMOE_Q4_0) {
    const uint32_t w = b ? r.s1 : r.s0;
    return half_bits_to_f32(h ? (w >> 16) : (w & 0xFFFFu));
  } else {
    return e8m0_to_f32((r.s0 >> (8 * (b * 2 + h))) & 0xFFu);
  }
}

template <int QT>
__device__ __forceinline__ void decode_word(uint32_t w, uint32_t (&a)[4]) {
  if (QT == FTMOE_Q4_0) q4_word_to_bf16x2(w, a); else e2m1_word_to_bf16x2(w, a);
}

template <int QT, int MODE, int KS, class Tab>
__global__ void __launch_bounds__(GEMV_THREADS) gemv_ffn_kernel(const GemvArgs a,
                                                                const __grid_constant__ Tab tab) {
  constexpr int NT = MODE == 0 ? 2 : 1;  // gate/up: two row tiles per feature tile
  constexpr int RT = (GEMV_THREADS / 32) / KS;
  constexpr int RB = rec_bytes(QT);
  __shared__ int s_act[1024];
  __shared__ int s_wsum[GEMV_THREADS / 32];
  __shared__ float s_red[GEMV_THREADS / 32][NT][GEMV_TG][4][32];

  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int g = lane >> 2, c = lane & 3;
  const int ts = wid / KS, kp = wid % KS;
  const int s_begin = kp * a.S / KS, s_end = (kp + 1) * a.S / KS;
  const bool ragged = (a.K & 63) != 0;  // last slab holds one block only

  const int nact = build_active_list(a.offsets, a.E, s_act, s_wsum);
  const int total = nact * a.items_per_expert;

  for (int item = blockIdx.x; item < total; item += gridDim.x) {
    const int ui = item / a.items_per_expert;
    const int tile = (item - ui * a.items_per_expert) * RT + ts;
    const int e = s_act[ui];
    const int r0 = a.offsets[e], n_e = a.offsets[e + 1] - r0;
    const bool tile_ok = tile < a.tiles_total;
    const uint8_t* wexp = tab.get(e, a);
    const uint8_t* rec_base[NT];
    rec_base[0] = wexp + (long long)tile * a.S * RB;
    if (NT == 2) rec_base[NT - 1] = wexp + (long long)(a.up_rt + tile) * a.S * RB;

    for (int tok0 = 0; tok0 < n_e; tok0 += 8 * GEMV_TG) {
      float acc[NT][GEMV_TG][4];
#pragma unroll
      for (int i = 0; i < NT; ++i)
#pragma unroll
        for (int t = 0; t < GEMV_TG; ++t)
#pragma unroll
          for (int q = 0; q < 4; ++q) acc[i][t][q] = 0.f;

      // B-operand rows of this lane (token g of each group), or null for padding
      const uint16_t* brow[GEMV_TG];
#pragma unroll
      for (int t = 0; t < GEMV_TG; ++t) {
        const int rr = tok0 + 8 * t + g;
        brow[t] = nullptr;
        if (rr < n_e) {
          long long row;
          if (MODE == 0) row = a.sorted_pair ? a.sorted_pair[r0 + rr] / a.k : (r0 + rr);
          else row = r0 + rr;
          brow[t] = a.act + row * a.act_ld;
        }
      }

      if (tile_ok) {
        RecRegs<QT> cur[NT];
        if (s_begin < s_end) {
#pragma unroll
          for (int i = 0; i < NT; ++i) cur[i] = load_rec<QT>(rec_base[i] + (long long)s_begin * RB, lane);
        }
        for (int s = s_begin; s < s_end; ++s) {
          RecRegs<QT> nxt[NT];
          if (s + 1 < s_end) {
#pragma unroll
            for (int i = 0; i < NT; ++i) nxt[i] = load_rec<QT>(rec_base[i] + (long long)(s + 1) * RB, lane);
          }
          const bool half = ragged && (s == a.S - 1);
#pragma unroll
          for (int b = 0; b < 2; ++b) {
            if (b == 1 && half) break;
            float part[NT][GEMV_TG][4];
#pragma unroll
            for (int i = 0; i < NT; ++i)
#pragma unroll
              for (int t = 0; t < GEMV_TG; ++t)
#pragma unroll
                for (int q = 0; q < 4; ++q) part[i][t][q] = 0.f;
#pragma unroll
            for (int jj = 0; jj < 2; ++jj) {
              const int j = 2 * b + jj;
              uint32_t bb[GEMV_TG][2];
#pragma unroll
              for (int t = 0; t < GEMV_TG; ++t) {
                bb[t][0] = bb[t][1] = 0u;
                if (brow[t]) {
                  const uint2 v = *reinterpret_cast<const uint2*>(brow[t] + s * 64 + 16 * j + 4 * c);
                  bb[t][0] = v.x;
                  bb[t][1] = v.y;
                }
              }
#pragma unroll
              for (int i = 0; i < NT; ++i) {
                const uint32_t w = j == 0 ? cur[i].q.x : j == 1 ? cur[i].q.y : j == 2 ? cur[i].q.z : cur[i].q.w;
                uint32_t av[4];
                decode_word<QT>(w, av);
#pragma unroll
                for (int t = 0; t < GEMV_TG; ++t)
                  if (t == 0 || tok0 + 8 * t < n_e) mma_16816(part[i][t], av, bb[t][0], bb[t][1]);
              }
            }
#pragma unroll
            for (int i = 0; i < NT; ++i) {
              const float sc0 = rec_scale<QT>(cur[i], b, 0), sc1 = rec_scale<QT>(cur[i], b, 1);
#pragma unroll
              for (int t = 0; t < GEMV_TG; ++t) {
                acc[i][t][0] = fmaf(sc0, part[i][t][0], acc[i][t][0]);
                acc[i][t][1] = fmaf(sc0, part[i][t][1], acc[i][t][1]);
                acc[i][t][2] = fmaf(sc1, part[i][t][2], acc[i][t][2]);
                acc[i][t][3] = fmaf(sc1, part[i][t][3], acc[i][t][3]);
              }
            }
          }
          if (s + 1 < s_end) {
#pragma unroll
            for (int i = 0; i < NT; ++i) cur[i] = nxt[i];
          }
        }
      }

      if (KS > 1) {
#pragma unroll
        for (int i = 0; i < NT; ++i)
#pragma unroll
          for (int t = 0; t < GEMV_TG; ++t)
#pragma unroll
            for (int q = 0; q < 4; ++q) s_red[wid][i][t][q][lane] = acc[i][t][q];
        __syncthreads();
        if (kp == 0) {
#pragma unroll
          for (int o = 1; o < KS; ++o)
#pragma unroll
            for (int i = 0; i < NT; ++i)
#pragma unroll
              for (int t = 0; t < GEMV_TG; ++t)
#pragma unroll
                for (int q = 0; q < 4; ++q) acc[i][t][q] += s_red[wid + o][i][t][q][lane];
        }
        __syncthreads();
      }

      if (kp == 0 && tile_ok) {
#pragma unroll
        for (int t = 0; t < GEMV_TG; ++t) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int rr = tok0 + 8 * t + 2 * c + (q & 1);
            if (rr >= n_e) continue;
            const int feat = tile * 16 + g + 8 * (q >> 1);
            float v;
            if (MODE == 0) v = silu_f32(acc[0][t][q]) * acc[NT - 1][t][q];
            else v = acc[0][t][q];
            a.out[(long long)(r0 + rr) * a.out_ld + feat] = f32_to_bf16_bits(v);
          }
        }
      }
    }
  }
}

template <int QT, int MODE, int KS, class Tab>
static cudaError_t launch_one(const GemvArgs& a, const Tab& tab, int upper_items, cudaStream_t st) {
  const DeviceInfo* di = device_info();
  if (!di) return cudaErrorUnknown;
  int per_sm = 0;
  cudaError_t err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
      &per_sm, gemv_ffn_kernel<QT, MODE, KS, Tab>, GEMV_THREADS, 0);
  if (err != cudaSuccess) return err;
  if (per_sm < 1) per_sm = 1;
  int grid = di->sm_count * per_sm;
  if (upper_items < grid) grid = upper_items;
  if (grid < 1) grid = 1;
  gemv_ffn_kernel<QT, MODE, KS, Tab><<<grid, GEMV_THREADS, 0, st>>>(a, tab);
  return cudaGetLastError();
}

// Split of the reduction over warps: enough slabs per warp to keep loads in flight.
static int pick_ks(int S) {
  if (S >= 32) return 8;
  if (S >= 12) return 4;
  if (S >= 4) return 2;
  return 1;
}

template <int QT, int MODE, class Tab>
static cudaError_t launch_mode(GemvArgs a, const Tab& tab, int max_active, cudaStream_t st) {
  const int ks = pick_ks(a.S);
  const int rt = 8 / ks;
  a.items_per_expert = (a.tiles_total + rt - 1) / rt;
  const int upper = max_active * a.items_per_expert;
  switch (ks) {
    case 8: return launch_one<QT, MODE, 8>(a, tab, upper, st);
    case 4: return launch_one<QT, MODE, 4>(a, tab, upper, st);
    case 2: return launch_one<QT, MODE, 2>(a, tab, upper, st);
    default: return launch_one<QT, MODE, 1>(a, tab, upper, st);
  }
}

template <int QT, class Tab>
static cudaError_t launch_qt(const FfnProblem& pb, const Tab& tab, cudaStream_t st) {
  const int max_active = pb.P < pb.E ? pb.P : pb.E;
  GemvArgs a{};
  a.offsets = pb.offsets;
  a.sorted_pair = pb.sorted_pair;
  a.k = pb.k;
  a.E = pb.E;
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
  a.tiles_total = pb.I / 16;
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
  a.tiles_total = pb.H / 16;
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
