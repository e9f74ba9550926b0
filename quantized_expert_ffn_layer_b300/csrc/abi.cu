// The libftmoe C ABI: host-side argument checks, workspace carving and launches.
// Every entry point validates before enqueueing and maps CUDA errors to a status.
#include <mutex>
#include <new>

#include "common.cuh"
#include "internal.h"

namespace ftmoe {

// One status word per device (module globals are instantiated on every device).
__device__ int g_device_status;

namespace {
constexpr int MAX_DEVICES = 64;
DeviceInfo g_info[MAX_DEVICES];
std::once_flag g_once[MAX_DEVICES];
bool g_ok[MAX_DEVICES];
int g_ffn_path = FTMOE_PATH_AUTO;

void init_device(int dev) {
  DeviceInfo& d = g_info[dev];
  g_ok[dev] = false;
  if (cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return;
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess) return;
  d.status = (int*)p;
  g_ok[dev] = true;
}

ftmoe_status from_cuda(cudaError_t e) { return e == cudaSuccess ? FTMOE_OK : FTMOE_ERR_CUDA; }

inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

bool qtype_ok(int q) { return q >= FTMOE_Q4_0 && q <= FTMOE_MXFP8; }
bool dim_ok(int v) { return v > 0 && v <= 16384 && v % 32 == 0; }
bool tke_ok(int T, int k, int E) {
  return T >= 0 && E >= 1 && E <= 1024 && k >= 1 && k <= E && k <= 32 &&
         (long long)T * k < (1LL << 31);
}

// Workspace carve-up shared by ftmoe_expert_ffn and ftmoe_layer.
// Workspace of the FFN: [gemv scratch (zero region first; 0 bytes: the GEMV's split
// reductions meet in shared memory)][h_act][gemm scratch: x rows in the permuted order].
struct FfnWs {
  void* gemv_ws;
  size_t gemv_zero_bytes;
  uint16_t* h_act;
  void* gemm_ws;
  size_t gemm_bytes;
};
size_t ffn_ws_bytes(int T, int k, int E, int H, int I) {
  const long long P = (long long)T * k;
  return align256(ffn_gemv_ws_bytes(T, k, E, H, I)) + align256((size_t)P * I * 2) +
         align256(ffn_gemm_ws_bytes(T, k, E, H, I));
}
FfnWs carve_ffn(void* ws, int T, int k, int E, int H, int I) {
  const long long P = (long long)T * k;
  char* b = (char*)ws;
  FfnWs w;
  w.gemv_ws = b;
  w.gemv_zero_bytes = ffn_gemv_zero_bytes(T, k, E, H, I);
  b += align256(ffn_gemv_ws_bytes(T, k, E, H, I));
  w.h_act = (uint16_t*)b;
  b += align256((size_t)P * I * 2);
  w.gemm_ws = b;
  w.gemm_bytes = ffn_gemm_ws_bytes(T, k, E, H, I);
  return w;
}

__global__ void set_pair_kernel(int32_t* p, int a, int b) {
  p[0] = a;
  p[1] = b;
}

bool weights_ok(const ftmoe_weights* w) {
  if (!w || !qtype_ok(w->qtype) || !dim_ok(w->H) || !dim_ok(w->I) || w->E < 1 || w->E > 1024)
    return false;
  if (w->expert_blob) {
    if (w->E > MAX_TABLE_EXPERTS) return false;
  } else if (!w->w13 || !w->w2) {
    return false;
  }
  if ((w->shared_w13 == nullptr) != (w->shared_w2 == nullptr)) return false;
  return true;
}

ftmoe_status run_ffn(const ftmoe_weights* wts, int E, const uint16_t* x, int T, int k,
                     const int32_t* offsets, const int32_t* sorted_pair, uint16_t* y_perm,
                     const void* w13, const void* w2, bool use_table, void* ws, bool ws_zeroed,
                     cudaStream_t st) {
  FfnProblem pb{};
  pb.qtype = wts->qtype;
  pb.E = E;
  pb.H = wts->H;
  pb.I = wts->I;
  pb.T = T;
  pb.k = k;
  pb.P = T * k;
  pb.x = x;
  pb.offsets = offsets;
  pb.sorted_pair = sorted_pair;
  pb.y_perm = y_perm;
  pb.w13 = (const uint8_t*)w13;
  pb.w2 = (const uint8_t*)w2;
  pb.w13_bytes = tiles_bytes_per_expert(wts->qtype, 2 * wts->I, wts->H);
  ExpertTable tab;
  if (use_table) {
    for (int e = 0; e < E; ++e) tab.p[e] = (const uint8_t*)wts->expert_blob[e];
    pb.table = &tab;
  }
  FfnWs fw = carve_ffn(ws, T, k, E, wts->H, wts->I);
  pb.h_act = fw.h_act;
  const int path = g_ffn_path;
  // measured crossovers (decode layer shape on B300): the grouped GEMV wins below about
  // 8 rows per expert, the decode GEMM between 8 and 32, the prefill GEMM above.  A
  // tensor-core path also needs work for the whole GPU: its items (token tiles of 256 or
  // 16 rows x 128- or 256-row weight slices) must number at least half the SMs, which a
  // single shared expert at decode sizes (E = 1, a few dozen rows) does not reach.
  const DeviceInfo* di = device_info();
  const long long half_sms = di ? di->sm_count / 2 : 74;
  const long long tiles256 = ((long long)pb.P + 255) / 256 + (E > 1 ? E - 1 : 0);
  const long long tiles16 = ((long long)pb.P + 15) / 16;
  const bool many_rows = (long long)pb.P >= 32LL * E && tiles256 * ((pb.I + 127) / 128) >= half_sms;
  const bool mid_rows = (long long)pb.P >= 8LL * E && tiles16 * ((pb.I + 127) / 128) >= half_sms;
  if (path == FTMOE_PATH_GEMM || (path == FTMOE_PATH_AUTO && many_rows)) {
    cudaError_t e = launch_ffn_gemm(pb, fw.gemm_ws, fw.gemm_bytes, st);
    if (e == cudaSuccess) return FTMOE_OK;
    if (e != cudaErrorNotSupported) return FTMOE_ERR_CUDA;
    if (path == FTMOE_PATH_GEMM) return FTMOE_ERR_UNSUPPORTED;
  }
  if (path == FTMOE_PATH_GEMM_DECODE || (path == FTMOE_PATH_AUTO && mid_rows)) {
    cudaError_t e = launch_ffn_gemm_decode(pb, st);
    if (e == cudaSuccess) return FTMOE_OK;
    if (e != cudaErrorNotSupported) return FTMOE_ERR_CUDA;
    if (path == FTMOE_PATH_GEMM_DECODE) return FTMOE_ERR_UNSUPPORTED;
  }
  const cudaError_t e = launch_ffn_gemv(pb, fw.gemv_ws, ws_zeroed, st);
  return e == cudaErrorNotSupported ? FTMOE_ERR_UNSUPPORTED : from_cuda(e);
}
}  // namespace

const DeviceInfo* device_info() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) return nullptr;
  std::call_once(g_once[dev], init_device, dev);
  return g_ok[dev] ? &g_info[dev] : nullptr;
}

}  // namespace ftmoe

using namespace ftmoe;

extern "C" {

const char* ftmoe_status_string(int s) {
  switch (s) {
    case FTMOE_OK: return "ok";
    case FTMOE_ERR_INVALID_ARG: return "invalid argument";
    case FTMOE_ERR_UNSUPPORTED: return "unsupported configuration";
    case FTMOE_ERR_CUDA: return "CUDA error";
    case FTMOE_ERR_NO_SLOT: return "no free cache slot";
    case FTMOE_ERR_TIMEOUT: return "bounded device wait timed out";
    case FTMOE_ERR_DEVICE_CHECK: return "device-side check failed";
    case FTMOE_ERR_WORKSPACE: return "workspace too small";
    default: return "unknown status";
  }
}

int ftmoe_version(void) { return 100; }

size_t ftmoe_tiled_bytes(int qtype, int E, int N, int K) {
  if (!qtype_ok(qtype) || E < 1 || N < 16 || N % 16 || K < 32 || K % 32) return 0;
  return (size_t)E * tiles_bytes_per_expert(qtype, N, K);
}

ftmoe_status ftmoe_repack(int qtype, const void* canon, void* tiles, int E, int N, int K,
                          ftmoe_stream_t stream) {
  if (!ftmoe_tiled_bytes(qtype, E, N, K) || !canon || !tiles) return FTMOE_ERR_INVALID_ARG;
  return from_cuda(launch_repack(qtype, canon, tiles, E, N, K, (cudaStream_t)stream));
}

ftmoe_status ftmoe_dequant(int qtype, const void* tiles, int E, int N, int K, float* out,
                           ftmoe_stream_t stream) {
  if (!ftmoe_tiled_bytes(qtype, E, N, K) || !tiles || !out) return FTMOE_ERR_INVALID_ARG;
  return from_cuda(launch_dequant(qtype, tiles, E, N, K, out, (cudaStream_t)stream));
}

ftmoe_status ftmoe_dequant_operand(int qtype, int which, const void* tiles, int E, int N, int K,
                                   uint16_t* out, ftmoe_stream_t stream) {
  if (!ftmoe_tiled_bytes(qtype, E, N, K) || !tiles || !out || ((uintptr_t)out & 15) ||
      (which != FTMOE_OPERAND_PREFILL && which != FTMOE_OPERAND_CODES))
    return FTMOE_ERR_INVALID_ARG;
  return from_cuda(launch_operand(qtype, which, tiles, E, N, K, out, (cudaStream_t)stream));
}

ftmoe_status ftmoe_route(const float* logits, int T, int E, int k, int32_t* ids, float* w,
                         ftmoe_stream_t stream) {
  if (!tke_ok(T, k, E)) return FTMOE_ERR_INVALID_ARG;
  if (T == 0) return FTMOE_OK;
  if (!logits || !ids || !w) return FTMOE_ERR_INVALID_ARG;
  return from_cuda(launch_route(logits, T, E, k, ids, w, (cudaStream_t)stream));
}

size_t ftmoe_permute_workspace_bytes(int T, int k, int E) {
  if (!tke_ok(T, k, E)) return 0;
  return permute_ws_bytes(T, k, E);
}

ftmoe_status ftmoe_permute(const int32_t* ids, int T, int k, int E, int32_t* offsets,
                           int32_t* sorted_pair, int32_t* inv_pos, void* ws, size_t ws_bytes,
                           ftmoe_stream_t stream) {
  if (!tke_ok(T, k, E) || !offsets) return FTMOE_ERR_INVALID_ARG;
  const size_t need = permute_ws_bytes(T, k, E);
  if (ws_bytes < need || (need && !ws)) return FTMOE_ERR_WORKSPACE;
  if (T > 0 && (!ids || !sorted_pair || !inv_pos)) return FTMOE_ERR_INVALID_ARG;
  const DeviceInfo* di = device_info();
  if (!di) return FTMOE_ERR_CUDA;
  if (T == 0) return from_cuda(cudaMemsetAsync(offsets, 0, (E + 1) * sizeof(int32_t), (cudaStream_t)stream));
  return from_cuda(launch_permute(ids, T, k, E, offsets, sorted_pair, inv_pos, ws, di->status,
                                  nullptr, 0, (cudaStream_t)stream));
}

size_t ftmoe_expert_blob_bytes(int qtype, int H, int I) {
  if (!qtype_ok(qtype) || !dim_ok(H) || !dim_ok(I)) return 0;
  return tiles_bytes_per_expert(qtype, 2 * I, H) + tiles_bytes_per_expert(qtype, H, I);
}

size_t ftmoe_ffn_workspace_bytes(int T, int k, int E, int H, int I) {
  if (!tke_ok(T, k, E) || !dim_ok(H) || !dim_ok(I)) return 0;
  return ffn_ws_bytes(T, k, E, H, I);
}

int ftmoe_set_ffn_path(int path) {
  const int old = g_ffn_path;
  if (path >= FTMOE_PATH_AUTO && path <= FTMOE_PATH_GEMM_DECODE) g_ffn_path = path;
  return old;
}

ftmoe_status ftmoe_expert_ffn(const ftmoe_weights* wts, const uint16_t* x, int T, int k,
                              const int32_t* offsets, const int32_t* sorted_pair,
                              uint16_t* y_perm, void* ws, size_t ws_bytes, ftmoe_stream_t stream) {
  if (!weights_ok(wts) || !tke_ok(T, k, wts->E)) return FTMOE_ERR_INVALID_ARG;
  if (!sorted_pair && k != 1) return FTMOE_ERR_INVALID_ARG;
  if (T == 0) return FTMOE_OK;
  if (!x || !offsets || !y_perm) return FTMOE_ERR_INVALID_ARG;
  if (ws_bytes < ffn_ws_bytes(T, k, wts->E, wts->H, wts->I) || !ws) return FTMOE_ERR_WORKSPACE;
  if (!device_info()) return FTMOE_ERR_CUDA;
  return run_ffn(wts, wts->E, x, T, k, offsets, sorted_pair, y_perm, wts->w13, wts->w2,
                 wts->expert_blob != nullptr, ws, false, (cudaStream_t)stream);
}

ftmoe_status ftmoe_combine(const uint16_t* y_perm, const float* w, const int32_t* inv_pos,
                           const uint16_t* shared_y, int T, int k, int H, uint16_t* out,
                           ftmoe_stream_t stream) {
  if (T < 0 || k < 1 || k > 32 || !dim_ok(H)) return FTMOE_ERR_INVALID_ARG;
  if (T == 0) return FTMOE_OK;
  if (!y_perm || !w || !inv_pos || !out) return FTMOE_ERR_INVALID_ARG;
  return from_cuda(launch_combine(y_perm, w, inv_pos, shared_y, T, k, H, out, (cudaStream_t)stream));
}

namespace {
struct LayerWs {
  int32_t *ids, *sorted_pair, *inv_pos, *offsets, *sh_offsets;
  float* w;
  void* perm_ws;
  uint16_t *y_perm, *y_sh;
  void* ffn_ws;
  size_t total;
};
LayerWs carve_layer(void* ws, int T, int k, int E, int H, int I, bool shared) {
  const size_t P = (size_t)T * k;
  LayerWs L{};
  char* b = (char*)ws;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    char* p = b ? b + off : nullptr;
    off += align256(bytes);
    return p;
  };
  L.ids = (int32_t*)take(P * 4);
  L.w = (float*)take(P * 4);
  L.sorted_pair = (int32_t*)take(P * 4);
  L.inv_pos = (int32_t*)take(P * 4);
  L.offsets = (int32_t*)take((E + 1) * 4);
  L.perm_ws = take(permute_ws_bytes(T, k, E));
  L.y_perm = (uint16_t*)take(P * H * 2);
  if (shared) {
    L.sh_offsets = (int32_t*)take(8);
    L.y_sh = (uint16_t*)take((size_t)T * H * 2);
  }
  const size_t f1 = ffn_ws_bytes(T, k, E, H, I);
  const size_t f2 = shared ? ffn_ws_bytes(T, 1, 1, H, I) : 0;
  L.ffn_ws = take(f1 > f2 ? f1 : f2);
  L.total = off;
  return L;
}
}  // namespace

size_t ftmoe_layer_workspace_bytes(int T, int k, int E, int H, int I, int has_shared) {
  if (!tke_ok(T, k, E) || !dim_ok(H) || !dim_ok(I)) return 0;
  return carve_layer(nullptr, T, k, E, H, I, has_shared != 0).total;
}

ftmoe_status ftmoe_layer(const ftmoe_weights* wts, const float* logits, const uint16_t* x, int T,
                         int k, uint16_t* out, int32_t* ids_out, float* w_out, void* ws,
                         size_t ws_bytes, ftmoe_stream_t stream) {
  if (!weights_ok(wts) || !tke_ok(T, k, wts->E)) return FTMOE_ERR_INVALID_ARG;
  if (T == 0) return FTMOE_OK;
  if (!logits || !x || !out) return FTMOE_ERR_INVALID_ARG;
  const bool shared = wts->shared_w13 != nullptr;
  const int E = wts->E, H = wts->H, I = wts->I;
  LayerWs L = carve_layer(ws, T, k, E, H, I, shared);
  if (!ws || ws_bytes < L.total) return FTMOE_ERR_WORKSPACE;
  const DeviceInfo* di = device_info();
  if (!di) return FTMOE_ERR_CUDA;
  cudaStream_t st = (cudaStream_t)stream;
  int32_t* ids = ids_out ? ids_out : L.ids;
  float* w = w_out ? w_out : L.w;
  // the permutation kernel also clears the FFN scratch that must start at zero; a small
  // batch is routed by the same one-CTA launch
  cudaError_t e;
  if (route_permute_fits(T, k)) {
    e = launch_route_permute(logits, T, E, k, ids, w, L.offsets, L.sorted_pair, L.inv_pos, di->status,
                             L.ffn_ws, ffn_gemv_zero_bytes(T, k, E, H, I), st);
  } else {
    e = launch_route(logits, T, E, k, ids, w, st);
    if (e == cudaSuccess)
      e = launch_permute(ids, T, k, E, L.offsets, L.sorted_pair, L.inv_pos, L.perm_ws, di->status,
                         L.ffn_ws, ffn_gemv_zero_bytes(T, k, E, H, I), st);
  }
  if (e != cudaSuccess) return FTMOE_ERR_CUDA;
  ftmoe_status s = run_ffn(wts, E, x, T, k, L.offsets, L.sorted_pair, L.y_perm, wts->w13, wts->w2,
                           wts->expert_blob != nullptr, L.ffn_ws, true, st);
  if (s != FTMOE_OK) return s;
  if (shared) {
    set_pair_kernel<<<1, 1, 0, st>>>(L.sh_offsets, 0, T);
    if (cudaGetLastError() != cudaSuccess) return FTMOE_ERR_CUDA;
    s = run_ffn(wts, 1, x, T, 1, L.sh_offsets, nullptr, L.y_sh, wts->shared_w13, wts->shared_w2,
                false, L.ffn_ws, false, st);
    if (s != FTMOE_OK) return s;
  }
  return from_cuda(launch_combine(L.y_perm, w, L.inv_pos, shared ? L.y_sh : nullptr, T, k, H, out, st));
}

ftmoe_status ftmoe_device_status(int* code_out, ftmoe_stream_t stream) {
  if (!code_out) return FTMOE_ERR_INVALID_ARG;
  const DeviceInfo* di = device_info();
  if (!di) return FTMOE_ERR_CUDA;
  cudaStream_t st = (cudaStream_t)stream;
  int v = 0;
  cudaError_t e = cudaMemcpyAsync(&v, di->status, sizeof(int), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaMemsetAsync(di->status, 0, sizeof(int), st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return FTMOE_ERR_CUDA;
  *code_out = v;
  return FTMOE_OK;
}

}  // extern "C"
