/*
 * libftmoe — quantized MoE expert layer for NVIDIA B300 (sm_103a).
 *
 * The layer: router logits -> softmax / top-k / renormalise -> permutation of
 * the (token, expert) pairs into per-expert groups -> expert SwiGLU FFN on 4-bit
 * block-quantized weights (GGUF Q4_0 or MXFP4) -> weighted combine back to
 * token order; plus an LRU cache that streams a pinned-host expert bank into a
 * device slot pool on a side stream.
 *
 * Sources (page title, section):
 *  [P5] "深入FreeToken架构从HTTP API到CUDA内核的本地MoE推理引擎全链路剖析"
 *       §五 (ExpertFFN banks per format incl. GGUF Q4_0 and MXFP4; hot experts
 *       on the GPU, cold experts in pinned host memory; global LRU; full-layer
 *       double-buffered prefill) and §六 (GGUF dequant + Q4_0 MoE kernels,
 *       pinned tensors, batched async copies).
 *  [P3] "从双缓冲 Prefill、带宽自适应 CPU–GPU 协同到 Agent 状态复用…"
 *       机制一 (copy the next layer while computing this one) and 机制四
 *       (global LRU expert cache); "为什么 MoE 模型适合做 CPU–GPU 协同" (only a
 *       subset of experts is active per token).
 *  [P4] "FreeToken：高效的边缘原生 MoE 服务与带宽自适应执行", 方法 (pipelined
 *       loading, expert caching) and 核心洞察 (CUDA-graph-compatible LRU).
 *  OCP Microscaling Formats (MX) v1.0 for E2M1 / E8M0.
 *
 * Conventions for every call:
 *  - Plain pointers.  "device" pointers are CUDA global memory of the current
 *    device; "host" pointers are ordinary (or pinned) CPU memory.  The caller
 *    allocates and owns every buffer; the library keeps no pointer beyond the
 *    call, except the cache, which keeps the bank / pool pointers it was
 *    created with.
 *  - bf16 tensors are passed as uint16_t bit patterns (row-major).
 *  - Every compute call is asynchronous on `stream` (NULL = legacy default
 *    stream) and returns after enqueueing; only ftmoe_device_status and
 *    ftmoe_cache_stats synchronize.
 *  - Arguments are validated on the host before anything is enqueued; an
 *    invalid call returns FTMOE_ERR_INVALID_ARG and enqueues nothing.  A CUDA
 *    launch error returns FTMOE_ERR_CUDA.  The library never aborts, never
 *    throws across this boundary and never traps on the device.
 *  - Sizes: T >= 0 tokens (T == 0 is a successful no-op), 1 <= E <= 1024
 *    experts, 1 <= k <= min(E, 32), H and I positive multiples of 32 up to
 *    16384, T * k < 2^31.
 */
#ifndef FTMOE_H
#define FTMOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t / CUstream. */
typedef struct CUstream_st* ftmoe_stream_t;

typedef enum {
  FTMOE_OK = 0,
  FTMOE_ERR_INVALID_ARG = 1,
  FTMOE_ERR_UNSUPPORTED = 2,
  FTMOE_ERR_CUDA = 3,
  FTMOE_ERR_NO_SLOT = 4,
  FTMOE_ERR_TIMEOUT = 5,
  FTMOE_ERR_DEVICE_CHECK = 6,
  FTMOE_ERR_WORKSPACE = 7
} ftmoe_status;

/* Block formats ([P5] §五 bank schemas).  Q4_0: 32 weights per block, fp16
 * scale d, weight = (q - 8) * d.  MXFP4: 32 E2M1 codes sharing an E8M0 scale
 * 2^(e - 127) (e = 255 is NaN).  NVFP4: 16 E2M1 codes sharing an E4M3 scale s,
 * and one fp32 tensor scale t per expert matrix: weight = E2M1 * s * t.  MXFP8
 * (the block-scaled FP8 bank; OCP MX v1.0): 32 E4M3 elements sharing an E8M0
 * scale 2^(e - 127). */
typedef enum { FTMOE_Q4_0 = 1, FTMOE_MXFP4 = 2, FTMOE_NVFP4 = 3, FTMOE_MXFP8 = 4 } ftmoe_qtype;

/* Expert FFN path selection (ftmoe_set_ffn_path). */
typedef enum {
  FTMOE_PATH_AUTO = 0,        /* GEMV below 8 E rows, GEMM_DECODE below 32 E, else GEMM */
  FTMOE_PATH_GEMV = 1,        /* grouped GEMV on mma.sync with split reductions for tiny batches */
  FTMOE_PATH_GEMM = 2,        /* tcgen05 grouped GEMM, 256-token tiles, bf16 weights staged in smem */
  FTMOE_PATH_GEMM_DECODE = 3  /* tcgen05 grouped GEMM, 16-token tiles, codes in tensor memory */
} ftmoe_path;

/* Human-readable name of a status code (static string; never NULL). */
const char* ftmoe_status_string(int status);

/* Library ABI version (major * 100 + minor). */
int ftmoe_version(void);

/* ------------------------------------------------------------------ weights
 *
 * Canonical block layout of one weight matrix W[E][N][K] (reduction dim K
 * last, blocks along K): E * N * (K / 32) blocks, block = scale then 16 code
 * bytes, element i < 16 in the low nibble of code byte i and element i >= 16
 * in the high nibble of code byte i - 16 (18 bytes per Q4_0 block, 17 per
 * MXFP4 block).  Expert e's gate/up matrix w13[e] is [2I][H] (rows [0, I)
 * gate, [I, 2I) up); its down matrix w2[e] is [H][I].
 *
 * MXFP8 blocks hold 32 weights in 33 bytes (E8M0 scale, then the 32 E4M3
 * element bytes in order).
 * NVFP4 blocks hold 16 weights in 9 bytes (E4M3 scale, then 8 code bytes:
 * element i < 8 in the low nibble of code byte i, i >= 8 in the high nibble of
 * byte i - 8), and the canonical buffer ends with the E fp32 tensor scales
 * (little-endian): E * N * (K / 16) * 9 + 4 E bytes.
 *
 * The kernels read a tiled layout instead ("tiles"): for each expert and
 * each group of 16 rows, ceil(K / 64) records of 64 reduction elements; a
 * record is 512 code bytes (1024 element bytes for MXFP8) followed by the
 * block scales of its 16 rows (64 bytes of fp16 for Q4_0 and 32 bytes of E8M0
 * for MXFP4 and MXFP8, 2 blocks per row; 64 E4M3 bytes for NVFP4, 4 blocks per
 * row), so records are 576 / 544 / 576 / 1056 bytes and every record starts
 * 16-byte aligned.  For NVFP4 each expert's
 * records are followed by a 16-byte trailer holding its tensor scale.  A ragged
 * last record (K % 64 == 32) is padded with zero weights.  N must be a
 * multiple of 16.
 */

/* Bytes of the tiled layout of W[E][N][K]; 0 for invalid arguments. */
size_t ftmoe_tiled_bytes(int qtype, int E, int N, int K);

/* Canonical blocks (device, E*N*K/32 blocks) -> tiles (device,
 * ftmoe_tiled_bytes bytes).  One-time load-time conversion; lossless. */
ftmoe_status ftmoe_repack(int qtype, const void* canon, void* tiles, int E, int N, int K,
                          ftmoe_stream_t stream);

/* Exact decode of tiles (device) to fp32 out[E][N][K] (device).  Every Q4_0
 * and MXFP4 weight is exactly representable in fp32 except MXFP4 values beyond
 * the fp32 range (-> +-inf) and subnormal-range scales, which stay exact as
 * fp32 subnormals.  Verification aid: the FFN kernels decode in registers /
 * shared memory without it. */
ftmoe_status ftmoe_dequant(int qtype, const void* tiles, int E, int N, int K, float* out,
                           ftmoe_stream_t stream);

/* Tensor-core operands built from the tiles (verification aid, [P5] §六 GGUF dequant):
 * which of the FFN kernels' decode steps to reproduce.  Each runs the same device
 * functions as that kernel and reads the result back through that kernel's layout. */
typedef enum {
  FTMOE_OPERAND_PREFILL = 0, /* prefill grouped GEMM A tile: each weight rounded once to
                                bf16, round-to-nearest-even of the exact decoded value
                                ((q - 8) * d for Q4_0, E2M1 * 2^(e - 127) for MXFP4);
                                beyond the bf16 range -> +-inf; NaN scales -> NaN */
  FTMOE_OPERAND_CODES = 1    /* decode GEMM A operand: the unscaled code value, q - 8
                                (Q4_0) or the E2M1 value (MXFP4, NVFP4), exact; for MXFP8
                                the grouped GEMV's: the E4M3 element value, exact for
                                every finite code (the NaN code reads as +-480) */
} ftmoe_operand;

/* Writes operand `which` of tiles (device) as bf16 bit patterns out[E][N][K] (device,
 * 16-byte aligned).  Same argument rules as ftmoe_dequant; an unknown `which` or a
 * misaligned `out` returns FTMOE_ERR_INVALID_ARG. */
ftmoe_status ftmoe_dequant_operand(int qtype, int which, const void* tiles, int E, int N, int K,
                                   uint16_t* out, ftmoe_stream_t stream);

/* ------------------------------------------------------------------ gate
 * The scores the router selects from ([P3] sparse expert activation), from the
 * hidden state: logits[t][e] = sum over h of x[t][h] * wg[e][h].
 *   x:      device bf16 [T][H];  wg: device bf16 [E][H] (gate matrix, one row per
 *           expert, the reduction dimension last);
 *   logits: device fp32 [T][E] (out).
 * fp32 accumulation in a fixed order that depends only on H (16-element steps
 * taken by 16 interleaved slices, the slices added in order), so a token's logits
 * do not depend on the batch.  H a multiple of 32 up to 16384, 1 <= E <= 1024;
 * T == 0 is a no-op.  Not part of ftmoe_layer, which starts from logits. */
ftmoe_status ftmoe_gate(const uint16_t* x, const uint16_t* wg, int T, int H, int E, float* logits,
                        ftmoe_stream_t stream);

/* ------------------------------------------------------------------ route
 * Per token t ([P3] sparse expert activation): ids[t][0..k) = the k experts
 * with the largest logits[t][:], in descending logit order, ties to the lower
 * expert id; w[t][j] = exp(l_j - l_max) / sum over the selected of
 * exp(l - l_max) (= softmax over all E, then renormalised over the selection).
 *   logits: device fp32 [T][E], finite values.
 *   ids:    device int32 [T][k] (out).   w: device fp32 [T][k] (out).
 * One warp per token. */
ftmoe_status ftmoe_route(const float* logits, int T, int E, int k, int32_t* ids, float* w,
                         ftmoe_stream_t stream);

/* ------------------------------------------------------------------ permute
 * Pairs p = t * k + j (P = T * k) grouped by expert, stable in p:
 *   offsets:     device int32 [E + 1] (out), exclusive prefix sum of the
 *                per-expert counts, offsets[E] = P;
 *   sorted_pair: device int32 [P] (out), pairs of expert e at
 *                [offsets[e], offsets[e+1]) in ascending p;
 *   inv_pos:     device int32 [P] (out), inv_pos[sorted_pair[r]] = r.
 * ids must hold values in [0, E) (out-of-range ids are counted in the device
 * status word and skipped).  ws: device scratch of at least
 * ftmoe_permute_workspace_bytes(T, k, E) bytes (may be NULL when that is 0). */
size_t ftmoe_permute_workspace_bytes(int T, int k, int E);
ftmoe_status ftmoe_permute(const int32_t* ids, int T, int k, int E, int32_t* offsets,
                           int32_t* sorted_pair, int32_t* inv_pos, void* ws, size_t ws_bytes,
                           ftmoe_stream_t stream);

/* Same result as ftmoe_permute, for callers that can neither call cudaMalloc nor
 * pass a workspace: a host program that owns all device memory through its own
 * fixed pool, or a plugin interface with no workspace hook.  It allocates nothing;
 * the scratch lives in a fixed 1 MiB device array inside the library (held on every
 * device that loads the library until the process exits).  The pages have no
 * counterpart to this call; it exists only for such callers.
 *   Limit: when T * k > 16384 the call needs ceil(T * k / 1024) * E int32 of
 *   scratch, at most 262144 (e.g. T * k <= 2,097,152 at E = 128); larger problems
 *   return FTMOE_ERR_WORKSPACE and enqueue nothing.
 *   Set-up: the first call on each device resolves the array's device address
 *   (cudaGetSymbolAddress) with that device current; make that first call before
 *   any stream capture.
 *   Sharing: every call on a device uses the same array, and nothing in it needs to
 *   start at zero.  Calls whose kernels overlap on the GPU (different streams with
 *   no ordering between them) race on the array and give undefined results. */
ftmoe_status ftmoe_permute_noalloc(const int32_t* ids, int T, int k, int E, int32_t* offsets,
                                   int32_t* sorted_pair, int32_t* inv_pos, ftmoe_stream_t stream);

/* ------------------------------------------------------------------ expert FFN
 * [P5] §五 ExpertFFN: for every expert e and every row r in
 * [offsets[e], offsets[e+1]) with token t = sorted_pair[r] / k:
 *   g = W_gate[e] x[t], u = W_up[e] x[t], h = silu(g) * u (rounded to bf16),
 *   y_perm[r] = W_down[e] h (rounded to bf16); silu(g) = g / (1 + exp(-g)).
 * Weights are decoded from their 4-bit blocks inside the kernels ([P5] §六).
 */
typedef struct {
  int qtype;                        /* ftmoe_qtype */
  int E, H, I;
  const void* w13;                  /* device tiles of w13 [E][2I][H] (NULL if expert_blob) */
  const void* w2;                   /* device tiles of w2  [E][H][I]  (NULL if expert_blob) */
  const void* const* expert_blob;   /* HOST array of E device pointers or NULL: expert e's
                                       tiles of w13[e] immediately followed by those of w2[e]
                                       (a cache slot).  Read at enqueue time only. */
  const void* shared_w13;           /* device tiles [1][2I][H] of an always-on shared expert, or NULL */
  const void* shared_w2;            /* device tiles [1][H][I], NULL iff shared_w13 is NULL */
} ftmoe_weights;

/* Bytes of one expert blob (tiles of w13[e] then w2[e]). */
size_t ftmoe_expert_blob_bytes(int qtype, int H, int I);

/* Scratch for ftmoe_expert_ffn / ftmoe_layer (device, 256-byte aligned, owned by the
 * caller, contents undefined between calls): the intermediate h (bf16 [T*k][I]) and,
 * for the tensor-core prefill path, the x rows in the permuted order (bf16 [T*k][H]);
 * ftmoe_layer adds the routing and permutation arrays. */
size_t ftmoe_ffn_workspace_bytes(int T, int k, int E, int H, int I);
size_t ftmoe_layer_workspace_bytes(int T, int k, int E, int H, int I, int has_shared);

/*   x:      device bf16 [T][H];  offsets / sorted_pair as produced by ftmoe_permute
 *           (sorted_pair == NULL means the identity, one row per token, k == 1);
 *   y_perm: device bf16 [T*k][H] (out), row r as above. */
ftmoe_status ftmoe_expert_ffn(const ftmoe_weights* wts, const uint16_t* x, int T, int k,
                              const int32_t* offsets, const int32_t* sorted_pair,
                              uint16_t* y_perm, void* ws, size_t ws_bytes, ftmoe_stream_t stream);

/* Kernel choice for ftmoe_expert_ffn / ftmoe_layer (ftmoe_path): AUTO picks the
 * GEMV when T * k < 8 E, GEMM_DECODE when 8 E <= T * k < 32 E and GEMM otherwise
 * (the crossovers measured on the decode layer shape).  Every path computes the
 * same definition; the reduction order (and so the last bits) differs between
 * paths, but within one path a token's output does not depend on the other tokens
 * of the batch.  Process-wide setting; returns the previous value. */
int ftmoe_set_ffn_path(int path);

/* ------------------------------------------------------------------ combine
 * out[t] = sum over j = 0..k-1 (in that order) of w[t][j] * y_perm[inv_pos[t*k+j]]
 *          (+ shared_y[t]), accumulated in fp32, stored as bf16.
 *   y_perm: device bf16 [T*k][H];  w: device fp32 [T][k];  inv_pos: device int32 [T*k];
 *   shared_y: device bf16 [T][H] or NULL;  out: device bf16 [T][H]. */
ftmoe_status ftmoe_combine(const uint16_t* y_perm, const float* w, const int32_t* inv_pos,
                           const uint16_t* shared_y, int T, int k, int H, uint16_t* out,
                           ftmoe_stream_t stream);

/* ------------------------------------------------------------------ layer
 * route -> permute -> expert FFN (+ shared expert over all tokens, weight 1)
 * -> combine, all enqueued on `stream`.
 *   logits: device fp32 [T][E];  x: device bf16 [T][H];  out: device bf16 [T][H];
 *   ids_out / w_out: device int32 / fp32 [T][k] copies of the routing, or NULL;
 *   ws: device scratch of ftmoe_layer_workspace_bytes(...) bytes. */
ftmoe_status ftmoe_layer(const ftmoe_weights* wts, const float* logits, const uint16_t* x,
                         int T, int k, uint16_t* out, int32_t* ids_out, float* w_out, void* ws,
                         size_t ws_bytes, ftmoe_stream_t stream);

/* Reads and clears the device status word that kernels set on a detected
 * problem (an out-of-range expert id, a bounded wait that ran out).  Blocks
 * until `stream` is idle.  *code_out = 0 if nothing was recorded. */
ftmoe_status ftmoe_device_status(int* code_out, ftmoe_stream_t stream);

/* Self-check of the bounded waits (no counterpart on the pages).  Launches one
 * CTA that waits on an mbarrier nothing arrives on, with the bounded wait the
 * pipelined kernels use and a limit of limit_ns nanoseconds of GPU wall time
 * (1e3 <= limit_ns <= 1e9, else FTMOE_ERR_INVALID_ARG).  The wait gives up, ORs
 * 2 (wait ran out) into the status word that ftmoe_device_status reads, writes 0
 * to *waited_ok (device int, nullable) and the kernel returns normally: the
 * context stays usable.  Asynchronous on `stream`. */
ftmoe_status ftmoe_check_wait_timeout(long long limit_ns, int* waited_ok, ftmoe_stream_t stream);

/* ------------------------------------------------------------------ expert cache
 * [P5] §五 / [P3] 机制四: cold experts live in a pinned host bank, hot ones in a
 * device slot pool managed by LRU; [P3] 机制一: the next layer's experts are
 * copied on a side stream while the current layer computes.
 *
 * Bank: pinned host memory, layers * E blobs of ftmoe_expert_blob_bytes each,
 * blob (l, e) at bank + (l * E + e) * blob_bytes.  Pool: device memory of
 * layers * slots_per_layer blobs.  Policy FTMOE_LRU_PER_LAYER keeps a pool of
 * slots_per_layer slots per layer; FTMOE_LRU_GLOBAL shares all slots among
 * all layers.  Every request touches its ids in order with a new recency stamp;
 * a resident expert is a hit, a missing one is copied into the lowest empty
 * slot of its pool, else the least recently used slot that is neither touched by
 * the same request nor pinned.  An acquire pins the slots it touched until the
 * layer's ftmoe_cache_release ([P4] 核心洞察: a layer, possibly replayed as a CUDA
 * graph, reads its experts in place), so no later prefetch or acquire overwrites
 * them; a prefetch pins nothing.  A request that finds no slot for a missing id
 * returns FTMOE_ERR_NO_SLOT and changes nothing (no slot, stamp or copy).  Copies
 * go on `copy_stream` and a slot is not overwritten before the compute work
 * released on it finished.
 */
typedef enum { FTMOE_LRU_PER_LAYER = 0, FTMOE_LRU_GLOBAL = 1 } ftmoe_cache_policy;

typedef struct {
  int layers, E;
  size_t blob_bytes;          /* bytes per expert blob (multiple of 16) */
  const void* bank;           /* pinned host bank (see above) */
  void* pool;                 /* device pool, >= layers * slots_per_layer * blob_bytes bytes */
  int slots_per_layer;
  int policy;                 /* ftmoe_cache_policy */
  ftmoe_stream_t copy_stream; /* side stream for host->device copies (not the compute stream) */
} ftmoe_cache_desc;

typedef struct {
  uint64_t lookups, hits, misses;          /* acquire requests' ids */
  uint64_t prefetch_lookups, prefetch_copies;
  uint64_t h2d_bytes;                      /* all copies */
  double h2d_ms;                           /* sum of copy durations measured with events */
} ftmoe_cache_stats;

typedef struct ftmoe_cache ftmoe_cache;

ftmoe_status ftmoe_cache_create(const ftmoe_cache_desc* desc, ftmoe_cache** out);

/* Start copies for the missing experts of `layer` (host ids[0..n)) on the copy
 * stream; returns at once.  slots_out (host int32 [n], nullable) receives the
 * slot index of each id (index within the layer's pool, or within the single
 * pool for the global policy) and copied_out (host uint8 [n], nullable) 1
 * where a copy was issued. */
ftmoe_status ftmoe_cache_prefetch(ftmoe_cache* c, int layer, const int32_t* ids, int n,
                                  int32_t* slots_out, uint8_t* copied_out);

/* Predictive prefetch from routing history ([P4] 方法: the decode phase predicts
 * the experts it needs; 核心洞察: consecutive agent steps reuse experts), in its
 * plainest form: ftmoe_cache_prefetch of the ids that `layer`'s most recent
 * ftmoe_cache_acquire asked for, in that order.  ids_out (host int32 [E],
 * nullable) receives those ids and *n_out their count (0, and nothing issued,
 * when the layer has not been acquired yet); slots_out / copied_out (host,
 * nullable, at least E entries) as for prefetch. */
ftmoe_status ftmoe_cache_prefetch_history(ftmoe_cache* c, int layer, int32_t* ids_out, int* n_out,
                                          int32_t* slots_out, uint8_t* copied_out);

/* Make `layer`'s experts ids[0..n) resident (copying misses), make `compute`
 * wait for their copies and pin their slots until ftmoe_cache_release(layer).
 * blob_out: host array of E pointers, filled for the requested ids (other entries
 * untouched), ready for ftmoe_weights.expert_blob.  slots_out / copied_out as for
 * prefetch.  FTMOE_ERR_NO_SLOT (nothing changed) when the pool has fewer unpinned
 * slots than the request needs. */
ftmoe_status ftmoe_cache_acquire(ftmoe_cache* c, int layer, const int32_t* ids, int n,
                                 ftmoe_stream_t compute, const void** blob_out,
                                 int32_t* slots_out, uint8_t* copied_out);

/* Unpin the slots of every acquire of `layer` since its previous release and mark
 * them as in use by the work enqueued on `compute` so far: a later copy into one of
 * them waits for that work. */
ftmoe_status ftmoe_cache_release(ftmoe_cache* c, int layer, ftmoe_stream_t compute);

/* Counters; synchronizes the copy stream so that h2d_ms is complete. */
ftmoe_status ftmoe_cache_stats_get(ftmoe_cache* c, ftmoe_cache_stats* out);

ftmoe_status ftmoe_cache_destroy(ftmoe_cache* c);

#ifdef __cplusplus
}
#endif

#endif /* FTMOE_H */
