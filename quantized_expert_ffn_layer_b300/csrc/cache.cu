// Expert slot cache: a pinned-host bank of expert blobs streamed into a device slot
// pool with LRU eviction, copies on a side stream ahead of use.
//
// FreeToken pages: hot experts stay on the GPU and cold ones in pinned host memory
// under a global LRU (architecture walkthrough §五; 机制四 of the double-buffered-
// prefill article), and the next layer is copied while the current one computes
// (机制一; "pipelined loading" in the paper digest's 方法).  The bookkeeping rules
// (stamps, victim choice) are stated in ftmoe.h.
#include <cstring>
#include <unordered_map>
#include <vector>

#include "common.cuh"
#include "internal.h"

struct ftmoe_cache {
  ftmoe_cache_desc d{};
  int npools = 0, nslot = 0;  // pools and slots per pool
  std::vector<int> owner_layer, owner_expert;  // [npools * nslot], -1 = empty
  std::vector<uint64_t> stamp;
  std::vector<cudaEvent_t> copy_done, busy;
  std::vector<char> copy_unwaited, has_busy;
  std::vector<int> pins;                       // per global slot: acquires not yet released
  std::unordered_map<long long, int> where;   // (layer * E + e) -> global slot
  std::vector<std::vector<int>> pinned;        // per layer: slots its acquires pinned
  std::vector<std::vector<int32_t>> last_ids;   // per layer: expert ids of the last acquire
  std::vector<cudaEvent_t> layer_done;          // per layer, recorded at release
  std::vector<std::pair<cudaEvent_t, cudaEvent_t>> timing_pending;
  std::vector<cudaEvent_t> timing_free;
  uint64_t clock = 0;
  ftmoe_cache_stats st{};
};

namespace {

int pool_of(const ftmoe_cache* c, int layer) {
  return c->d.policy == FTMOE_LRU_PER_LAYER ? layer : 0;
}

cudaEvent_t timing_event(ftmoe_cache* c) {
  if (!c->timing_free.empty()) {
    cudaEvent_t e = c->timing_free.back();
    c->timing_free.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

// Touches ids in order (see ftmoe.h); issues the copies of misses on the copy stream.
// All or nothing: the slot of every id is planned first, and a request that finds no
// slot for a missing id returns FTMOE_ERR_NO_SLOT before any record changes.  With
// `pin` (an acquire) the touched slots stay pinned until the layer's release.
ftmoe_status request(ftmoe_cache* c, int layer, const int32_t* ids, int n, int32_t* slots_out,
                     uint8_t* copied_out, std::vector<int>* gslots, int* ncopies, bool pin) {
  if (layer < 0 || layer >= c->d.layers || n < 0 || (n > 0 && !ids)) return FTMOE_ERR_INVALID_ARG;
  for (int i = 0; i < n; ++i)
    if (ids[i] < 0 || ids[i] >= c->d.E) return FTMOE_ERR_INVALID_ARG;
  if (n > c->nslot) return FTMOE_ERR_NO_SLOT;
  const int pool = pool_of(c, layer);
  const int base = pool * c->nslot;
  cudaStream_t cs = (cudaStream_t)c->d.copy_stream;
  // ---- plan (no record changes): a slot taken for a miss is touched, so it is taken at
  // most once per request, and the stamps of untouched slots do not change meanwhile
  std::vector<char> touched(c->nslot, 0), retaken(c->nslot, 0);
  std::unordered_map<long long, int> taken;  // keys placed by this request -> pool slot
  std::vector<int> plan_slot(n);
  std::vector<char> plan_copy(n);
  for (int i = 0; i < n; ++i) {
    const long long key = (long long)layer * c->d.E + ids[i];
    int s = -1;
    auto tk = taken.find(key);
    if (tk != taken.end()) {
      s = tk->second;
    } else {
      auto it = c->where.find(key);
      if (it != c->where.end() && !retaken[it->second - base]) s = it->second - base;
    }
    const bool copied = s < 0;
    if (copied) {
      for (int q = 0; q < c->nslot && s < 0; ++q)
        if (!touched[q] && !c->pins[base + q] && c->owner_layer[base + q] < 0) s = q;
      if (s < 0) {
        uint64_t best = UINT64_MAX;
        for (int q = 0; q < c->nslot; ++q)
          if (!touched[q] && !c->pins[base + q] && c->stamp[base + q] < best) {
            best = c->stamp[base + q];
            s = q;
          }
      }
      if (s < 0) return FTMOE_ERR_NO_SLOT;
      retaken[s] = 1;
      taken[key] = s;
    }
    touched[s] = 1;
    plan_slot[i] = s;
    plan_copy[i] = copied ? 1 : 0;
  }
  // ---- commit
  std::vector<int> to_copy;  // global slots whose blob must be copied
  std::vector<long long> to_copy_key;
  for (int i = 0; i < n; ++i) {
    const long long key = (long long)layer * c->d.E + ids[i];
    const int s = plan_slot[i], gs = base + s;
    ++c->clock;
    if (plan_copy[i]) {
      if (c->owner_layer[gs] >= 0)
        c->where.erase((long long)c->owner_layer[gs] * c->d.E + c->owner_expert[gs]);
      c->owner_layer[gs] = layer;
      c->owner_expert[gs] = ids[i];
      c->where[key] = gs;
      to_copy.push_back(gs);
      to_copy_key.push_back(key);
    }
    c->stamp[gs] = c->clock;
    if (slots_out) slots_out[i] = s;
    if (copied_out) copied_out[i] = plan_copy[i];
    if (gslots) gslots->push_back(gs);
  }
  if (pin)
    for (int q = 0; q < c->nslot; ++q)
      if (touched[q]) {
        ++c->pins[base + q];
        c->pinned[layer].push_back(base + q);
      }
  *ncopies = (int)to_copy.size();
  if (to_copy.empty()) return FTMOE_OK;
  // a victim slot may still be read by compute work released on it: wait for that first
  for (int gs : to_copy)
    if (c->has_busy[gs] && cudaStreamWaitEvent(cs, c->busy[gs], 0) != cudaSuccess) return FTMOE_ERR_CUDA;
  cudaEvent_t t0 = timing_event(c), t1 = timing_event(c);
  if (!t0 || !t1 || cudaEventRecord(t0, cs) != cudaSuccess) return FTMOE_ERR_CUDA;
  for (size_t i = 0; i < to_copy.size(); ++i) {
    const int gs = to_copy[i];
    const char* src = (const char*)c->d.bank + (size_t)to_copy_key[i] * c->d.blob_bytes;
    char* dst = (char*)c->d.pool + (size_t)gs * c->d.blob_bytes;
    if (cudaMemcpyAsync(dst, src, c->d.blob_bytes, cudaMemcpyHostToDevice, cs) != cudaSuccess)
      return FTMOE_ERR_CUDA;
    if (cudaEventRecord(c->copy_done[gs], cs) != cudaSuccess) return FTMOE_ERR_CUDA;
    c->copy_unwaited[gs] = 1;
    c->st.h2d_bytes += c->d.blob_bytes;
  }
  if (cudaEventRecord(t1, cs) != cudaSuccess) return FTMOE_ERR_CUDA;
  c->timing_pending.emplace_back(t0, t1);
  return FTMOE_OK;
}

void destroy_events(ftmoe_cache* c) {
  for (auto e : c->copy_done) if (e) cudaEventDestroy(e);
  // busy[] entries alias layer_done[] events
  for (auto e : c->layer_done) if (e) cudaEventDestroy(e);
  for (auto& p : c->timing_pending) { cudaEventDestroy(p.first); cudaEventDestroy(p.second); }
  for (auto e : c->timing_free) cudaEventDestroy(e);
}

}  // namespace

extern "C" {

ftmoe_status ftmoe_cache_create(const ftmoe_cache_desc* d, ftmoe_cache** out) {
  if (!d || !out || d->layers < 1 || d->E < 1 || d->slots_per_layer < 1 || !d->bank || !d->pool ||
      d->blob_bytes == 0 || d->blob_bytes % 16 || !d->copy_stream ||
      (d->policy != FTMOE_LRU_PER_LAYER && d->policy != FTMOE_LRU_GLOBAL))
    return FTMOE_ERR_INVALID_ARG;
  ftmoe_cache* c = new (std::nothrow) ftmoe_cache();
  if (!c) return FTMOE_ERR_INVALID_ARG;
  c->d = *d;
  c->npools = d->policy == FTMOE_LRU_PER_LAYER ? d->layers : 1;
  c->nslot = d->policy == FTMOE_LRU_PER_LAYER ? d->slots_per_layer : d->slots_per_layer * d->layers;
  const int total = c->npools * c->nslot;
  c->owner_layer.assign(total, -1);
  c->owner_expert.assign(total, -1);
  c->stamp.assign(total, 0);
  c->copy_done.assign(total, nullptr);
  c->busy.assign(total, nullptr);
  c->copy_unwaited.assign(total, 0);
  c->has_busy.assign(total, 0);
  c->pins.assign(total, 0);
  c->pinned.resize(d->layers);
  c->last_ids.resize(d->layers);
  c->layer_done.assign(d->layers, nullptr);
  bool ok = true;
  for (int i = 0; i < total && ok; ++i)
    ok = cudaEventCreateWithFlags(&c->copy_done[i], cudaEventDisableTiming) == cudaSuccess;
  for (int l = 0; l < d->layers && ok; ++l)
    ok = cudaEventCreateWithFlags(&c->layer_done[l], cudaEventDisableTiming) == cudaSuccess;
  if (!ok) {
    destroy_events(c);
    delete c;
    return FTMOE_ERR_CUDA;
  }
  *out = c;
  return FTMOE_OK;
}

ftmoe_status ftmoe_cache_prefetch(ftmoe_cache* c, int layer, const int32_t* ids, int n,
                                  int32_t* slots_out, uint8_t* copied_out) {
  if (!c) return FTMOE_ERR_INVALID_ARG;
  int nc = 0;
  ftmoe_status s = request(c, layer, ids, n, slots_out, copied_out, nullptr, &nc, false);
  if (s == FTMOE_OK) {
    c->st.prefetch_lookups += (uint64_t)n;
    c->st.prefetch_copies += (uint64_t)nc;
  }
  return s;
}

ftmoe_status ftmoe_cache_acquire(ftmoe_cache* c, int layer, const int32_t* ids, int n,
                                 ftmoe_stream_t compute, const void** blob_out, int32_t* slots_out,
                                 uint8_t* copied_out) {
  if (!c || !blob_out) return FTMOE_ERR_INVALID_ARG;
  std::vector<int> gs;
  int nc = 0;
  ftmoe_status s = request(c, layer, ids, n, slots_out, copied_out, &gs, &nc, true);
  if (s != FTMOE_OK) return s;
  c->st.lookups += (uint64_t)n;
  c->st.misses += (uint64_t)nc;
  c->st.hits += (uint64_t)(n - nc);
  cudaStream_t cs = (cudaStream_t)compute;
  for (int i = 0; i < n; ++i) {
    const int g = gs[i];
    if (c->copy_unwaited[g]) {
      if (cudaStreamWaitEvent(cs, c->copy_done[g], 0) != cudaSuccess) return FTMOE_ERR_CUDA;
      c->copy_unwaited[g] = 0;
    }
    blob_out[ids[i]] = (const char*)c->d.pool + (size_t)g * c->d.blob_bytes;
  }
  c->last_ids[layer].assign(ids, ids + n);
  return FTMOE_OK;
}

// Semantic-aware expert caching (the edge-serving digest, 方法: the decode phase
// predicts the experts it will need to raise the hit rate; 核心洞察: consecutive agent
// steps reuse experts) in its plainest form: predict that a layer needs what it needed
// at its last acquire.
ftmoe_status ftmoe_cache_prefetch_history(ftmoe_cache* c, int layer, int32_t* ids_out, int* n_out,
                                          int32_t* slots_out, uint8_t* copied_out) {
  if (!c || !n_out || layer < 0 || layer >= c->d.layers) return FTMOE_ERR_INVALID_ARG;
  const std::vector<int32_t> ids = c->last_ids[layer];  // (request() may not change it, but copy)
  *n_out = (int)ids.size();
  if (ids_out && !ids.empty()) std::memcpy(ids_out, ids.data(), ids.size() * sizeof(int32_t));
  if (ids.empty()) return FTMOE_OK;
  return ftmoe_cache_prefetch(c, layer, ids.data(), (int)ids.size(), slots_out, copied_out);
}

ftmoe_status ftmoe_cache_release(ftmoe_cache* c, int layer, ftmoe_stream_t compute) {
  if (!c || layer < 0 || layer >= c->d.layers) return FTMOE_ERR_INVALID_ARG;
  cudaEvent_t ev = c->layer_done[layer];
  if (cudaEventRecord(ev, (cudaStream_t)compute) != cudaSuccess) return FTMOE_ERR_CUDA;
  for (int g : c->pinned[layer]) {
    c->busy[g] = ev;
    c->has_busy[g] = 1;
    --c->pins[g];
  }
  c->pinned[layer].clear();
  return FTMOE_OK;
}

ftmoe_status ftmoe_cache_stats_get(ftmoe_cache* c, ftmoe_cache_stats* out) {
  if (!c || !out) return FTMOE_ERR_INVALID_ARG;
  if (cudaStreamSynchronize((cudaStream_t)c->d.copy_stream) != cudaSuccess) return FTMOE_ERR_CUDA;
  for (auto& p : c->timing_pending) {
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, p.first, p.second) == cudaSuccess) c->st.h2d_ms += ms;
    c->timing_free.push_back(p.first);
    c->timing_free.push_back(p.second);
  }
  c->timing_pending.clear();
  *out = c->st;
  return FTMOE_OK;
}

ftmoe_status ftmoe_cache_destroy(ftmoe_cache* c) {
  if (!c) return FTMOE_ERR_INVALID_ARG;
  cudaStreamSynchronize((cudaStream_t)c->d.copy_stream);
  destroy_events(c);
  delete c;
  return FTMOE_OK;
}

}  // extern "C"
