// cache.cu — the delta cache (host code).  Interface and policy:
// include/bitdelta_cache.h.
//
// Page "BitDelta: serving 14 Zen models from one GPU cluster", section
// "Infrastructure details": cold loads on first request, eviction by LRU
// weighted by request rate with the highest-traffic variants pinned, and
// requests for a variant whose delta is loading queued behind that one load.
#include <climits>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <unordered_map>
#include <vector>

#include <cuda_runtime.h>

#include "bitdelta_cache.h"

namespace {

struct Variant {
  const void* src = nullptr;
  size_t bytes = 0;
  uint64_t requests = 0;  // traffic: acquire calls so far
  uint64_t last_use = 0;  // logical time of the last acquire
  int32_t slot = -1;      // -1: not resident
  int32_t holders = 0;    // acquires not yet released
};

}  // namespace

struct bd_cache {
  std::mutex mu;
  uint8_t* arena = nullptr;
  size_t slot_bytes = 0;
  int32_t n_slots = 0;
  int32_t pin_top_k = 0;
  bd_cache_arena_kind kind = BD_CACHE_DEVICE_ARENA;
  cudaStream_t copy = nullptr;
  std::vector<int32_t> slot_owner;      // variant per slot, -1 = free
  std::vector<cudaEvent_t> slot_loaded; // device arena: completion of the slot's load
  cudaEvent_t released = nullptr;       // device arena: readers' progress at a release
  std::unordered_map<int32_t, Variant> vars;
  uint64_t clock = 0;
  bd_cache_stats stats{};
};

namespace {

bool device_arena(const bd_cache* c) { return c->kind == BD_CACHE_DEVICE_ARENA; }

// The pin_top_k registered variants with the most requests (ties: lower id).
bool is_pinned(const bd_cache* c, int32_t id) {
  if (c->pin_top_k <= 0) return false;
  const Variant& v = c->vars.at(id);
  int32_t ahead = 0;  // variants ranked before `id`
  for (const auto& kv : c->vars) {
    const Variant& o = kv.second;
    if (o.requests > v.requests || (o.requests == v.requests && kv.first < id)) {
      if (++ahead >= c->pin_top_k) return false;
    }
  }
  return true;
}

// A free slot, else the least recently used resident variant that nobody
// holds and that is not pinned (evicted); -1 when there is none.
int32_t take_slot(bd_cache* c, int32_t for_id) {
  for (int32_t s = 0; s < c->n_slots; ++s)
    if (c->slot_owner[s] < 0) return s;
  int32_t victim = -1;
  uint64_t oldest = UINT64_MAX;
  for (int32_t s = 0; s < c->n_slots; ++s) {
    const int32_t id = c->slot_owner[s];
    if (id == for_id) continue;
    const Variant& v = c->vars.at(id);
    if (v.holders > 0 || is_pinned(c, id)) continue;
    if (v.last_use < oldest) {
      oldest = v.last_use;
      victim = s;
    }
  }
  if (victim >= 0) {
    c->vars.at(c->slot_owner[victim]).slot = -1;
    c->slot_owner[victim] = -1;
    ++c->stats.evictions;
  }
  return victim;
}

}  // namespace

extern "C" {

bd_status bd_cache_create(void* arena, size_t arena_bytes, size_t slot_bytes, int32_t pin_top_k,
                          bd_cache_arena_kind kind, bd_stream_t copy_stream, bd_cache_t** out) {
  if (out == nullptr || arena == nullptr || slot_bytes == 0 || slot_bytes % 256 != 0 ||
      pin_top_k < 0 || (reinterpret_cast<uintptr_t>(arena) & 255u) != 0 ||
      (kind != BD_CACHE_DEVICE_ARENA && kind != BD_CACHE_HOST_ARENA))
    return BD_ERR_INVALID_ARG;
  const size_t n = arena_bytes / slot_bytes;
  if (n == 0 || n > INT32_MAX) return BD_ERR_INVALID_ARG;
  bd_cache* c = new bd_cache();
  c->arena = static_cast<uint8_t*>(arena);
  c->slot_bytes = slot_bytes;
  c->n_slots = static_cast<int32_t>(n);
  c->pin_top_k = pin_top_k;
  c->kind = kind;
  c->copy = reinterpret_cast<cudaStream_t>(copy_stream);
  c->slot_owner.assign(n, -1);
  if (device_arena(c)) {
    c->slot_loaded.assign(n, nullptr);
    bool ok = cudaEventCreateWithFlags(&c->released, cudaEventDisableTiming) == cudaSuccess;
    for (size_t s = 0; ok && s < n; ++s)
      ok = cudaEventCreateWithFlags(&c->slot_loaded[s], cudaEventDisableTiming) == cudaSuccess;
    if (!ok) {
      bd_cache_destroy(c);
      return BD_ERR_CUDA;
    }
  }
  *out = c;
  return BD_OK;
}

bd_status bd_cache_destroy(bd_cache_t* c) {
  if (c == nullptr) return BD_ERR_INVALID_ARG;
  for (cudaEvent_t e : c->slot_loaded)
    if (e != nullptr) cudaEventDestroy(e);
  if (c->released != nullptr) cudaEventDestroy(c->released);
  delete c;
  return BD_OK;
}

bd_status bd_cache_register(bd_cache_t* c, int32_t variant, const void* host_src, size_t bytes) {
  if (c == nullptr || variant < 0 || host_src == nullptr || bytes == 0 || bytes > c->slot_bytes)
    return BD_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(c->mu);
  Variant& v = c->vars[variant];
  if (v.slot >= 0) {
    if (v.holders > 0) return BD_ERR_INVALID_ARG;
    c->slot_owner[v.slot] = -1;  // the old bytes are stale: free the slot
    v.slot = -1;
  }
  v.src = host_src;
  v.bytes = bytes;
  return BD_OK;
}

bd_status bd_cache_acquire(bd_cache_t* c, int32_t variant, bd_stream_t stream, void** ptr) {
  if (c == nullptr || ptr == nullptr) return BD_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(c->mu);
  auto it = c->vars.find(variant);
  if (it == c->vars.end()) return BD_ERR_INVALID_ARG;
  Variant& v = it->second;
  ++v.requests;
  v.last_use = ++c->clock;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (v.slot >= 0) {
    bool in_flight = false;
    if (device_arena(c)) {
      const cudaError_t q = cudaEventQuery(c->slot_loaded[v.slot]);
      if (q != cudaSuccess && q != cudaErrorNotReady) return BD_ERR_CUDA;
      in_flight = q == cudaErrorNotReady;
      // queue behind the one load of this delta (a no-op once it is done)
      if (cudaStreamWaitEvent(s, c->slot_loaded[v.slot], 0) != cudaSuccess) return BD_ERR_CUDA;
    }
    ++v.holders;
    ++c->stats.acquires;
    ++(in_flight ? c->stats.queued_behind_load : c->stats.hits);
    *ptr = c->arena + static_cast<size_t>(v.slot) * c->slot_bytes;
    return BD_OK;
  }
  const int32_t slot = take_slot(c, variant);
  if (slot < 0) return BD_ERR_CACHE_FULL;
  uint8_t* dst = c->arena + static_cast<size_t>(slot) * c->slot_bytes;
  if (device_arena(c)) {
    // the copy stream has already waited for every earlier release's readers
    if (cudaMemcpyAsync(dst, v.src, v.bytes, cudaMemcpyHostToDevice, c->copy) != cudaSuccess ||
        cudaEventRecord(c->slot_loaded[slot], c->copy) != cudaSuccess ||
        cudaStreamWaitEvent(s, c->slot_loaded[slot], 0) != cudaSuccess) {
      return BD_ERR_CUDA;  // the slot stays free
    }
  } else {
    std::memcpy(dst, v.src, v.bytes);
  }
  c->slot_owner[slot] = variant;
  v.slot = slot;
  v.holders = 1;
  ++c->stats.loads;
  ++c->stats.acquires;
  c->stats.bytes_loaded += v.bytes;
  *ptr = dst;
  return BD_OK;
}

bd_status bd_cache_release(bd_cache_t* c, int32_t variant, bd_stream_t stream) {
  if (c == nullptr) return BD_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(c->mu);
  auto it = c->vars.find(variant);
  if (it == c->vars.end() || it->second.holders <= 0) return BD_ERR_INVALID_ARG;
  if (device_arena(c)) {
    // A later load into this slot runs on the copy stream: order it after the
    // work this holder queued on `stream` up to now (its reads of the slot).
    if (cudaEventRecord(c->released, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess ||
        cudaStreamWaitEvent(c->copy, c->released, 0) != cudaSuccess)
      return BD_ERR_CUDA;
  }
  --it->second.holders;
  return BD_OK;
}

bd_status bd_cache_get_stats(const bd_cache_t* c, bd_cache_stats* out) {
  if (c == nullptr || out == nullptr) return BD_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(const_cast<bd_cache*>(c)->mu);
  *out = c->stats;
  return BD_OK;
}

bd_status bd_cache_slot_of(const bd_cache_t* c, int32_t variant, int32_t* slot) {
  if (c == nullptr || slot == nullptr) return BD_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(const_cast<bd_cache*>(c)->mu);
  auto it = c->vars.find(variant);
  *slot = it == c->vars.end() ? -1 : it->second.slot;
  return BD_OK;
}

}  // extern "C"
