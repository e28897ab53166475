// kmerge.cu — the K-Merge adapter pool (host code, no CUDA calls).
// Interface, policy and readings: include/bitdelta_kmerge.h.
//
// Page "BitDelta: serving 14 Zen models from one GPU cluster", section
// "K-Merge": a pool of merged adapters whose total storage never exceeds the
// budget B; a requested adapter outside the pool is compared with every
// member by the cosine similarity of task vectors and merged into the most
// similar one.
#include <cmath>
#include <cstdint>
#include <mutex>
#include <unordered_map>
#include <vector>

#include "bitdelta_kmerge.h"

namespace {

struct Entry {
  uint64_t bytes = 0;
  std::vector<int32_t> adapters;
};

}  // namespace

struct bd_kmerge_pool {
  std::mutex mu;
  uint64_t budget = 0;
  uint64_t used = 0;
  std::vector<Entry> entries;
  std::unordered_map<int32_t, int32_t> entry_of;  // adapter -> entry
  int32_t pending_adapter = -1;                   // merge proposed, not yet committed
  int32_t pending_entry = -1;
  bd_kmerge_stats stats{};
};

extern "C" {

bd_status bd_kmerge_create(uint64_t budget_bytes, bd_kmerge_pool_t** out) {
  if (out == nullptr || budget_bytes == 0) return BD_ERR_INVALID_ARG;
  bd_kmerge_pool* p = new bd_kmerge_pool;
  p->budget = budget_bytes;
  *out = p;
  return BD_OK;
}

bd_status bd_kmerge_destroy(bd_kmerge_pool_t* pool) {
  if (pool == nullptr) return BD_ERR_INVALID_ARG;
  delete pool;
  return BD_OK;
}

bd_status bd_kmerge_request(bd_kmerge_pool_t* pool, int32_t adapter, uint64_t bytes,
                            const double* cos, int32_t n_cos, bd_kmerge_action* action,
                            int32_t* entry) {
  if (pool == nullptr || action == nullptr || entry == nullptr || adapter < 0 || bytes == 0)
    return BD_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(pool->mu);
  const auto hit = pool->entry_of.find(adapter);
  if (hit != pool->entry_of.end()) {
    *action = BD_KMERGE_HIT;
    *entry = hit->second;
    ++pool->stats.hits;
    return BD_OK;
  }
  if (bytes > pool->budget) {
    *action = BD_KMERGE_REJECT;
    *entry = -1;
    ++pool->stats.rejects;
    return BD_OK;
  }
  if (pool->used + bytes <= pool->budget) {
    // fits within B: an entry of its own (a pending merge re-checks B at
    // its commit)
    Entry e;
    e.bytes = bytes;
    e.adapters.push_back(adapter);
    pool->entries.push_back(e);
    pool->used += bytes;
    const int32_t idx = static_cast<int32_t>(pool->entries.size()) - 1;
    pool->entry_of[adapter] = idx;
    *action = BD_KMERGE_STORE;
    *entry = idx;
    ++pool->stats.stores;
    return BD_OK;
  }
  // storing would exceed B: steps 1-2, the most similar entry
  if (cos == nullptr) {
    *action = BD_KMERGE_NEED_SIMILARITY;
    *entry = -1;
    return BD_OK;
  }
  if (n_cos != static_cast<int32_t>(pool->entries.size())) return BD_ERR_INVALID_ARG;
  if (pool->pending_adapter >= 0 && pool->pending_adapter != adapter) return BD_ERR_INVALID_ARG;
  int32_t best = -1;
  for (int32_t i = 0; i < n_cos; ++i) {
    const double c = cos[i];
    if (!std::isfinite(c) || c < -1.000001 || c > 1.000001) return BD_ERR_INVALID_ARG;
    if (best < 0 || c > cos[best]) best = i;  // strict: ties keep the lower index
  }
  pool->pending_adapter = adapter;
  pool->pending_entry = best;
  *action = BD_KMERGE_MERGE;
  *entry = best;
  ++pool->stats.merges_proposed;
  return BD_OK;
}

bd_status bd_kmerge_commit(bd_kmerge_pool_t* pool, int32_t adapter, int32_t entry,
                           int32_t accepted, uint64_t merged_bytes) {
  if (pool == nullptr) return BD_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(pool->mu);
  if (pool->pending_adapter < 0 || pool->pending_adapter != adapter ||
      pool->pending_entry != entry)
    return BD_ERR_INVALID_ARG;
  if (accepted) {
    Entry& e = pool->entries[static_cast<size_t>(entry)];
    if (merged_bytes == 0 || pool->used - e.bytes + merged_bytes > pool->budget)
      return BD_ERR_INVALID_ARG;  // still pending: the caller may commit again
    pool->used = pool->used - e.bytes + merged_bytes;
    e.bytes = merged_bytes;
    e.adapters.push_back(adapter);
    pool->entry_of[adapter] = entry;
    ++pool->stats.merges_accepted;
  } else {
    ++pool->stats.merges_rejected;
  }
  pool->pending_adapter = -1;
  pool->pending_entry = -1;
  return BD_OK;
}

bd_status bd_kmerge_entry_of(const bd_kmerge_pool_t* pool, int32_t adapter, int32_t* entry) {
  if (pool == nullptr || entry == nullptr) return BD_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(const_cast<bd_kmerge_pool*>(pool)->mu);
  const auto it = pool->entry_of.find(adapter);
  *entry = it == pool->entry_of.end() ? -1 : it->second;
  return BD_OK;
}

bd_status bd_kmerge_entry_info(const bd_kmerge_pool_t* pool, int32_t entry, uint64_t* bytes,
                               int32_t* adapters) {
  if (pool == nullptr || bytes == nullptr || adapters == nullptr) return BD_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(const_cast<bd_kmerge_pool*>(pool)->mu);
  if (entry < 0 || entry >= static_cast<int32_t>(pool->entries.size())) return BD_ERR_INVALID_ARG;
  *bytes = pool->entries[static_cast<size_t>(entry)].bytes;
  *adapters = static_cast<int32_t>(pool->entries[static_cast<size_t>(entry)].adapters.size());
  return BD_OK;
}

bd_status bd_kmerge_get_stats(const bd_kmerge_pool_t* pool, bd_kmerge_stats* out) {
  if (pool == nullptr || out == nullptr) return BD_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(const_cast<bd_kmerge_pool*>(pool)->mu);
  *out = pool->stats;
  out->entries = static_cast<int32_t>(pool->entries.size());
  out->adapters = static_cast<int32_t>(pool->entry_of.size());
  out->used_bytes = pool->used;
  out->budget_bytes = pool->budget;
  return BD_OK;
}

}  // extern "C"
