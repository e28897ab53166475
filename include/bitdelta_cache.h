/* bitdelta_cache.h — the delta cache: variants' packed deltas (signs + α)
 * kept resident in a caller-owned arena, loaded on first request.
 *
 * Page "BitDelta: serving 14 Zen models from one GPU cluster", section
 * "Infrastructure details": a variant whose delta is not cached pays a cold
 * load on its first request and then stays cached until the eviction policy
 * removes it; eviction is LRU weighted by request rate — the variants with
 * the most traffic (the page: the top 6 of 14) always stay resident and the
 * rest share the remaining space under LRU; requests for a variant whose
 * delta is being loaded queue behind that one load instead of each starting
 * a load of its own.
 *
 * Reading of "LRU weighted by request rate" (the page gives no formula):
 * a variant's traffic is its count of acquire calls; the pin_top_k variants
 * with the highest counts (ties: lower id) are never evicted; among the other
 * resident variants that no caller holds, the least recently acquired one is
 * evicted first.
 *
 * Memory: everything is caller-owned.  The arena (device memory, or host
 * memory for a host-only cache) is split into equal slots; each variant's
 * delta is one contiguous blob of at most slot_bytes, registered with its
 * host address (pinned host memory lets the copy run asynchronously).  The
 * cache allocates only its own host bookkeeping and, for a device arena, one
 * CUDA event per slot.
 *
 * Streams: loads are cudaMemcpyAsync calls on the caller's copy stream,
 * followed by an event; bd_cache_acquire makes the caller's stream wait for
 * that event, so work queued on it after acquire sees the loaded bytes.
 * All calls are thread-safe (one mutex per cache).
 */
#ifndef BITDELTA_CACHE_H_
#define BITDELTA_CACHE_H_

#include <stddef.h>
#include <stdint.h>

#include "bitdelta.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct bd_cache bd_cache_t;

typedef enum {
  BD_CACHE_DEVICE_ARENA = 0, /* arena in device memory; loads are async H2D copies */
  BD_CACHE_HOST_ARENA = 1    /* arena in host memory; loads are memcpy (no CUDA calls) */
} bd_cache_arena_kind;

typedef struct {
  uint64_t acquires;           /* bd_cache_acquire calls that returned BD_OK */
  uint64_t hits;               /* ... that found the delta resident and loaded */
  uint64_t queued_behind_load; /* ... that found its load still in flight and waited on it */
  uint64_t loads;              /* loads started (one per miss) */
  uint64_t evictions;          /* resident variants evicted to make room */
  uint64_t bytes_loaded;       /* bytes copied into the arena */
} bd_cache_stats;

/* Create a cache over arena [arena, arena + arena_bytes) cut into
 * floor(arena_bytes / slot_bytes) slots.  slot_bytes must be a positive
 * multiple of 256 and the arena 256-byte aligned; pin_top_k >= 0.
 * copy_stream: the stream loads run on (device arena; ignored for a host
 * arena).  BD_ERR_INVALID_ARG for bad arguments, BD_ERR_CUDA if an event
 * cannot be created.  *out receives the cache. */
bd_status bd_cache_create(void* arena, size_t arena_bytes, size_t slot_bytes, int32_t pin_top_k,
                          bd_cache_arena_kind kind, bd_stream_t copy_stream, bd_cache_t** out);

/* Destroy the cache (after the caller's streams are done with its slots). */
bd_status bd_cache_destroy(bd_cache_t* cache);

/* Register (or re-register) variant `variant` (>= 0) as `bytes` (<= slot
 * bytes) at host address host_src, which must stay valid while the cache
 * lives.  Re-registering a resident variant invalidates its slot (the next
 * acquire loads the new bytes) unless a caller holds it (then
 * BD_ERR_INVALID_ARG). */
bd_status bd_cache_register(bd_cache_t* cache, int32_t variant, const void* host_src, size_t bytes);

/* Acquire variant `variant`: *ptr receives the address of its delta in the
 * arena, valid until the matching bd_cache_release.  If it is not resident a
 * slot is taken (free, else by eviction) and its load is queued on the copy
 * stream; if its load is already in flight the call shares it.  For a device
 * arena, `stream` is made to wait for the load.  BD_ERR_INVALID_ARG for an
 * unregistered variant; BD_ERR_CACHE_FULL when every slot is held by callers
 * or by pinned variants (nothing is evicted, nothing loaded); BD_ERR_CUDA if
 * a copy or event call fails. */
bd_status bd_cache_acquire(bd_cache_t* cache, int32_t variant, bd_stream_t stream, void** ptr);

/* Release one acquire of `variant` (BD_ERR_INVALID_ARG if it holds none).
 * `stream`: the stream on which the holder queued its reads of the slot; a
 * later load that reuses the slot is ordered after that work (device arena:
 * the copy stream waits for an event recorded on `stream` now). */
bd_status bd_cache_release(bd_cache_t* cache, int32_t variant, bd_stream_t stream);

/* Counters since creation. */
bd_status bd_cache_get_stats(const bd_cache_t* cache, bd_cache_stats* out);

/* Slot of `variant` (-1 when not resident). */
bd_status bd_cache_slot_of(const bd_cache_t* cache, int32_t variant, int32_t* slot);

#ifdef __cplusplus
}
#endif

#endif /* BITDELTA_CACHE_H_ */
