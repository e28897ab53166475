/* bitdelta_kmerge.h — the K-Merge adapter pool: which requested adapters are
 * stored, under a fixed storage budget B, and which stored entry a new
 * adapter is merged into when storing it would exceed B.
 *
 * Page "BitDelta: serving 14 Zen models from one GPU cluster", section
 * "K-Merge: online LoRA adapter management for the edge": the pool of (merged)
 * adapters never holds more than B bytes in all.  When an adapter that is not
 * in the pool is requested, (1) its cosine similarity with every pool member
 * is computed on the task vectors, (2) the most similar member is found,
 * (3) the new adapter is merged into it (OPCM), and (4) if the merged adapter
 * passes a quality threshold on both tasks, it replaces the original.
 *
 * Readings (the page leaves these open):
 *   - An adapter that fits within B next to the current entries is stored as
 *     an entry of its own; steps 1-4 run only when storing it would exceed B
 *     (the policy's purpose is to stay within B, and merging adapters that
 *     both fit would only lose quality).
 *   - The similarity of step 1 is the 1-bit task-vector cosine of
 *     bitdelta_sign_similarity (include/bitdelta.h); the caller computes it
 *     against each entry's stored delta.  The most similar entry is the
 *     argmax, ties to the lowest entry index.
 *   - OPCM (step 3) and the quality threshold (step 4) are not specified by
 *     the page and need evaluation data: they are the caller's.  The pool
 *     names the merge target, the caller merges and evaluates, and reports
 *     the outcome with bd_kmerge_commit (accepted: the entry now covers both
 *     adapters and holds the merged adapter's bytes; rejected: nothing
 *     changes and the adapter stays outside the pool).
 *   - Entries are never removed: a merge replaces an entry's contents in
 *     place, so entry indices are stable for the caller's own storage.
 *
 * Memory: the pool keeps only host bookkeeping (ids and byte counts); the
 * adapters' deltas live wherever the caller stores them.  All calls are
 * host-only (no CUDA calls) and thread-safe (one mutex per pool).
 */
#ifndef BITDELTA_KMERGE_H_
#define BITDELTA_KMERGE_H_

#include <stddef.h>
#include <stdint.h>

#include "bitdelta.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct bd_kmerge_pool bd_kmerge_pool_t;

typedef enum {
  BD_KMERGE_HIT = 0,              /* already covered by entry *entry */
  BD_KMERGE_STORE = 1,            /* stored as the new entry *entry (it fit within B) */
  BD_KMERGE_NEED_SIMILARITY = 2,  /* storing would exceed B: call again with cos[] */
  BD_KMERGE_MERGE = 3,            /* merge into entry *entry (most similar), then commit */
  BD_KMERGE_REJECT = 4            /* larger than B by itself: never stored */
} bd_kmerge_action;

typedef struct {
  int32_t entries;        /* entries stored */
  int32_t adapters;       /* adapters covered by the entries */
  uint64_t used_bytes;    /* bytes the entries hold (<= budget) */
  uint64_t budget_bytes;  /* B */
  uint64_t stores, merges_proposed, merges_accepted, merges_rejected, rejects, hits;
} bd_kmerge_stats;

/* Create a pool with budget B = budget_bytes (> 0). */
bd_status bd_kmerge_create(uint64_t budget_bytes, bd_kmerge_pool_t** out);
bd_status bd_kmerge_destroy(bd_kmerge_pool_t* pool);

/* Request adapter `adapter` (>= 0) whose delta takes `bytes` (> 0) bytes.
 *   Covered by an entry            -> BD_KMERGE_HIT, *entry = that entry.
 *   used + bytes <= B              -> BD_KMERGE_STORE, *entry = new entry index
 *                                     (the caller stores the delta there).
 *   otherwise, cos == NULL         -> BD_KMERGE_NEED_SIMILARITY, *entry = -1,
 *                                     nothing changes.
 *   otherwise, cos of n_cos = number of entries values (the adapter's
 *   similarity with each entry, in entry order, finite, in [-1, 1] up to
 *   rounding)                     -> BD_KMERGE_MERGE, *entry = argmax (ties:
 *                                     lowest index); the merge is pending until
 *                                     bd_kmerge_commit (one pending merge at a
 *                                     time; requesting the same adapter again
 *                                     proposes again).
 *   bytes > B                      -> BD_KMERGE_REJECT.
 * BD_ERR_INVALID_ARG for bad arguments (n_cos not the entry count, a value
 * not finite or outside [-1.000001, 1.000001], a merge already pending for
 * another adapter). */
bd_status bd_kmerge_request(bd_kmerge_pool_t* pool, int32_t adapter, uint64_t bytes,
                            const double* cos, int32_t n_cos, bd_kmerge_action* action,
                            int32_t* entry);

/* Outcome of the pending merge of `adapter` into `entry` (the caller's OPCM
 * merge and quality check).  accepted != 0: the entry covers `adapter` too and
 * now holds merged_bytes bytes (BD_ERR_INVALID_ARG, and nothing changes, if
 * that would take the pool over B).  accepted == 0: nothing changes.  Either
 * way the merge is no longer pending.  BD_ERR_INVALID_ARG if no merge of
 * `adapter` into `entry` is pending. */
bd_status bd_kmerge_commit(bd_kmerge_pool_t* pool, int32_t adapter, int32_t entry,
                           int32_t accepted, uint64_t merged_bytes);

/* Entry covering `adapter` (-1 when none). */
bd_status bd_kmerge_entry_of(const bd_kmerge_pool_t* pool, int32_t adapter, int32_t* entry);

/* Bytes held by entry `entry`, and how many adapters it covers. */
bd_status bd_kmerge_entry_info(const bd_kmerge_pool_t* pool, int32_t entry, uint64_t* bytes,
                               int32_t* adapters);

bd_status bd_kmerge_get_stats(const bd_kmerge_pool_t* pool, bd_kmerge_stats* out);

#ifdef __cplusplus
}
#endif

#endif /* BITDELTA_KMERGE_H_ */
