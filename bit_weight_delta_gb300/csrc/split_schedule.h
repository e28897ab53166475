// split_schedule.h — index arithmetic of the prefill kernel's split schedule
// (gemm_pair.cu), shared with a host test hook so that the CPU tests check
// the kernel's own formulas.
//
// A split region is sk_tiles tiles of the call's flat tile order starting at
// sk_lo (row tiles outer, t_total token tiles inner).  When it is whole row
// tiles and the token tiles divide the pairs, it splits into g = t_total
// groups, one per token tile, of n_pairs / g pairs each; else into one group.
// Group g_id holds the region's tiles of token tile g_id (its local tile u is
// flat tile sk_lo + u·g + g_id); the k-blocks of those tiles, tile after tile
// (w in all), are cut into one contiguous range per pair of the group:
// [a, b) for the pair of index g_idx.  With at least as many tiles as pairs
// every range spans more than one tile, so a tile is shared by at most two
// pairs: the pairs of index q_lo and q_hi whose ranges meet its first and
// last k-block.
#pragma once

#include <cstdint>

#if defined(__CUDACC__)
#define BD_SPLIT_FN __host__ __device__ __forceinline__
#else
#define BD_SPLIT_FN inline
#endif

namespace bd {

struct SplitPair {
  int64_t g;        // groups
  int64_t g_pairs;  // pairs per group
  int64_t g_id;     // this pair's group
  int64_t g_idx;    // this pair's index in its group
  int64_t w;        // k-blocks of a group's tiles
  int64_t a, b;     // this pair's k-blocks [a, b)
  int64_t n_items;  // tiles its range meets
};

// The share of pair pair_id of n_pairs (sk_tiles == 0: no split region).
BD_SPLIT_FN SplitPair split_pair(int64_t pair_id, int64_t n_pairs, int64_t t_total, int64_t sk_lo,
                                 int64_t sk_tiles, int64_t n_kb) {
  SplitPair sp;
  sp.g = sk_tiles > 0 && t_total > 0 && n_pairs % t_total == 0 && sk_lo % t_total == 0 &&
                 sk_tiles % t_total == 0
             ? t_total
             : 1;
  sp.g_pairs = n_pairs / sp.g;
  sp.g_id = pair_id % sp.g;
  sp.g_idx = pair_id / sp.g;
  sp.w = sk_tiles / sp.g * n_kb;
  sp.a = sp.g_idx * sp.w / sp.g_pairs;
  sp.b = (sp.g_idx + 1) * sp.w / sp.g_pairs;
  sp.n_items = sp.b > sp.a ? (sp.b - 1) / n_kb - sp.a / n_kb + 1 : 0;
  return sp;
}

struct SplitItem {
  int64_t tile;   // flat tile index
  int64_t su;     // the group's local tile index
  int kb0, kb1;   // k-blocks [kb0, kb1) of the tile
  int j;          // this pair's partial slot: 0 for its first split item, else 1
  bool partial;   // shared with another pair (not all of the tile's k-blocks)
};

// The k-th of the pair's split items (0 <= k < n_items).
BD_SPLIT_FN SplitItem split_item(const SplitPair& sp, int64_t k, int64_t sk_lo, int64_t n_kb) {
  SplitItem it;
  it.su = sp.a / n_kb + k;
  const int64_t base = it.su * n_kb;
  it.tile = sk_lo + it.su * sp.g + sp.g_id;
  it.kb0 = static_cast<int>((sp.a > base ? sp.a : base) - base);
  it.kb1 = static_cast<int>((sp.b < base + n_kb ? sp.b : base + n_kb) - base);
  it.j = k == 0 ? 0 : 1;
  it.partial = !(it.kb0 == 0 && it.kb1 == n_kb);
  return it;
}

struct SplitShare {
  int64_t pair_lo, pair_hi;  // the two contributors (pair ids), k order
  int j_lo;                  // pair_lo's slot for this tile (pair_hi's is 0)
  int64_t counter;           // the tile's index among the region's tiles
};

// The contributors of the group's local tile su (a partial tile): the
// largest index q with q·w / g_pairs <= x is ((x + 1)·g_pairs − 1) / w.
// pair_hi's range starts in the tile (slot 0); pair_lo's part is its slot 1
// unless the tile also holds the start of pair_lo's range.
BD_SPLIT_FN SplitShare split_share(const SplitPair& sp, int64_t su, int64_t n_kb) {
  const int64_t x0 = su * n_kb, x1 = x0 + n_kb - 1;
  const int64_t q_lo = ((x0 + 1) * sp.g_pairs - 1) / sp.w;
  const int64_t q_hi0 = ((x1 + 1) * sp.g_pairs - 1) / sp.w;
  const int64_t q_hi = q_hi0 < sp.g_pairs - 1 ? q_hi0 : sp.g_pairs - 1;
  SplitShare sh;
  sh.pair_lo = q_lo * sp.g + sp.g_id;
  sh.pair_hi = q_hi * sp.g + sp.g_id;
  sh.j_lo = (q_lo * sp.w / sp.g_pairs) / n_kb == su ? 0 : 1;
  sh.counter = su * sp.g + sp.g_id;
  return sh;
}

}  // namespace bd
