// gemm_pair.cu — fused BitDelta linear for many rows (prefill) on pairs of
// CTAs sharing one tcgen05 MMA (cta_group::2).
//
// Page "BitDelta: serving 14 Zen models from one GPU cluster", section
// "Serving architecture": the fused kernel reads the base weight and the delta
// bits, builds the effective weight on chip — never the whole W_eff in HBM —
// and multiplies in the same pass (conceptual fused_bitdelta_linear:
// F.linear(x, W_base + α·unpack(bits))).
//
// Two tile widths share this file.
//
// Narrow pair tile: 256 output rows x 256 tokens x 64 K per stage.  CTA rank
// r of the pair owns output rows n0 + 128r .. +127: it loads those W_base
// rows, builds their W_eff in its own tensor memory (the MMA's A operand) and
// holds their fp32 accumulator (128 lanes x 256 token columns).  Each CTA
// loads half of the x tile (tokens tok0 + 128r .. +127, the MMA's B operand,
// split in N).  Rank 0 issues one 256x256x16 MMA that reads both CTAs'
// operands.  Six 32 KB stages.
//
// Wide pair tile: 256 output rows x 512 tokens.  The two accumulators (tokens
// tok0 .. +255 and tok0 + 256 .. +511) fill the 512 tensor-memory columns, so
// W_eff is written back over the W_base stage in shared memory, in the same
// swizzled layout the TMA wrote, and both N = 256 MMAs of a K step read it
// from there.  Each W_eff value then feeds 512 tokens: half the transform
// work per FLOP of the narrow tile.  Each CTA loads two 128-token x boxes
// per stage (tok0 + 128r and tok0 + 256 + 128r); eight 24 KB stages of
// 32 K (64-byte swizzle).
//
// Work of a pair: a list of items, each a tile and a range of its k-blocks:
// whole tiles of the call's flat tile order (pair p takes tiles p, p + n_pairs,
// ...), then, in the split schedule, the k-block range of a split region
// that falls to the pair (a tile there is shared by at most two pairs, whose
// fp32 partials the later of the two adds up).  Every role walks the same
// list.
//
// Warp roles per CTA (448 threads, one CTA per SM, persistent over items):
//   warps 0-7   transform: two warpgroups take the stages in turn; thread i
//               of a warpgroup owns W row i (TMEM lane i), forms the stage's
//               W_eff values of its row and stores them to the stage's A
//               slot (tcgen05.st, narrow) or back to shared memory (wide),
//               then its warp arrives on rank 0's xform barrier.
//   warps 8-11  epilogue: tcgen05.ld this CTA's accumulator, store bf16 y
//               (or a split tile's fp32 partial, or the pair sum).
//   warp 12     TMA producer for this CTA's W_base rows and its x rows.
//   warp 13     rank 0: MMA issuer; rank 1: waits for the pair's last MMA.
// Barriers: full[s] (TMA -> transform, local), xform[s] (both CTAs'
// transforms -> rank 0's MMA), empty[s] and accfull (rank 0's MMA commits,
// multicast to both CTAs), accempty (both CTAs' epilogues -> rank 0).  Every
// wait is bounded; TMEM is released on every exit path.
#include <cstdint>

#include "gemm_common.cuh"
#include "split_schedule.h"

namespace bd {
namespace {
using namespace gemm_detail;

#ifndef BD_PAIR_BK
#define BD_PAIR_BK 64
#endif
#ifndef BD_PAIR_XF_GROUPS
#define BD_PAIR_XF_GROUPS 2
#endif
// K per stage of the wide tile: 32 (eight 24 KB stages) measured 4-7%
// faster than 64 (four 48 KB stages) on M = 2048 projections.
#ifndef BD_PAIR_WIDE_BK
#define BD_PAIR_WIDE_BK 32
#endif

constexpr int kBM = 128;         // output rows per CTA
constexpr int kPairM = 2 * kBM;  // output rows per pair tile (UMMA M)
constexpr int kMmaN = 256;       // tokens per MMA (UMMA N)
constexpr int kXBox = kMmaN / 2; // x rows per TMA box (one CTA's half of an MMA's N)
constexpr int kPrefetch = 2;     // sign/α prefetch distance (own stages)
constexpr int kRing = kPrefetch + 2;  // private ring slots per thread
constexpr int kTmemCols = 512;
constexpr int kXfGroups = BD_PAIR_XF_GROUPS;  // transform warpgroups, stages in turn
constexpr int kXfWarps = 4 * kXfGroups;
constexpr int kEpiWarp0 = kXfWarps;
constexpr int kTmaWarp = kEpiWarp0 + 4;
constexpr int kMmaWarp = kTmaWarp + 1;
constexpr int kThreads = (kMmaWarp + 1) * 32;
static_assert(kEpiWarp0 % 4 == 0, "epilogue warps must start a warpgroup");
constexpr uint32_t kIdesc = idesc_bf16_f32(kPairM, kMmaN);
constexpr uint32_t kXformArrivals = 2 * 4;     // 4 transform warps per stage, both CTAs
constexpr uint32_t kAccEmptyArrivals = 2 * 4;  // 4 epilogue warps, both CTAs

template <bool kWide>
struct Cfg {
  static constexpr int kNMma = kWide ? 2 : 1;  // N = 256 MMAs per K step
  static constexpr int kBN = kNMma * kMmaN;    // tokens per pair tile
  // K per stage: one row of a swizzle atom, 128 bytes of bf16 (BK = 64,
  // 128-byte swizzle) or 64 bytes (BK = 32, 64-byte swizzle).
  static constexpr int kBK = kWide ? BD_PAIR_WIDE_BK : BD_PAIR_BK;
  static constexpr int kStages = kWide ? 256 / kBK : 384 / kBK;
  static constexpr int kABytes = kBM * kBK * 2;             // W_base (W_eff) per stage
  static constexpr int kXBoxBytes = kXBox * kBK * 2;        // one x box
  static constexpr int kBBytes = kNMma * kXBoxBytes;        // x per stage
  static constexpr int kChunks = kBK / 8;                   // 16-byte chunks per W row
  static constexpr int kSwzShift = kBK == 64 ? 0 : 1;       // row bits that select the XOR
  static constexpr int kSignBytes = kBK / 8;                // sign bytes per row per stage
  static constexpr int kACol0 = kBN;                        // narrow: first A slot column
  static constexpr int kAColsPerStage = kBK / 2;            // narrow: two bf16 per column
  // Shared memory layout (offsets from a 1024-byte aligned base; identical
  // in both CTAs, so one offset names the same buffer in either).
  static constexpr int kOffA = 0;
  static constexpr int kOffB = kOffA + kStages * kABytes;
  static constexpr int kOffSign = kOffB + kStages * kBBytes;                // [G][kRing][128] x 8 B
  static constexpr int kOffAlpha = kOffSign + kXfGroups * kRing * kBM * 8;  // [G][kRing][128] f32
  static constexpr int kOffBar = kOffAlpha + kXfGroups * kRing * kBM * 4;
  static constexpr int kNumBars = 3 * kStages + 3;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;  // tmem slot, abort flag, counts
  static constexpr int kOffSeg = kOffMisc + 64;            // grouped-mode tables
  static constexpr int kSegBytes = (3 * kGemmMaxSegs + 2) * 4;
  static constexpr int kSmemBytes = kOffSeg + kSegBytes + 1024;  // + alignment slack
  static_assert(kBK == 32 || kBK == 64, "BK is one 64- or 128-byte swizzle row");
  static_assert(kXfGroups <= kStages, "a warpgroup's stages must not alias in the ring");
  static_assert(kWide ? kNMma * kMmaN <= kTmemCols
                      : kACol0 + kStages * kAColsPerStage <= kTmemCols,
                "tensor memory budget");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
  static_assert(kABytes % 1024 == 0 && kXBoxBytes % 1024 == 0, "swizzle atoms stay aligned");
};

struct Misc {
  uint32_t tmem_base;
  int abort;
  int64_t t_total;  // token tiles over all segments
};

// kGrouped: the multi-tenant call (segment table, per-tile variant); the
// single-variant instance drops its per-stage variant and alignment cases.
template <bool kWide, bool kGrouped>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    bitdelta_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmap_w,
                              const __grid_constant__ CUtensorMap tmap_x, const GemmArgs p) {
  using C = Cfg<kWide>;
  constexpr int kStages = C::kStages;
  constexpr int kBK = C::kBK;
  constexpr int kBN = C::kBN;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* full_bar = bars;                 // own TMA -> own transform
  uint64_t* xform_bar = bars + kStages;      // both transforms -> rank 0's MMA (rank 0 only)
  uint64_t* empty_bar = bars + 2 * kStages;  // rank 0's MMA -> both TMA producers
  uint64_t* accfull_bar = bars + 3 * kStages;
  uint64_t* accempty_bar = accfull_bar + 1;  // both epilogues -> rank 0's MMA (rank 0 only)
  uint64_t* drain_bar = accempty_bar + 1;
  Misc* misc = reinterpret_cast<Misc*>(smem + C::kOffMisc);
  int32_t* s_seg_off = reinterpret_cast<int32_t*>(smem + C::kOffSeg);
  int32_t* s_seg_var = s_seg_off + (kGemmMaxSegs + 1);
  int32_t* s_prefix = s_seg_var + kGemmMaxSegs;
  volatile int* abort = &misc->abort;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  constexpr bool grouped = kGrouped;
  const uint32_t rank = cluster_rank();

  // ---------------------------------------------------------------- set-up
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&xform_bar[s], kXformArrivals);
      mbar_init(&empty_bar[s], 1);
    }
    mbar_init(accfull_bar, 1);
    mbar_init(accempty_bar, kAccEmptyArrivals);
    mbar_init(drain_bar, 1);
    misc->abort = 0;
    fence_mbar_init();
  }
  if (grouped) {
    load_segments<kBN>(p, s_seg_off, s_seg_var, s_prefix, &misc->t_total);
  } else if (threadIdx.x == 0) {
    misc->t_total = (p.M + kBN - 1) / kBN;
  }
  if (warp == kMmaWarp) {
    // one warp in each CTA of the pair allocates, collectively
    tmem_alloc_pair(&misc->tmem_base, kTmemCols);
    tmem_relinquish_pair();
  }
  if (warp == kTmaWarp && lane == 0) {
    prefetch_tmap(&tmap_w);
    prefetch_tmap(&tmap_x);
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // the peer's barriers are initialised before anyone arrives on them
  tc_fence_after();

  const uint32_t tmem_base = misc->tmem_base;
  const int64_t t_total = misc->t_total;
  const int64_t n_tiles_n = (p.d_out + kPairM - 1) / kPairM;
  const int64_t all_tiles = n_tiles_n * t_total;
  // a range of the flat tile order (single-variant mode), else all of it
  const bool split = !grouped && p.sk_tiles > 0 && p.sk_lo >= 0 && p.sk_lo < all_tiles;
  const bool ranged = !grouped && (p.tile_hi > 0 || split);
  const int64_t t_lo = ranged ? p.tile_lo : 0;
  const int64_t t_hi = ranged && p.tile_hi < all_tiles ? p.tile_hi : all_tiles;
  const int64_t num_tiles = t_hi > t_lo ? t_hi - t_lo : 0;
  const int64_t pair_id = blockIdx.x >> 1;
  const int64_t n_pairs = gridDim.x >> 1;
  const int64_t my_tiles = pair_id < num_tiles ? (num_tiles - 1 - pair_id) / n_pairs + 1 : 0;
  const int n_kb = static_cast<int>(p.d_in / kBK);
  const int32_t* seg_off_tbl = grouped ? s_seg_off : nullptr;
  auto my_tile = [&](int64_t i) {
    return tile_at<kPairM, kBN>(p, t_lo + pair_id + i * n_pairs, t_total, seg_off_tbl, s_seg_var,
                                s_prefix);
  };
  // Split region (split_schedule.h): this pair's k-block range of its
  // group's tiles, after its whole tiles.  A pair's work is a list of items
  // (a tile and a k-block range of it): its whole tiles, then the split
  // tiles its range meets.
  int64_t sk_tiles =
      split ? (p.sk_tiles < all_tiles - p.sk_lo ? p.sk_tiles : all_tiles - p.sk_lo) : 0;
  if (sk_tiles > 0 && sk_tiles < n_pairs) {
    // fewer tiles than pairs would give a tile more than two contributors
    // (the sum below takes two): the host never launches this
    if (blockIdx.x == 0 && threadIdx.x == 0) record_error(p.ctx, kErrBounds);
    sk_tiles = 0;
  }
  const SplitPair sp = split_pair(pair_id, n_pairs, t_total, p.sk_lo, sk_tiles, n_kb);
  const int64_t n_items = my_tiles + sp.n_items;
  struct Item {
    Tile t;
    int kb0, kb1;  // k-blocks [kb0, kb1) of the tile
    int64_t su;    // the group's local tile index, -1 for a whole tile of the range
    int j;         // partial slot of this pair: 0 first split item, 1 later
  };
  auto item_at = [&](int64_t it) {
    Item im;
    if (it < my_tiles) {
      im.t = my_tile(it);
      im.kb0 = 0;
      im.kb1 = n_kb;
      im.su = -1;
      im.j = 0;
      return im;
    }
    const SplitItem si = split_item(sp, it - my_tiles, p.sk_lo, n_kb);
    im.t = tile_at<kPairM, kBN>(p, si.tile, t_total, nullptr, nullptr, nullptr);
    im.kb0 = si.kb0;
    im.kb1 = si.kb1;
    im.su = si.su;
    im.j = si.j;
    return im;
  };
  const int64_t row0 = static_cast<int64_t>(rank) * kBM;     // this CTA's rows in the tile
  const int64_t tok_half = static_cast<int64_t>(rank) * kXBox;  // this CTA's x rows per MMA

  if (warp < kXfWarps) {
    // ============================================================ transform
    const int wg = warp >> 2;
    const int r = threadIdx.x & 127;  // the W row (and TMEM lane) of this thread
    const int quarter = warp & 3;     // TMEM lane quarter of this warp
    uint8_t* sign_ring = smem + C::kOffSign + wg * (kRing * kBM * 8);
    float* alpha_ring = reinterpret_cast<float*>(smem + C::kOffAlpha) + wg * (kRing * kBM);
    const int64_t row_bytes = p.d_in / 8;

    const uint32_t a_lane = tmem_base + (static_cast<uint32_t>(32 * quarter) << 16);
    const uint32_t xform_rank0 = map_to_rank(smem_addr(xform_bar), 0);

    // Cursors over this warpgroup's stages: flat positions wg, wg + G, ...
    // of the pair's k-block stream (the items in turn, k-blocks [kb0, kb1)
    // of each).  kb < kb0g marks the warpgroup's first stage of an item; the
    // per-stage step is kb += G and one compare, the item change a slow path.
    // The prefetch cursor also holds where this row's sign bytes come from
    // (mode 1), or a fill of +1 signs for a variant table entry that is not
    // aligned (mode 2, recorded as a bounds error), or nothing for base rows
    // and past the last item (mode 0), so the per-stage copy is one cp.async.
    // Each thread later reads only what it copied itself, from private ring
    // slot (own stage index) % kRing.
    struct Cur {
      int it, kb, kb1, kb0g, var;
    };
    const int n_it = static_cast<int>(n_items);
    int pf_mode = 0;
    const uint8_t* pf_src = nullptr;
    const float* pf_alpha = nullptr;
    auto pf_load_item = [&](const Tile& t) {
      pf_mode = 0;
      if (t.variant <= 0) return;
      const uint8_t* pk = grouped ? p.packed_table[t.variant - 1] : p.packed;
      const float* al = grouped ? p.alpha_table[t.variant - 1] : p.alpha;
      // a row past d_out reads row d_out - 1: its products land in
      // accumulator rows that the epilogue never stores
      int64_t row = t.n0 + row0 + r;
      row = row < p.d_out ? row : p.d_out - 1;
      pf_alpha = p.per_row ? al + row : al;
      if ((reinterpret_cast<uintptr_t>(pk) & (C::kSignBytes - 1)) == 0) {
        pf_src = pk + row * row_bytes;
        pf_mode = 1;
      } else {
        // a variant table entry off its boundary (the single-variant call's
        // pointer is checked on the host): recorded, and read as +1 signs
        if (blockIdx.x == 0) record_error(p.ctx, kErrBounds);
        pf_mode = kGrouped ? 2 : 0;
      }
    };
    auto cur_set = [&](Cur& c, const Item& im, int over, bool is_pf) {
      c.kb = im.kb0 + over;
      c.kb1 = im.kb1;
      c.kb0g = im.kb0 + kXfGroups;
      c.var = im.t.variant;
      if (is_pf) pf_load_item(im.t);
    };
    auto cur_carry = [&](Cur& c, bool is_pf) {
      do {
        const int over = c.kb - c.kb1;
        if (++c.it >= n_it) {
          c.kb1 = 0x7FFFFFFF;
          if (is_pf) pf_mode = 0;
          return;
        }
        cur_set(c, item_at(c.it), over, is_pf);
      } while (c.kb >= c.kb1);
    };
    auto cur_start = [&](Cur& c, bool is_pf) {
      c.it = 0;
      c.kb = 0;
      c.kb1 = 0x7FFFFFFF;
      c.kb0g = 0;
      c.var = 0;
      if (n_it <= 0) return;
      cur_set(c, item_at(0), wg, is_pf);
      if (c.kb >= c.kb1) cur_carry(c, is_pf);
    };

    Cur pf;
    cur_start(pf, true);
    int pf_slot = 0;
    auto prefetch_next = [&]() {
      uint8_t* dst = sign_ring + (pf_slot * kBM + r) * 8;
      if (pf_mode == 1) {
        if constexpr (C::kSignBytes == 8)
          cp_async_8(dst, pf_src + pf.kb * C::kSignBytes);
        else
          cp_async_4(dst, pf_src + pf.kb * C::kSignBytes);
      } else if (kGrouped && pf_mode == 2) {
        *reinterpret_cast<uint2*>(dst) = make_uint2(0xFFFFFFFFu, 0xFFFFFFFFu);
      }
      if (pf_mode != 0 && pf.kb < pf.kb0g) cp_async_4(alpha_ring + pf_slot * kBM + r, pf_alpha);
      cp_async_commit();
      pf_slot = pf_slot + 1 == kRing ? 0 : pf_slot + 1;
      pf.kb += kXfGroups;
      if (pf.kb >= pf.kb1) cur_carry(pf, true);
    };

    for (int d = 0; d < kPrefetch; ++d) prefetch_next();
    uint32_t alpha_bits = 0u;  // α of the current item's rows (fp32 bits)
    // s / ph: ring stage and phase parity of the flat position
    Cur cu;
    cur_start(cu, false);
    int slot = 0;
    int s = wg;
    uint32_t ph = 0u;
    while (cu.it < n_it) {
      prefetch_next();
      cp_async_wait<kPrefetch>();
      int ok = 0;
      if (lane == 0) ok = mbar_wait(&full_bar[s], ph, p.ctx, abort) ? 1 : 0;
      ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
      __syncwarp();
      if (!ok) break;
      const bool has_delta = !kGrouped || cu.var > 0;
      if (cu.kb < cu.kb0g && has_delta) alpha_bits = __float_as_uint(alpha_ring[slot * kBM + r]);
      uint2 sg = make_uint2(0u, 0u);
      if (has_delta) {
        if constexpr (C::kSignBytes == 8)
          sg = *reinterpret_cast<const uint2*>(sign_ring + (slot * kBM + r) * 8);
        else
          sg.x = *reinterpret_cast<const uint32_t*>(sign_ring + (slot * kBM + r) * 8);
      }
      uint8_t* w_row = smem + C::kOffA + s * C::kABytes + r * (kBK * 2);
      const int swz = (r >> C::kSwzShift) & (C::kChunks - 1);
      if constexpr (kWide) {
        // W_eff over W_base in place (same swizzled chunk positions); base
        // rows are already the operand.  The fence makes these generic-proxy
        // writes visible to the tensor core's reads of the stage.
        if (has_delta) {
          uint4 wv[C::kChunks];
#pragma unroll
          for (int c = 0; c < C::kChunks; ++c)
            wv[c] = *reinterpret_cast<const uint4*>(w_row + ((c ^ swz) << 4));
          uint32_t packed[kBK / 2];
          weff_chunks<C::kChunks>(wv, sg, alpha_bits, packed);
#pragma unroll
          for (int c = 0; c < C::kChunks; ++c)
            *reinterpret_cast<uint4*>(w_row + ((c ^ swz) << 4)) =
                make_uint4(packed[4 * c], packed[4 * c + 1], packed[4 * c + 2], packed[4 * c + 3]);
          fence_proxy_async_smem();
        }
        __syncwarp();
      } else {
        uint4 wv[C::kChunks];
#pragma unroll
        for (int c = 0; c < C::kChunks; ++c) {
          // logical 16-byte chunk c sits at physical chunk c ^ swz: the TMA's
          // 128-byte (64-byte) swizzle XORs the chunk index with address bits
          // 7-9 (7-8), i.e. with row bits 0-2 (1-2)
          wv[c] = *reinterpret_cast<const uint4*>(w_row + ((c ^ swz) << 4));
        }
        uint32_t packed[kBK / 2];
        if (has_delta) {
          weff_chunks<C::kChunks>(wv, sg, alpha_bits, packed);
        } else {
#pragma unroll
          for (int c = 0; c < C::kChunks; ++c) {
            packed[4 * c + 0] = wv[c].x;
            packed[4 * c + 1] = wv[c].y;
            packed[4 * c + 2] = wv[c].z;
            packed[4 * c + 3] = wv[c].w;
          }
        }
        tmem_st_32x32b(a_lane + static_cast<uint32_t>(C::kACol0 + C::kAColsPerStage * s), packed);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
      }
      // the A operand is written and this CTA's x of the stage has landed
      if (lane == 0) mbar_arrive_cluster(xform_rank0 + static_cast<uint32_t>(8 * s));
      s += kXfGroups;
      if (s >= kStages) {
        s -= kStages;
        ph ^= 1u;
      }
      slot = slot + 1 == kRing ? 0 : slot + 1;
      cu.kb += kXfGroups;
      if (cu.kb >= cu.kb1) cur_carry(cu, false);
    }
    cp_async_wait<0>();
  } else if (warp < kTmaWarp) {
    // ============================================================ epilogue
    const int quarter = warp - kEpiWarp0;  // TMEM lanes 32*quarter ..
    const uint32_t accempty_rank0 = map_to_rank(smem_addr(accempty_bar), 0);
    const uint32_t taddr = tmem_base + (static_cast<uint32_t>(32 * quarter) << 16);
    const int rr = 32 * quarter + lane;  // this thread's row of the CTA's 128
    for (int64_t i = 0; i < n_items; ++i) {
      const uint32_t ph = static_cast<uint32_t>(i & 1);
      int ok = 0;
      if (lane == 0) ok = mbar_wait_cluster(accfull_bar, ph, p.ctx, abort) ? 1 : 0;
      ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
      __syncwarp();
      if (!ok) break;
      tc_fence_after();
      const Item im = item_at(i);
      const int64_t n = im.t.n0 + row0 + rr;
      if (im.su < 0 || (im.kb0 == 0 && im.kb1 == n_kb)) {
        store_acc_rows<kBN>(taddr, p.y, p.d_out, n, im.t.tok0, im.t.tok_end);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(accempty_rank0);
        continue;
      }
      // A part of a split tile, shared with one other pair of the group
      // (split_share: the two contributors in k order and their slots).  One
      // counter per tile, CTA half and epilogue warp counts the parts stored.
      const int64_t span = im.t.tok_end - im.t.tok0;
      const int cols = span <= 0 ? 0 : (span < kBN ? static_cast<int>(span) : kBN);
      constexpr int64_t kSlot = static_cast<int64_t>(kBN) * kBM;
      const SplitShare sh = split_share(sp, im.su, n_kb);
      const int64_t pair_lo = sh.pair_lo;
      const float* slot_lo = p.sk_part + ((sh.pair_lo * 2 + sh.j_lo) * 2 + rank) * kSlot;
      const float* slot_hi = p.sk_part + ((sh.pair_hi * 2 + 0) * 2 + rank) * kSlot;
      unsigned int* cnt = p.sk_count + (sh.counter * 2 + rank) * 4 + quarter;
      int other_done = 0;
      if (lane == 0) other_done = ld_acquire_u32(cnt) != 0u ? 1 : 0;
      other_done = __shfl_sync(0xFFFFFFFFu, other_done, 0);
      if (other_done) {
        // the other part is stored: add it to this one straight from tensor
        // memory (nothing else reads this part, so it is neither stored nor
        // counted)
        __threadfence();
        sum_tmem_partial_store(taddr, pair_id == pair_lo ? slot_hi : slot_lo, rr, p.y, p.d_out, n,
                               im.t.tok0, cols);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(accempty_rank0);
        continue;
      }
      store_acc_partial(taddr, p.sk_part + ((pair_id * 2 + im.j) * 2 + rank) * kSlot, rr, cols);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(accempty_rank0);
      __threadfence();
      __syncwarp();
      int last = 0;
      if (lane == 0) last = atomicAdd(cnt, 1u) == 1u ? 1 : 0;
      last = __shfl_sync(0xFFFFFFFFu, last, 0);
      if (!last) continue;
      // both parts were stored at about the same time: sum the two slots
      __threadfence();
      sum_pair_partials_store(slot_lo, slot_hi, rr, p.y, p.d_out, n, im.t.tok0, cols);
    }
  } else if (warp == kTmaWarp) {
    // ============================================================ TMA producer
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_first();
      const uint64_t pol_x = policy_evict_last();
      int64_t q = 0;
      bool ok = true;
      for (int64_t i = 0; i < n_items && ok; ++i) {
        const Item im = item_at(i);
        const Tile& tl = im.t;
        for (int kb = im.kb0; kb < im.kb1; ++kb, ++q) {
          const int s = static_cast<int>(q % kStages);
          const uint32_t ph = static_cast<uint32_t>((q / kStages) & 1);
          if (!mbar_wait_cluster(&empty_bar[s], ph ^ 1u, p.ctx, abort)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full_bar[s], C::kABytes + C::kBBytes);
          tma_load_2d(smem + C::kOffA + s * C::kABytes, &tmap_w, &full_bar[s], kb * kBK,
                      static_cast<int32_t>(tl.n0 + row0), pol_w);
#pragma unroll
          for (int j = 0; j < C::kNMma; ++j)
            tma_load_2d(smem + C::kOffB + s * C::kBBytes + j * C::kXBoxBytes, &tmap_x,
                        &full_bar[s], kb * kBK,
                        static_cast<int32_t>(tl.tok0 + j * kMmaN + tok_half), pol_x);
        }
      }
      // Drain: wait (bounded, ignoring abort) until every issued copy landed.
      const int64_t first = q > kStages ? q - kStages : 0;
      for (int64_t qq = first; qq < q; ++qq)
        mbar_wait(&full_bar[qq % kStages], static_cast<uint32_t>((qq / kStages) & 1), p.ctx,
                  nullptr);
    }
  } else if (warp == kMmaWarp) {
    // ============================================================ MMA issuer
    if (lane == 0 && rank == 0) {
      const uint32_t a_base = smem_addr(smem + C::kOffA);
      const uint32_t b_base = smem_addr(smem + C::kOffB);
      int64_t q = 0;
      bool ok = true;
      bool issued = false;
      for (int64_t i = 0; i < n_items && ok; ++i) {
        const Item im = item_at(i);
        // N = 256 MMAs with at least one output token (the wide tile's second
        // half is skipped when the tile ends in its first half)
        int n_mma = 1;
        if constexpr (kWide) n_mma = im.t.tok0 + kMmaN < im.t.tok_end ? 2 : 1;
        // both CTAs' accumulators must have been drained by their epilogues
        if (!mbar_wait_cluster(accempty_bar, static_cast<uint32_t>((i & 1) ^ 1), p.ctx, abort))
          break;
        tc_fence_after();
        for (int kb = im.kb0; kb < im.kb1; ++kb, ++q) {
          const int s = static_cast<int>(q % kStages);
          const uint32_t ph = static_cast<uint32_t>((q / kStages) & 1);
          if (!mbar_wait_cluster(&xform_bar[s], ph, p.ctx, abort)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t b_desc = kBK == 64 ? sdesc_k_sw128(b_base + s * C::kBBytes)
                                            : sdesc_k_sw64(b_base + s * C::kBBytes);
          if constexpr (kWide) {
            const uint64_t a_desc = kBK == 64 ? sdesc_k_sw128(a_base + s * C::kABytes)
                                              : sdesc_k_sw64(a_base + s * C::kABytes);
            constexpr uint64_t kBoxStep = C::kXBoxBytes >> 4;  // descriptor address units
#pragma unroll
            for (int k = 0; k < kBK / 16; ++k) {
              // K step 16: +32 bytes inside both operands' swizzle atoms
              const uint32_t acc = (kb > im.kb0 || k > 0) ? 1u : 0u;
              umma_bf16_pair(tmem_base, a_desc + 2 * k, b_desc + 2 * k, kIdesc, acc);
              if (n_mma > 1)
                umma_bf16_pair(tmem_base + kMmaN, a_desc + 2 * k, b_desc + kBoxStep + 2 * k,
                               kIdesc, acc);
            }
          } else {
            const uint32_t a_tmem =
                tmem_base + static_cast<uint32_t>(C::kACol0 + C::kAColsPerStage * s);
#pragma unroll
            for (int k = 0; k < kBK / 16; ++k) {
              // K step 16: 8 TMEM columns of A; +32 bytes inside B's swizzle atom
              umma_bf16_tmem_a_pair(tmem_base, a_tmem + 8 * k, b_desc + 2 * k, kIdesc,
                                    (kb > im.kb0 || k > 0) ? 1u : 0u);
            }
          }
          issued = true;
          umma_commit_pair(&empty_bar[s]);
        }
        if (!ok) break;
        umma_commit_pair(accfull_bar);
      }
      if (issued) umma_commit_pair(drain_bar);
      if (issued) mbar_wait_cluster(drain_bar, 0, p.ctx, nullptr);
    } else if (lane == 0 && n_items > 0) {
      // rank 1: its shared and tensor memory are operands of rank 0's MMAs;
      // stay until the last of them has completed
      mbar_wait_cluster(drain_bar, 0, p.ctx, nullptr);
    }
  }

  // ---------------------------------------------------------------- teardown
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // no CTA leaves while the other may still touch its memory
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc_pair(tmem_base, kTmemCols);
}

// Per device: kernel attributes set and the number of pairs that fit at once
// (occupancy query), once per instantiation.
template <bool kWide>
cudaError_t pair_capacity(int* pairs) {
  static bool done[64] = {};
  static int max_pairs[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(host_cache_mutex());
  if (!done[dev]) {
    e = cudaFuncSetAttribute(bitdelta_gemm_pair_kernel<kWide, false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<kWide>::kSmemBytes);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(bitdelta_gemm_pair_kernel<kWide, true>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<kWide>::kSmemBytes);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = Cfg<kWide>::kSmemBytes;
    cfg.gridDim = dim3(2);
    int n = 0;
    e = cudaOccupancyMaxActiveClusters(&n, bitdelta_gemm_pair_kernel<kWide, false>, &cfg);
    if (e != cudaSuccess) return e;
    max_pairs[dev] = n;
    done[dev] = true;
  }
  *pairs = max_pairs[dev];
  return cudaSuccess;
}

template <bool kWide>
cudaError_t launch_pair_instance(const GemmArgs& p, const CUtensorMap& tmap_w,
                                 const CUtensorMap& tmap_x, int64_t pair_tiles_bound,
                                 cudaStream_t stream) {
  int max_pairs = 0;
  cudaError_t e = pair_capacity<kWide>(&max_pairs);
  if (e != cudaSuccess) return e;
  if (max_pairs < 1) return cudaErrorInvalidConfiguration;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = Cfg<kWide>::kSmemBytes;
  cfg.stream = stream;
  const int64_t pairs = pair_tiles_bound < max_pairs ? pair_tiles_bound : max_pairs;
  cfg.gridDim = dim3(static_cast<unsigned>(2 * (pairs > 0 ? pairs : 1)));
  if (p.seg_off != nullptr)
    return cudaLaunchKernelEx(&cfg, bitdelta_gemm_pair_kernel<kWide, true>, tmap_w, tmap_x, p);
  return cudaLaunchKernelEx(&cfg, bitdelta_gemm_pair_kernel<kWide, false>, tmap_w, tmap_x, p);
}

}  // namespace

int gemm_block_rows() { return kBM; }
int gemm_pair_x_rows() { return kXBox; }
int gemm_pair_block_k() { return Cfg<false>::kBK; }
int gemm_pair_wide_block_k() { return Cfg<true>::kBK; }
int gemm_pair_tokens(bool wide) { return wide ? Cfg<true>::kBN : Cfg<false>::kBN; }
int gemm_pair_capacity(bool wide) {
  int n = 0;
  const cudaError_t e = wide ? pair_capacity<true>(&n) : pair_capacity<false>(&n);
  return e == cudaSuccess ? n : -static_cast<int>(e);
}

size_t gemm_split_count_bytes(int64_t sk_tiles) {
  const size_t b = static_cast<size_t>(sk_tiles > 0 ? sk_tiles : 0) * 2 * 4 * sizeof(unsigned int);
  return (b + 255) & ~static_cast<size_t>(255);
}
size_t gemm_split_part_bytes(int64_t pairs) {
  return static_cast<size_t>(pairs > 0 ? pairs : 0) * 2 * 2 * Cfg<true>::kBN * kBM * sizeof(float);
}

cudaError_t launch_gemm_pair(const GemmArgs& p, const CUtensorMap& tmap_w,
                             const CUtensorMap& tmap_x, int64_t pair_tiles_bound, bool wide,
                             cudaStream_t stream) {
  return wide ? launch_pair_instance<true>(p, tmap_w, tmap_x, pair_tiles_bound, stream)
              : launch_pair_instance<false>(p, tmap_w, tmap_x, pair_tiles_bound, stream);
}

// ------------------------------------------------------------------ test hook

namespace {
__global__ void wait_timeout_probe_kernel(DevCtx ctx) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
    // Nothing ever arrives on `bar`: the bounded wait must give up.
    mbar_wait(&bar, 0, ctx, nullptr);
  }
  __syncthreads();
}
}  // namespace

cudaError_t launch_wait_timeout_probe(DevCtx ctx, cudaStream_t stream) {
  wait_timeout_probe_kernel<<<1, 32, 0, stream>>>(ctx);
  return cudaGetLastError();
}

}  // namespace bd
