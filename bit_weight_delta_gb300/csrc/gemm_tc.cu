// gemm_tc.cu — fused BitDelta linear for many rows (prefill) on the tcgen05
// tensor cores.
//
// Page "BitDelta: serving 14 Zen models from one GPU cluster", section
// "Serving architecture": the fused kernel reads the base weight and the delta
// bits, builds the effective weight in registers or shared memory — never the
// whole W_eff in HBM — and multiplies in the same pass (conceptual
// fused_bitdelta_linear: F.linear(x, W_base + α·unpack(bits))).
//
// Tile: 128 output rows (n, UMMA M, operand A = W_eff) x 256 tokens (UMMA N,
// operand B = x) x 64 K per stage; D = W_eff·xᵀ = yᵀ accumulates in TMEM
// (fp32, 128 lanes x 256 columns, double-buffered).
//
// Shared transform.  A thread-block cluster of C CTAs (C = 1, 2 or 4) works
// on the same 128 output rows for C consecutive token tiles.  Each CTA loads
// only its 128/C rows of W_base and rewrites them in place as
// W_eff = bf16_rne(fp32(W_base) ± α); each transform warp then copies its
// finished rows into the A buffers of the other C-1 CTAs with one bulk copy
// per peer (distributed shared memory), which completes as transaction bytes
// on the peer's "transformed" barrier.  Every CTA's MMA commit is multicast to
// every CTA's "empty" barrier, so a stage is reloaded (and overwritten by a
// peer's copy) only when all C CTAs are done with it.  The transform work and
// the W_base traffic per CTA both drop by C.
//
// Warp roles (448 threads, one CTA per SM, persistent over cluster tiles):
//   warps 0-7   transform: the CTA's 128/C W rows split over 8 warps; lanes
//               prefetch their rows' sign bytes (8 per row per stage) and α
//               with cp.async into a ring several stages ahead.
//   warps 8-11  epilogue: tcgen05.ld the finished accumulator (lane = n,
//               column = token), round to bf16, store y.
//   warp 12     TMA producer: W_base rows [128/C x 64] and x tile [256 x 64].
//   warp 13     MMA issuer: 4 x tcgen05.mma (128x256x16) per stage, commit.
// Every wait is bounded (the kernel records a timeout and unwinds); TMEM is
// released on every exit path; the cluster synchronises before any CTA exits.
#include <cstdint>

#include "common.cuh"
#include "kernels.h"

namespace bd {
namespace {

#ifndef BD_GEMM_STAGES
#define BD_GEMM_STAGES 4
#endif
constexpr int kBM = 128;  // d_out rows per tile
constexpr int kBN = 256;  // tokens per tile
constexpr int kBK = 64;   // K per stage: one 128-byte swizzle atom of bf16
constexpr int kStages = BD_GEMM_STAGES;
constexpr int kABytes = kBM * kBK * 2;  // 16 KB
constexpr int kBBytes = kBN * kBK * 2;  // 32 KB
constexpr int kPrefetch = 4;            // sign/α prefetch distance (stages)
constexpr int kRing = kPrefetch + 2;    // ring slots
constexpr int kAccCols = kBN;           // fp32 accumulator columns per buffer
constexpr int kTmemCols = 2 * kAccCols;
constexpr int kXfWarps = 8;                     // transform warps (independent)
constexpr int kEpiWarp0 = kXfWarps;             // 4 epilogue warps: TMEM lane quarters 0..3
constexpr int kTmaWarp = kEpiWarp0 + 4;
constexpr int kMmaWarp = kTmaWarp + 1;
constexpr int kThreads = (kMmaWarp + 1) * 32;
static_assert(kEpiWarp0 % 4 == 0, "epilogue warps must start a warpgroup");
constexpr uint32_t kIdesc = idesc_bf16_f32(kBM, kBN);

// Shared memory layout (offsets from a 1024-byte aligned base).
constexpr int kOffA = 0;
constexpr int kOffB = kOffA + kStages * kABytes;
constexpr int kOffSign = kOffB + kStages * kBBytes;     // [kRing][128][8] bytes
constexpr int kOffAlpha = kOffSign + kRing * kBM * 8;   // [kRing][128] floats
constexpr int kOffBar = kOffAlpha + kRing * kBM * 4;
constexpr int kNumBars = 3 * kStages + 2 + 2 + 1;
constexpr int kOffMisc = kOffBar + kNumBars * 8;        // tmem slot, abort flag, counts
constexpr int kOffSeg = kOffMisc + 64;                  // grouped-mode tables
constexpr int kSegBytes = (3 * kGemmMaxSegs + 2) * 4;
constexpr int kSmemBytes = kOffSeg + kSegBytes + 1024;  // + alignment slack

struct Misc {
  uint32_t tmem_base;
  int abort;
  int64_t groups;  // token-tile groups over all segments (a group = C tiles)
};

struct Tile {
  int64_t n0;
  int64_t tok0;
  int64_t tok_end;  // rows [tok0, min(tok0 + 256, tok_end)) are this CTA's outputs
  int32_t variant;  // 0 = base (no delta)
};

// ------------------------------------------------------------------ cluster PTX

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t map_to_rank(uint32_t local_smem_addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local_smem_addr), "r"(rank));
  return r;
}
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity,
                                                      uint32_t suspend_ns) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity), "r"(suspend_ns)
      : "memory");
  return done != 0;
}
// Bounded wait on a barrier that other CTAs of the cluster arrive on.
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity,
                                                  const DevCtx& ctx, volatile int* abort) {
  if (mbar_try_wait_cluster(bar, parity, 0)) return true;
  const long long t0 = clock64();
  const long long limit = static_cast<long long>(ctx.wait_limit_ns) * 2;
  while (true) {
    if (mbar_try_wait_cluster(bar, parity, 20000u)) return true;
    if (abort != nullptr && *abort) return false;
    if (clock64() - t0 > limit) {
      record_error(ctx, kErrTimeout);
      if (abort != nullptr) *abort = 1;
      return false;
    }
  }
}
// Bulk copy of `bytes` from this CTA's shared memory to a peer's (both
// addresses 16-byte aligned); completes as transaction bytes on the peer's
// mbarrier at cluster address `peer_bar`.
__device__ __forceinline__ void bulk_copy_to_peer(uint32_t peer_dst, uint32_t local_src,
                                                  uint32_t bytes, uint32_t peer_bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, "
      "[%3];" ::"r"(peer_dst),
      "r"(local_src), "r"(bytes), "r"(peer_bar)
      : "memory");
}
// Arrive on `bar` (same offset) in every CTA of `mask` when this thread's
// previously issued MMAs complete.
__device__ __forceinline__ void umma_commit_multicast(uint64_t* bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 "
      "[%0], %1;" ::"r"(smem_addr(bar)),
      "h"(mask)
      : "memory");
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}

// ------------------------------------------------------------------ schedule

// Tile of this CTA (cluster rank `rank`) for cluster tile `ct`.  Plain mode:
// token tiles of [0, M) in groups of C.  Grouped mode: the same per long
// segment; `prefix` is the prefix sum of groups per segment.  A rank whose
// token tile lies past its segment gets an empty token range (it still loads
// and transforms its W rows for the other CTAs).
template <int C>
__device__ __forceinline__ Tile tile_at(const GemmArgs& p, int64_t ct, int64_t groups,
                                        uint32_t rank, const int32_t* seg_off,
                                        const int32_t* seg_var, const int32_t* prefix) {
  Tile tl;
  const int64_t nt = ct / groups;
  const int64_t j = ct - nt * groups;
  tl.n0 = nt * kBM;
  if (seg_off == nullptr) {
    tl.tok0 = (j * C + rank) * kBN;
    tl.tok_end = p.M;
    tl.variant = 1;
  } else {
    // largest s with prefix[s] <= j (prefix is non-decreasing, prefix[0] = 0)
    int lo = 0, hi = p.n_seg;  // invariant: prefix[lo] <= j < prefix[hi]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (prefix[mid] <= j)
        lo = mid;
      else
        hi = mid;
    }
    tl.tok0 = seg_off[lo] + ((j - prefix[lo]) * C + rank) * kBN;
    tl.tok_end = seg_off[lo + 1];
    tl.variant = seg_var[lo];
  }
  return tl;
}

// ±α by the sign bit at `col` of `byte` (bit 1 -> +α); neg_alpha = α | sign.
__device__ __forceinline__ float signed_alpha(uint32_t byte, int col, uint32_t neg_alpha) {
  return __uint_as_float(neg_alpha ^ ((byte << (31 - col)) & 0x80000000u));
}

template <int C>
__global__ void __launch_bounds__(kThreads, 1)
    bitdelta_gemm_kernel(const __grid_constant__ CUtensorMap tmap_w,
                         const __grid_constant__ CUtensorMap tmap_x, const GemmArgs p) {
  constexpr int kRowsPerCta = kBM / C;           // W rows this CTA loads and transforms
  constexpr int kWBytes = kRowsPerCta * 128;     // its W_base bytes per stage
  constexpr int kRowsPerWarp = kRowsPerCta / kXfWarps;  // 16, 8 or 4
  constexpr int kChunksPerLane = kRowsPerWarp / 4;      // 4, 2 or 1
  static_assert(kRowsPerWarp % 4 == 0 && kRowsPerWarp >= 4, "transform lane mapping");

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint64_t* full_bar = bars;                 // own TMA -> own transform and MMA
  uint64_t* xform_bar = bars + kStages;      // all transforms -> MMA
  uint64_t* empty_bar = bars + 2 * kStages;  // all MMAs -> TMA
  uint64_t* accfull_bar = bars + 3 * kStages;
  uint64_t* accempty_bar = accfull_bar + 2;
  uint64_t* drain_bar = accempty_bar + 2;
  Misc* misc = reinterpret_cast<Misc*>(smem + kOffMisc);
  int32_t* s_seg_off = reinterpret_cast<int32_t*>(smem + kOffSeg);
  int32_t* s_seg_var = s_seg_off + (kGemmMaxSegs + 1);
  int32_t* s_prefix = s_seg_var + kGemmMaxSegs;
  volatile int* abort = &misc->abort;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const bool grouped = p.seg_off != nullptr;
  const uint32_t rank = C > 1 ? cluster_rank() : 0u;

  // ---------------------------------------------------------------- set-up
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&xform_bar[s], kXfWarps);
      mbar_init(&empty_bar[s], C);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&accfull_bar[a], 1);
      mbar_init(&accempty_bar[a], 128);
    }
    mbar_init(drain_bar, 1);
    misc->abort = 0;
    fence_mbar_init();
  }
  if (grouped) {
    // Copy the segment table, then count token-tile groups per valid long
    // segment.  One malformed entry rejects the whole table (no tiles at all).
    for (int s = threadIdx.x; s <= p.n_seg; s += blockDim.x) s_seg_off[s] = __ldg(p.seg_off + s);
    for (int s = threadIdx.x; s < p.n_seg; s += blockDim.x) s_seg_var[s] = __ldg(p.seg_var + s);
    __syncthreads();
    int bad_local = 0;
    for (int s = threadIdx.x; s < p.n_seg; s += blockDim.x) {
      const int32_t a = s_seg_off[s], b = s_seg_off[s + 1], v = s_seg_var[s];
      bad_local |= (a < 0 || b < a || b > p.M || v < 0 || v > p.n_var) ? 1 : 0;
    }
    const bool table_bad = __syncthreads_or(bad_local) != 0;
    if (table_bad && blockIdx.x == 0 && threadIdx.x == 0) record_error(p.ctx, kErrBounds);
    for (int s = threadIdx.x; s < p.n_seg; s += blockDim.x) {
      const int32_t len = table_bad ? 0 : s_seg_off[s + 1] - s_seg_off[s];
      const int32_t tiles = len > p.max_short ? (len + kBN - 1) / kBN : 0;
      s_prefix[s + 1] = (tiles + C - 1) / C;
    }
    __syncthreads();
    if (warp == 0) {  // inclusive scan of the group counts
      int32_t carry = 0;
      if (lane == 0) s_prefix[0] = 0;
      for (int base = 0; base < p.n_seg; base += 32) {
        const int s = base + lane;
        int32_t v = s < p.n_seg ? s_prefix[s + 1] : 0;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const int32_t o = __shfl_up_sync(0xFFFFFFFFu, v, off);
          if (lane >= off) v += o;
        }
        if (s < p.n_seg) s_prefix[s + 1] = carry + v;
        carry += __shfl_sync(0xFFFFFFFFu, v, 31);
      }
      if (lane == 0) misc->groups = carry;
    }
  } else if (threadIdx.x == 0) {
    const int64_t t_total = (p.M + kBN - 1) / kBN;
    misc->groups = (t_total + C - 1) / C;
  }
  if (warp == kMmaWarp) {
    tmem_alloc(&misc->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  if (warp == kTmaWarp && lane == 0) {
    prefetch_tmap(&tmap_w);
    prefetch_tmap(&tmap_x);
  }
  tc_fence_before();
  __syncthreads();
  if (C > 1) cluster_sync();  // every CTA's barriers exist before any remote arrive
  tc_fence_after();

  const uint32_t tmem_base = misc->tmem_base;
  const int64_t groups = misc->groups;
  const int64_t n_tiles_n = (p.d_out + kBM - 1) / kBM;
  const int64_t num_ctiles = n_tiles_n * groups;
  const int64_t cluster_id = blockIdx.x / C;
  const int64_t n_clusters = gridDim.x / C;
  const int64_t my_tiles =
      cluster_id < num_ctiles ? (num_ctiles - 1 - cluster_id) / n_clusters + 1 : 0;
  const int n_kb = static_cast<int>(p.d_in / kBK);
  const int64_t total_q = my_tiles * n_kb;
  const int32_t* seg_off_tbl = grouped ? s_seg_off : nullptr;
  auto my_tile = [&](int64_t i) {
    return tile_at<C>(p, cluster_id + i * n_clusters, groups, rank, seg_off_tbl, s_seg_var,
                      s_prefix);
  };

  if (warp < kXfWarps) {
    // ============================================================ transform
    const int p8 = lane & 7;    // physical 16-byte chunk within a 128-byte row
    const int rsub = lane >> 3;  // rows of this lane: row0 + 4*k + rsub
    const int row0 = static_cast<int>(rank) * kRowsPerCta + kRowsPerWarp * warp;
    uint8_t* sign_ring = smem + kOffSign;
    float* alpha_ring = reinterpret_cast<float*>(smem + kOffAlpha);
    const int64_t row_bytes = p.d_in / 8;

    // Lanes 0..kRowsPerWarp-1 copy the sign bytes (and, at k-block 0, α) of
    // row row0+lane for the next stage in flat order into its ring slot.
    // Every lane commits a group per stage, so cp.async.wait_group counts
    // stages.  The cursor advances incrementally.
    int pf_i = 0, pf_kb = 0, pf_slot = 0;
    Tile pf_tl = my_tiles > 0 ? my_tile(0) : Tile{0, 0, 0, 0};
    auto prefetch_next = [&]() {
      if (pf_i < my_tiles && lane < kRowsPerWarp && pf_tl.variant > 0) {
        const uint8_t* pk = grouped ? p.packed_table[pf_tl.variant - 1] : p.packed;
        const float* al = grouped ? p.alpha_table[pf_tl.variant - 1] : p.alpha;
        const int r = row0 + lane;
        const int64_t row = pf_tl.n0 + r;
        uint8_t* dst = sign_ring + (pf_slot * kBM + r) * 8;
        if (row < p.d_out && (reinterpret_cast<uintptr_t>(pk) & 7u) == 0) {
          cp_async_8(dst, pk + row * row_bytes + static_cast<int64_t>(pf_kb) * 8);
        } else {
          if (row < p.d_out && blockIdx.x == 0 && pf_kb == 0) record_error(p.ctx, kErrBounds);
          *reinterpret_cast<uint2*>(dst) = make_uint2(0xFFFFFFFFu, 0xFFFFFFFFu);
        }
        if (pf_kb == 0) {
          float* adst = alpha_ring + pf_slot * kBM + r;
          if (row < p.d_out)
            cp_async_4(adst, p.per_row ? al + row : al);
          else
            *adst = 0.f;
        }
      }
      cp_async_commit();
      pf_slot = pf_slot + 1 == kRing ? 0 : pf_slot + 1;
      if (pf_i < my_tiles && ++pf_kb == n_kb) {
        pf_kb = 0;
        if (++pf_i < my_tiles) pf_tl = my_tile(pf_i);
      }
    };

    for (int d = 0; d < kPrefetch; ++d) prefetch_next();
    uint32_t neg_alpha[kChunksPerLane];
    Tile tl{0, 0, 0, 0};
    int kb = 0, i = 0, s = 0, slot = 0;
    uint32_t ph = 0;
    for (int64_t q = 0; q < total_q; ++q) {
      prefetch_next();
      cp_async_wait<kPrefetch>();
      // lane 0 waits for this CTA's W rows of the stage; the shuffle makes the
      // verdict warp-uniform and __syncwarp publishes the ring bytes.  The own
      // TMA load of a stage is issued only after every CTA's MMA released the
      // stage, so the peers' A buffers are free to be written as well.
      int ok = 0;
      if (lane == 0) ok = mbar_wait(&full_bar[s], ph, p.ctx, abort) ? 1 : 0;
      ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
      __syncwarp();
      if (!ok) break;
      if (kb == 0) tl = my_tile(i);
      const bool has_delta = tl.variant > 0;
      if (has_delta || C > 1) {  // base rows still go to the peers' A buffers
        if (has_delta && kb == 0) {
#pragma unroll
          for (int k = 0; k < kChunksPerLane; ++k) {
            const int r = row0 + 4 * k + rsub;
            neg_alpha[k] = __float_as_uint(alpha_ring[slot * kBM + r]) | 0x80000000u;
          }
        }
        uint8_t* a_tile = smem + kOffA + s * kABytes;
        uint4 w[kChunksPerLane];
        uint32_t byte[kChunksPerLane];
#pragma unroll
        for (int k = 0; k < kChunksPerLane; ++k) {
          const int r = row0 + 4 * k + rsub;
          const int c = p8 ^ (r & 7);  // logical chunk: columns 8c .. 8c+7
          byte[k] = has_delta ? sign_ring[(slot * kBM + r) * 8 + c] : 0u;
          w[k] = *reinterpret_cast<const uint4*>(a_tile + r * 128 + p8 * 16);
        }
#pragma unroll
        for (int k = 0; k < kChunksPerLane; ++k) {
          const int r = row0 + 4 * k + rsub;
          const uint32_t in[4] = {w[k].x, w[k].y, w[k].z, w[k].w};
          uint32_t out[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            if (has_delta) {
              const float lo =
                  __fadd_rn(bf16lo_to_f32(in[j]), signed_alpha(byte[k], 2 * j, neg_alpha[k]));
              const float hi = __fadd_rn(bf16hi_to_f32(in[j]),
                                         signed_alpha(byte[k], 2 * j + 1, neg_alpha[k]));
              out[j] = pack_bf16x2_rn(lo, hi);
            } else {
              out[j] = in[j];
            }
          }
          if (has_delta)
            *reinterpret_cast<uint4*>(a_tile + r * 128 + p8 * 16) =
                make_uint4(out[0], out[1], out[2], out[3]);
        }
        fence_proxy_async_smem();  // the MMA and the bulk copies read these rows
      }
      __syncwarp();
      if (lane == 0) {
        if (C > 1) {
          // this warp's rows are contiguous in the stage: send them to every peer
          const uint32_t src = smem_addr(smem + kOffA + s * kABytes + row0 * 128);
#pragma unroll
          for (int c = 1; c < C; ++c) {
            const uint32_t peer = (rank + c) % C;
            bulk_copy_to_peer(map_to_rank(src, peer), src, kRowsPerWarp * 128,
                              map_to_rank(smem_addr(&xform_bar[s]), peer));
          }
          // the peers' rows of this stage arrive as transaction bytes here
          if (warp == 0)
            mbar_arrive_expect_tx(&xform_bar[s], (C - 1) * kWBytes);
          else
            mbar_arrive(&xform_bar[s]);
        } else {
          mbar_arrive(&xform_bar[s]);
        }
      }
      // advance the stage cursor
      if (++s == kStages) {
        s = 0;
        ph ^= 1u;
      }
      slot = slot + 1 == kRing ? 0 : slot + 1;
      if (++kb == n_kb) {
        kb = 0;
        ++i;
      }
    }
    cp_async_wait<0>();
  } else if (warp < kTmaWarp) {
    // ============================================================ epilogue
    const int quarter = warp - kEpiWarp0;  // TMEM lanes 32*quarter ..
    for (int64_t i = 0; i < my_tiles; ++i) {
      const int acc = static_cast<int>(i & 1);
      const uint32_t ph = static_cast<uint32_t>((i >> 1) & 1);
      // lane 0 waits, the verdict is warp-uniform (tcgen05.ld below runs on
      // all 32 lanes)
      int ok = 0;
      if (lane == 0) ok = mbar_wait(&accfull_bar[acc], ph, p.ctx, abort) ? 1 : 0;
      ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
      __syncwarp();
      if (!ok) break;
      tc_fence_after();
      const Tile tl = my_tile(i);
      const int64_t n = tl.n0 + 32 * quarter + lane;
      const bool n_ok = n < p.d_out;
      const int64_t tok_limit = tl.tok_end < tl.tok0 + kBN ? tl.tok_end : tl.tok0 + kBN;
      const int chunks = tok_limit > tl.tok0 ? static_cast<int>((tok_limit - tl.tok0 + 31) / 32) : 0;
#pragma unroll 1
      for (int c = 0; c < chunks; ++c) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(tmem_base + (static_cast<uint32_t>(32 * quarter) << 16) +
                               static_cast<uint32_t>(acc * kAccCols + 32 * c),
                           r);
        tmem_ld_wait();
        const int64_t tok_base = tl.tok0 + 32 * c;
        if (n_ok) {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int64_t tok = tok_base + j;
            if (tok < tok_limit) {
              const uint32_t pk = pack_bf16x2_rn(__uint_as_float(r[j]), 0.f);
              p.y[tok * p.d_out + n] = static_cast<uint16_t>(pk & 0xFFFFu);
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&accempty_bar[acc]);
    }
  } else if (warp == kTmaWarp) {
    // ============================================================ TMA producer
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_first();
      const uint64_t pol_x = policy_evict_last();
      int64_t q = 0;
      bool ok = true;
      for (int64_t i = 0; i < my_tiles && ok; ++i) {
        const Tile tl = my_tile(i);
        for (int kb = 0; kb < n_kb; ++kb, ++q) {
          const int s = static_cast<int>(q % kStages);
          const uint32_t ph = static_cast<uint32_t>((q / kStages) & 1);
          // every CTA's MMA must be done with this stage (its A buffer is
          // rewritten by the cluster's transforms after the load lands)
          const bool got = C == 1 ? mbar_wait(&empty_bar[s], ph ^ 1u, p.ctx, abort)
                                  : mbar_wait_cluster(&empty_bar[s], ph ^ 1u, p.ctx, abort);
          if (!got) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full_bar[s], kWBytes + kBBytes);
          tma_load_2d(smem + kOffA + s * kABytes + rank * kWBytes, &tmap_w, &full_bar[s],
                      kb * kBK, static_cast<int32_t>(tl.n0 + rank * kRowsPerCta), pol_w);
          tma_load_2d(smem + kOffB + s * kBBytes, &tmap_x, &full_bar[s], kb * kBK,
                      static_cast<int32_t>(tl.tok0), pol_x);
        }
      }
      // Drain: wait (bounded, ignoring abort) until every issued copy landed.
      const int64_t first = q > kStages ? q - kStages : 0;
      for (int64_t qq = first; qq < q; ++qq)
        mbar_wait(&full_bar[qq % kStages], static_cast<uint32_t>((qq / kStages) & 1), p.ctx,
                  nullptr);
      // With a cluster, also wait until the last commit of every stage from
      // every CTA and the last rows copied in by the peers have landed here,
      // so no remote arrive or copy reaches this CTA's shared memory after it
      // exits.
      if (C > 1) {
        const int64_t first_done = total_q > kStages ? total_q - kStages : 0;
        for (int64_t qq = first_done; qq < total_q; ++qq) {
          const uint32_t ph_done = static_cast<uint32_t>((qq / kStages) & 1);
          mbar_wait_cluster(&xform_bar[qq % kStages], ph_done, p.ctx, nullptr);
          mbar_wait_cluster(&empty_bar[qq % kStages], ph_done, p.ctx, nullptr);
        }
      }
    }
  } else if (warp == kMmaWarp) {
    // ============================================================ MMA issuer
    if (lane == 0) {
      const uint32_t a_base = smem_addr(smem + kOffA);
      const uint32_t b_base = smem_addr(smem + kOffB);
      const uint16_t all_ctas = static_cast<uint16_t>((1u << C) - 1u);
      int64_t q = 0;
      bool ok = true;
      bool issued = false;
      for (int64_t i = 0; i < my_tiles && ok; ++i) {
        const int acc = static_cast<int>(i & 1);
        const uint32_t aph = static_cast<uint32_t>((i >> 1) & 1);
        if (!mbar_wait(&accempty_bar[acc], aph ^ 1u, p.ctx, abort)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * kAccCols);
        for (int kb = 0; kb < n_kb; ++kb, ++q) {
          const int s = static_cast<int>(q % kStages);
          const uint32_t ph = static_cast<uint32_t>((q / kStages) & 1);
          const bool got_x = mbar_wait(&full_bar[s], ph, p.ctx, abort);
          const bool got_a = got_x && (C == 1 ? mbar_wait(&xform_bar[s], ph, p.ctx, abort)
                                              : mbar_wait_cluster(&xform_bar[s], ph, p.ctx, abort));
          if (!got_a) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t a_desc = sdesc_k_sw128(a_base + s * kABytes);
          const uint64_t b_desc = sdesc_k_sw128(b_base + s * kBBytes);
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k) {
            // +32 bytes along K inside the swizzle atom = +2 in the address field
            umma_bf16(d_tmem, a_desc + 2 * k, b_desc + 2 * k, kIdesc,
                      (kb > 0 || k > 0) ? 1u : 0u);
          }
          issued = true;
          if (C == 1)
            umma_commit(&empty_bar[s]);
          else
            umma_commit_multicast(&empty_bar[s], all_ctas);
        }
        if (!ok) break;
        umma_commit(&accfull_bar[acc]);
      }
      if (issued) {
        umma_commit(drain_bar);
        mbar_wait(drain_bar, 0, p.ctx, nullptr);
      }
    }
  }

  // ---------------------------------------------------------------- teardown
  tc_fence_before();
  __syncthreads();
  // No CTA leaves while a peer may still store into its shared memory or
  // arrive on its barriers.
  if (C > 1) cluster_sync();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tmem_base, kTmemCols);
}

template <int C>
cudaError_t launch_c(const GemmArgs& p, const CUtensorMap& tmap_w, const CUtensorMap& tmap_x,
                     int max_clusters_wanted, cudaStream_t stream) {
  static bool attr_done[64] = {};
  static int max_clusters[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (!attr_done[dev]) {
    e = cudaFuncSetAttribute(bitdelta_gemm_kernel<C>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmemBytes);
    if (e != cudaSuccess) return e;
    int n = 0;
    cfg.gridDim = dim3(C);
    e = cudaOccupancyMaxActiveClusters(&n, bitdelta_gemm_kernel<C>, &cfg);
    if (e != cudaSuccess) return e;
    if (n < 1) return cudaErrorInvalidConfiguration;
    max_clusters[dev] = n;
    attr_done[dev] = true;
  }
  const int clusters = max_clusters_wanted < max_clusters[dev] ? max_clusters_wanted
                                                               : max_clusters[dev];
  cfg.gridDim = dim3(C * (clusters > 0 ? clusters : 1));
  return cudaLaunchKernelEx(&cfg, bitdelta_gemm_kernel<C>, tmap_w, tmap_x, p);
}

}  // namespace

int gemm_block_rows() { return kBM; }
int gemm_block_tokens() { return kBN; }

cudaError_t launch_gemm(const GemmArgs& p, const CUtensorMap& tmap_w, const CUtensorMap& tmap_x,
                        int cluster_size, int64_t cluster_tiles_bound, cudaStream_t stream) {
  const int want = static_cast<int>(cluster_tiles_bound < (1 << 20) ? cluster_tiles_bound
                                                                     : (1 << 20));
  switch (cluster_size) {
    case 1:
      return launch_c<1>(p, tmap_w, tmap_x, want, stream);
    case 2:
      return launch_c<2>(p, tmap_w, tmap_x, want, stream);
    case 4:
      return launch_c<4>(p, tmap_w, tmap_x, want, stream);
    default:
      return cudaErrorInvalidValue;
  }
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
