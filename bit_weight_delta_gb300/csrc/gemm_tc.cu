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
// Warp roles (448 threads, one CTA per SM, persistent over tiles):
//   warps 0-7   transform: each warp owns 16 of the 128 W rows.  It waits for
//               the TMA'd W_base stage, rewrites its rows in place as
//               W_eff = bf16_rne(fp32(W_base) ± α) (same 128-byte swizzled
//               layout, so each 16-byte chunk maps to itself), makes the writes
//               visible to the async proxy and arrives once.  Its lanes
//               prefetch their rows' sign bytes (8 per row per stage) and α
//               with cp.async into a ring several stages ahead.  The warps
//               never synchronise with one another.
//   warps 8-11  epilogue: tcgen05.ld the finished accumulator (lane = n,
//               column = token), round to bf16, store y.
//   warp 12     TMA producer: W_base tile [128 x 64] and x tile [256 x 64].
//   warp 13     MMA issuer: 4 x tcgen05.mma (128x256x16) per stage, commit.
// Every wait is bounded (kernel records a timeout and unwinds); TMEM is
// released on every exit path.
#include <cstdint>

#include "common.cuh"
#include "kernels.h"

namespace bd {
namespace {

#ifndef BD_GEMM_BN
#define BD_GEMM_BN 256
#endif
#ifndef BD_GEMM_STAGES
#define BD_GEMM_STAGES 4
#endif
constexpr int kBM = 128;         // d_out rows per tile
constexpr int kBN = BD_GEMM_BN;  // tokens per tile
constexpr int kBK = 64;          // K per stage: one 128-byte swizzle atom of bf16
constexpr int kStages = BD_GEMM_STAGES;
constexpr int kABytes = kBM * kBK * 2;  // 16 KB
constexpr int kBBytes = kBN * kBK * 2;  // 32 KB
constexpr int kPrefetch = 4;            // sign/α prefetch distance (stages)
constexpr int kRing = kPrefetch + 2;    // ring slots (see the transform loop)
constexpr int kAccCols = kBN;           // fp32 accumulator columns per buffer
constexpr int kTmemCols = 2 * kAccCols;
constexpr int kXfWarps = 8;                     // transform warps (independent)
constexpr int kXfRows = kBM / kXfWarps;         // W rows each transform warp owns
constexpr int kEpiWarp0 = kXfWarps;             // 4 epilogue warps: TMEM lane quarters 0..3
constexpr int kTmaWarp = kEpiWarp0 + 4;
constexpr int kMmaWarp = kTmaWarp + 1;
constexpr int kThreads = (kMmaWarp + 1) * 32;
static_assert(kEpiWarp0 % 4 == 0, "epilogue warps must start a warpgroup");
static_assert(kXfRows == 16, "transform lane mapping assumes 16 rows per warp");
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
  int64_t t_total;  // token tiles over all segments
};

struct Tile {
  int64_t n0;
  int64_t tok0;
  int64_t tok_end;
  int32_t variant;  // 0 = base (no delta)
};

__device__ __forceinline__ Tile tile_at(const GemmArgs& p, int64_t t, int64_t t_total,
                                        const int32_t* seg_off, const int32_t* seg_var,
                                        const int32_t* prefix) {
  Tile tl;
  const int64_t nt = t / t_total;
  const int64_t j = t - nt * t_total;
  tl.n0 = nt * kBM;
  if (seg_off == nullptr) {
    tl.tok0 = j * kBN;
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
    tl.tok0 = seg_off[lo] + (j - prefix[lo]) * kBN;
    tl.tok_end = seg_off[lo + 1];
    tl.variant = seg_var[lo];
  }
  return tl;
}

// ±α by the sign bit at `col` of `byte` (bit 1 -> +α); neg_alpha = α | sign.
__device__ __forceinline__ float signed_alpha(uint32_t byte, int col, uint32_t neg_alpha) {
  return __uint_as_float(neg_alpha ^ ((byte << (31 - col)) & 0x80000000u));
}

__global__ void __launch_bounds__(kThreads, 1)
    bitdelta_gemm_kernel(const __grid_constant__ CUtensorMap tmap_w,
                         const __grid_constant__ CUtensorMap tmap_x, const GemmArgs p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint64_t* full_bar = bars;                 // TMA -> transform
  uint64_t* xform_bar = bars + kStages;      // transform -> MMA
  uint64_t* empty_bar = bars + 2 * kStages;  // MMA -> TMA
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

  // ---------------------------------------------------------------- set-up
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&xform_bar[s], kXfWarps);
      mbar_init(&empty_bar[s], 1);
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
    // Copy the segment table, then count token tiles per valid long segment.
    // A malformed segment gets no tiles (so tile_at never selects it).
    for (int s = threadIdx.x; s <= p.n_seg; s += blockDim.x) s_seg_off[s] = __ldg(p.seg_off + s);
    for (int s = threadIdx.x; s < p.n_seg; s += blockDim.x) s_seg_var[s] = __ldg(p.seg_var + s);
    __syncthreads();
    // One malformed entry rejects the whole table (no tiles at all).
    int bad_local = 0;
    for (int s = threadIdx.x; s < p.n_seg; s += blockDim.x) {
      const int32_t a = s_seg_off[s], b = s_seg_off[s + 1], v = s_seg_var[s];
      bad_local |= (a < 0 || b < a || b > p.M || v < 0 || v > p.n_var) ? 1 : 0;
    }
    const bool table_bad = __syncthreads_or(bad_local) != 0;
    if (table_bad && blockIdx.x == 0 && threadIdx.x == 0) record_error(p.ctx, kErrBounds);
    for (int s = threadIdx.x; s < p.n_seg; s += blockDim.x) {
      const int32_t len = table_bad ? 0 : s_seg_off[s + 1] - s_seg_off[s];
      s_prefix[s + 1] = len > p.max_short ? (len + kBN - 1) / kBN : 0;
    }
    __syncthreads();
    if (warp == 0) {  // inclusive scan of the tile counts
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
      if (lane == 0) misc->t_total = carry;
    }
  } else if (threadIdx.x == 0) {
    misc->t_total = (p.M + kBN - 1) / kBN;
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
  tc_fence_after();

  const uint32_t tmem_base = misc->tmem_base;
  const int64_t t_total = misc->t_total;
  const int64_t n_tiles_n = (p.d_out + kBM - 1) / kBM;
  const int64_t num_tiles = n_tiles_n * t_total;
  const int64_t my_tiles =
      blockIdx.x < num_tiles ? (num_tiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;
  const int64_t n_kb = p.d_in / kBK;
  const int64_t total_q = my_tiles * n_kb;
  const int32_t* seg_off_tbl = grouped ? s_seg_off : nullptr;

  if (warp < kXfWarps) {
    // ============================================================ transform
    const int p8 = lane & 7;    // physical 16-byte chunk within a 128-byte row
    const int rsub = lane >> 3;  // rows of this lane: kXfRows*warp + 4*i + rsub
    const int row0 = kXfRows * warp;
    uint8_t* sign_ring = smem + kOffSign;
    float* alpha_ring = reinterpret_cast<float*>(smem + kOffAlpha);
    const int64_t row_bytes = p.d_in / 8;

    // Lanes 0..15 copy the sign bytes (and, at k-block 0, α) of row row0+lane
    // for flat stage q into ring slot q % kRing.  Every lane commits a group.
    auto prefetch = [&](int64_t q) {
      if (q < total_q && lane < kXfRows) {
        const int64_t i = q / n_kb;
        const int64_t kb = q - i * n_kb;
        const Tile tl = tile_at(p, blockIdx.x + i * gridDim.x, t_total, seg_off_tbl, s_seg_var,
                                s_prefix);
        const int slot = static_cast<int>(q % kRing);
        if (tl.variant > 0) {
          const uint8_t* pk = grouped ? p.packed_table[tl.variant - 1] : p.packed;
          const float* al = grouped ? p.alpha_table[tl.variant - 1] : p.alpha;
          const int r = row0 + lane;
          const int64_t row = tl.n0 + r;
          uint8_t* dst = sign_ring + (slot * kBM + r) * 8;
          if (row < p.d_out && (reinterpret_cast<uintptr_t>(pk) & 7u) == 0) {
            cp_async_8(dst, pk + row * row_bytes + kb * 8);
          } else {
            if (row < p.d_out && blockIdx.x == 0 && kb == 0) record_error(p.ctx, kErrBounds);
            *reinterpret_cast<uint2*>(dst) = make_uint2(0xFFFFFFFFu, 0xFFFFFFFFu);
          }
          if (kb == 0) {
            float* adst = alpha_ring + slot * kBM + r;
            if (row < p.d_out)
              cp_async_4(adst, p.per_row ? al + row : al);
            else
              *adst = 0.f;
          }
        }
      }
      cp_async_commit();
    };

    for (int d = 0; d < kPrefetch; ++d) prefetch(d);
    uint32_t neg_alpha[4];
    Tile tl{0, 0, 0, 0};
    for (int64_t q = 0; q < total_q; ++q) {
      prefetch(q + kPrefetch);
      cp_async_wait<kPrefetch>();
      const int64_t i = q / n_kb;
      const int64_t kb = q - i * n_kb;
      const int s = static_cast<int>(q % kStages);
      const uint32_t ph = static_cast<uint32_t>((q / kStages) & 1);
      // lane 0 waits; the shuffle makes the verdict warp-uniform, __syncwarp
      // publishes the lanes' ring bytes of stage q to the whole warp
      int ok = 0;
      if (lane == 0) ok = mbar_wait(&full_bar[s], ph, p.ctx, abort) ? 1 : 0;
      ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
      __syncwarp();
      if (!ok) break;
      if (kb == 0)
        tl = tile_at(p, blockIdx.x + i * gridDim.x, t_total, seg_off_tbl, s_seg_var, s_prefix);
      if (tl.variant > 0) {
        const int slot = static_cast<int>(q % kRing);
        if (kb == 0) {
#pragma unroll
          for (int r4 = 0; r4 < 4; ++r4) {
            const int r = row0 + 4 * r4 + rsub;
            neg_alpha[r4] = __float_as_uint(alpha_ring[slot * kBM + r]) | 0x80000000u;
          }
        }
        uint8_t* a_tile = smem + kOffA + s * kABytes;
        uint4 w[4];
        uint32_t byte[4];
#pragma unroll
        for (int r4 = 0; r4 < 4; ++r4) {
          const int r = row0 + 4 * r4 + rsub;
          const int c = p8 ^ (r & 7);  // logical chunk: columns 8c .. 8c+7
          byte[r4] = sign_ring[(slot * kBM + r) * 8 + c];
          w[r4] = *reinterpret_cast<const uint4*>(a_tile + r * 128 + p8 * 16);
        }
#pragma unroll
        for (int r4 = 0; r4 < 4; ++r4) {
          const int r = row0 + 4 * r4 + rsub;
          const uint32_t in[4] = {w[r4].x, w[r4].y, w[r4].z, w[r4].w};
          uint32_t out[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float lo =
                __fadd_rn(bf16lo_to_f32(in[j]), signed_alpha(byte[r4], 2 * j, neg_alpha[r4]));
            const float hi =
                __fadd_rn(bf16hi_to_f32(in[j]), signed_alpha(byte[r4], 2 * j + 1, neg_alpha[r4]));
            out[j] = pack_bf16x2_rn(lo, hi);
          }
          *reinterpret_cast<uint4*>(a_tile + r * 128 + p8 * 16) =
              make_uint4(out[0], out[1], out[2], out[3]);
        }
        fence_proxy_async_smem();
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&xform_bar[s]);
    }
    cp_async_wait<0>();
  } else if (warp < kTmaWarp) {
    // ============================================================ epilogue
    const int quarter = warp - kEpiWarp0;  // TMEM lanes 32*quarter ..
    for (int64_t i = 0; i < my_tiles; ++i) {
      const int acc = static_cast<int>(i & 1);
      const uint32_t ph = static_cast<uint32_t>((i >> 1) & 1);
      // warp-uniform verdict: tcgen05.ld below must run on all 32 lanes
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(&accfull_bar[acc], ph, p.ctx, abort))) break;
      tc_fence_after();
      const Tile tl =
          tile_at(p, blockIdx.x + i * gridDim.x, t_total, seg_off_tbl, s_seg_var, s_prefix);
      const int64_t n = tl.n0 + 32 * quarter + lane;
      const bool n_ok = n < p.d_out;
#pragma unroll 1
      for (int c = 0; c < kBN / 32; ++c) {
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
            if (tok < tl.tok_end) {
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
        const Tile tl =
            tile_at(p, blockIdx.x + i * gridDim.x, t_total, seg_off_tbl, s_seg_var, s_prefix);
        for (int64_t kb = 0; kb < n_kb; ++kb, ++q) {
          const int s = static_cast<int>(q % kStages);
          const uint32_t ph = static_cast<uint32_t>((q / kStages) & 1);
          if (!mbar_wait(&empty_bar[s], ph ^ 1u, p.ctx, abort)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full_bar[s], kABytes + kBBytes);
          tma_load_2d(smem + kOffA + s * kABytes, &tmap_w, &full_bar[s],
                      static_cast<int32_t>(kb * kBK), static_cast<int32_t>(tl.n0), pol_w);
          tma_load_2d(smem + kOffB + s * kBBytes, &tmap_x, &full_bar[s],
                      static_cast<int32_t>(kb * kBK), static_cast<int32_t>(tl.tok0), pol_x);
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
    if (lane == 0) {
      const uint32_t a_base = smem_addr(smem + kOffA);
      const uint32_t b_base = smem_addr(smem + kOffB);
      int64_t q = 0;
      bool ok = true;
      bool issued = false;
      for (int64_t i = 0; i < my_tiles && ok; ++i) {
        const int acc = static_cast<int>(i & 1);
        const uint32_t aph = static_cast<uint32_t>((i >> 1) & 1);
        if (!mbar_wait(&accempty_bar[acc], aph ^ 1u, p.ctx, abort)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * kAccCols);
        for (int64_t kb = 0; kb < n_kb; ++kb, ++q) {
          const int s = static_cast<int>(q % kStages);
          const uint32_t ph = static_cast<uint32_t>((q / kStages) & 1);
          if (!mbar_wait(&full_bar[s], ph, p.ctx, abort) ||
              !mbar_wait(&xform_bar[s], ph, p.ctx, abort)) {
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
          umma_commit(&empty_bar[s]);
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
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tmem_base, kTmemCols);
}

}  // namespace

int gemm_block_rows() { return kBM; }
int gemm_block_tokens() { return kBN; }

cudaError_t launch_gemm(const GemmArgs& p, const CUtensorMap& tmap_w, const CUtensorMap& tmap_x,
                        int grid, cudaStream_t stream) {
  static bool attr_done[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_done[dev]) {
    e = cudaFuncSetAttribute(bitdelta_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_done[dev] = true;
  }
  bitdelta_gemm_kernel<<<grid, kThreads, kSmemBytes, stream>>>(tmap_w, tmap_x, p);
  return cudaGetLastError();
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
