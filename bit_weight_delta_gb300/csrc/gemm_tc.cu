// gemm_tc.cu — fused BitDelta linear for many rows (prefill) on the tcgen05
// tensor cores.
//
// Page "BitDelta: serving 14 Zen models from one GPU cluster", section
// "Serving architecture": the fused kernel reads the base weight and the delta
// bits, builds the effective weight in registers or on-chip memory — never the
// whole W_eff in HBM — and multiplies in the same pass (conceptual
// fused_bitdelta_linear: F.linear(x, W_base + α·unpack(bits))).
//
// Tile: 128 output rows (n, UMMA M, operand A = W_eff) x 256 tokens (UMMA N,
// operand B = x) x 64 K per stage; D = W_eff·xᵀ = yᵀ accumulates in tensor
// memory (fp32, 128 lanes x 256 columns).
//
// The effective weight goes to tensor memory, not shared memory: the MMA takes
// its A operand from TMEM (row = lane, two bf16 along K per 32-bit column), so
// shared memory carries only the TMA writes of W_base and x, one read of
// W_base by the transform and the MMA's reads of x.
//
// Warp roles (one CTA per SM, persistent over tiles):
//   warps 0..4G-1  transform, G warpgroups taking the flat stages in turn.  Thread
//               i of a warpgroup owns W row i: it reads the row's 64 W_base
//               values of the stage from the TMA'd (128-byte swizzled) tile,
//               forms W_eff = bf16_rne(fp32(W_base) ± α) and writes the 32
//               packed columns to the stage's A slot with tcgen05.st.  Its
//               row's sign bytes and α are prefetched with cp.async into a
//               private ring several stages ahead.
//   next 4      epilogue: tcgen05.ld the finished accumulator (lane = n,
//               column = token), round to bf16, store y.
//   next 1      TMA producer: W_base tile [128 x 64] and x tile [256 x 64].
//   last        MMA issuer: 4 x tcgen05.mma (128x256x16, A in TMEM) per stage.
// G = 2 (448 threads).  Measured on 8192-wide projections at 2048 tokens, a
// third warpgroup made the kernel about 10% slower.
// Every wait is bounded (the kernel records a timeout and unwinds); TMEM is
// released on every exit path.
#include <cstdint>

#include "gemm_common.cuh"

namespace bd {
namespace {
using namespace gemm_detail;

constexpr int kBM = 128;  // d_out rows per tile
constexpr int kBN = 256;  // tokens per tile
#ifndef BD_GEMM_BK
#define BD_GEMM_BK 64
#endif
// K per stage: one row of a swizzle atom, 128 bytes of bf16 (BK = 64, 128-byte
// swizzle) or 64 bytes (BK = 32, 64-byte swizzle).  The ring holds 192 KB
// either way.  Measured on 8192-wide projections at 2048 tokens, BK = 64 is
// about 13% faster: the per-stage handoffs cost more than the deeper ring gains.
constexpr int kBK = BD_GEMM_BK;
static_assert(kBK == 32 || kBK == 64, "BK is one 64- or 128-byte swizzle row");
constexpr int kStages = 256 / kBK;       // 8 stages of 24 KB or 4 of 48 KB
constexpr int kABytes = kBM * kBK * 2;   // W_base per stage
constexpr int kBBytes = kBN * kBK * 2;   // x per stage
constexpr int kChunks = kBK / 8;         // 16-byte chunks per W row per stage
constexpr int kSwzShift = kBK == 64 ? 0 : 1;  // row bits that select the chunk XOR
constexpr int kSignBytes = kBK / 8;      // packed sign bytes per row per stage
constexpr int kPrefetch = kBK == 64 ? 2 : 4;  // sign/α prefetch distance (own stages)
constexpr int kRing = kPrefetch + 2;     // private ring slots per thread
constexpr int kDCols = kBN;              // accumulator columns
constexpr int kACol0 = kDCols;           // first column of the A slots
constexpr int kAColsPerStage = kBK / 2;  // two bf16 per 32-bit column
constexpr int kTmemCols = 512;           // D (256) + A slots (128), power of two
#ifndef BD_GEMM_XF_GROUPS
#define BD_GEMM_XF_GROUPS 2
#endif
constexpr int kXfGroups = BD_GEMM_XF_GROUPS;  // transform warpgroups
#ifndef BD_GEMM_SPLIT
#define BD_GEMM_SPLIT 0
#endif
// Split stages: every warpgroup works on every stage, warpgroup w on columns
// [w·BK/G, (w+1)·BK/G) of it, so a stage is transformed in 1/G of the time
// (the ring slot's round trip is TMA latency + transform + MMA, and it bounds
// the stage rate).  Otherwise the warpgroups take whole stages in turn.
constexpr bool kSplit = BD_GEMM_SPLIT != 0;
constexpr int kStep = kSplit ? 1 : kXfGroups;  // flat stages between a warpgroup's stages
constexpr int kXfChunks = kSplit ? kChunks / kXfGroups : kChunks;  // per thread per stage
constexpr int kXfSignBytes = kXfChunks;        // one sign byte per 8 columns
constexpr int kXfCols = 4 * kXfChunks;         // TMEM columns per thread per stage
constexpr uint32_t kXformArrivals = kSplit ? 4 * kXfGroups : 4;
static_assert(!kSplit || kXfSignBytes == 4, "split stages take 4 sign bytes per thread");
constexpr int kXfWarps = 4 * kXfGroups;
constexpr int kEpiWarp0 = kXfWarps;      // 4 epilogue warps: TMEM lane quarters 0..3
constexpr int kTmaWarp = kEpiWarp0 + 4;
constexpr int kMmaWarp = kTmaWarp + 1;
constexpr int kThreads = (kMmaWarp + 1) * 32;
static_assert(kEpiWarp0 % 4 == 0, "epilogue warps must start a warpgroup");
static_assert(kACol0 + kStages * kAColsPerStage <= kTmemCols, "tensor memory budget");
static_assert(kXfGroups <= kStages, "a warpgroup's stages must not alias in the ring");
constexpr uint32_t kIdesc = idesc_bf16_f32(kBM, kBN);

// Shared memory layout (offsets from a 1024-byte aligned base).
constexpr int kOffA = 0;
constexpr int kOffB = kOffA + kStages * kABytes;
constexpr int kOffSign = kOffB + kStages * kBBytes;                // [G][kRing][128] x 8 B
constexpr int kOffAlpha = kOffSign + kXfGroups * kRing * kBM * 8;  // [G][kRing][128] floats
constexpr int kOffBar = kOffAlpha + kXfGroups * kRing * kBM * 4;
constexpr int kNumBars = 4 * kStages + 2 + 1;
constexpr int kOffMisc = kOffBar + kNumBars * 8;  // tmem slot, abort flag, counts
constexpr int kOffSeg = kOffMisc + 64;            // grouped-mode tables
constexpr int kSegBytes = (3 * kGemmMaxSegs + 2) * 4;
constexpr int kSmemBytes = kOffSeg + kSegBytes + 1024;  // + alignment slack
static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");

struct Misc {
  uint32_t tmem_base;
  int abort;
  int64_t t_total;  // token tiles over all segments
};

__global__ void __launch_bounds__(kThreads, 1)
    bitdelta_gemm_kernel(const __grid_constant__ CUtensorMap tmap_w,
                         const __grid_constant__ CUtensorMap tmap_x, const GemmArgs p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  // Each stage's W_base and x complete on separate barriers: the transform
  // starts as soon as its 16 KB of W_base has landed, while x is still
  // arriving (the MMA waits for x and the transform).
  uint64_t* full_bar = bars;                 // TMA (W_base) -> transform
  uint64_t* xfull_bar = bars + kStages;      // TMA (x) -> MMA
  uint64_t* xform_bar = bars + 2 * kStages;  // transform -> MMA (A slot written)
  uint64_t* empty_bar = bars + 3 * kStages;  // MMA -> TMA (stage and A slot free)
  uint64_t* accfull_bar = bars + 4 * kStages;
  uint64_t* accempty_bar = accfull_bar + 1;
  uint64_t* drain_bar = accempty_bar + 1;
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
      mbar_init(&xfull_bar[s], 1);
      mbar_init(&xform_bar[s], kXformArrivals);  // the transform warps of the stage
      mbar_init(&empty_bar[s], 1);
    }
    mbar_init(accfull_bar, 1);
    mbar_init(accempty_bar, 128);
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
  const int n_kb = static_cast<int>(p.d_in / kBK);
  const int64_t total_q = my_tiles * n_kb;  // flat stages q = i * n_kb + kb
  const int32_t* seg_off_tbl = grouped ? s_seg_off : nullptr;
  auto my_tile = [&](int64_t i) {
    return tile_at<kBM, kBN>(p, blockIdx.x + i * gridDim.x, t_total, seg_off_tbl, s_seg_var,
                             s_prefix);
  };

  if (warp < kXfWarps) {
    // ============================================================ transform
    const int wg = warp >> 2;          // warpgroup
    const int c0 = kSplit ? wg * kXfChunks : 0;  // first 16-byte chunk of this warpgroup
    const int r = threadIdx.x & 127;   // the W row (and TMEM lane) of this thread
    const int quarter = warp & 3;      // TMEM lane quarter of this warp
    uint8_t* sign_ring = smem + kOffSign + wg * (kRing * kBM * 8);
    float* alpha_ring = reinterpret_cast<float*>(smem + kOffAlpha) + wg * (kRing * kBM);
    const int64_t row_bytes = p.d_in / 8;

    // A cursor over this warpgroup's flat stages (q = wg, wg + G, ... taking
    // stages in turn; every q with split stages) as (tile i, k-block kb);
    // kb < kStep marks the warpgroup's first stage of a tile.
    struct Cursor {
      int64_t q, i;
      int kb;
    };
    auto advance = [&](Cursor& c, int64_t step) {
      c.q += step;
      c.kb += static_cast<int>(step);
      bool moved = false;
      while (c.kb >= n_kb && c.i < my_tiles) {
        c.kb -= n_kb;
        ++c.i;
        moved = true;
      }
      return moved;
    };

    // Prefetch cursor: row r's sign bytes (and α at the warpgroup's first
    // stage of each tile) into private ring slot (own index) % kRing.  Each
    // thread later reads only what it copied itself.
    Cursor pf{0, 0, 0};
    advance(pf, kSplit ? 0 : wg);
    int pf_slot = 0;
    Tile pf_tl = pf.i < my_tiles ? my_tile(pf.i) : Tile{0, 0, 0, 0};
    auto prefetch_next = [&]() {
      if (pf.q < total_q && pf_tl.variant > 0) {
        const uint8_t* pk = grouped ? p.packed_table[pf_tl.variant - 1] : p.packed;
        const float* al = grouped ? p.alpha_table[pf_tl.variant - 1] : p.alpha;
        const int64_t row = pf_tl.n0 + r;
        uint8_t* dst = sign_ring + (pf_slot * kBM + r) * 8;
        if (row < p.d_out && (reinterpret_cast<uintptr_t>(pk) & (kXfSignBytes - 1)) == 0) {
          const uint8_t* src =
              pk + row * row_bytes + static_cast<int64_t>(pf.kb) * kSignBytes + c0;
          if constexpr (kXfSignBytes == 8)
            cp_async_8(dst, src);
          else
            cp_async_4(dst, src);
        } else {
          if (row < p.d_out && blockIdx.x == 0 && pf.kb < kStep) record_error(p.ctx, kErrBounds);
          *reinterpret_cast<uint2*>(dst) = make_uint2(0xFFFFFFFFu, 0xFFFFFFFFu);
        }
        if (pf.kb < kStep) {
          float* adst = alpha_ring + pf_slot * kBM + r;
          if (row < p.d_out)
            cp_async_4(adst, p.per_row ? al + row : al);
          else
            *adst = 0.f;
        }
      }
      cp_async_commit();
      pf_slot = pf_slot + 1 == kRing ? 0 : pf_slot + 1;
      if (pf.q < total_q && advance(pf, kStep) && pf.i < my_tiles) pf_tl = my_tile(pf.i);
    };

    for (int d = 0; d < kPrefetch; ++d) prefetch_next();
    uint32_t alpha_bits = 0u;  // α of the current tile's rows (fp32 bits)
    Cursor cur{0, 0, 0};
    advance(cur, kSplit ? 0 : wg);
    Tile tl = cur.i < my_tiles ? my_tile(cur.i) : Tile{0, 0, 0, 0};
    int slot = 0;
    int s = static_cast<int>(cur.q % kStages);                      // stage / A slot of q
    uint32_t ph = static_cast<uint32_t>((cur.q / kStages) & 1);     // parity of q's round
    const uint32_t a_lane = tmem_base + (static_cast<uint32_t>(32 * quarter) << 16);
    while (cur.q < total_q) {
      prefetch_next();
      cp_async_wait<kPrefetch>();
      int ok = 0;
      if (lane == 0) ok = mbar_wait(&full_bar[s], ph, p.ctx, abort) ? 1 : 0;
      ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
      __syncwarp();
      if (!ok) break;
      if (cur.kb < kStep && tl.variant > 0)
        alpha_bits = __float_as_uint(alpha_ring[slot * kBM + r]);
      const bool has_delta = tl.variant > 0;
      uint2 sg = make_uint2(0u, 0u);
      if (has_delta) {
        if constexpr (kXfSignBytes == 8)
          sg = *reinterpret_cast<const uint2*>(sign_ring + (slot * kBM + r) * 8);
        else
          sg.x = *reinterpret_cast<const uint32_t*>(sign_ring + (slot * kBM + r) * 8);
      }
      const uint8_t* w_row = smem + kOffA + s * kABytes + r * (kBK * 2);
      const int swz = (r >> kSwzShift) & (kChunks - 1);
      uint4 wv[kXfChunks];
#pragma unroll
      for (int c = 0; c < kXfChunks; ++c) {
        // logical 16-byte chunk c0+c (columns 8(c0+c) ..) sits at physical
        // chunk (c0+c) ^ swz: the TMA's 128-byte (64-byte) swizzle XORs the
        // chunk index with address bits 7-9 (7-8), i.e. with row bits 0-2 (1-2)
        wv[c] = *reinterpret_cast<const uint4*>(w_row + (((c0 + c) ^ swz) << 4));
      }
      uint32_t packed[kXfCols];
      if (has_delta) {
        weff_chunks<kXfChunks>(wv, sg, alpha_bits, packed);
      } else {
        // base rows (grouped mode, variant 0): W_base unchanged
#pragma unroll
        for (int c = 0; c < kXfChunks; ++c) {
          packed[4 * c + 0] = wv[c].x;
          packed[4 * c + 1] = wv[c].y;
          packed[4 * c + 2] = wv[c].z;
          packed[4 * c + 3] = wv[c].w;
        }
      }
      tmem_st_32x32b(a_lane + static_cast<uint32_t>(kACol0 + kAColsPerStage * s + 4 * c0),
                     packed);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&xform_bar[s]);
      // advance to this warpgroup's next stage (kStep flat stages later)
      s += kStep;
      if (s >= kStages) {
        s -= kStages;
        ph ^= 1u;
      }
      slot = slot + 1 == kRing ? 0 : slot + 1;
      if (advance(cur, kStep) && cur.i < my_tiles) tl = my_tile(cur.i);
    }
    cp_async_wait<0>();
  } else if (warp < kTmaWarp) {
    // ============================================================ epilogue
    const int quarter = warp - kEpiWarp0;  // TMEM lanes 32*quarter ..
    for (int64_t i = 0; i < my_tiles; ++i) {
      const uint32_t ph = static_cast<uint32_t>(i & 1);
      // lane 0 waits, the verdict is warp-uniform (tcgen05.ld below runs on
      // all 32 lanes)
      int ok = 0;
      if (lane == 0) ok = mbar_wait(accfull_bar, ph, p.ctx, abort) ? 1 : 0;
      ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
      __syncwarp();
      if (!ok) break;
      tc_fence_after();
      const Tile tl = my_tile(i);
      store_acc_rows<kBN>(tmem_base + (static_cast<uint32_t>(32 * quarter) << 16), p.y, p.d_out,
                          tl.n0 + 32 * quarter + lane, tl.tok0, tl.tok_end);
      tc_fence_before();
      mbar_arrive(accempty_bar);
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
          if (!mbar_wait(&empty_bar[s], ph ^ 1u, p.ctx, abort)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full_bar[s], kABytes);
          tma_load_2d(smem + kOffA + s * kABytes, &tmap_w, &full_bar[s], kb * kBK,
                      static_cast<int32_t>(tl.n0), pol_w);
          mbar_arrive_expect_tx(&xfull_bar[s], kBBytes);
          tma_load_2d(smem + kOffB + s * kBBytes, &tmap_x, &xfull_bar[s], kb * kBK,
                      static_cast<int32_t>(tl.tok0), pol_x);
        }
      }
      // Drain: wait (bounded, ignoring abort) until every issued copy landed.
      const int64_t first = q > kStages ? q - kStages : 0;
      for (int64_t qq = first; qq < q; ++qq) {
        const uint32_t par = static_cast<uint32_t>((qq / kStages) & 1);
        mbar_wait(&full_bar[qq % kStages], par, p.ctx, nullptr);
        mbar_wait(&xfull_bar[qq % kStages], par, p.ctx, nullptr);
      }
    }
  } else if (warp == kMmaWarp) {
    // ============================================================ MMA issuer
    if (lane == 0) {
      const uint32_t b_base = smem_addr(smem + kOffB);
      int64_t q = 0;
      bool ok = true;
      bool issued = false;
      for (int64_t i = 0; i < my_tiles && ok; ++i) {
        // the single accumulator must have been drained by the epilogue
        if (!mbar_wait(accempty_bar, static_cast<uint32_t>((i & 1) ^ 1), p.ctx, abort)) break;
        tc_fence_after();
        for (int kb = 0; kb < n_kb; ++kb, ++q) {
          const int s = static_cast<int>(q % kStages);
          const uint32_t ph = static_cast<uint32_t>((q / kStages) & 1);
          if (!mbar_wait(&xfull_bar[s], ph, p.ctx, abort)) { ok = false; break; }
          if (!mbar_wait(&xform_bar[s], ph, p.ctx, abort)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_tmem = tmem_base + static_cast<uint32_t>(kACol0 + kAColsPerStage * s);
          const uint64_t b_desc = kBK == 64 ? sdesc_k_sw128(b_base + s * kBBytes)
                                            : sdesc_k_sw64(b_base + s * kBBytes);
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k) {
            // K step 16: 8 TMEM columns of A; +32 bytes inside B's swizzle atom
            umma_bf16_tmem_a(tmem_base, a_tmem + 8 * k, b_desc + 2 * k, kIdesc,
                             (kb > 0 || k > 0) ? 1u : 0u);
          }
          issued = true;
          umma_commit(&empty_bar[s]);
        }
        if (!ok) break;
        umma_commit(accfull_bar);
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
int gemm_block_k() { return kBK; }

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
