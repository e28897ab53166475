// gemv.cu — fused BitDelta linear for few rows (decode), bandwidth-bound.
//
// Page "BitDelta: serving 14 Zen models from one GPU cluster", section
// "Serving architecture": one fused kernel reads the base weight and the delta
// bits together and never materialises W_eff in HBM; the conceptual
// fused_bitdelta_linear computes F.linear(x, W_base + α·unpack(bits)).
//
// Arithmetic (exact rewriting of x·W_effᵀ with W_eff = W_base + α·S, S = ±1):
//     y[m][n] = Σ_k x[m][k]·W_base[n][k]  +  α_n · Σ_k x[m][k]·S[n][k]
// Both sums run on the tensor cores with warp-level mma.sync m16n8k16 (bf16
// in, fp32 accumulate): the raw W_base words are the B fragments as loaded,
// and S is turned into ±1 bf16 pairs with three integer ops per two weights.
// The only difference from the canonical bf16-rounded W_eff is that W_eff is
// not rounded to bf16 before the product (a half-ulp change per weight).
//
// Work layout: a CTA owns 8·NG output rows (n) and one group of up to 16 x
// rows (m); its KW warps split d_in and reduce through shared memory in a
// fixed order.  Each thread loads, per 32-column chunk, one 16-byte word of a
// W_base row (8 adjacent columns; the 4 threads of a quad cover 64 contiguous
// bytes) and the matching 8 columns of two x rows.  The columns inside a
// fragment are permuted consistently for A and B, which a dot product allows.
// Sign bits arrive as one 16-byte load per row per super-chunk of 128 columns;
// each warp keeps two super-chunks of loads in flight in registers (M = 9..16,
// and shapes without 16-byte sign rows).  For M <= 8 the "deep queue" kernel
// instead routes W_base, signs and x through a per-warp cp.async ring in
// shared memory (three super-chunks in flight per warp, no registers held) and
// puts the W rows on the MMA's A side.  Per weight the kernels move
// 2 + 1/8 bytes from HBM; x stays in L1/L2.  Launched with programmatic
// dependent launch: both kernels issue their first weight loads (and the
// register kernel an L2 prefetch of the head of its weight slice) before
// they wait for the previous kernel in the stream; x is read after the wait.
#include <cstdint>
#include <type_traits>

#include "common.cuh"
#include "kernels.h"

namespace bd {
namespace {

// Launch shape: kNG groups of 8 output rows per CTA, kKW warps splitting d_in,
// super-chunks of kCPS x 32 columns (two in flight per warp).  The defaults
// were the fastest of a sweep on the 4096x4096 decode layer.
#ifndef BD_GEMV_NG
#define BD_GEMV_NG 2
#endif
#ifndef BD_GEMV_KW
#define BD_GEMV_KW 4
#endif
#ifndef BD_GEMV_CPS
#define BD_GEMV_CPS 4
#endif
constexpr int kNG = BD_GEMV_NG;
constexpr int kKW = BD_GEMV_KW;
constexpr int kCPS = BD_GEMV_CPS;
static_assert(kCPS == 4, "sign words are fetched 16 bytes (128 columns) at a time");
constexpr int kMaxGroupRows = 16;

__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// bf16x2 of ±1 for sign bits (2i, 2i+1) of `byte` (< 256): bit 1 -> +1.0
// (0x3F80), bit 0 -> −1.0 (0xBF80); column 2i in the low half.  One multiply
// and one logic op: byte·(0x40008000 >> 2i) puts bit 2i at bit 15 and bit
// 2i+1 at bit 31, and its two partial products (bits 9..22 and 24..37 at
// most) never overlap, so no carry reaches either bit.
__device__ __forceinline__ uint32_t pm_one_pair(uint32_t byte, int i) {
  return ((byte * (0x40008000u >> (2 * i))) & 0x80008000u) ^ 0xBF80BF80u;
}

// One 32-column chunk for NG groups of 8 W rows: base and sign products.
template <int NG>
__device__ __forceinline__ void chunk_mma(float (&acc_b)[NG][4], float (&acc_s)[NG][4],
                                          const uint4 (&wv)[NG], const uint32_t (&sb)[NG],
                                          uint4 xa, uint4 xb, bool has_delta) {
#pragma unroll
  for (int ng = 0; ng < NG; ++ng) {
    mma_16816(acc_b[ng], xa.x, xb.x, xa.y, xb.y, wv[ng].x, wv[ng].y);
    mma_16816(acc_b[ng], xa.z, xb.z, xa.w, xb.w, wv[ng].z, wv[ng].w);
    if (has_delta) {
      const uint32_t b = sb[ng];
      mma_16816(acc_s[ng], xa.x, xb.x, xa.y, xb.y, pm_one_pair(b, 0), pm_one_pair(b, 1));
      mma_16816(acc_s[ng], xa.z, xb.z, xa.w, xb.w, pm_one_pair(b, 2), pm_one_pair(b, 3));
    }
  }
}

struct RowGroup {
  int32_t rows[kMaxGroupRows];  // x/y row index per slot, −1 = empty
  int32_t variant;              // 0 = base model
};

// Register-resident operands of one super-chunk (CPS chunks of 32 columns).
template <int NG, int CPS, bool kM16>
struct Frag {
  uint4 w[CPS][NG];
  uint32_t s[CPS][NG];  // raw sign data: a 4-byte word per chunk, or one byte
  uint4 xa[CPS];
  uint4 xb[kM16 ? CPS : 1];
};

// Warp 0 sums the KW warps' partial products in a fixed order and writes the
// group's y rows (bf16, round to nearest even).
template <int NG>
__device__ __forceinline__ void store_group_rows(const GemvArgs& p, const RowGroup& grp,
                                                 const float* red, int64_t n0, int lane) {
  const int g = lane >> 2, t = lane & 3;
  const int64_t d_out = p.d_out;
#pragma unroll
  for (int ng = 0; ng < NG; ++ng) {
    float v[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      float s = 0.f;
      for (int w = 0; w < kKW; ++w) s += red[(w * NG * 4 + ng * 4 + e) * 32 + lane];
      v[e] = s;
    }
    const int64_t n = n0 + 8 * ng + 2 * t;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int slot = g + 8 * h;
      const int row = grp.rows[slot];
      if (row < 0 || n >= d_out) continue;
      uint16_t* yr = p.y + static_cast<int64_t>(row) * d_out;
      const uint32_t pk = pack_bf16x2_rn(v[2 * h], v[2 * h + 1]);
      if (n + 1 < d_out && (d_out % 2) == 0) {
        *reinterpret_cast<uint32_t*>(yr + n) = pk;
      } else {
        yr[n] = static_cast<uint16_t>(pk & 0xFFFFu);
        if (n + 1 < d_out) yr[n + 1] = static_cast<uint16_t>(pk >> 16);
      }
    }
  }
}

template <int NG, int CPS, bool kM16, bool kSignVec>
__device__ __forceinline__ void gemv_group(const GemvArgs& p, const RowGroup& grp,
                                           const uint8_t* __restrict__ packed,
                                           const float* __restrict__ alpha, bool has_delta,
                                           float* red) {
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int64_t d_in = p.d_in, d_out = p.d_out;
  const int64_t row_bytes = d_in / 8;
  const int64_t n0 = static_cast<int64_t>(blockIdx.x) * (8 * NG);

  const int ra_idx = grp.rows[g];
  const int rb_idx = kM16 ? grp.rows[g + 8] : -1;
  const uint16_t* xra = ra_idx >= 0 ? p.x + static_cast<int64_t>(ra_idx) * d_in : nullptr;
  const uint16_t* xrb = rb_idx >= 0 ? p.x + static_cast<int64_t>(rb_idx) * d_in : nullptr;

  const uint16_t* wrow[NG];
  const uint8_t* srow[NG];
#pragma unroll
  for (int ng = 0; ng < NG; ++ng) {
    const int64_t n = n0 + 8 * ng + g;
    wrow[ng] = n < d_out ? p.w + n * d_in : nullptr;
    srow[ng] = n < d_out ? packed + n * row_bytes : nullptr;
  }

  float acc_b[NG][4], acc_s[NG][4];
#pragma unroll
  for (int ng = 0; ng < NG; ++ng)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc_b[ng][e] = acc_s[ng][e] = 0.f;

  const uint4 zero4 = make_uint4(0u, 0u, 0u, 0u);
  using F = Frag<NG, CPS, kM16>;

  // the weight operands of a super-chunk (W_base words, sign words) ...
  auto load_w = [&](F& f, int64_t kc0) {
#pragma unroll
    for (int ng = 0; ng < NG; ++ng) {
      if (wrow[ng] != nullptr) {
#pragma unroll
        for (int j = 0; j < CPS; ++j) f.w[j][ng] = ldg_stream_v4(wrow[ng] + kc0 + 32 * j + 8 * t);
        if (has_delta) {
          if (kSignVec) {
            const uint4 v = ldg_v4(srow[ng] + kc0 / 8);
            f.s[0][ng] = v.x;
            f.s[1 % CPS][ng] = v.y;
            f.s[2 % CPS][ng] = v.z;
            f.s[3 % CPS][ng] = v.w;
          } else {
#pragma unroll
            for (int j = 0; j < CPS; ++j) f.s[j][ng] = __ldg(srow[ng] + kc0 / 8 + 4 * j + t);
          }
        }
      } else {
#pragma unroll
        for (int j = 0; j < CPS; ++j) {
          f.w[j][ng] = zero4;
          f.s[j][ng] = 0u;
        }
      }
    }
  };
  // ... and its activations
  auto load_x = [&](F& f, int64_t kc0) {
#pragma unroll
    for (int j = 0; j < CPS; ++j) {
      f.xa[j] = xra != nullptr ? ldg_v4(xra + kc0 + 32 * j + 8 * t) : zero4;
      if (kM16) f.xb[j] = xrb != nullptr ? ldg_v4(xrb + kc0 + 32 * j + 8 * t) : zero4;
    }
  };
  auto load = [&](F& f, int64_t kc0) {
    load_w(f, kc0);
    load_x(f, kc0);
  };
  auto compute = [&](const F& f) {
#pragma unroll
    for (int j = 0; j < CPS; ++j) {
      uint32_t sb[NG];
#pragma unroll
      for (int ng = 0; ng < NG; ++ng)
        sb[ng] = kSignVec ? (f.s[j][ng] >> (8 * t)) & 0xFFu : f.s[j][ng];
      chunk_mma<NG>(acc_b, acc_s, f.w[j], sb, f.xa[j], kM16 ? f.xb[kM16 ? j : 0] : zero4,
                    has_delta);
    }
  };

  const int64_t n_sc = d_in / (32 * CPS);
  if constexpr (kSignVec) {
    // Two super-chunks in flight per warp: the loads of the next one are
    // issued before the products of the current one.
    // The first super-chunk's weight loads go out before the wait for the
    // previous kernel in the stream (weights are never its output), its x
    // loads after it.
    F f0, f1;
    int64_t sc = warp;
    if (sc < n_sc) load_w(f0, sc * 32 * CPS);
    griddep_wait();
    if (sc < n_sc) load_x(f0, sc * 32 * CPS);
    while (sc < n_sc) {
      const int64_t sc1 = sc + kKW;
      if (sc1 < n_sc) load(f1, sc1 * 32 * CPS);
      compute(f0);
      if (sc1 >= n_sc) break;
      const int64_t sc2 = sc1 + kKW;
      if (sc2 < n_sc) load(f0, sc2 * 32 * CPS);
      compute(f1);
      sc = sc2;
    }
  } else {
    // Sign rows not 16-byte aligned: byte-wise sign loads, one super-chunk
    // at a time.
    griddep_wait();
    for (int64_t sc = warp; sc < n_sc; sc += kKW) {
      F f;
      load(f, sc * 32 * CPS);
      compute(f);
    }
  }
  // Tail: 32-column chunks past the last full super-chunk.  d_in is a
  // multiple of 8, so each thread's 8 columns are wholly inside or outside.
  for (int64_t c32 = n_sc * CPS + warp; c32 * 32 < d_in; c32 += kKW) {
    const int64_t col = c32 * 32 + 8 * t;
    const bool ok = col < d_in;
    uint4 wv[NG];
    uint32_t sb[NG];
#pragma unroll
    for (int ng = 0; ng < NG; ++ng) {
      const bool v = ok && wrow[ng] != nullptr;
      wv[ng] = v ? ldg_stream_v4(wrow[ng] + col) : zero4;
      sb[ng] = (v && has_delta) ? static_cast<uint32_t>(__ldg(srow[ng] + col / 8)) : 0xFFu;
    }
    const uint4 xa = (ok && xra != nullptr) ? ldg_v4(xra + col) : zero4;
    const uint4 xb = (kM16 && ok && xrb != nullptr) ? ldg_v4(xrb + col) : zero4;
    chunk_mma<NG>(acc_b, acc_s, wv, sb, xa, xb, has_delta);
  }

  // y_part = acc_b + α_n·acc_s for (m = g, g+8; n = n0 + 8ng + 2t + {0,1}).
#pragma unroll
  for (int ng = 0; ng < NG; ++ng) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      float v = acc_b[ng][e];
      if (has_delta) {
        const int64_t n = n0 + 8 * ng + 2 * t + (e & 1);
        const float a = n < d_out ? (p.per_row ? __ldg(alpha + n) : __ldg(alpha)) : 0.f;
        v = fmaf(a, acc_s[ng][e], v);
      }
      red[(warp * NG * 4 + ng * 4 + e) * 32 + lane] = v;
    }
  }
  __syncthreads();
  if (warp == 0) store_group_rows<NG>(p, grp, red, n0, lane);
  __syncthreads();
}

// ------------------------------------------------------------------ deep queue

// The same products with W_base, the sign words and x routed through shared
// memory by cp.async (the decode path for M <= 8): each warp keeps several
// super-chunks of its rows in flight in its own slice of a ring, holding no
// registers while they travel, where the register pipeline above holds two.
// The copies are mapped for coalescing, not for the MMA fragments: one copy
// instruction moves two whole 256-byte row segments (lanes 0-15 one row,
// 16-31 the next), and the fragment reads come back from shared memory after
// a warp barrier.  Row r's 16-byte word w sits at r·16 + (w ^ 4·(r & 1)), so
// the fragment reads (rows g and g+1 in one 128-byte phase) hit distinct
// banks.  The products use the swapped operands of chunk_mma_t.  Requires
// d_in % 128 == 0 and 16-byte aligned sign rows.
#ifndef BD_GEMV_ASYNC_MAX_M
#define BD_GEMV_ASYNC_MAX_M 8
#endif
constexpr int kStageRows = 8 * kNG;  // W rows of a CTA
// One warp's stage: W row segments, sign words, then the x segments of the
// NT·8 token rows (x goes through the ring too: every CTA reads it from L2,
// and a load issued one iteration ahead would not hide that latency).
template <int NT>
__host__ __device__ constexpr int stage_bytes() { return kStageRows * 256 + kStageRows * 16 + NT * 8 * 256; }
// Ring depth: two CTAs per SM.  With one token tile (M <= 8) 3 stages (77 KB
// per CTA) measured a few percent faster than 4 on 4096 x 4096 layers and 2
// far slower there (12.1 against 7.4 µs at M = 1); 2 stages at four CTAs
// per SM gained 2% on 57344 x 8192 and lost 7% on 8192 x 28672.  Two token
// tiles (M = 9..16, one-wave grids only): 3 stages, 101 KB.
#ifndef BD_GEMV_RING_STAGES
#define BD_GEMV_RING_STAGES 3
#endif
template <int NT>
__host__ __device__ constexpr int ring_stages() { return NT == 1 ? BD_GEMV_RING_STAGES : 3; }
template <int NT>
constexpr size_t gemv_ring_bytes() {
  return static_cast<size_t>(ring_stages<NT>()) * kKW * stage_bytes<NT>();
}

__device__ __forceinline__ void cp_async_16_cg(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
// x rows are read by every CTA at the same K position at about the same
// time: keep them in L1 too (.ca), so the CTAs of an SM fetch each line from
// L2 once instead of every warp queueing on the same few L2 lines.
// CTA pairs (clusters of two) for the grouped pass split over d_in.
__device__ __forceinline__ uint32_t pair_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void pair_store_f32(const float* local, uint32_t rank, float v) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
               : "=r"(remote)
               : "r"(smem_addr(local)), "r"(rank));
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(remote), "f"(v) : "memory");
}
// Every thread of both CTAs: release of the CTA's shared-memory writes
// (local and remote), acquire of the other's.
__device__ __forceinline__ void pair_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}

__device__ __forceinline__ void cp_async_16_x(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

// Operands swapped for the deep-queue path: the CTA's 16 W rows are the
// m16 A operand (rows g and g+8 of the fragment are W rows n0+g and n0+8+g)
// and up to 8 tokens are the n8 B operand, so M <= 8 issues half the MMAs of
// the x-as-A form.  Same column permutation as chunk_mma: thread t's 16-byte
// word (columns 8t..8t+7 of the chunk) feeds k-slots {2t, 2t+1, 2t+8, 2t+9}
// of two MMAs.  C: c0/c1 = (row g, tokens 2t, 2t+1), c2/c3 = row g+8.
template <int NT>
__device__ __forceinline__ void chunk_mma_t(float (&acc_b)[NT][4], float (&acc_s)[NT][4],
                                            const uint4 (&wv)[2], const uint32_t (&sb)[2],
                                            const uint4 (&xv)[NT], bool has_delta) {
  uint32_t s0[4], s1[4];
  if (has_delta) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      s0[i] = pm_one_pair(sb[0], i);
      s1[i] = pm_one_pair(sb[1], i);
    }
  }
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    mma_16816(acc_b[nt], wv[0].x, wv[1].x, wv[0].y, wv[1].y, xv[nt].x, xv[nt].y);
    mma_16816(acc_b[nt], wv[0].z, wv[1].z, wv[0].w, wv[1].w, xv[nt].z, xv[nt].w);
    if (has_delta) {
      mma_16816(acc_s[nt], s0[0], s1[0], s0[1], s1[1], xv[nt].x, xv[nt].y);
      mma_16816(acc_s[nt], s0[2], s1[2], s0[3], s1[3], xv[nt].z, xv[nt].w);
    }
  }
}

// Warp 0 sums the KW warps' partial products (transposed fragments) in a
// fixed order and writes y[token][n] (bf16, round to nearest even).
template <int NT, class Grp>
__device__ __forceinline__ void store_group_rows_t(const GemvArgs& p, const Grp& grp,
                                                   const float* red, int64_t n0, int lane) {
  const int g = lane >> 2, t = lane & 3;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      float v = 0.f;
      for (int w = 0; w < kKW; ++w) v += red[(w * NT * 4 + nt * 4 + e) * 32 + lane];
      const int64_t n = n0 + g + 8 * (e >> 1);
      const int row = grp.rows[8 * nt + 2 * t + (e & 1)];
      if (row < 0 || n >= p.d_out) continue;
      p.y[static_cast<int64_t>(row) * p.d_out + n] =
          static_cast<uint16_t>(pack_bf16x2_rn(v, 0.f) & 0xFFFFu);
    }
  }
}

template <int NG, bool kM16>
__device__ __forceinline__ void gemv_group_async(const GemvArgs& p, const RowGroup& grp,
                                                 const uint8_t* __restrict__ packed,
                                                 const float* __restrict__ alpha, bool has_delta,
                                                 float* red, uint8_t* ring) {
  static_assert(NG == kNG, "ring sized for kNG row groups");
  constexpr int CPS = kCPS;
  constexpr int R = 8 * NG;
  constexpr int NT = kM16 ? 2 : 1;  // token tiles of 8
  constexpr int D = ring_stages<NT>();
  constexpr int kSB = stage_bytes<NT>();
  constexpr int kXOff = R * 256 + R * 16;  // x segments within a stage
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int64_t d_in = p.d_in, d_out = p.d_out;
  const int64_t row_bytes = d_in / 8;
  const int64_t n0 = static_cast<int64_t>(blockIdx.x) * R;
  const int64_t rows_here = d_out - n0 < R ? d_out - n0 : R;

  bool x_ok[NT];  // token slot g (+8) holds a row of x
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) x_ok[nt] = grp.rows[g + 8 * nt] >= 0;

  bool row_ok[NG];
#pragma unroll
  for (int ng = 0; ng < NG; ++ng) row_ok[ng] = 8 * ng + g < rows_here;

  float acc_b[NT][4], acc_s[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc_b[nt][e] = acc_s[nt][e] = 0.f;

  const uint4 zero4 = make_uint4(0u, 0u, 0u, 0u);
  uint8_t* const wring = ring + static_cast<size_t>(warp) * D * kSB;
  const uint32_t wring_sa = smem_addr(wring);

  // copy side: lane L moves word (L & 15) of rows 2k + (L >> 4), k = 0..R/2-1,
  // and lanes 0..R-1 the sign word of row L
  const int cr = lane >> 4, cw = lane & 15;
  const uint16_t* const wsrc0 = p.w + (n0 + cr) * d_in + 8 * cw;
  const uint8_t* const ssrc0 = packed + (n0 + lane) * row_bytes;
  // x rows copied by this lane: token slots 2k + cr, k = 0..4·NT-1
  const uint16_t* xsrc[4 * NT];
#pragma unroll
  for (int k = 0; k < 4 * NT; ++k) {
    const int row = grp.rows[2 * k + cr];
    xsrc[k] = row >= 0 ? p.x + static_cast<int64_t>(row) * d_in + 8 * cw : nullptr;
  }
  const int64_t n_sc = d_in / (32 * CPS);
  // the weight operands of a stage: W_base row segments and sign words
  auto issue_w = [&](int s, int64_t sc) {
    if (sc < n_sc) {
      const int64_t kc0 = sc * 32 * CPS;
      const uint32_t st = wring_sa + s * kSB;
#pragma unroll
      for (int k = 0; k < R / 2; ++k) {
        const int r = 2 * k + cr;
        if (r < rows_here)
          cp_async_16_cg(st + 16u * (r * 16 + (cw ^ ((r & 1) << 2))), wsrc0 + 2 * k * d_in + kc0);
      }
      if (has_delta && lane < rows_here && lane < R)
        cp_async_16_cg(st + R * 256 + 16u * lane, ssrc0 + kc0 / 8);
    }
  };
  // the activations of a stage: x row segments
  auto issue_x = [&](int s, int64_t sc) {
    if (sc < n_sc) {
      const int64_t kc0 = sc * 32 * CPS;
      const uint32_t st = wring_sa + s * kSB;
#pragma unroll
      for (int k = 0; k < 4 * NT; ++k) {
        const int r = 2 * k + cr;
        if (xsrc[k] != nullptr)
          cp_async_16_x(st + kXOff + 16u * (r * 16 + (cw ^ ((r & 1) << 2))), xsrc[k] + kc0);
      }
    }
  };

  // Prologue: the weight halves of the first D-1 stages are issued before
  // waiting for the previous kernel in the stream (weights are never its
  // output), the x halves after it.  That makes 2(D-1) commit groups
  // W_0..W_{D-2}, X_0..X_{D-2}; in iteration i the loop below commits one
  // more group (both halves of stage i+D-1) and waits until at most D-1
  // groups are pending, which leaves only groups newer than X_i (i < D-1) or
  // than stage i: stage i is complete in either case.
  int64_t next = warp;
#pragma unroll
  for (int s = 0; s < D - 1; ++s) {
    issue_w(s, next + s * kKW);
    cp_async_commit();
  }
  griddep_wait();
#pragma unroll
  for (int s = 0; s < D - 1; ++s) {
    issue_x(s, next + s * kKW);
    cp_async_commit();
  }
  next += (D - 1) * kKW;
  int s_rd = 0;
  for (int64_t sc = warp; sc < n_sc; sc += kKW) {
    __syncwarp();  // every lane is done reading the slot refilled next
    issue_w(s_rd == 0 ? D - 1 : s_rd - 1, next);
    issue_x(s_rd == 0 ? D - 1 : s_rd - 1, next);
    cp_async_commit();  // one group per stage, empty past the end
    next += kKW;
    cp_async_wait<D - 1>();  // this lane's copies of the stage have landed
    __syncwarp();            // ... and every other lane's
    const uint8_t* st = wring + s_rd * kSB;
    // No selects on the fragment reads: a W row past d_out or an empty token
    // slot holds whatever the ring held and feeds only products of that row
    // or token, which are never stored (nor are sign words without a delta).
    uint4 sw[NG];
#pragma unroll
    for (int ng = 0; ng < NG; ++ng)
      sw[ng] = *reinterpret_cast<const uint4*>(st + R * 256 + 16 * (8 * ng + g));
#pragma unroll
    for (int j = 0; j < CPS; ++j) {
      uint4 wv[NG];
      uint32_t sb[NG];
#pragma unroll
      for (int ng = 0; ng < NG; ++ng) {
        const int r = 8 * ng + g;
        wv[ng] = *reinterpret_cast<const uint4*>(st + 16 * (r * 16 + ((4 * j + t) ^ ((r & 1) << 2))));
        const uint32_t word = j == 0 ? sw[ng].x : j == 1 ? sw[ng].y : j == 2 ? sw[ng].z : sw[ng].w;
        sb[ng] = (word >> (8 * t)) & 0xFFu;
      }
      uint4 xv[NT];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const int r = 8 * nt + g;
        xv[nt] = *reinterpret_cast<const uint4*>(
            st + kXOff + 16 * (r * 16 + ((4 * j + t) ^ ((r & 1) << 2))));
      }
      chunk_mma_t<NT>(acc_b, acc_s, wv, sb, xv, has_delta);
    }
    s_rd = s_rd == D - 1 ? 0 : s_rd + 1;
  }
  cp_async_wait<0>();

  // y_part = acc_b + α_n·acc_s (n = W row of the fragment), then the
  // fixed-order reduction over warps
  float a_row[2] = {0.f, 0.f};
  if (has_delta) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int64_t n = n0 + g + 8 * h;
      a_row[h] = n < d_out ? (p.per_row ? __ldg(alpha + n) : __ldg(alpha)) : 0.f;
    }
  }
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e)
      red[(warp * NT * 4 + nt * 4 + e) * 32 + lane] =
          has_delta ? fmaf(a_row[e >> 1], acc_s[nt][e], acc_b[nt][e]) : acc_b[nt][e];
  __syncthreads();
  if (warp == 0) store_group_rows_t<NT>(p, grp, red, n0, lane);
  __syncthreads();
}

// ------------------------------------------------------------------ mixed groups

// Up to 16 short rows of up to kMaxGroupVars distinct delta variants (and any
// number of base rows) computed in ONE pass over this CTA's W_base rows: the
// base product x·W_baseᵀ covers every row of the group at once, and the delta
// product of variant v uses x fragments in which the rows of other variants
// are zero, so each row collects exactly its own variant's α_v·(x·S_vᵀ).
constexpr int kMaxGroupVars = 4;
constexpr int kMixedAhead = 2;  // super-chunks of L2 prefetch ahead per warp

struct MixedGroup {
  int32_t rows[kMaxGroupRows];     // x/y row per slot, −1 = empty
  int32_t slot_var[kMaxGroupRows]; // index into vars[] of the slot's variant; −1 = base or empty
  int32_t vars[kMaxGroupVars];     // the group's delta variant ids (>= 1)
  int32_t n_vars;
};

template <int NG, bool kSignVec>
__device__ __forceinline__ void gemv_group_mixed(const GemvArgs& p, const MixedGroup& grp,
                                                 float* red) {
  constexpr int CPS = kCPS;
  constexpr int V = kMaxGroupVars;
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int64_t d_in = p.d_in, d_out = p.d_out;
  const int64_t row_bytes = d_in / 8;
  const int64_t n0 = static_cast<int64_t>(blockIdx.x) * (8 * NG);
  const int nv = grp.n_vars;

  const int ra_idx = grp.rows[g], rb_idx = grp.rows[g + 8];
  const int va = grp.slot_var[g], vb = grp.slot_var[g + 8];
  const uint16_t* xra = ra_idx >= 0 ? p.x + static_cast<int64_t>(ra_idx) * d_in : nullptr;
  const uint16_t* xrb = rb_idx >= 0 ? p.x + static_cast<int64_t>(rb_idx) * d_in : nullptr;

  const uint16_t* wrow[NG];
  const uint8_t* srow[V][NG];
#pragma unroll
  for (int ng = 0; ng < NG; ++ng) {
    const int64_t n = n0 + 8 * ng + g;
    wrow[ng] = n < d_out ? p.w + n * d_in : nullptr;
#pragma unroll
    for (int v = 0; v < V; ++v)
      srow[v][ng] = (v < nv && n < d_out) ? p.packed_table[grp.vars[v] - 1] + n * row_bytes
                                          : nullptr;
  }

  float acc_b[NG][4], acc_s[V][NG][4];
#pragma unroll
  for (int ng = 0; ng < NG; ++ng)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      acc_b[ng][e] = 0.f;
#pragma unroll
      for (int v = 0; v < V; ++v) acc_s[v][ng][e] = 0.f;
    }
  const uint4 zero4 = make_uint4(0u, 0u, 0u, 0u);

  // one 32-column chunk: base product for all rows, delta product per variant
  auto chunk = [&](const uint4 (&wv)[NG], const uint32_t (&sb)[V][NG], uint4 xa, uint4 xb) {
#pragma unroll
    for (int ng = 0; ng < NG; ++ng) {
      mma_16816(acc_b[ng], xa.x, xb.x, xa.y, xb.y, wv[ng].x, wv[ng].y);
      mma_16816(acc_b[ng], xa.z, xb.z, xa.w, xb.w, wv[ng].z, wv[ng].w);
    }
#pragma unroll
    for (int v = 0; v < V; ++v) {
      if (v < nv) {
        const uint4 xav = va == v ? xa : zero4;
        const uint4 xbv = vb == v ? xb : zero4;
#pragma unroll
        for (int ng = 0; ng < NG; ++ng) {
          const uint32_t b = sb[v][ng];
          mma_16816(acc_s[v][ng], xav.x, xbv.x, xav.y, xbv.y, pm_one_pair(b, 0),
                    pm_one_pair(b, 1));
          mma_16816(acc_s[v][ng], xav.z, xbv.z, xav.w, xbv.w, pm_one_pair(b, 2),
                    pm_one_pair(b, 3));
        }
      }
    }
  };

  const int64_t n_sc = d_in / (32 * CPS);
  // L2 prefetch of the super-chunk kMixedAhead steps ahead (this warp's next
  // but one): lane L takes one 128-byte line of the 16 W row segments and of
  // the x row segments, and the variants' sign words of rows 0..7 of each
  // group of 8 rows
  const int pr = lane >> 1, ph = lane & 1;  // row, half (line) of a 256-byte segment
  const int64_t n_pf = n0 + pr;
  const uint16_t* w_pf = n_pf < d_out && pr < 8 * NG ? p.w + n_pf * d_in + 64 * ph : nullptr;
  const int xr_pf = pr < kMaxGroupRows ? grp.rows[pr] : -1;
  const uint16_t* x_pf = xr_pf >= 0 ? p.x + static_cast<int64_t>(xr_pf) * d_in + 64 * ph : nullptr;
  auto prefetch_sc = [&](int64_t sc_pf) {
    if (sc_pf >= n_sc) return;
    const int64_t kc = sc_pf * 32 * CPS;
    if (w_pf != nullptr) prefetch_l2(w_pf + kc);
    if (x_pf != nullptr) prefetch_l2(x_pf + kc);
#pragma unroll
    for (int v = 0; v < V; ++v) {
      const int row = lane & 15, half = lane >> 4;  // row of group `half`
      if (v < nv && half < NG && row < 8 && n0 + 8 * half + row < d_out)
        prefetch_l2(p.packed_table[grp.vars[v] - 1] + (n0 + 8 * half + row) * row_bytes + kc / 8);
    }
  };
  prefetch_sc(warp + kKW);
  for (int64_t sc = warp; sc < n_sc; sc += kKW) {
    prefetch_sc(sc + kMixedAhead * kKW);
    const int64_t kc0 = sc * 32 * CPS;
    uint4 w[CPS][NG];
    uint32_t sw[CPS][V][NG];
    uint4 xa[CPS], xb[CPS];
#pragma unroll
    for (int ng = 0; ng < NG; ++ng) {
#pragma unroll
      for (int j = 0; j < CPS; ++j)
        w[j][ng] = wrow[ng] != nullptr ? ldg_stream_v4(wrow[ng] + kc0 + 32 * j + 8 * t) : zero4;
#pragma unroll
      for (int v = 0; v < V; ++v) {
        if (kSignVec) {
          const uint4 q = srow[v][ng] != nullptr ? ldg_v4(srow[v][ng] + kc0 / 8) : zero4;
          sw[0][v][ng] = q.x;
          sw[1][v][ng] = q.y;
          sw[2][v][ng] = q.z;
          sw[3][v][ng] = q.w;
        } else {
#pragma unroll
          for (int j = 0; j < CPS; ++j)
            sw[j][v][ng] = srow[v][ng] != nullptr ? __ldg(srow[v][ng] + kc0 / 8 + 4 * j + t) : 0u;
        }
      }
    }
#pragma unroll
    for (int j = 0; j < CPS; ++j) {
      xa[j] = xra != nullptr ? ldg_v4(xra + kc0 + 32 * j + 8 * t) : zero4;
      xb[j] = xrb != nullptr ? ldg_v4(xrb + kc0 + 32 * j + 8 * t) : zero4;
    }
#pragma unroll
    for (int j = 0; j < CPS; ++j) {
      uint32_t sb[V][NG];
#pragma unroll
      for (int v = 0; v < V; ++v)
#pragma unroll
        for (int ng = 0; ng < NG; ++ng)
          sb[v][ng] = kSignVec ? (sw[j][v][ng] >> (8 * t)) & 0xFFu : sw[j][v][ng];
      uint4 wj[NG];
#pragma unroll
      for (int ng = 0; ng < NG; ++ng) wj[ng] = w[j][ng];
      chunk(wj, sb, xa[j], xb[j]);
    }
  }
  // tail: 32-column chunks past the last full super-chunk
  for (int64_t c32 = n_sc * CPS + warp; c32 * 32 < d_in; c32 += kKW) {
    const int64_t col = c32 * 32 + 8 * t;
    const bool ok = col < d_in;
    uint4 wv[NG];
    uint32_t sb[V][NG];
#pragma unroll
    for (int ng = 0; ng < NG; ++ng) {
      wv[ng] = (ok && wrow[ng] != nullptr) ? ldg_stream_v4(wrow[ng] + col) : zero4;
#pragma unroll
      for (int v = 0; v < V; ++v)
        sb[v][ng] = (ok && srow[v][ng] != nullptr)
                        ? static_cast<uint32_t>(__ldg(srow[v][ng] + col / 8))
                        : 0xFFu;
    }
    const uint4 xa = (ok && xra != nullptr) ? ldg_v4(xra + col) : zero4;
    const uint4 xb = (ok && xrb != nullptr) ? ldg_v4(xrb + col) : zero4;
    chunk(wv, sb, xa, xb);
  }

  // y_part = acc_b + Σ_v α_v[n]·acc_s[v]  (for m = g, g+8; n = n0 + 8ng + 2t + {0,1})
#pragma unroll
  for (int ng = 0; ng < NG; ++ng) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int64_t n = n0 + 8 * ng + 2 * t + (e & 1);
      float val = acc_b[ng][e];
#pragma unroll
      for (int v = 0; v < V; ++v) {
        if (v < nv && n < d_out) {
          const float* al = p.alpha_table[grp.vars[v] - 1];
          val = fmaf(p.per_row ? __ldg(al + n) : __ldg(al), acc_s[v][ng][e], val);
        }
      }
      red[(warp * NG * 4 + ng * 4 + e) * 32 + lane] = val;
    }
  }
  __syncthreads();
  if (warp == 0) {
#pragma unroll
    for (int ng = 0; ng < NG; ++ng) {
      float vsum[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float sum = 0.f;
        for (int w = 0; w < kKW; ++w) sum += red[(w * NG * 4 + ng * 4 + e) * 32 + lane];
        vsum[e] = sum;
      }
      const int64_t n = n0 + 8 * ng + 2 * t;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int row = grp.rows[g + 8 * h];
        if (row < 0 || n >= d_out) continue;
        uint16_t* yr = p.y + static_cast<int64_t>(row) * d_out;
        const uint32_t pk = pack_bf16x2_rn(vsum[2 * h], vsum[2 * h + 1]);
        if (n + 1 < d_out && (d_out % 2) == 0) {
          *reinterpret_cast<uint32_t*>(yr + n) = pk;
        } else {
          yr[n] = static_cast<uint16_t>(pk & 0xFFFFu);
          if (n + 1 < d_out) yr[n + 1] = static_cast<uint16_t>(pk >> 16);
        }
      }
    }
  }
  __syncthreads();
}

// Single variant: blockIdx.y (strided) picks 16 consecutive x rows.
// Before waiting on the previous kernel in the stream, the register kernel
// pulls the first kPrefetchCols columns of its W_base rows (and the first
// line of each sign row) towards L2, so that its first loads, which it can
// only keep two super-chunks deep, hit L2.  Only a bounded head of the slice:
// prefetching whole slices (measured first) put the resident CTAs' slices
// beyond L2 on large layers (8192 x 28672: 917 KB per CTA) and took both
// decode kernels from 5.4-6.0 TB/s to 3.8-4.7 TB/s on 57344 x 8192 and
// 8192 x 28672; with the head only, the register kernel at 16 rows runs
// 4.9 TB/s there (3.9 without any prefetch), and the cp.async ring kernel
// is fastest with none at all.  L2 is the point of coherence, so a
// prefetch before griddep_wait cannot return stale data.
constexpr int64_t kPrefetchCols = 1024;
template <int NG>
__device__ __forceinline__ void prefetch_weights(const GemvArgs& p) {
  const int64_t rows = 8 * NG;
  const int64_t n0 = static_cast<int64_t>(blockIdx.x) * rows;
  const int64_t n_rows = p.d_out - n0 < rows ? p.d_out - n0 : rows;
  const int64_t cols = p.d_in < kPrefetchCols ? p.d_in : kPrefetchCols;
  const int64_t row_lines = (cols * 2 + 127) / 128;
  for (int64_t i = threadIdx.x; i < n_rows * row_lines; i += blockDim.x) {
    const int64_t r = i / row_lines, l = i - r * row_lines;
    prefetch_l2(reinterpret_cast<const uint8_t*>(p.w + (n0 + r) * p.d_in) + 128 * l);
  }
  for (int64_t r = threadIdx.x; r < n_rows; r += blockDim.x)
    prefetch_l2(p.packed + (n0 + r) * (p.d_in / 8));
}

// gemv_group waits for the previous kernel itself, after its first weight
// loads.
template <int NG, bool kM16, bool kSignVec>
__global__ void __launch_bounds__(kKW * 32) gemv_single_kernel(GemvArgs p) {
  __shared__ float red[kKW * NG * 4 * 32];
  __shared__ RowGroup grp;
  if (blockIdx.y == 0) prefetch_weights<NG>(p);
  griddep_launch_dependents();
  const int64_t n_chunks = (p.M + kMaxGroupRows - 1) / kMaxGroupRows;
  for (int64_t c = blockIdx.y; c < n_chunks; c += gridDim.y) {
    if (threadIdx.x < kMaxGroupRows) {
      const int64_t r = c * kMaxGroupRows + threadIdx.x;
      grp.rows[threadIdx.x] = r < p.M ? static_cast<int32_t>(r) : -1;
    }
    if (threadIdx.x == 0) grp.variant = 1;
    __syncthreads();
    gemv_group<NG, kCPS, kM16, kSignVec>(p, grp, p.packed, p.alpha, true, red);
  }
}

// Single variant through the deep cp.async queue (d_in % 128 == 0, aligned
// sign rows); same grid as above.  It waits for the previous kernel in the
// stream only after it has issued the weight loads of its first ring stages
// (inside gemv_group_async): W_base, the signs and α are inputs that no
// kernel still in flight writes, so a CTA that starts while the previous
// launch drains fills most of its ring before x is ready.
template <int NG, bool kM16>
__global__ void __launch_bounds__(kKW * 32) gemv_single_async_kernel(GemvArgs p) {
  extern __shared__ __align__(16) uint8_t ring[];
  __shared__ float red[kKW * NG * 4 * 32];
  __shared__ RowGroup grp;
  griddep_launch_dependents();
  const int64_t n_chunks = (p.M + kMaxGroupRows - 1) / kMaxGroupRows;
  for (int64_t c = blockIdx.y; c < n_chunks; c += gridDim.y) {
    if (threadIdx.x < kMaxGroupRows) {
      const int64_t r = c * kMaxGroupRows + threadIdx.x;
      grp.rows[threadIdx.x] = r < p.M ? static_cast<int32_t>(r) : -1;
    }
    if (threadIdx.x == 0) grp.variant = 1;
    __syncthreads();
    gemv_group_async<NG, kM16>(p, grp, p.packed, p.alpha, true, red, ring);
  }
}

// Mixed groups through the deep queue: W_base rows, every variant's sign
// words and the group's x rows travel by cp.async into a per-warp ring (as in
// gemv_group_async), the W rows are the MMA's A operand and NT tiles of 8
// tokens its B operand.  Each variant's sign product runs over all the
// group's tokens; a token reads only its own variant's accumulator, so no
// masking is needed.  Groups hold at most V delta variants (2 when the call
// has no more, else 4).  Requires d_in % 128 == 0; a variant table entry off
// a 16-byte boundary has its sign words fetched with plain loads.
template <int NT, int V>
__host__ __device__ constexpr int mixed_stage_bytes() {
  return kStageRows * 256 + V * kStageRows * 16 + NT * 8 * 256;
}
// Ring depth D (stages per warp): 3 while the grid's 16-row blocks fit one
// wave at two CTAs per SM (each warp then needs two stages in flight), 2 on
// larger grids, whose CTAs then fit four per SM (52 KB of ring and no other
// large buffer: the cross-warp sum goes through the ring): on the 40-layer
// slice's projections (8192-57344 rows, two variants) 2 stages took 4.1 ->
// 5.3 TB/s on 57344 x 8192 and 3.0 -> 4.0 on 10240 x 8192, and 15.0 -> 16.5
// µs on a 4096-row layer (one wave) against 3 stages.  With a separate 4 KB
// reduction buffer only three CTAs fitted per SM, and a grid of 512 blocks
// (8192 x 28672, two variants) took 125 µs against 99 µs at four.
template <int NT, int V, int D>
constexpr size_t mixed_ring_bytes() {
  return static_cast<size_t>(D) * kKW * mixed_stage_bytes<NT, V>();
}

template <int NT, int V, int D, bool kSplit>
__device__ __forceinline__ void gemv_group_mixed_async(const GemvArgs& p, const MixedGroup& grp,
                                                       uint8_t* ring, bool w_ahead, float* xfer) {
  constexpr int CPS = kCPS;
  constexpr int R = kStageRows;  // 16 W rows
  static_assert(R == 16 && V % 2 == 0, "two 8-row halves; variants copied in pairs");
  constexpr int kSB = mixed_stage_bytes<NT, V>();
  constexpr int kSOff = R * 256;              // sign words: [variant][row] × 16 bytes
  constexpr int kXOff = R * 256 + V * R * 16; // x segments of NT·8 token rows
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int64_t d_in = p.d_in, d_out = p.d_out;
  const int64_t row_bytes = d_in / 8;
  // kSplit: CTAs 2b and 2b + 1 (one cluster) share row block b, CTA `half`
  // taking the stages half·kKW + warp + 2·kKW·i
  const int half = kSplit ? static_cast<int>(pair_rank()) : 0;
  constexpr int kStep = kSplit ? 2 * kKW : kKW;
  const int64_t n0 = static_cast<int64_t>(kSplit ? blockIdx.x >> 1 : blockIdx.x) * R;
  const int64_t rows_here = d_out - n0 < R ? d_out - n0 : R;
  const int nv = grp.n_vars;

  bool x_ok[NT];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) x_ok[nt] = grp.rows[g + 8 * nt] >= 0;
  bool row_ok[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) row_ok[h] = 8 * h + g < rows_here;

  float acc_b[NT][4], acc_s[V][NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      acc_b[nt][e] = 0.f;
#pragma unroll
      for (int v = 0; v < V; ++v) acc_s[v][nt][e] = 0.f;
    }
  const uint4 zero4 = make_uint4(0u, 0u, 0u, 0u);
  uint8_t* const wring = ring + static_cast<size_t>(warp) * D * kSB;
  const uint32_t wring_sa = smem_addr(wring);

  // copy side (lane L): W word L & 15 of rows 2k + (L >> 4); the sign word of
  // row L & 15 of variants 2k + (L >> 4); x word L & 15 of token rows 2k + (L >> 4)
  const int cr = lane >> 4, cw = lane & 15;
  const uint16_t* const wsrc0 = p.w + (n0 + cr) * d_in + 8 * cw;
  const uint8_t* ssrc[V / 2];
  bool s_al[V / 2];  // 16-byte aligned sign row: cp.async; else plain loads
#pragma unroll
  for (int k = 0; k < V / 2; ++k) {
    const int v = 2 * k + cr;
    ssrc[k] = (v < nv && cw < rows_here)
                  ? p.packed_table[grp.vars[v] - 1] + (n0 + cw) * row_bytes
                  : nullptr;
    s_al[k] = (reinterpret_cast<uintptr_t>(ssrc[k]) & 15u) == 0;
  }
  const uint16_t* xsrc[4 * NT];
#pragma unroll
  for (int k = 0; k < 4 * NT; ++k) {
    const int row = grp.rows[2 * k + cr];
    xsrc[k] = row >= 0 ? p.x + static_cast<int64_t>(row) * d_in + 8 * cw : nullptr;
  }
  const int64_t n_sc = d_in / (32 * CPS);
  auto issue_w = [&](int s, int64_t sc) {
    if (sc < n_sc) {
      const int64_t kc0 = sc * 32 * CPS;
      const uint32_t st = wring_sa + s * kSB;
#pragma unroll
      for (int k = 0; k < R / 2; ++k) {
        const int r = 2 * k + cr;
        if (r < rows_here)
          cp_async_16_cg(st + 16u * (r * 16 + (cw ^ ((r & 1) << 2))), wsrc0 + 2 * k * d_in + kc0);
      }
    }
  };
  auto issue_sx = [&](int s, int64_t sc) {
    if (sc < n_sc) {
      const int64_t kc0 = sc * 32 * CPS;
      const uint32_t st = wring_sa + s * kSB;
#pragma unroll
      for (int k = 0; k < V / 2; ++k) {
        if (ssrc[k] == nullptr) continue;
        const uint32_t dst = st + kSOff + 16u * ((2 * k + cr) * R + cw);
        if (s_al[k]) {
          cp_async_16_cg(dst, ssrc[k] + kc0 / 8);
        } else {
          // read by the other lanes after the stage's __syncwarp, like the copies
          const uint8_t* src = ssrc[k] + kc0 / 8;
          uint32_t wv[4];
#pragma unroll
          for (int b = 0; b < 4; ++b)
            wv[b] = static_cast<uint32_t>(__ldg(src + 4 * b)) |
                    (static_cast<uint32_t>(__ldg(src + 4 * b + 1)) << 8) |
                    (static_cast<uint32_t>(__ldg(src + 4 * b + 2)) << 16) |
                    (static_cast<uint32_t>(__ldg(src + 4 * b + 3)) << 24);
          asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(wv[0]),
                       "r"(wv[1]), "r"(wv[2]), "r"(wv[3])
                       : "memory");
        }
      }
#pragma unroll
      for (int k = 0; k < 4 * NT; ++k) {
        const int r = 2 * k + cr;
        if (xsrc[k] != nullptr)
          cp_async_16_x(st + kXOff + 16u * (r * 16 + (cw ^ ((r & 1) << 2))), xsrc[k] + kc0);
      }
    }
  };
  auto issue = [&](int s, int64_t sc) {
    issue_w(s, sc);
    issue_sx(s, sc);
    cp_async_commit();  // one group per stage, empty past the end
  };

  // Prologue.  With w_ahead the W rows of stages 0..D-2 are already in
  // flight as D-1 commit groups of their own (issued by mixed_issue_w before
  // the kernel waited for the previous one); their sign words and x follow
  // as D-1 more groups.  Iteration i of the loop below commits one group and
  // then waits until at most D-1 are pending: for i < D-1 that leaves only
  // groups newer than stage i's signs and x, later only groups newer than
  // stage i, so stage i has landed either way.
  int64_t next = half * kKW + warp;
#pragma unroll
  for (int s = 0; s < D - 1; ++s) {
    if (w_ahead) {
      issue_sx(s, next);
      cp_async_commit();
    } else {
      issue(s, next);
    }
    next += kStep;
  }
  int s_rd = 0;
  for (int64_t sc = half * kKW + warp; sc < n_sc; sc += kStep) {
    __syncwarp();  // every lane is done reading the slot refilled next
    issue(s_rd == 0 ? D - 1 : s_rd - 1, next);
    next += kStep;
    cp_async_wait<D - 1>();
    __syncwarp();
    const uint8_t* st = wring + s_rd * kSB;
    // No selects on the fragment reads: a W row past d_out, an empty token
    // slot or a variant slot past nv holds whatever the ring held, and feeds
    // only products of that row, token or slot, which are never stored.
    uint4 sw[V][2];
#pragma unroll
    for (int v = 0; v < V; ++v)
#pragma unroll
      for (int h = 0; h < 2; ++h)
        sw[v][h] = *reinterpret_cast<const uint4*>(st + kSOff + 16 * (v * R + 8 * h + g));
#pragma unroll
    for (int j = 0; j < CPS; ++j) {
      uint4 wv[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int r = 8 * h + g;
        wv[h] = *reinterpret_cast<const uint4*>(st + 16 * (r * 16 + ((4 * j + t) ^ ((r & 1) << 2))));
      }
      uint4 xv[NT];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const int r = 8 * nt + g;
        xv[nt] = *reinterpret_cast<const uint4*>(
            st + kXOff + 16 * (r * 16 + ((4 * j + t) ^ ((r & 1) << 2))));
      }
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        mma_16816(acc_b[nt], wv[0].x, wv[1].x, wv[0].y, wv[1].y, xv[nt].x, xv[nt].y);
        mma_16816(acc_b[nt], wv[0].z, wv[1].z, wv[0].w, wv[1].w, xv[nt].z, xv[nt].w);
      }
#pragma unroll
      for (int v = 0; v < V; ++v) {
        if (v < nv) {
          const uint32_t w0 = j == 0 ? sw[v][0].x : j == 1 ? sw[v][0].y : j == 2 ? sw[v][0].z : sw[v][0].w;
          const uint32_t w1 = j == 0 ? sw[v][1].x : j == 1 ? sw[v][1].y : j == 2 ? sw[v][1].z : sw[v][1].w;
          const uint32_t b0 = (w0 >> (8 * t)) & 0xFFu, b1 = (w1 >> (8 * t)) & 0xFFu;
          uint32_t s0[4], s1[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            s0[i] = pm_one_pair(b0, i);
            s1[i] = pm_one_pair(b1, i);
          }
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            mma_16816(acc_s[v][nt], s0[0], s1[0], s0[1], s1[1], xv[nt].x, xv[nt].y);
            mma_16816(acc_s[v][nt], s0[2], s1[2], s0[3], s1[3], xv[nt].z, xv[nt].w);
          }
        }
      }
    }
    s_rd = s_rd == D - 1 ? 0 : s_rd + 1;
  }
  cp_async_wait<0>();

  // y_part = acc_b + α_v[n]·acc_s[v], v the token's own variant (fragment
  // rows: W rows n0+g, n0+8+g; columns: tokens 8nt + 2t, 8nt + 2t + 1).
  // Each warp leaves its part at the head of its own ring, which it has
  // finished reading and has no copy in flight to; no separate reduction
  // buffer keeps the CTA small enough for four per SM with two stages.
  __syncwarp();  // every lane has read its last stage and seen its copies land
  float* red = reinterpret_cast<float*>(wring);
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int m = 8 * nt + 2 * t + (e & 1);
      const int64_t n = n0 + g + 8 * (e >> 1);
      const int mv = grp.slot_var[m];
      float sv = 0.f;
#pragma unroll
      for (int v = 0; v < V; ++v)
        if (v == mv) sv = acc_s[v][nt][e];
      float val = acc_b[nt][e];
      if (mv >= 0 && n < d_out) {
        const float* al = p.alpha_table[grp.vars[mv] - 1];
        val = fmaf(p.per_row ? __ldg(al + n) : __ldg(al), sv, val);
      }
      red[(nt * 4 + e) * 32 + lane] = val;
    }
  }
  __syncthreads();
  // the kKW warps' parts summed in warp order, as store_group_rows_t does;
  // kSplit: CTA 1 hands its sums to CTA 0, which adds them after its own
  float v[NT][4];
  if (warp == 0) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float a = 0.f;
        for (int w = 0; w < kKW; ++w)
          a += reinterpret_cast<const float*>(ring + static_cast<size_t>(w) * D * kSB)
              [(nt * 4 + e) * 32 + lane];
        v[nt][e] = a;
        if (kSplit && half == 1) pair_store_f32(xfer + (nt * 4 + e) * 32 + lane, 0, a);
      }
    }
  }
  if constexpr (kSplit) pair_sync();  // CTA 1's sums are in CTA 0's xfer
  if (warp == 0 && half == 0) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float a = kSplit ? v[nt][e] + xfer[(nt * 4 + e) * 32 + lane] : v[nt][e];
        const int64_t n = n0 + g + 8 * (e >> 1);
        const int row = grp.rows[8 * nt + 2 * t + (e & 1)];
        if (row < 0 || n >= d_out) continue;
        p.y[static_cast<int64_t>(row) * d_out + n] =
            static_cast<uint16_t>(pack_bf16x2_rn(a, 0.f) & 0xFFFFu);
      }
    }
  }
  // the rings are refilled by the next group (and, kSplit, CTA 0 is done
  // with xfer before CTA 1 writes it again)
  if constexpr (kSplit)
    pair_sync();
  else
    __syncthreads();
}

// The short rows of a grouped call (segments of at most max_short rows),
// bucketed by variant in this CTA's shared memory: dyn holds [n_var+2] bucket
// counts, [n_var+2] bucket starts and the row list; rows
// [start[v], start[v+1]) of the list belong to variant v (0 = base).  The
// whole table is validated first: offsets non-decreasing inside [0, M], ids
// inside [0, n_var].  One bad entry rejects the table (the error word records
// it, no row is computed and false is returned to every thread), so segments
// never overlap and the list never exceeds its bound.  Called by all threads.
__device__ bool bucket_short_rows(const GemvArgs& p, int32_t* dyn) {
  const int nb = p.n_var + 1;
  int32_t* cnt = dyn;
  int32_t* start = dyn + (nb + 1);
  int32_t* rows = dyn + 2 * (nb + 1);
  for (int i = threadIdx.x; i < nb + 1; i += blockDim.x) cnt[i] = 0;
  __syncthreads();
  int bad_local = 0;
  for (int s = threadIdx.x; s < p.n_seg; s += blockDim.x) {
    const int32_t a = __ldg(p.seg_off + s), b = __ldg(p.seg_off + s + 1);
    const int32_t v = __ldg(p.seg_var + s);
    bad_local |= (a < 0 || b < a || b > p.M || v < 0 || v > p.n_var) ? 1 : 0;
  }
  if (__syncthreads_or(bad_local)) {
    if (blockIdx.x == 0 && threadIdx.x == 0) record_error(p.ctx, kErrBounds);
    return false;
  }
  // pass 1: count short-segment rows per variant
  for (int s = threadIdx.x; s < p.n_seg; s += blockDim.x) {
    const int32_t a = __ldg(p.seg_off + s), b = __ldg(p.seg_off + s + 1);
    const int32_t v = __ldg(p.seg_var + s);
    if (b - a > 0 && b - a <= p.max_short) atomicAdd(&cnt[v], b - a);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int32_t acc = 0;
    for (int v = 0; v < nb; ++v) {
      start[v] = acc;
      acc += cnt[v];
      cnt[v] = 0;  // reused as fill cursor
    }
    start[nb] = acc;
  }
  __syncthreads();
  // pass 2: scatter row indices into their bucket
  for (int s = threadIdx.x; s < p.n_seg; s += blockDim.x) {
    const int32_t a = __ldg(p.seg_off + s), b = __ldg(p.seg_off + s + 1);
    const int32_t v = __ldg(p.seg_var + s);
    if (b - a <= 0 || b - a > p.max_short) continue;
    const int32_t pos = start[v] + atomicAdd(&cnt[v], b - a);
    for (int32_t r = a; r < b; ++r) rows[pos + (r - a)] = r;
  }
  __syncthreads();
  return true;
}

// The W_base rows of this warp's first D-1 ring stages for the first group
// of gemv_group_mixed_async (same slots and copy mapping), one commit group
// per stage.  W_base is never the output of a kernel still in flight, so
// this runs before the grouped kernel waits for the previous kernel.
template <int NT, int V, int D, bool kSplit>
__device__ __forceinline__ void mixed_issue_w(const GemvArgs& p, uint8_t* ring) {
  constexpr int R = kStageRows;
  constexpr int kSB = mixed_stage_bytes<NT, V>();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int cr = lane >> 4, cw = lane & 15;
  const int64_t d_in = p.d_in;
  const int half = kSplit ? static_cast<int>(pair_rank()) : 0;
  constexpr int kStep = kSplit ? 2 * kKW : kKW;
  const int64_t n0 = static_cast<int64_t>(kSplit ? blockIdx.x >> 1 : blockIdx.x) * R;
  const int64_t rows_here = p.d_out - n0 < R ? p.d_out - n0 : R;
  const int64_t n_sc = d_in / (32 * kCPS);
  const uint32_t wring_sa = smem_addr(ring + static_cast<size_t>(warp) * D * kSB);
  const uint16_t* const wsrc0 = p.w + (n0 + cr) * d_in + 8 * cw;
#pragma unroll
  for (int s = 0; s < D - 1; ++s) {
    const int64_t sc = half * kKW + warp + static_cast<int64_t>(s) * kStep;
    if (sc < n_sc) {
      const int64_t kc0 = sc * 32 * kCPS;
      const uint32_t st = wring_sa + s * kSB;
#pragma unroll
      for (int k = 0; k < R / 2; ++k) {
        const int r = 2 * k + cr;
        if (r < rows_here)
          cp_async_16_cg(st + 16u * (r * 16 + (cw ^ ((r & 1) << 2))), wsrc0 + 2 * k * d_in + kc0);
      }
    }
    cp_async_commit();
  }
}

// Multi-tenant: rows of short segments, bucketed by variant, then taken in
// groups of up to 16 rows of up to kMaxGroupVars delta variants.  Every CTA
// builds the same grouping in shared memory, then covers its 8·NG output
// columns for every group.
// One token tile with a two-stage ring: four CTAs per SM, so at most 128
// registers per thread.
// kSplit (ring pass only): launched in clusters of two CTAs that share a row
// block and split d_in (see gemv_group_mixed_async).
template <int NG, int kAsyncNT, int V, int D, bool kSplit = false>
__global__ void __launch_bounds__(kKW * 32, (kAsyncNT == 1 && D == 2) ? 4 : 1)
    gemv_grouped_kernel(GemvArgs p, int ring_off) {
  // the ring pass reduces through its ring; only the register pass needs this
  __shared__ float red[kAsyncNT > 0 ? 1 : kKW * NG * 4 * 32];
  // kSplit: CTA 1's sums, written into CTA 0's copy of this array
  __shared__ float xfer[kSplit ? (kAsyncNT > 0 ? kAsyncNT : 1) * 4 * 32 : 1];
  extern __shared__ __align__(16) int32_t dyn[];
  griddep_launch_dependents();
  if constexpr (kAsyncNT > 0)
    mixed_issue_w<kAsyncNT, V, D, kSplit>(p, reinterpret_cast<uint8_t*>(dyn) + ring_off);
  griddep_wait();
  if (!bucket_short_rows(p, dyn)) {
    cp_async_wait<0>();  // no copy may land after the CTA has left
    return;
  }
  const int nb = p.n_var + 1;
  const int32_t* start = dyn + (nb + 1);
  const int32_t* rows = dyn + 2 * (nb + 1);
  // Groups of up to 16 rows taken in bucket (variant) order, closed early
  // when a fifth delta variant would join: each group is one pass over this
  // CTA's W_base rows.  Thread 0 forms the next group in shared memory.
  __shared__ MixedGroup mg;
  __shared__ int32_t cursor, bucket;
  __shared__ int mg_vec;
  const int32_t total = start[nb];
  if (threadIdx.x == 0) {
    cursor = 0;
    bucket = 0;
  }
  __syncthreads();
  bool first = true;  // the first group (its W rows are in flight already)
  while (cursor < total) {
    if (threadIdx.x == 0) {
      int i = 0, nvars = 0;
      int32_t c = cursor, bk = bucket;
      bool vec = p.d_in % 128 == 0;
      while (i < kMaxGroupRows && c < total) {
        while (c >= start[bk + 1]) ++bk;  // the bucket (variant) of sorted row c
        int slot = -1;
        if (bk > 0) {
          if (nvars == 0 || mg.vars[nvars - 1] != bk) {
            if (nvars == V) break;
            mg.vars[nvars++] = bk;
            vec = vec && (reinterpret_cast<uintptr_t>(p.packed_table[bk - 1]) & 15u) == 0;
          }
          slot = nvars - 1;
        }
        mg.rows[i] = rows[c];
        mg.slot_var[i] = slot;
        ++i;
        ++c;
      }
      for (; i < kMaxGroupRows; ++i) {
        mg.rows[i] = -1;
        mg.slot_var[i] = -1;
      }
      mg.n_vars = nvars;
      mg_vec = vec ? 1 : 0;
      cursor = c;
      bucket = bk;
    }
    __syncthreads();
    if constexpr (kAsyncNT > 0) {
      // the ring (d_in % 128 == 0): unaligned variant tables included; the
      // first group's W rows were issued before the dependency wait
      gemv_group_mixed_async<kAsyncNT, V, D, kSplit>(
          p, mg, reinterpret_cast<uint8_t*>(dyn) + ring_off, first, xfer);
      first = false;
    } else {
      if (mg_vec)
        gemv_group_mixed<NG, true>(p, mg, red);
      else
        gemv_group_mixed<NG, false>(p, mg, red);
    }
  }
  cp_async_wait<0>();  // no short rows: the early W copies still land before exit
}

// ------------------------------------------------------------------ wide passes

// The short rows of a grouped call when there can be more of them than one
// group holds: up to kWideTok rows of up to kWideVars delta variants (and any
// number of base rows) in ONE pass over the CTA's 16 W_base rows, instead of
// one pass per group of 16 rows and 4 variants.  y = x·W_baseᵀ + α_v ⊙
// (x·S_vᵀ), the two products in separate accumulators over all of d_in and α
// applied once at the end, as in the other decode kernels.  The base product
// runs over the pass's rows in dense groups of 8; the sign product per tile
// of at most 8 rows of ONE variant (the rows in bucket order; base rows have
// no tile), so no masking is needed.  The CTA shares one cp.async ring of
// 128-column stages, each holding the W_base row segments, the sign words of
// every variant of the pass and the x segments of every row; warp w owns
// groups and tiles w, w + W, ... (W warps) over all columns and reads each
// W_base fragment once for them.  At the end the base sums meet the sign
// products through shared memory.  The inner loop has no data-dependent
// branch, and lanes past a tile's rows compute on its first row.
// On 14336 x 4096 with 14 variants and 64 rows, where the legacy tensor path
// (mma.sync m16n8k16, measured at most ~600 TFLOP/s on this part) bounds the
// pass: 274 µs for groups of 16 rows and 4 variants; 158 µs for one pass with
// a base product per tile (tiles of ~4 rows, so half of each n8 product
// wasted, and a useless sign product on base tiles); 151 µs with the dense
// base groups (27% fewer MMAs).  Tracking the variant of the previous tile
// to skip a conversion, and predicated zero operands, each cost more issue
// slots than they saved (208 µs), and so did a tile loop with an exit on the
// warp's tile count (173 µs: the compiler cannot interleave tiles across the
// exits), hence one body per count; eight warps per CTA took 161 µs.
constexpr int kWideTok = 64;    // rows of x per pass (the ring's x segments)
constexpr int kWideTiles = 16;  // tiles of at most 8 rows of one variant per pass
#ifndef BD_WIDE_WARPS
#define BD_WIDE_WARPS 4
#endif
constexpr int kWideWarps = BD_WIDE_WARPS;  // warps of a CTA
constexpr int kWideThreads = 32 * kWideWarps;
constexpr int kWideTilesPerWarp = kWideTiles / kWideWarps;
constexpr int kWideVars = 16;   // delta variants per pass
#ifndef BD_WIDE_COLS
#define BD_WIDE_COLS 128
#endif
struct WidePass {
  int32_t rows[kWideTok];         // x/y row of the pass's row slot i, −1 = empty
  int32_t vars[kWideVars];        // the pass's delta variant ids (>= 1)
  int32_t tile_r0[kWideTiles];    // first row slot of the tile
  int32_t tile_n[kWideTiles];     // row slots of the tile (1..8; 0 = no tile)
  int32_t tile_var[kWideTiles];   // index into vars[] of the tile's variant, −1 = base
  int32_t n_tok, n_vars, n_tiles;
  int32_t n_base;      // the first n_base row slots are base-model rows (no tile)
  uint32_t unaligned;  // bit v: variant v's sign table is off the copy size (C/8 bytes)
};
// A ring stage of C columns (64 or 128): W_base row segments (16 × 2C
// bytes, swizzled), the sign segments of every variant ([variant][row] ×
// C/8 bytes), then the x segments of every row slot (64 × 2C bytes, swizzled).
template <int C>
__host__ __device__ constexpr int wide_s_off() { return 16 * 2 * C; }
template <int C>
__host__ __device__ constexpr int wide_x_off() { return wide_s_off<C>() + kWideVars * 16 * (C / 8); }
template <int C>
__host__ __device__ constexpr int wide_stage_bytes() { return wide_x_off<C>() + kWideTok * 2 * C; }
template <int C, int D>
constexpr size_t wide_ring_bytes() {
  return static_cast<size_t>(D) * wide_stage_bytes<C>();
}

// CTAs per SM the wide kernel is compiled for (registers per thread capped
// so that they fit): as many of four-warp CTAs as the ring leaves room for,
// three with the 72 KB ring of three 128-column stages.
template <int C, int D>
constexpr int wide_min_blocks() {
  const int by_smem = wide_ring_bytes<C, D>() <= 50 * 1024 ? 4 : 3;
  const int b = by_smem * 128 / kWideThreads;
  return b > 0 ? b : 1;
}

__device__ __forceinline__ uint4 lds128(const uint8_t* a) {
  return *reinterpret_cast<const uint4*>(a);
}

template <int C, int D>
__device__ __forceinline__ void gemv_wide_pass(const GemvArgs& p, const WidePass& wp,
                                               const float2 (&al_s)[kWideVars][8],
                                               uint8_t* ring, int64_t n0) {
  constexpr int R = 16;
  constexpr int TW = kWideTilesPerWarp;
  static_assert(C == 64 || C == 128, "stages of 64 or 128 columns");
  constexpr int WPR = C / 8;                 // 16-byte words per row segment
  constexpr int RPR = kWideThreads / WPR;    // row segments one round of the CTA's threads copies
  constexpr int SPR = kWideThreads;          // (variant, row) sign segments per round
  constexpr int SB = C / 8;             // sign bytes per row segment
  constexpr int kSOff = wide_s_off<C>(), kXOff = wide_x_off<C>(), kSB = wide_stage_bytes<C>();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int64_t d_in = p.d_in, d_out = p.d_out;
  const int64_t row_bytes = d_in / 8;
  const int64_t rows_here = d_out - n0 < R ? d_out - n0 : R;
  const int n_tok = wp.n_tok, nv = wp.n_vars;
  const uint32_t ring_sa = smem_addr(ring);
  const uint4 zero4 = make_uint4(0u, 0u, 0u, 0u);

  // copy side: thread T moves word T % WPR of W rows T / WPR + RPR·k, the
  // sign segment of (variant, row) pairs T + SPR·k, and word T % WPR of row
  // slots T / WPR + RPR·k
  constexpr int kSK = kWideVars * 16 / SPR;
  const int cw = tid % WPR, cr = tid / WPR;
  const uint8_t* ssrc[kSK];
  bool s_al[kSK];
#pragma unroll
  for (int k = 0; k < kSK; ++k) {
    const int i = tid + SPR * k, v = i >> 4, r = i & 15;
    ssrc[k] = (v < nv && r < rows_here) ? p.packed_table[wp.vars[v] - 1] + (n0 + r) * row_bytes
                                        : nullptr;
    s_al[k] = v < nv && ((wp.unaligned >> v) & 1u) == 0;
  }
  int32_t xrow[kWideTok / RPR];
#pragma unroll
  for (int k = 0; k < kWideTok / RPR; ++k) {
    const int slot = cr + RPR * k;
    xrow[k] = slot < n_tok ? wp.rows[slot] : -1;
  }
  const int64_t n_sc = d_in / C;
  auto issue = [&](int s, int64_t sc) {
    if (sc < n_sc) {
      const int64_t kc0 = sc * C;
      const uint32_t st = ring_sa + s * kSB;
#pragma unroll
      for (int k = 0; k < R / RPR; ++k) {
        const int r = cr + RPR * k;
        if (r < rows_here)
          cp_async_16_cg(st + 16u * (r * WPR + (cw ^ ((r & 1) << 2))),
                         p.w + (n0 + r) * d_in + kc0 + 8 * cw);
      }
#pragma unroll
      for (int k = 0; k < kSK; ++k) {
        if (ssrc[k] == nullptr) continue;
        const uint32_t dst = st + kSOff + SB * (tid + SPR * k);
        const uint8_t* src = ssrc[k] + kc0 / 8;
        if (s_al[k]) {
          if constexpr (SB == 16)
            cp_async_16_cg(dst, src);
          else
            asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(dst), "l"(src)
                         : "memory");
        } else {
          // read by the other warps after the stage's barrier, like the copies
          uint32_t w4[4];
#pragma unroll
          for (int b = 0; b < SB / 4; ++b)
            w4[b] = static_cast<uint32_t>(__ldg(src + 4 * b)) |
                    (static_cast<uint32_t>(__ldg(src + 4 * b + 1)) << 8) |
                    (static_cast<uint32_t>(__ldg(src + 4 * b + 2)) << 16) |
                    (static_cast<uint32_t>(__ldg(src + 4 * b + 3)) << 24);
          if constexpr (SB == 16)
            asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(w4[0]),
                         "r"(w4[1]), "r"(w4[2]), "r"(w4[3])
                         : "memory");
          else
            asm volatile("st.shared.v2.u32 [%0], {%1, %2};" ::"r"(dst), "r"(w4[0]), "r"(w4[1])
                         : "memory");
        }
      }
#pragma unroll
      for (int k = 0; k < kWideTok / RPR; ++k) {
        const int slot = cr + RPR * k;
        if (xrow[k] >= 0)
          cp_async_16_x(st + kXOff + 16u * (slot * WPR + (cw ^ ((slot & 1) << 2))),
                        p.x + static_cast<int64_t>(xrow[k]) * d_in + kc0 + 8 * cw);
      }
    }
    cp_async_commit();  // one group per stage, empty past the end
  };

  // compute side.  Base products over the pass's row slots in groups of 8
  // (group q: slots 8q .. 8q+7), warp w owning groups w, w + W (W warps);
  // sign products per tile of one delta variant (base rows have none), warp
  // w owning tiles w, w + W, ....  Groups and tiles are numbered densely, so
  // a warp's are a prefix of its list.  The lane's B column is slot 8q + g
  // (group) or r0 + g (tile; lanes past a tile's rows read its first row,
  // and their columns of the products are never stored); W rows past d_out
  // and empty slots hold whatever the ring held, and feed only products
  // that are never stored, so no fragment read needs a select.
  constexpr int GW = kWideTok / 8 / kWideWarps;  // groups per warp
  int goff[GW], gpar[GW];
  int my_groups = 0;
#pragma unroll
  for (int q = 0; q < GW; ++q) {
    const int grp = warp + kWideWarps * q;
    const int xs = 8 * grp + g;
    goff[q] = kXOff + 16 * (xs * WPR + t);
    gpar[q] = (xs & 1) << 6;
    my_groups += 8 * grp < n_tok ? 1 : 0;
  }
  int tvar[TW], xoff[TW], xpar[TW], soff[TW];
  int my_tiles = 0;
#pragma unroll
  for (int k = 0; k < TW; ++k) {
    const int kt = warp + kWideWarps * k;
    const int n = wp.tile_n[kt];
    my_tiles += n > 0 ? 1 : 0;
    tvar[k] = wp.tile_var[kt];
    const int xs = wp.tile_r0[kt] + (g < n ? g : 0);
    xoff[k] = kXOff + 16 * (xs * WPR + t);
    xpar[k] = (xs & 1) << 6;
    const int vs = tvar[k] > 0 ? tvar[k] : 0;
    soff[k] = kSOff + SB * (vs * 16 + g) + t;
  }
  const int w_off0 = 16 * (g * WPR + t), w_off1 = 16 * ((g + 8) * WPR + t);
  const int wpar = (g & 1) << 6;
  float acc_b[GW][4], acc_s[TW][4];
#pragma unroll
  for (int q = 0; q < GW; ++q)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc_b[q][e] = 0.f;
#pragma unroll
  for (int k = 0; k < TW; ++k)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc_s[k][e] = 0.f;

#pragma unroll
  for (int s = 0; s < D - 1; ++s) issue(s, s);
  int slot = 0;
  for (int64_t sc = 0; sc < n_sc; ++sc) {
    cp_async_wait<D - 2>();  // this thread's copies of stage sc have landed
    __syncthreads();         // ... everyone's; and the slot refilled next is free
    issue(slot == 0 ? D - 1 : slot - 1, sc + D - 1);
    const uint8_t* st = ring + slot * kSB;
    // The stage's products for this warp's first NGR groups and NTK tiles,
    // both known at compile time: one straight-line block the compiler can
    // interleave (a loop with an exit on a count cannot be).
    auto stage = [&](auto ngr, auto ntk) {
      constexpr int NGR = decltype(ngr)::value, NTK = decltype(ntk)::value;
#pragma unroll
      for (int j = 0; j < C / 32; ++j) {  // 32-column chunks: word 4j + t of a row
        const uint4 wv0 = lds128(st + w_off0 + ((64 * j) ^ wpar));
        const uint4 wv1 = lds128(st + w_off1 + ((64 * j) ^ wpar));
#pragma unroll
        for (int q = 0; q < NGR; ++q) {
          const uint4 xv = lds128(st + goff[q] + ((64 * j) ^ gpar[q]));
          mma_16816(acc_b[q], wv0.x, wv1.x, wv0.y, wv1.y, xv.x, xv.y);
          mma_16816(acc_b[q], wv0.z, wv1.z, wv0.w, wv1.w, xv.z, xv.w);
        }
#pragma unroll
        for (int k = 0; k < NTK; ++k) {
          const uint4 xv = lds128(st + xoff[k] + ((64 * j) ^ xpar[k]));
          const uint32_t b0 = st[soff[k] + 4 * j];
          const uint32_t b1 = st[soff[k] + 8 * SB + 4 * j];
          uint32_t s0[4], s1[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            s0[i] = pm_one_pair(b0, i);
            s1[i] = pm_one_pair(b1, i);
          }
          mma_16816(acc_s[k], s0[0], s1[0], s0[1], s1[1], xv.x, xv.y);
          mma_16816(acc_s[k], s0[2], s1[2], s0[3], s1[3], xv.z, xv.w);
        }
      }
    };
    static_assert(TW <= 4 && GW <= 2, "stage bodies for 0..4 tiles and 0..2 groups per warp");
    auto tiles = [&](auto ngr) {
      if (TW >= 4 && my_tiles >= 4)
        stage(ngr, std::integral_constant<int, (TW >= 4 ? 4 : 0)>{});
      else if (TW >= 3 && my_tiles == 3)
        stage(ngr, std::integral_constant<int, (TW >= 3 ? 3 : 0)>{});
      else if (TW >= 2 && my_tiles == 2)
        stage(ngr, std::integral_constant<int, (TW >= 2 ? 2 : 0)>{});
      else if (my_tiles == 1)
        stage(ngr, std::integral_constant<int, 1>{});
      else
        stage(ngr, std::integral_constant<int, 0>{});
    };
    if (GW >= 2 && my_groups >= 2)
      tiles(std::integral_constant<int, (GW >= 2 ? 2 : 0)>{});
    else if (my_groups == 1)
      tiles(std::integral_constant<int, 1>{});
    else
      tiles(std::integral_constant<int, 0>{});
    slot = slot == D - 1 ? 0 : slot + 1;
  }
  cp_async_wait<0>();
  __syncthreads();  // every warp is done with the ring, which now takes the base sums

  // Base sums of every slot through shared memory: bsum[r][slot] for the
  // CTA's W row r (fragment rows g, g + 8; columns 2t, 2t + 1 of a group).
  constexpr int kBS = kWideTok + 1;  // row stride (floats)
  float* bsum = reinterpret_cast<float*>(ring);
#pragma unroll
  for (int q = 0; q < GW; ++q) {
    if (q >= my_groups) continue;
    const int grp = warp + kWideWarps * q;
#pragma unroll
    for (int e = 0; e < 4; ++e)
      bsum[(g + 8 * (e >> 1)) * kBS + 8 * grp + 2 * t + (e & 1)] = acc_b[q][e];
  }
  __syncthreads();
  // delta rows: y = base + α_v[n]·(x·S_vᵀ); base rows (the pass's first
  // n_base slots): y = base
#pragma unroll
  for (int k = 0; k < TW; ++k) {
    if (k >= my_tiles) continue;
    const int kt = warp + kWideWarps * k;
    const int n_rows = wp.tile_n[kt], r0 = wp.tile_r0[kt];
    const float2 al = al_s[tvar[k]][g];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int c = 2 * t + (e & 1);
      const int r = g + 8 * (e >> 1);
      const int64_t n = n0 + r;
      if (c >= n_rows || n >= d_out) continue;
      const float v = fmaf((e >> 1) ? al.y : al.x, acc_s[k][e], bsum[r * kBS + r0 + c]);
      p.y[static_cast<int64_t>(wp.rows[r0 + c]) * d_out + n] =
          static_cast<uint16_t>(pack_bf16x2_rn(v, 0.f) & 0xFFFFu);
    }
  }
  for (int i = tid; i < wp.n_base * R; i += kWideThreads) {
    const int s = i / R, r = i - s * R;
    if (r >= rows_here) continue;
    p.y[static_cast<int64_t>(wp.rows[s]) * d_out + n0 + r] =
        static_cast<uint16_t>(pack_bf16x2_rn(bsum[r * kBS + s], 0.f) & 0xFFFFu);
  }
  __syncthreads();  // the ring and the pass tables are reused by the next pass
}

// The next pass from the bucketed row list (run by one thread): rows in
// bucket (variant) order take the pass's row slots; base rows (bucket 0)
// first, without tiles, then each delta variant's rows cut into tiles of at
// most 8 rows of that variant.  The pass closes when it holds kWideTok rows
// or kWideTiles tiles, or when a (kWideVars+1)-th delta variant would join.
// A variant whose sign table does not start on a `copy_bytes` boundary is
// flagged in wp.unaligned (its signs are then fetched with plain loads).
__device__ void form_wide_pass(const GemvArgs& p, const int32_t* start, const int32_t* rows,
                               int32_t total, int copy_bytes, int32_t& cursor, int32_t& bucket,
                               WidePass& wp) {
  int n = 0, nvars = 0, ntl = 0, n_base = 0;
  uint32_t unal = 0;
  int32_t c = cursor, bk = bucket;
  while (c < total && n < kWideTok && ntl < kWideTiles) {
    while (c >= start[bk + 1]) ++bk;  // the bucket (variant) of sorted row c
    const int32_t end = start[bk + 1];
    if (bk == 0) {  // base rows (bucket 0, so a pass's first slots): no tile
      while (c < end && n < kWideTok) {
        wp.rows[n++] = rows[c++];
        ++n_base;
      }
      continue;
    }
    if (nvars == kWideVars) break;
    const int vslot = nvars;
    wp.vars[nvars] = bk;
    if ((reinterpret_cast<uintptr_t>(p.packed_table[bk - 1]) & (copy_bytes - 1)) != 0)
      unal |= 1u << nvars;
    ++nvars;
    while (c < end && n < kWideTok && ntl < kWideTiles) {
      int32_t cnt = end - c;
      cnt = cnt < 8 ? cnt : 8;
      cnt = cnt < kWideTok - n ? cnt : kWideTok - n;
      wp.tile_r0[ntl] = n;
      wp.tile_n[ntl] = cnt;
      wp.tile_var[ntl] = vslot;
      ++ntl;
      for (int32_t i = 0; i < cnt; ++i) wp.rows[n++] = rows[c++];
    }
  }
  for (int i = n; i < kWideTok; ++i) wp.rows[i] = -1;
  for (int k = ntl; k < kWideTiles; ++k) {
    wp.tile_r0[k] = 0;
    wp.tile_n[k] = 0;
    wp.tile_var[k] = -1;
  }
  wp.n_tok = n;
  wp.n_vars = nvars;
  wp.n_tiles = ntl;
  wp.n_base = n_base;
  wp.unaligned = unal;
  cursor = c;
  bucket = bk;
}

// Requires d_in % 128 == 0.  One CTA per 16 W_base rows; every CTA buckets
// the short rows (as the grouped kernel does), then runs the passes: thread 0
// cuts the rows, in bucket order, into tiles of at most 8 rows of one
// variant, closing the pass when it holds kWideTok rows or kWideTiles tiles,
// or when a (kWideVars+1)-th delta variant would join.
template <int C, int D>
__global__ void __launch_bounds__(kWideThreads, wide_min_blocks<C, D>())
    gemv_wide_kernel(GemvArgs p, int ring_off) {
  extern __shared__ __align__(16) int32_t dyn[];
  __shared__ WidePass wp;
  __shared__ float2 al_s[kWideVars][8];  // α of the pass's variants: rows n0+g, n0+8+g
  __shared__ int32_t cursor, bucket;
  griddep_launch_dependents();
  griddep_wait();
  if (!bucket_short_rows(p, dyn)) return;
  const int nb = p.n_var + 1;
  const int32_t* start = dyn + (nb + 1);
  const int32_t* rows = dyn + 2 * (nb + 1);
  const int32_t total = start[nb];
  uint8_t* ring = reinterpret_cast<uint8_t*>(dyn) + ring_off;
  const int64_t n0 = static_cast<int64_t>(blockIdx.x) * 16;
  if (threadIdx.x == 0) {
    cursor = 0;
    bucket = 0;
  }
  __syncthreads();
  while (cursor < total) {
    if (threadIdx.x == 0) form_wide_pass(p, start, rows, total, C / 8, cursor, bucket, wp);
    __syncthreads();
    for (int i = threadIdx.x; i < wp.n_vars * 16; i += blockDim.x) {
      const int v = i >> 4, r = i & 15;
      const int64_t n = n0 + r;
      const float* a = p.alpha_table[wp.vars[v] - 1];
      const float val = n < p.d_out ? (p.per_row ? __ldg(a + n) : __ldg(a)) : 0.f;
      if (r < 8)
        al_s[v][r].x = val;
      else
        al_s[v][r - 8].y = val;
    }
    __syncthreads();
    gemv_wide_pass<C, D>(p, wp, al_s, ring, n0);
  }
}

// The ring kernel takes M <= 8, and M = 9..16 (two token tiles) when the
// grid is one wave at two CTAs per SM: there it beats the register kernel
// (4096 x 4096: 9.3 / 10.0 µs against 10.1 / 10.2 at M = 12 / 16), while on
// multi-wave grids the two tiles' x copies cost it more than it gains
// (57344 x 8192 at M = 16: 218 against 204 µs).
template <int NG>
cudaError_t launch_single(const GemvArgs& p, bool sign_vec, int num_sms, cudaStream_t stream) {
  const int64_t n_blocks = (p.d_out + 8 * NG - 1) / (8 * NG);
  const int64_t n_chunks = (p.M + kMaxGroupRows - 1) / kMaxGroupRows;
  dim3 grid(static_cast<unsigned>(n_blocks),
            static_cast<unsigned>(n_chunks < 65535 ? n_chunks : 65535));
  const bool m16 = p.M > 8;
  const dim3 block(kKW * 32);
  const bool one_wave = n_blocks <= 2 * static_cast<int64_t>(num_sms);
  const int64_t ring_max_m = one_wave ? kMaxGroupRows : BD_GEMV_ASYNC_MAX_M;
  if (sign_vec && p.M <= ring_max_m) {
    // The ring needs more than the default 48 KB of dynamic shared memory:
    // raise the limit once per device (outside any capture in practice: the
    // first call on a device).
    static bool attr_set[64][2] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    const size_t smem = m16 ? gemv_ring_bytes<2>() : gemv_ring_bytes<1>();
    std::lock_guard<std::mutex> lock(host_cache_mutex());
    if (!attr_set[dev][m16 ? 1 : 0]) {
      e = cudaFuncSetAttribute(m16 ? gemv_single_async_kernel<NG, true>
                                   : gemv_single_async_kernel<NG, false>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(smem));
      if (e != cudaSuccess) return e;
      attr_set[dev][m16 ? 1 : 0] = true;
    }
    if (m16) return launch_pdl(gemv_single_async_kernel<NG, true>, grid, block, smem, stream, p);
    return launch_pdl(gemv_single_async_kernel<NG, false>, grid, block, smem, stream, p);
  }
  if (m16 && sign_vec)
    return launch_pdl(gemv_single_kernel<NG, true, true>, grid, block, 0, stream, p);
  if (m16) return launch_pdl(gemv_single_kernel<NG, true, false>, grid, block, 0, stream, p);
  if (sign_vec) return launch_pdl(gemv_single_kernel<NG, false, true>, grid, block, 0, stream, p);
  return launch_pdl(gemv_single_kernel<NG, false, false>, grid, block, 0, stream, p);
}

}  // namespace

size_t gemv_grouped_smem_bytes(int32_t n_var, int64_t max_rows) {
  return sizeof(int32_t) * (2 * (static_cast<size_t>(n_var) + 2) + static_cast<size_t>(max_rows));
}

cudaError_t launch_gemv(const GemvArgs& p, int num_sms, cudaStream_t stream) {
  const bool sign_vec = (p.d_in % 128 == 0) &&
                        (reinterpret_cast<uintptr_t>(p.packed) % 16 == 0);
  return launch_single<kNG>(p, sign_vec, num_sms, stream);
}

template <int NT, int V, int D, bool kSplit = false>
cudaError_t launch_grouped_instance(const GemvArgs& p, size_t smem, int ring_off, dim3 grid,
                                    cudaStream_t stream) {
  // Raise the dynamic shared-memory limit only when a call needs more than
  // any earlier call on this device (so captured calls make no attribute call).
  static size_t smem_set[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  {
    std::lock_guard<std::mutex> lock(host_cache_mutex());
    if (smem > 48 * 1024 && smem > smem_set[dev]) {
      e = cudaFuncSetAttribute(gemv_grouped_kernel<kNG, NT, V, D, kSplit>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(smem));
      if (e != cudaSuccess) return e;
      smem_set[dev] = smem;
    }
  }
  if constexpr (kSplit) {
    // clusters of two CTAs (one row block each pair), with programmatic
    // dependent launch as the others
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * grid.x);
    cfg.blockDim = dim3(kKW * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = 2;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    const cudaError_t le =
        cudaLaunchKernelEx(&cfg, gemv_grouped_kernel<kNG, NT, V, D, true>, p, ring_off);
    if (le == cudaSuccess) return le;
    // a device that cannot place the clusters: nothing was launched; the
    // unsplit grid computes the same rows
    (void)cudaGetLastError();
    return launch_grouped_instance<NT, V, D, false>(p, smem, ring_off, grid, stream);
  } else {
    return launch_pdl(gemv_grouped_kernel<kNG, NT, V, D>, grid, dim3(kKW * 32), smem, stream, p,
                      ring_off);
  }
}

template <int C, int D>
cudaError_t launch_wide_instance(const GemvArgs& p, size_t smem, int ring_off, dim3 grid,
                                 cudaStream_t stream) {
  static size_t smem_set[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  {
    std::lock_guard<std::mutex> lock(host_cache_mutex());
    if (smem > 48 * 1024 && smem > smem_set[dev]) {
      e = cudaFuncSetAttribute(gemv_wide_kernel<C, D>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(smem));
      if (e != cudaSuccess) return e;
      smem_set[dev] = smem;
    }
  }
  return launch_pdl(gemv_wide_kernel<C, D>, grid, dim3(kWideThreads), smem, stream, p,
                    ring_off);
}

cudaError_t launch_gemv_grouped(const GemvArgs& p, int64_t max_rows, int num_sms,
                                cudaStream_t stream) {
  const size_t group_smem = gemv_grouped_smem_bytes(p.n_var, max_rows);
  const int64_t n_blocks = (p.d_out + 8 * kNG - 1) / (8 * kNG);
  const dim3 grid(static_cast<unsigned>(n_blocks));
  // The deep-queue pass (d_in % 128 == 0) with one token tile when no group
  // can hold more than 8 rows, else two; groups of at most two delta
  // variants when the call has no more (half the ring's sign slots, fewer
  // registers); a two-stage ring on grids of more than one wave at two CTAs
  // per SM (see mixed_ring_bytes).  The ring follows the grouping lists.
  const size_t ring_off = (group_smem + 15) / 16 * 16;
  const size_t kMaxDyn = 200 * 1024;
  const int ro = static_cast<int>(ring_off);
#ifndef BD_WIDE_STAGES
#define BD_WIDE_STAGES 3
#endif
  // More short rows than one group holds: the wide pass (all of them, up to
  // 64 rows and 16 variants per pass, in one pass over W_base).
  constexpr size_t kWideRing = wide_ring_bytes<BD_WIDE_COLS, BD_WIDE_STAGES>();
  if (p.d_in % 128 == 0 && max_rows > kMaxGroupRows && ring_off + kWideRing <= kMaxDyn)
    return launch_wide_instance<BD_WIDE_COLS, BD_WIDE_STAGES>(p, ring_off + kWideRing, ro, grid,
                                                               stream);
  if (p.d_in % 128 == 0) {
    const bool two = p.n_var <= 2;
    const bool shallow = n_blocks > 2 * static_cast<int64_t>(num_sms);
    // Row blocks split over d_in between the two CTAs of a cluster when that
    // evens out the per-SM load of a grid of a few waves, ceil(2b / SMs) / 2
    // against ceil(b / SMs) row blocks on the busiest SM (b = 512 on 152
    // SMs: 3.5 against 4), and each CTA keeps a long run of stages: on 8192
    // x 28672 (two variants, 8 rows) 99.8 -> 94.4 µs, while on 8192 x 8192
    // the half-length CTAs lost (32.7 -> 37.0 µs) and 10240 x 8192 gained
    // nothing.
    const int64_t sms = num_sms > 0 ? num_sms : 1;
    const int64_t per1 = (n_blocks + sms - 1) / sms, per2 = (2 * n_blocks + sms - 1) / sms;
    const bool split = per2 < 2 * per1 && per1 <= 8 && p.d_in >= 16384;
    if (max_rows <= 8) {
      if (two && shallow && split && ring_off + mixed_ring_bytes<1, 2, 2>() <= kMaxDyn)
        return launch_grouped_instance<1, 2, 2, true>(p, ring_off + mixed_ring_bytes<1, 2, 2>(),
                                                      ro, grid, stream);
      if (two && shallow && ring_off + mixed_ring_bytes<1, 2, 2>() <= kMaxDyn)
        return launch_grouped_instance<1, 2, 2>(p, ring_off + mixed_ring_bytes<1, 2, 2>(), ro,
                                                grid, stream);
      if (two && ring_off + mixed_ring_bytes<1, 2, 3>() <= kMaxDyn)
        return launch_grouped_instance<1, 2, 3>(p, ring_off + mixed_ring_bytes<1, 2, 3>(), ro,
                                                grid, stream);
      if (shallow && ring_off + mixed_ring_bytes<1, 4, 2>() <= kMaxDyn)
        return launch_grouped_instance<1, 4, 2>(p, ring_off + mixed_ring_bytes<1, 4, 2>(), ro,
                                                grid, stream);
      if (ring_off + mixed_ring_bytes<1, 4, 3>() <= kMaxDyn)
        return launch_grouped_instance<1, 4, 3>(p, ring_off + mixed_ring_bytes<1, 4, 3>(), ro,
                                                grid, stream);
    }
    if (two && ring_off + mixed_ring_bytes<2, 2, 2>() <= kMaxDyn)
      return launch_grouped_instance<2, 2, 2>(p, ring_off + mixed_ring_bytes<2, 2, 2>(), ro, grid,
                                              stream);
    if (ring_off + mixed_ring_bytes<2, 4, 2>() <= kMaxDyn)
      return launch_grouped_instance<2, 4, 2>(p, ring_off + mixed_ring_bytes<2, 4, 2>(), ro, grid,
                                              stream);
  }
  return launch_grouped_instance<0, kMaxGroupVars, 2>(p, group_smem, 0, grid, stream);
}

}  // namespace bd
