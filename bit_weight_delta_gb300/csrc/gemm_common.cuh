// gemm_common.cuh — pieces of the prefill kernel (CTA pairs, gemm_pair.cu):
// the tile schedule, the W_eff transform arithmetic, tensor-memory stores and
// loads, and the cluster forms of the tcgen05 and mbarrier primitives.
#pragma once

#include <cstdint>

#include "common.cuh"
#include "kernels.h"

namespace bd {
namespace gemm_detail {

struct Tile {
  int64_t n0;       // first output row (d_out) of the tile
  int64_t tok0;     // first token (x row) of the tile
  int64_t tok_end;  // rows [tok0, min(tok0 + BN, tok_end)) are outputs
  int32_t variant;  // 0 = base (no delta)
};

// Tile t of the flat schedule: t = nt * t_total + j, output rows
// [nt*BM, nt*BM + BM), token tile j.  Plain mode: token tiles of [0, M).
// Grouped mode: token tiles of each long segment in turn; `prefix` is the
// inclusive prefix sum of tiles per segment (prefix[0] = 0).
template <int BM, int BN>
__device__ __forceinline__ Tile tile_at(const GemmArgs& p, int64_t t, int64_t t_total,
                                        const int32_t* seg_off, const int32_t* seg_var,
                                        const int32_t* prefix) {
  Tile tl;
  const int64_t nt = t / t_total;
  const int64_t j = t - nt * t_total;
  tl.n0 = nt * BM;
  if (seg_off == nullptr) {
    tl.tok0 = j * BN;
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
    tl.tok0 = seg_off[lo] + (j - prefix[lo]) * BN;
    tl.tok_end = seg_off[lo + 1];
    tl.variant = seg_var[lo];
  }
  return tl;
}

// Grouped mode set-up, run by every thread of the CTA: copy the segment table
// to shared memory, validate it (one malformed entry rejects the whole table:
// no tiles at all, error word set), and build the prefix sum of token tiles
// (of BN rows) over the long segments.  Returns the total number of token
// tiles through *t_total (written by warp 0, lane 0; visible after the
// caller's next __syncthreads).
template <int BN>
__device__ __forceinline__ void load_segments(const GemmArgs& p, int32_t* s_seg_off,
                                              int32_t* s_seg_var, int32_t* s_prefix,
                                              int64_t* t_total) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
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
    s_prefix[s + 1] = len > p.max_short ? (len + BN - 1) / BN : 0;
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
    if (lane == 0) *t_total = carry;
  }
}

// ------------------------------------------------------------------ W_eff

// Sign-flip mask of one bf16 pair: bit 15 (the low element, column 2j of the
// chunk) and bit 31 (the high element, column 2j+1) are set where the sign
// bit is 0 (s = -1).  nb = the chunk's inverted sign byte (8 bits); the
// multiply places nb bit 2j at bit 15 and bit 2j+1 at bit 31 (the two partial
// products do not overlap, so no carry reaches either bit).
template <int J>
__device__ __forceinline__ uint32_t pair_flip_mask(uint32_t nb) {
  return (nb * (0x40008000u >> (2 * J))) & 0x80008000u;
}

// bf16x2_rne(fp32(w.lo) + a, fp32(w.hi) + a): two mixed-precision adds (the
// bf16 operand widened exactly to fp32 inside the add, one fp32 rounding)
// and one packing conversion, with no shifts to unpack the halves.
__device__ __forceinline__ uint32_t add_round_bf16x2(uint32_t w, uint32_t a) {
  uint32_t r;
  asm("{\n\t.reg .b16 l, h;\n\t.reg .f32 fl, fh;\n\t"
      "mov.b32 {l, h}, %1;\n\t"
      "add.rn.f32.bf16 fl, l, %2;\n\t"
      "add.rn.f32.bf16 fh, h, %2;\n\t"
      "cvt.rn.bf16x2.f32 %0, fh, fl;\n\t}"
      : "=r"(r)
      : "r"(w), "f"(__uint_as_float(a)));
  return r;
}

// W_eff of one row's 8·C columns held as C 16-byte chunks of bf16 W_base:
// W + s·α = s·(s·W + α).  The sign flip of W is exact and round-to-nearest-
// even is symmetric, so flipping W where s = -1, adding α in fp32, rounding
// to bf16 and flipping back gives bf16_rne(fp32(W) + s·α) (up to the sign of
// an exact zero, which no product or sum of the MMA can tell apart).
// sg: the row's sign bits for these columns (bit 1 = +1), 8 per chunk.
template <int C>
__device__ __forceinline__ void weff_chunks(const uint4 (&wv)[C], uint2 sg, uint32_t alpha_bits,
                                            uint32_t (&packed)[4 * C]) {
  const uint32_t nsx = ~sg.x, nsy = ~sg.y;
#pragma unroll
  for (int c = 0; c < C; ++c) {
    const uint32_t nb = ((c < 4 ? nsx : nsy) >> (8 * (c & 3))) & 0xFFu;
    const uint32_t f0 = pair_flip_mask<0>(nb), f1 = pair_flip_mask<1>(nb);
    const uint32_t f2 = pair_flip_mask<2>(nb), f3 = pair_flip_mask<3>(nb);
    packed[4 * c + 0] = add_round_bf16x2(wv[c].x ^ f0, alpha_bits) ^ f0;
    packed[4 * c + 1] = add_round_bf16x2(wv[c].y ^ f1, alpha_bits) ^ f1;
    packed[4 * c + 2] = add_round_bf16x2(wv[c].z ^ f2, alpha_bits) ^ f2;
    packed[4 * c + 3] = add_round_bf16x2(wv[c].w ^ f3, alpha_bits) ^ f3;
  }
}

// fp32 -> bf16 bits, round to nearest even.
__device__ __forceinline__ uint16_t bf16_rn(float f) {
  uint16_t h;
  asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(h) : "f"(f));
  return h;
}

// ------------------------------------------------------------------ TMEM

// 32 lanes x 32 consecutive 32-bit columns: thread i writes lane (base+i).
__device__ __forceinline__ void tmem_st_32x32b_x32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
      "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
      "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
// 32 lanes x 16 consecutive 32-bit columns.
__device__ __forceinline__ void tmem_st_32x32b_x16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15])
      : "memory");
}
template <int N>
__device__ __forceinline__ void tmem_st_32x32b(uint32_t taddr, const uint32_t (&r)[N]) {
  static_assert(N == 16 || N == 32, "16 or 32 columns");
  if constexpr (N == 32)
    tmem_st_32x32b_x32(taddr, r);
  else
    tmem_st_32x32b_x16(taddr, r);
}
__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Epilogue of one warp: its 32 accumulator lanes (lane = output row n, which
// is this thread's row) x the tile's token columns (column c = token
// tok0 + c, c < BN), rounded to bf16 and stored to y[tok][n] (row-major
// [M, d_out]).  Tokens at or past tok_end and rows at or past d_out are not
// stored.  taddr: TMEM address of the warp's lane quarter, column 0.
template <int BN>
__device__ __forceinline__ void store_acc_rows(uint32_t taddr, uint16_t* y, int64_t d_out,
                                               int64_t n, int64_t tok0, int64_t tok_end) {
  const int64_t span = tok_end - tok0;
  const int cols = span <= 0 ? 0 : (span < BN ? static_cast<int>(span) : BN);
  const bool n_ok = n < d_out;
  uint16_t* yp = y + tok0 * d_out + n;
#pragma unroll 1
  for (int c = 0; c < cols; c += 32) {
    uint32_t rr[32];
    tmem_ld_32x32b_x32(taddr + static_cast<uint32_t>(c), rr);
    tmem_ld_wait();
    if (n_ok) {
      uint16_t* q = yp;
      if (cols - c >= 32) {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          *q = bf16_rn(__uint_as_float(rr[j]));
          q += d_out;
        }
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          if (j < cols - c) *q = bf16_rn(__uint_as_float(rr[j]));
          q += d_out;
        }
      }
    }
    yp += 32 * d_out;
  }
}

// Partial slots of a split tile (one per CTA half): 128 rows x BN tokens of
// fp32, four tokens of a row together: (token c, row r) at float
// ((c / 4) * 128 + r) * 4 + c % 4.  A warp's 16-byte access for four tokens
// of its 32 rows is then 512 contiguous bytes, in the store and in the sum.

__device__ __forceinline__ void st_global_v4_hint(float4* p, float4 v, uint64_t policy) {
  asm volatile("st.global.L2::cache_hint.v4.f32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(p), "f"(v.x),
               "f"(v.y), "f"(v.z), "f"(v.w), "l"(policy)
               : "memory");
}
__device__ __forceinline__ unsigned int ld_acquire_u32(const unsigned int* p) {
  unsigned int v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Epilogue of one warp for a part of a split tile: its 32 accumulator lanes
// (row r = this thread's row of the CTA's 128) x the first `cols` tokens
// (rounded up to four), stored as fp32 to the slot under an L2 evict-last
// policy (the partner reads it, often at the end of the kernel, while the
// weight stream passes through L2 as evict-first).
__device__ __forceinline__ void store_acc_partial(uint32_t taddr, float* slot, int r, int cols) {
  const uint64_t keep = policy_evict_last();
  float4* s4 = reinterpret_cast<float4*>(slot) + r;
#pragma unroll 1
  for (int c = 0; c < cols; c += 32) {
    uint32_t v[32];
    tmem_ld_32x32b_x32(taddr + static_cast<uint32_t>(c), v);
    tmem_ld_wait();
#pragma unroll
    for (int k = 0; k < 8; ++k)
      if (c + 4 * k < cols)
        st_global_v4_hint(s4 + static_cast<int64_t>(c / 4 + k) * 128,
                          make_float4(__uint_as_float(v[4 * k]), __uint_as_float(v[4 * k + 1]),
                                      __uint_as_float(v[4 * k + 2]), __uint_as_float(v[4 * k + 3])),
                          keep);
  }
}

// The second contributor's sum of a split tile while it still holds its own
// part in tensor memory: own accumulator + the partner's partial (fp32
// addition of two terms is commutative, so the result equals the sum in k
// order), rounded once to bf16 and stored to y[tok0 + c][n].  The partner's
// eight 16-byte loads of a step are issued before the tensor-memory load
// completes.
__device__ __forceinline__ void sum_tmem_partial_store(uint32_t taddr, const float* slot, int r,
                                                       uint16_t* y, int64_t d_out, int64_t n,
                                                       int64_t tok0, int cols) {
  const bool n_ok = n < d_out;
  const float4* s4 = reinterpret_cast<const float4*>(slot) + r;
  uint16_t* yp = y + tok0 * d_out + n;
#pragma unroll 1
  for (int c = 0; c < cols; c += 32) {
    uint32_t v[32];
    tmem_ld_32x32b_x32(taddr + static_cast<uint32_t>(c), v);
    float4 pv[8];
#pragma unroll
    for (int k = 0; k < 8; ++k)
      pv[k] = n_ok && c + 4 * k < cols ? __ldcg(s4 + static_cast<int64_t>(c / 4 + k) * 128)
                                       : make_float4(0.f, 0.f, 0.f, 0.f);
    tmem_ld_wait();
    if (n_ok) {
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const float sum[4] = {__uint_as_float(v[4 * k]) + pv[k].x,
                              __uint_as_float(v[4 * k + 1]) + pv[k].y,
                              __uint_as_float(v[4 * k + 2]) + pv[k].z,
                              __uint_as_float(v[4 * k + 3]) + pv[k].w};
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (c + 4 * k + e < cols)
            yp[static_cast<int64_t>(c + 4 * k + e) * d_out] = bf16_rn(sum[e]);
      }
    }
  }
}

// The last contributor's sum of a split tile: for row r and each of the
// tile's `cols` tokens, the partials in slot a then slot b (the k order of
// the two contributors' ranges), rounded once to bf16 and stored to
// y[tok0 + c][n].  Eight 16-byte loads in flight per thread per step.
__device__ __forceinline__ void sum_pair_partials_store(const float* slot_a, const float* slot_b,
                                                        int r, uint16_t* y, int64_t d_out,
                                                        int64_t n, int64_t tok0, int cols) {
  if (n >= d_out) return;
  const float4* a4 = reinterpret_cast<const float4*>(slot_a) + r;
  const float4* b4 = reinterpret_cast<const float4*>(slot_b) + r;
  uint16_t* yp = y + tok0 * d_out + n;
#pragma unroll 1
  for (int c = 0; c < cols; c += 16) {
    float4 va[4], vb[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int64_t off = static_cast<int64_t>(c / 4 + k) * 128;
      va[k] = c + 4 * k < cols ? __ldcg(a4 + off) : make_float4(0.f, 0.f, 0.f, 0.f);
      vb[k] = c + 4 * k < cols ? __ldcg(b4 + off) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float s[4] = {va[k].x + vb[k].x, va[k].y + vb[k].y, va[k].z + vb[k].z,
                          va[k].w + vb[k].w};
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (c + 4 * k + e < cols) yp[static_cast<int64_t>(c + 4 * k + e) * d_out] = bf16_rn(s[e]);
    }
  }
}

// ------------------------------------------------------------------ CTA pairs

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Shared::cluster address of the variable at `local_smem_addr` in CTA `rank`.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t local_smem_addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local_smem_addr), "r"(rank));
  return r;
}
// Arrive on an mbarrier given by cluster address (possibly the other CTA's),
// with the instruction's default ordering.  A release at cluster scope here
// put a full memory barrier on every transform stage (ncu: 22% of the pair
// kernel's warp samples stalled on it on 256-token tiles; on the 512-token
// tiles' rank-1 arrivals alone it cost 45% of their throughput).  What the
// MMA needs from these arrivals stays on the arriving CTA's own SM: in a
// cta_group::2 MMA each CTA's tensor core reads that CTA's A rows (its W_eff),
// so rank 1's transform output is read by rank 1's tensor core.  On the
// 256-token tile that output is in rank 1's tensor memory, ordered before the
// arrival by tcgen05.wait::st and tcgen05.fence::before_thread_sync; on the
// 512-token tile it is in rank 1's shared memory, ordered by each writing
// thread's fence.proxy.async.shared::cta and the warp barrier before lane 0
// arrives.  The MMA that reads it is issued only after rank 0 has observed
// the arrival, so no read can start before those fences.  The bit-for-bit
// equality of the two tile widths on the same problem (a GPU test) is the
// measured side of that argument.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
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
// Bounded wait (acquire at cluster scope) on a barrier that the other CTA of
// the pair, or its MMAs, arrive on.  Same contract as mbar_wait.
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity,
                                                  const DevCtx& ctx, volatile int* abort) {
  if (mbar_try_wait_cluster(bar, parity, 0)) return true;
  const long long t0 = clock64();
  const long long limit = static_cast<long long>(ctx.wait_limit_ns) * 2;
  while (true) {
    if (mbar_try_wait_cluster(bar, parity, kSuspendNs)) return true;
    if (abort != nullptr && *abort) return false;
    if (clock64() - t0 > limit) {
      record_error(ctx, kErrTimeout);
      if (abort != nullptr) *abort = 1;
      return false;
    }
  }
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}

// Pair forms of the tcgen05 instructions (every tcgen05 instruction of a
// kernel that has a CTA-group qualifier must use the same group).
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* slot_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_addr(slot_smem)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
// D (+)= A · Bᵀ over the pair: M = 256 (128 rows of A and D in each CTA's
// tensor memory), B's N rows split in halves, rank 0's half first, each in
// its own CTA's shared memory at the same offset.  Issued by rank 0 only.
__device__ __forceinline__ void umma_bf16_tmem_a_pair(uint32_t d_tmem, uint32_t a_tmem,
                                                      uint64_t b_desc, uint32_t idesc,
                                                      uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// The same with A in shared memory: each CTA's 128 rows of A at the same
// shared-memory offset (descriptor a_desc), read by that CTA's tensor core.
__device__ __forceinline__ void umma_bf16_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                               uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive on `bar` (same offset) in both CTAs of the pair when the MMAs this
// thread issued so far complete.
__device__ __forceinline__ void umma_commit_pair(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 "
      "[%0], %1;" ::"r"(smem_addr(bar)),
      "h"(static_cast<uint16_t>(0x3))
      : "memory");
}

}  // namespace gemm_detail
}  // namespace bd
