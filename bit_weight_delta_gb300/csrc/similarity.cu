// similarity.cu — cosine similarity of task vectors in their 1-bit form.
//
// Page "BitDelta: serving 14 Zen models from one GPU cluster", section
// "K-Merge": when an adapter that is not in the pool is requested, compute its
// pairwise cosine similarity with every pool member on the task vectors and
// pick the most similar one.  Here the task vectors are the BitDelta deltas
// α ⊙ S (S = ±1 from the packed signs), which is what a server that keeps
// only the compressed deltas holds:
//     <α_a⊙S_a, α_b⊙S_b> = Σ_n α_a[n]·α_b[n]·(d_in − 2·popcount(S_a[n] ⊕ S_b[n]))
//     ‖α⊙S‖² = Σ_n α[n]²·d_in
// (one α for the matrix: the same with α constant).  The row's agreement
// count is an exact integer; the α products and sums are fp64.
//
// HBM-bound: the candidate's signs are read once, each member's once
// ((1 + n_b)/16 bytes per weight).  A warp takes one row of the candidate at
// a time into registers (16 bytes per lane per 4096 columns) and streams the
// pool members' same row, sixteen members per round of loads, and starts an
// L2 prefetch of the next row it will take.  The lanes'
// disagreement counts are summed by a transposing butterfly that leaves
// member j's row total in lanes 2j and 2j+1 (16 shuffles for 16 members),
// and the even lanes do the fp64 α arithmetic side by side.  Per-CTA partial
// sums go to the caller's workspace; the last CTA of each group of kGroup
// CTAs sums its group's partials, and the last group to finish sums the
// group partials and writes the cosines and the argmax: fixed orders
// (deterministic), and the fp64 reduction spread over many SMs instead of
// one.
#include <cstdint>

#include "common.cuh"
#include "kernels.h"

namespace bd {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kRound = 16;  // pool members whose row loads are in flight together
constexpr int kMaxGrid = 1024;  // CTAs of a launch at most
constexpr int kGroup = 32;      // CTA partials summed by one group reducer
constexpr int kMaxGroups = kMaxGrid / kGroup;
static_assert(4 * (1 + kMaxGroups) <= 256, "counters fit the workspace's first 256 bytes");

struct SimArgs {
  const uint8_t* pa;
  const float* aa;
  const uint8_t* const* pb_table;
  const float* const* ab_table;
  int32_t n_b;
  int per_row;
  int64_t d_out, d_in;
  double* cos_out;
  int32_t* best_out;
  double* partial;         // [gridDim.x][2·n_b + 1]: dot[b], norm_b[b], norm_a
  double* group_partial;   // [groups][2·n_b + 1]
  unsigned int* counter;   // [0]: groups finished; [1 + g]: CTAs of group g finished
                           // (each reset by the one that completes it)
  int vec;                 // 16-byte loads allowed (d_in % 128 == 0, candidate aligned)
};

__device__ __forceinline__ int popc4(uint4 a, uint4 b) {
  return __popc(a.x ^ b.x) + __popc(a.y ^ b.y) + __popc(a.z ^ b.z) + __popc(a.w ^ b.w);
}

// c[j]: this lane's count for member j of the round.  Each level halves the
// members a lane keeps (lanes with the level's bit set keep the upper half)
// and adds the partner's half it does not keep; after xor 16, 8, 4, 2 lane L
// holds its pair's share of member L >> 1, and xor 1 completes the total.
__device__ __forceinline__ int transpose_sum16(int (&c)[kRound], int lane) {
  static_assert(kRound == 16, "four halving levels");
#pragma unroll
  for (int lvl = 0; lvl < 4; ++lvl) {
    const int x = 16 >> lvl, half = 8 >> lvl;
    const bool up = (lane & x) != 0;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      if (k < half) {
        const int send = up ? c[k] : c[k + half];
        const int keep = up ? c[k + half] : c[k];
        c[k] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, x);
      }
    }
  }
  return c[0] + __shfl_xor_sync(0xFFFFFFFFu, c[0], 1);
}

// Four CTAs per SM (64 registers, no spills): the per-row sums are
// latency-bound, and 32 resident warps hide more of it than 24 (33 against
// 39 µs per call on 14336 x 4096, 1 vs 13; five CTAs at 48 registers spill).
__global__ void __launch_bounds__(kThreads, 4) sign_similarity_kernel(SimArgs p) {
  extern __shared__ double sm[];  // [kWarps][2·n_b + 1]
  __shared__ const uint8_t* s_pb[256];
  __shared__ const float* s_ab[256];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_b = p.n_b;
  const int stride_w = 2 * n_b + 1;
  double* mine = sm + warp * stride_w;
  for (int i = lane; i < stride_w; i += 32) mine[i] = 0.0;
  griddep_launch_dependents();
  griddep_wait();
  for (int b = threadIdx.x; b < n_b; b += kThreads) {
    s_pb[b] = p.pb_table[b];
    s_ab[b] = p.ab_table[b];
  }
  __syncthreads();

  const int64_t row_bytes = p.d_in / 8;
  const double d_in = static_cast<double>(p.d_in);
  const int64_t r_step = static_cast<int64_t>(gridDim.x) * kWarps;
  for (int64_t r = static_cast<int64_t>(blockIdx.x) * kWarps + warp; r < p.d_out; r += r_step) {
    const uint8_t* ra = p.pa + r * row_bytes;
    // The next row this warp takes, of the candidate and every member,
    // towards L2 while this row's loads and sums run (lane L takes every
    // 32nd 128-byte line of the (1 + n_b) row segments).
    if (r + r_step < p.d_out) {
      const int64_t rn = r + r_step;
      const int64_t lines = (row_bytes + 127) / 128;
      for (int64_t i = lane; i < (1 + n_b) * lines; i += 32) {
        const int64_t m = i / lines, l = i - m * lines;
        const uint8_t* base = m == 0 ? p.pa : s_pb[m - 1];
        prefetch_l2(base + rn * row_bytes + 128 * l);
      }
    }
    const double alpha_a = static_cast<double>(p.per_row ? __ldg(p.aa + r) : __ldg(p.aa));
    for (int b0 = 0; b0 < n_b; b0 += kRound) {
      int cnt[kRound];
#pragma unroll
      for (int q = 0; q < kRound; ++q) cnt[q] = 0;
      // lane pair (2j, 2j+1) ends with member b0 + j; the even lane fetches
      // its α for this row while the signs stream
      const int jm = lane >> 1;
      const bool mine_j = (lane & 1) == 0 && b0 + jm < n_b;
      const float ab_j = mine_j ? (p.per_row ? __ldg(s_ab[b0 + jm] + r) : __ldg(s_ab[b0 + jm]))
                                : 0.f;
      bool v4 = p.vec != 0;  // 16-byte loads when every member row is 16-byte aligned
#pragma unroll
      for (int q = 0; q < kRound; ++q)
        if (b0 + q < n_b) v4 = v4 && (reinterpret_cast<uintptr_t>(s_pb[b0 + q]) & 15u) == 0;
      if (v4) {
        for (int64_t off = 16 * lane; off < row_bytes; off += 512) {
          const uint4 va = ldg_stream_v4(ra + off);
          uint4 vb[kRound];
#pragma unroll
          for (int q = 0; q < kRound; ++q)
            vb[q] = b0 + q < n_b ? ldg_stream_v4(s_pb[b0 + q] + r * row_bytes + off) : va;
#pragma unroll
          for (int q = 0; q < kRound; ++q) cnt[q] += popc4(va, vb[q]);
        }
      } else {
        for (int64_t off = lane; off < row_bytes; off += 32) {
          const uint32_t a = __ldg(ra + off);
#pragma unroll
          for (int q = 0; q < kRound; ++q)
            if (b0 + q < n_b) cnt[q] += __popc(a ^ __ldg(s_pb[b0 + q] + r * row_bytes + off));
        }
      }
      // disagreeing signs of row r with member b0 + jm
      const int d_mine = transpose_sum16(cnt, lane);
      if (mine_j) {
        const double alpha_b = static_cast<double>(ab_j);
        mine[b0 + jm] += alpha_a * alpha_b * (d_in - 2.0 * d_mine);
        mine[n_b + b0 + jm] += alpha_b * alpha_b * d_in;
      }
    }
    if (lane == 0) mine[2 * n_b] += alpha_a * alpha_a * d_in;
  }
  __syncthreads();
  // CTA partials in a fixed warp order
  for (int i = threadIdx.x; i < stride_w; i += kThreads) {
    double s = 0.0;
    for (int w = 0; w < kWarps; ++w) s += sm[w * stride_w + i];
    p.partial[static_cast<int64_t>(blockIdx.x) * stride_w + i] = s;
  }
  __threadfence();
  __syncthreads();
  __shared__ unsigned int last;
  const unsigned int n_cta = gridDim.x;
  const unsigned int grp = blockIdx.x / kGroup, g0 = grp * kGroup;
  const unsigned int g_size = n_cta - g0 < kGroup ? n_cta - g0 : kGroup;
  if (threadIdx.x == 0) last = atomicAdd(p.counter + 1 + grp, 1u) == g_size - 1 ? 1u : 0u;
  __syncthreads();
  if (!last) return;
  __threadfence();
  // The last CTA of the group: its CTAs' partials in CTA order, value i by
  // thread i (loads bypass L1: other SMs wrote them).
  for (int i = threadIdx.x; i < stride_w; i += kThreads) {
    double v[kGroup];
#pragma unroll
    for (int q = 0; q < kGroup; ++q)
      v[q] = q < static_cast<int>(g_size)
                 ? __ldcg(p.partial + static_cast<int64_t>(g0 + q) * stride_w + i)
                 : 0.0;
    double s = 0.0;
#pragma unroll
    for (int q = 0; q < kGroup; ++q) s += v[q];
    p.group_partial[static_cast<int64_t>(grp) * stride_w + i] = s;
  }
  if (threadIdx.x == 0) p.counter[1 + grp] = 0u;
  __threadfence();
  __syncthreads();
  const unsigned int n_grp = (n_cta + kGroup - 1) / kGroup;
  if (threadIdx.x == 0) last = atomicAdd(p.counter, 1u) == n_grp - 1 ? 1u : 0u;
  __syncthreads();
  if (!last) return;
  __threadfence();
  // The last group: totals over the groups in group order, value i by
  // thread i, eight loads in flight at a time; then cosines and argmax.
  double* tot = sm;  // reuse: [stride_w]
  for (int i = threadIdx.x; i < stride_w; i += kThreads) {
    double s = 0.0;
    for (unsigned int q0 = 0; q0 < n_grp; q0 += 8) {
      double v[8];
#pragma unroll
      for (int q = 0; q < 8; ++q)
        v[q] = q0 + q < n_grp ? __ldcg(p.group_partial + static_cast<int64_t>(q0 + q) * stride_w + i)
                              : 0.0;
#pragma unroll
      for (int q = 0; q < 8; ++q) s += v[q];
    }
    tot[i] = s;
  }
  __syncthreads();
  double* cosv = tot + stride_w;  // [n_b]
  for (int b = threadIdx.x; b < n_b; b += kThreads) {
    const double c = tot[b] / sqrt(tot[2 * n_b] * tot[n_b + b]);
    cosv[b] = c;
    p.cos_out[b] = c;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int best = 0;
    double bv = -2.0;
    for (int b = 0; b < n_b; ++b) {
      if (cosv[b] > bv) {  // ties keep the lower index
        bv = cosv[b];
        best = b;
      }
    }
    *p.best_out = best;
    *p.counter = 0u;
  }
}

}  // namespace

int sign_similarity_grid(int64_t d_out) {
  const int64_t want = (d_out + kWarps - 1) / kWarps;
  return static_cast<int>(want < kMaxGrid ? want : kMaxGrid);
}

size_t sign_similarity_workspace_bytes(int64_t d_out, int32_t n_b) {
  const size_t grid = static_cast<size_t>(sign_similarity_grid(d_out));
  const size_t groups = (grid + kGroup - 1) / kGroup;
  return 256 + (grid + groups) * (2 * static_cast<size_t>(n_b) + 1) * sizeof(double);
}

cudaError_t launch_sign_similarity(const uint8_t* pa, const float* aa,
                                   const uint8_t* const* pb_table, const float* const* ab_table,
                                   int32_t n_b, bool per_row, int64_t d_out, int64_t d_in,
                                   double* cos_out, int32_t* best_out, void* workspace,
                                   bool vec, cudaStream_t stream) {
  SimArgs a{};
  a.pa = pa;
  a.aa = aa;
  a.pb_table = pb_table;
  a.ab_table = ab_table;
  a.n_b = n_b;
  a.per_row = per_row ? 1 : 0;
  a.d_out = d_out;
  a.d_in = d_in;
  a.cos_out = cos_out;
  a.best_out = best_out;
  a.counter = static_cast<unsigned int*>(workspace);
  a.partial = reinterpret_cast<double*>(static_cast<uint8_t*>(workspace) + 256);
  a.group_partial = a.partial + static_cast<int64_t>(sign_similarity_grid(d_out)) * (2 * n_b + 1);
  a.vec = vec ? 1 : 0;
  const size_t smem = static_cast<size_t>(kWarps) * (2 * n_b + 1) * sizeof(double);
  // One wave: at most the CTAs the device holds at once (a second, partial
  // wave of 56 CTAs made a third of the SMs idle for half of a 4096 x 14336
  // call), and rows spread evenly over the warps by the kernel's stride.
  int dev = 0, sms = 0, per_sm = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, sign_similarity_kernel, kThreads,
                                                    smem);
  if (e != cudaSuccess) return e;
  int grid = sign_similarity_grid(d_out);
  const int wave = sms * (per_sm > 0 ? per_sm : 1);
  if (grid > wave) grid = wave;
  return launch_pdl(sign_similarity_kernel, dim3(grid), dim3(kThreads), smem, stream, a);
}

}  // namespace bd
