// monosoup.cu — MonoSoup merge of k fine-tuned checkpoints of one base.
//
// Page "BitDelta: serving 14 Zen models from one GPU cluster", section
// "MonoSoup: complementing the single checkpoint with SVD":
//     Δ_i = W_i − W_base,   τ_i = rank-r truncated SVD of Δ_i,
//     W_merged = W_base + (1/k)·Σ_i τ_i.
//
// τ_i by block subspace iteration on Δ_i, which is formed on the fly in fp32
// from the two bf16 matrices and never stored:
//     Y = orth(Δ·Ω)                         Ω: d_in × r, entries ±1
//     q times:  Z = orth(Δᵀ·Y),  Y = orth(Δ·Z)
//     Y = orth(Y);  R = Δᵀ·Y                τ_i = Y·Rᵀ = Y·Yᵀ·Δ
// Y·Yᵀ·Δ is Δ projected onto the span of Y; once that span is the dominant
// r-dimensional left singular subspace of Δ, it equals the truncated SVD.
// Each product brings the span closer by the factor σ_{r+1}/σ_r, so with a
// gap after σ_r a few iterations reach the truncation to fp32 accuracy.
// orth() is Cholesky QR: G = AᵀA (r × r), G = L·Lᵀ, A ← A·L⁻ᵀ; a column whose
// pivot falls below 1e-6 of the largest diagonal entry is dependent and is
// dropped (zeroed).  The merge is one pass over W_base:
//     W_merged = bf16_rne(W_base + (1/k)·Σ_i Y_i·R_iᵀ).
//
// Factor matrices are fp32, row-major with RP columns (r padded to 16, 32 or
// 64; the padding columns stay zero).  Products with Δ are tall-skinny
// (64 rows of the long side × RP per CTA, split over the contracted side with
// a fixed-order reduction of the partial results); they run on the CUDA
// cores in fp32.
#include <cstdint>

#include "common.cuh"
#include "kernels.h"

namespace bd {
namespace {

constexpr int kMsThreads = 256;
constexpr int kTileA = 64;   // rows of the long side per CTA
constexpr int kTileB = 32;   // contracted indices per step
constexpr int kMaxSplit = 16;
constexpr int kMaxGramParts = 256;

__device__ __forceinline__ void bf16x8_to_f32(const uint4 v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

// Ω[c][j] = ±1 for j < r (a hash of (seed, c, j)), 0 for the padding columns.
__global__ void sketch_fill_kernel(float* omega, int64_t d_in, int r, int rp, uint64_t seed) {
  const int64_t n = d_in * rp;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int j = static_cast<int>(i % rp);
    uint64_t z = seed + 0x9E3779B97F4A7C15ull * static_cast<uint64_t>(i + 1);
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    z ^= z >> 31;
    omega[i] = j < r ? ((z & 1u) ? 1.f : -1.f) : 0.f;
  }
}

// out[a][j] = Σ_b Δ(a, b)·V[b][j] over b in this CTA's split.
//   kT = false: a = row n of Δ, b = column c   (Y = Δ·V,  V: d_in × RP)
//   kT = true:  a = column c,   b = row n      (Z = Δᵀ·V, V: d_out × RP)
// Grid (ceil(A / 64), S); split s covers b in [s·b_chunk, (s+1)·b_chunk) and
// writes part[s][a][j] (or out directly when S == 1).
template <int RP, bool kT>
__global__ void __launch_bounds__(kMsThreads) delta_mul_kernel(
    const uint16_t* __restrict__ wft, const uint16_t* __restrict__ wb, int64_t d_out,
    int64_t d_in, const float* __restrict__ v, float* __restrict__ out, int64_t b_chunk) {
  constexpr int JW = RP / 16;  // output columns per thread
  __shared__ __align__(16) float ds[kTileB][kTileA + 4];  // [b][a]
  __shared__ __align__(16) float vs[kTileB][RP];
  const int tid = threadIdx.x;
  const int ty = tid >> 4, tx = tid & 15;
  const int64_t A = kT ? d_in : d_out;
  const int64_t B = kT ? d_out : d_in;
  const int64_t a0 = static_cast<int64_t>(blockIdx.x) * kTileA;
  const int64_t b_lo = static_cast<int64_t>(blockIdx.y) * b_chunk;
  const int64_t b_hi = b_lo + b_chunk < B ? b_lo + b_chunk : B;

  float acc[4][JW];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < JW; ++j) acc[i][j] = 0.f;

  for (int64_t b0 = b_lo; b0 < b_hi; b0 += kTileB) {
    // Δ tile: 64 a × 32 b, 256 vectors of 8 bf16 (one per thread)
    if (!kT) {
      const int row = tid >> 2, vec = tid & 3;
      const int64_t n = a0 + row, c = b0 + 8 * vec;
      float f[8];
      if (n < d_out && c < b_hi) {
        float fb[8];
        bf16x8_to_f32(__ldg(reinterpret_cast<const uint4*>(wft + n * d_in + c)), f);
        bf16x8_to_f32(__ldg(reinterpret_cast<const uint4*>(wb + n * d_in + c)), fb);
#pragma unroll
        for (int e = 0; e < 8; ++e) f[e] -= fb[e];
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) f[e] = 0.f;
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) ds[8 * vec + e][row] = f[e];
    } else {
      const int row = tid >> 3, vec = tid & 7;
      const int64_t n = b0 + row, c = a0 + 8 * vec;
      float f[8];
      if (n < b_hi && c < d_in) {
        float fb[8];
        bf16x8_to_f32(__ldg(reinterpret_cast<const uint4*>(wft + n * d_in + c)), f);
        bf16x8_to_f32(__ldg(reinterpret_cast<const uint4*>(wb + n * d_in + c)), fb);
#pragma unroll
        for (int e = 0; e < 8; ++e) f[e] -= fb[e];
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) f[e] = 0.f;
      }
      *reinterpret_cast<float4*>(&ds[row][8 * vec]) = make_float4(f[0], f[1], f[2], f[3]);
      *reinterpret_cast<float4*>(&ds[row][8 * vec + 4]) = make_float4(f[4], f[5], f[6], f[7]);
    }
    // V tile: 32 b × RP
    for (int q = tid; q < kTileB * RP / 4; q += kMsThreads) {
      const int bb = q / (RP / 4), j4 = q % (RP / 4);
      const int64_t b = b0 + bb;
      *reinterpret_cast<float4*>(&vs[bb][4 * j4]) =
          b < b_hi ? __ldg(reinterpret_cast<const float4*>(v + b * RP) + j4)
                   : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    __syncthreads();
#pragma unroll 8
    for (int bb = 0; bb < kTileB; ++bb) {
      const float4 a4 = *reinterpret_cast<const float4*>(&ds[bb][4 * ty]);
      const float av[4] = {a4.x, a4.y, a4.z, a4.w};
      float vv[JW];
#pragma unroll
      for (int j = 0; j < JW; ++j) vv[j] = vs[bb][JW * tx + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < JW; ++j) acc[i][j] = fmaf(av[i], vv[j], acc[i][j]);
    }
    __syncthreads();
  }
  float* dst = out + static_cast<int64_t>(blockIdx.y) * A * RP;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int64_t a = a0 + 4 * ty + i;
    if (a >= A) continue;
#pragma unroll
    for (int j = 0; j < JW; ++j) dst[a * RP + JW * tx + j] = acc[i][j];
  }
}

// out[i] = Σ_s part[s][i], s in order.
__global__ void reduce_parts_kernel(const float* __restrict__ part, int n_part, int64_t n,
                                    float* __restrict__ out) {
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    float s = 0.f;
    for (int p = 0; p < n_part; ++p) s += part[p * n + i];
    out[i] = s;
  }
}

// gpart[cta] = Σ over this CTA's rows of A[row]ᵀ·A[row]  (RP × RP).
template <int RP>
__global__ void __launch_bounds__(kMsThreads) gram_partial_kernel(const float* __restrict__ a,
                                                                  int64_t m, int64_t rows_per_cta,
                                                                  float* __restrict__ gpart) {
  constexpr int JW = RP / 16;
  __shared__ __align__(16) float rows[32][RP];
  const int tid = threadIdx.x;
  const int ty = tid >> 4, tx = tid & 15;
  const int64_t r_lo = static_cast<int64_t>(blockIdx.x) * rows_per_cta;
  const int64_t r_hi = r_lo + rows_per_cta < m ? r_lo + rows_per_cta : m;
  float acc[JW][JW];
#pragma unroll
  for (int i = 0; i < JW; ++i)
#pragma unroll
    for (int j = 0; j < JW; ++j) acc[i][j] = 0.f;
  for (int64_t r0 = r_lo; r0 < r_hi; r0 += 32) {
    for (int q = tid; q < 32 * RP / 4; q += kMsThreads) {
      const int rr = q / (RP / 4), j4 = q % (RP / 4);
      const int64_t row = r0 + rr;
      *reinterpret_cast<float4*>(&rows[rr][4 * j4]) =
          row < r_hi ? __ldg(reinterpret_cast<const float4*>(a + row * RP) + j4)
                     : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    __syncthreads();
    for (int rr = 0; rr < 32; ++rr) {
      float ai[JW], aj[JW];
#pragma unroll
      for (int i = 0; i < JW; ++i) {
        ai[i] = rows[rr][JW * ty + i];
        aj[i] = rows[rr][JW * tx + i];
      }
#pragma unroll
      for (int i = 0; i < JW; ++i)
#pragma unroll
        for (int j = 0; j < JW; ++j) acc[i][j] = fmaf(ai[i], aj[j], acc[i][j]);
    }
    __syncthreads();
  }
  float* g = gpart + static_cast<int64_t>(blockIdx.x) * RP * RP;
#pragma unroll
  for (int i = 0; i < JW; ++i)
#pragma unroll
    for (int j = 0; j < JW; ++j) g[(JW * ty + i) * RP + JW * tx + j] = acc[i][j];
}

// One CTA: G = Σ gpart (in order), G = L·Lᵀ over the leading r × r block,
// T = L⁻ᵀ (RP × RP, zero outside r × r and in the columns of dropped pivots).
template <int RP>
__global__ void __launch_bounds__(kMsThreads) chol_inverse_kernel(const float* __restrict__ gpart,
                                                                  int n_part, int r,
                                                                  float* __restrict__ t_out) {
  __shared__ float g[RP][RP + 1];   // G, then L⁻¹ (lower) once L is complete
  __shared__ float l[RP][RP + 1];
  __shared__ float inv_d[RP];
  __shared__ float thr;
  const int tid = threadIdx.x;
  for (int q = tid; q < RP * RP; q += kMsThreads) {
    float s = 0.f;
    for (int p = 0; p < n_part; ++p) s += gpart[static_cast<int64_t>(p) * RP * RP + q];
    g[q / RP][q % RP] = s;
    l[q / RP][q % RP] = 0.f;
  }
  __syncthreads();
  if (tid == 0) {
    float mx = 0.f;
    for (int j = 0; j < r; ++j) mx = fmaxf(mx, g[j][j]);
    thr = 1e-6f * mx;
  }
  __syncthreads();
  for (int j = 0; j < r; ++j) {
    if (tid == 0) {
      const float d = g[j][j];
      const bool live = d > thr && thr > 0.f;
      const float sd = live ? sqrtf(d) : 0.f;
      l[j][j] = sd;
      inv_d[j] = live ? 1.f / sd : 0.f;
    }
    __syncthreads();
    for (int i = j + 1 + tid; i < r; i += kMsThreads) l[i][j] = g[i][j] * inv_d[j];
    __syncthreads();
    const int w = r - j - 1;  // trailing block (i, k) with j < k <= i < r
    for (int q = tid; q < w * w; q += kMsThreads) {
      const int i = j + 1 + q / w, k = j + 1 + q % w;
      if (k <= i) g[i][k] -= l[i][j] * l[k][j];
    }
    __syncthreads();
  }
  // X = L⁻¹ by forward substitution, one column per thread, into g
  float (*x)[RP + 1] = g;
  for (int q = tid; q < RP * RP; q += kMsThreads) x[q / RP][q % RP] = 0.f;
  __syncthreads();
  if (tid < r) {
    const int c = tid;
    x[c][c] = inv_d[c];
    for (int i = c + 1; i < r; ++i) {
      float s = 0.f;
      for (int m = c; m < i; ++m) s = fmaf(l[i][m], x[m][c], s);
      x[i][c] = -s * inv_d[i];
    }
  }
  __syncthreads();
  for (int q = tid; q < RP * RP; q += kMsThreads) {
    const int i = q / RP, j = q % RP;
    t_out[q] = (i < r && j < r) ? x[j][i] : 0.f;  // T = Xᵀ
  }
}

// A[row] ← A[row]·T in place, one warp per row.
template <int RP>
__global__ void __launch_bounds__(kMsThreads) apply_right_kernel(float* __restrict__ a, int64_t m,
                                                                 const float* __restrict__ t) {
  __shared__ float ts[RP][RP];
  for (int q = threadIdx.x; q < RP * RP; q += kMsThreads) ts[q / RP][q % RP] = t[q];
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  constexpr int PER = (RP + 31) / 32;
  for (int64_t row = static_cast<int64_t>(blockIdx.x) * (kMsThreads / 32) + warp; row < m;
       row += static_cast<int64_t>(gridDim.x) * (kMsThreads / 32)) {
    float* ar = a + row * RP;
    float av[PER];
#pragma unroll
    for (int p = 0; p < PER; ++p) av[p] = 32 * p + lane < RP ? ar[32 * p + lane] : 0.f;
    float out[PER];
#pragma unroll
    for (int p = 0; p < PER; ++p) out[p] = 0.f;
#pragma unroll
    for (int p = 0; p < PER; ++p) {
      for (int src = 0; src < 32 && 32 * p + src < RP; ++src) {
        const float ai = __shfl_sync(0xFFFFFFFFu, av[p], src);
        const int i = 32 * p + src;
#pragma unroll
        for (int o = 0; o < PER; ++o)
          if (32 * o + lane < RP) out[o] = fmaf(ai, ts[i][32 * o + lane], out[o]);
      }
    }
    __syncwarp();
#pragma unroll
    for (int p = 0; p < PER; ++p)
      if (32 * p + lane < RP) ar[32 * p + lane] = out[p];
  }
}

// W_merged = bf16_rne(W_base + inv_k·Σ_i P_i·R_iᵀ) over 64 × 64 tiles.
template <int RP>
__global__ void __launch_bounds__(kMsThreads) merge_kernel(
    const uint16_t* __restrict__ wb, const float* __restrict__ p_fac,
    const float* __restrict__ r_fac, int k, int64_t d_out, int64_t d_in, float inv_k,
    uint16_t* __restrict__ out, float* __restrict__ corr) {
  __shared__ __align__(16) float ps[16][64 + 4];  // [j][n]
  __shared__ __align__(16) float rs[16][64 + 4];  // [j][c]
  const int tid = threadIdx.x;
  const int ty = tid >> 4, tx = tid & 15;
  const int64_t n0 = static_cast<int64_t>(blockIdx.y) * 64;
  const int64_t c0 = static_cast<int64_t>(blockIdx.x) * 64;
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
  const int lr = tid >> 2, lj = tid & 3;  // loader: row of the tile, 4 columns of the step
  for (int i = 0; i < k; ++i) {
    const float* pi = p_fac + static_cast<int64_t>(i) * d_out * RP;
    const float* ri = r_fac + static_cast<int64_t>(i) * d_in * RP;
    for (int j0 = 0; j0 < RP; j0 += 16) {
      const int64_t n = n0 + lr, c = c0 + lr;
      const float4 pv = n < d_out ? __ldg(reinterpret_cast<const float4*>(pi + n * RP + j0) + lj)
                                  : make_float4(0.f, 0.f, 0.f, 0.f);
      const float4 rv = c < d_in ? __ldg(reinterpret_cast<const float4*>(ri + c * RP + j0) + lj)
                                 : make_float4(0.f, 0.f, 0.f, 0.f);
      ps[4 * lj + 0][lr] = pv.x;
      ps[4 * lj + 1][lr] = pv.y;
      ps[4 * lj + 2][lr] = pv.z;
      ps[4 * lj + 3][lr] = pv.w;
      rs[4 * lj + 0][lr] = rv.x;
      rs[4 * lj + 1][lr] = rv.y;
      rs[4 * lj + 2][lr] = rv.z;
      rs[4 * lj + 3][lr] = rv.w;
      __syncthreads();
#pragma unroll
      for (int jj = 0; jj < 16; ++jj) {
        const float4 p4 = *reinterpret_cast<const float4*>(&ps[jj][4 * ty]);
        const float4 r4 = *reinterpret_cast<const float4*>(&rs[jj][4 * tx]);
        const float pv4[4] = {p4.x, p4.y, p4.z, p4.w};
        const float rv4[4] = {r4.x, r4.y, r4.z, r4.w};
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
          for (int b = 0; b < 4; ++b) acc[a][b] = fmaf(pv4[a], rv4[b], acc[a][b]);
      }
      __syncthreads();
    }
  }
  const int64_t c = c0 + 4 * tx;
  if (c >= d_in) return;  // d_in % 8 == 0: the 4 columns are wholly inside or outside
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    const int64_t n = n0 + 4 * ty + a;
    if (n >= d_out) continue;
    const uint2 w = *reinterpret_cast<const uint2*>(wb + n * d_in + c);
    const float base[4] = {__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xFFFF0000u),
                           __uint_as_float(w.y << 16), __uint_as_float(w.y & 0xFFFF0000u)};
    float cv[4], mv[4];
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      cv[b] = inv_k * acc[a][b];
      mv[b] = base[b] + cv[b];
    }
    *reinterpret_cast<uint2*>(out + n * d_in + c) =
        make_uint2(pack_bf16x2_rn(mv[0], mv[1]), pack_bf16x2_rn(mv[2], mv[3]));
    if (corr != nullptr)
      *reinterpret_cast<float4*>(corr + n * d_in + c) = make_float4(cv[0], cv[1], cv[2], cv[3]);
  }
}

// ------------------------------------------------------------------ host side

struct MsLayout {
  int rp = 0;
  size_t omega = 0, z = 0, part = 0, gpart = 0, t = 0, p = 0, r = 0, total = 0;
};

int padded_rank(int r) { return r <= 16 ? 16 : r <= 32 ? 32 : 64; }

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

MsLayout ms_layout(int64_t d_out, int64_t d_in, int k, int r) {
  MsLayout L;
  L.rp = padded_rank(r);
  const size_t rp = static_cast<size_t>(L.rp);
  const size_t a_max = static_cast<size_t>(d_out > d_in ? d_out : d_in);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off += align256(bytes);
    return o;
  };
  L.omega = take(static_cast<size_t>(d_in) * rp * 4);
  L.z = take(static_cast<size_t>(d_in) * rp * 4);
  L.part = take(kMaxSplit * a_max * rp * 4);
  L.gpart = take(static_cast<size_t>(kMaxGramParts) * rp * rp * 4);
  L.t = take(rp * rp * 4);
  L.p = take(static_cast<size_t>(k) * d_out * rp * 4);
  L.r = take(static_cast<size_t>(k) * d_in * rp * 4);
  L.total = off;
  return L;
}

template <int RP>
struct MsRunner {
  const MonoSoupArgs& a;
  cudaStream_t s;
  uint8_t* ws;
  MsLayout L;
  int num_sms;

  float* f(size_t off) const { return reinterpret_cast<float*>(ws + off); }

  cudaError_t delta_mul(bool trans, const uint16_t* wft, const float* v, float* out) const {
    const int64_t A = trans ? a.d_in : a.d_out;
    const int64_t B = trans ? a.d_out : a.d_in;
    const int64_t a_blocks = (A + kTileA - 1) / kTileA;
    const int64_t want = 2 * static_cast<int64_t>(num_sms);
    int64_t split = (want + a_blocks - 1) / a_blocks;
    if (split < 1) split = 1;
    if (split > kMaxSplit) split = kMaxSplit;
    int64_t b_chunk = (B + split - 1) / split;
    if (b_chunk < 2 * kTileB) b_chunk = 2 * kTileB;
    b_chunk = (b_chunk + kTileB - 1) / kTileB * kTileB;
    split = (B + b_chunk - 1) / b_chunk;
    float* dst = split == 1 ? out : f(L.part);
    const dim3 grid(static_cast<unsigned>(a_blocks), static_cast<unsigned>(split));
    if (trans)
      delta_mul_kernel<RP, true><<<grid, kMsThreads, 0, s>>>(wft, a.w_base, a.d_out, a.d_in, v,
                                                             dst, b_chunk);
    else
      delta_mul_kernel<RP, false><<<grid, kMsThreads, 0, s>>>(wft, a.w_base, a.d_out, a.d_in, v,
                                                              dst, b_chunk);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || split == 1) return e;
    const int64_t n = A * RP;
    const int64_t blocks = (n + kMsThreads - 1) / kMsThreads;
    reduce_parts_kernel<<<static_cast<unsigned>(blocks < 4096 ? blocks : 4096), kMsThreads, 0, s>>>(
        f(L.part), static_cast<int>(split), n, out);
    return cudaGetLastError();
  }

  cudaError_t orth(float* m_ptr, int64_t m) const {
    int64_t rows_per_cta = (m + kMaxGramParts - 1) / kMaxGramParts;
    if (rows_per_cta < 32) rows_per_cta = 32;
    rows_per_cta = (rows_per_cta + 31) / 32 * 32;
    const int64_t parts = (m + rows_per_cta - 1) / rows_per_cta;
    gram_partial_kernel<RP><<<static_cast<unsigned>(parts), kMsThreads, 0, s>>>(
        m_ptr, m, rows_per_cta, f(L.gpart));
    chol_inverse_kernel<RP><<<1, kMsThreads, 0, s>>>(f(L.gpart), static_cast<int>(parts), a.rank,
                                                     f(L.t));
    const int64_t rows_blocks = (m + 7) / 8;
    apply_right_kernel<RP><<<static_cast<unsigned>(rows_blocks < 4096 ? rows_blocks : 4096),
                             kMsThreads, 0, s>>>(m_ptr, m, f(L.t));
    return cudaGetLastError();
  }

  cudaError_t run() const {
    cudaError_t e;
    if (a.rank > 0) {
      const int64_t n_om = a.d_in * RP;
      sketch_fill_kernel<<<static_cast<unsigned>((n_om + 255) / 256 < 4096 ? (n_om + 255) / 256
                                                                             : 4096),
                           256, 0, s>>>(f(L.omega), a.d_in, a.rank, RP, a.seed);
      if ((e = cudaGetLastError()) != cudaSuccess) return e;
      for (int i = 0; i < a.k; ++i) {
        const uint16_t* wft = a.w_ft[i];
        float* y = f(L.p) + static_cast<int64_t>(i) * a.d_out * RP;
        float* r = f(L.r) + static_cast<int64_t>(i) * a.d_in * RP;
        float* z = f(L.z);
        if ((e = delta_mul(false, wft, f(L.omega), y)) != cudaSuccess) return e;
        if ((e = orth(y, a.d_out)) != cudaSuccess) return e;
        for (int it = 0; it < a.power_iters; ++it) {
          if ((e = delta_mul(true, wft, y, z)) != cudaSuccess) return e;
          if ((e = orth(z, a.d_in)) != cudaSuccess) return e;
          if ((e = delta_mul(false, wft, z, y)) != cudaSuccess) return e;
          if ((e = orth(y, a.d_out)) != cudaSuccess) return e;
        }
        if ((e = orth(y, a.d_out)) != cudaSuccess) return e;  // second Cholesky QR pass
        if ((e = delta_mul(true, wft, y, r)) != cudaSuccess) return e;
      }
    }
    const dim3 grid(static_cast<unsigned>((a.d_in + 63) / 64),
                    static_cast<unsigned>((a.d_out + 63) / 64));
    merge_kernel<RP><<<grid, kMsThreads, 0, s>>>(a.w_base, f(L.p), f(L.r),
                                                 a.rank > 0 ? a.k : 0, a.d_out, a.d_in,
                                                 1.0f / static_cast<float>(a.k), a.w_merged,
                                                 a.correction);
    return cudaGetLastError();
  }
};

}  // namespace

size_t monosoup_workspace_bytes(int64_t d_out, int64_t d_in, int k, int rank) {
  return ms_layout(d_out, d_in, k, rank).total;
}

cudaError_t launch_monosoup(const MonoSoupArgs& a, void* workspace, int num_sms,
                            cudaStream_t stream) {
  const MsLayout L = ms_layout(a.d_out, a.d_in, a.k, a.rank);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  // factors start at zero: the padding columns stay zero and rank 0 merges nothing
  cudaError_t e = cudaMemsetAsync(ws + L.p, 0, L.total - L.p, stream);
  if (e != cudaSuccess) return e;
  switch (L.rp) {
    case 16:
      return MsRunner<16>{a, stream, ws, L, num_sms}.run();
    case 32:
      return MsRunner<32>{a, stream, ws, L, num_sms}.run();
    default:
      return MsRunner<64>{a, stream, ws, L, num_sms}.run();
  }
}

}  // namespace bd
