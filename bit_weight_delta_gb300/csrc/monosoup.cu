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
//     q times:  Z = Δᵀ·Y,  Y = orth(Δ·Z)
//     Y = orth(Y);  R = Δᵀ·Y                τ_i = Y·Rᵀ = Y·Yᵀ·Δ
// Y·Yᵀ·Δ is Δ projected onto the span of Y; once that span is the dominant
// r-dimensional left singular subspace of Δ, it equals the truncated SVD.
// Each product brings the span closer by the factor σ_{r+1}/σ_r, so with a
// gap after σ_r a few iterations reach the truncation to fp32 accuracy.
// orth() is Cholesky QR: G = AᵀA (r × r), G = L·Lᵀ, A ← A·L⁻ᵀ; a column whose
// pivot falls below 1e-6 of the largest diagonal entry is dependent and is
// dropped (zeroed).  The merge is one tensor-core pass over W_base:
//     W_merged = bf16_rne(W_base + (1/k)·Σ_i Y_i·R_iᵀ).
//
// Factor matrices are fp32, row-major with RP columns (r padded to 16, 32 or
// 64; the padding columns stay zero).  Products with Δ are tall-skinny (64
// rows of the long side × RP per CTA, split over the contracted side with a
// fixed-order reduction of the partial results); they run on the tensor
// cores as W_i·V − W_base·V with V split into two bf16 terms (four bf16
// products per tile, fp32 accumulation).
#include <cstdint>

#include "common.cuh"
#include "kernels.h"

namespace bd {
namespace {

constexpr int kMsThreads = 256;
constexpr int kMulThreads = 128;  // threads of a Δ-product CTA
constexpr int kTileA = 64;   // rows of the long side per Δ-product CTA (16 per warp)
constexpr int kTileB = 32;   // contracted indices per step
constexpr int kMaxSplit = 32;

constexpr int kMaxCkpt = 64;
struct CkptTable {  // the checkpoints' W_i, passed by value
  const uint16_t* p[kMaxCkpt];
};

// D += A·B, mma.sync m16n8k16 (bf16 A row-major, bf16 B column-major, fp32).
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1,
                                               uint32_t a2, uint32_t a3, uint32_t b0,
                                               uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Ω[c][j] = ±1 for j < r (a hash of (seed, c, j)), 0 for the padding columns.
__global__ void sketch_fill_kernel(float* omega, int64_t d_in, int r, int rp, uint64_t seed) {
  griddep_wait();
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
  // the next launch may start as this grid's last CTAs finish (a trigger at
  // the start let the next kernel's CTAs take the slots of this one's
  // later waves)
  griddep_launch_dependents();
}

// V split for the tensor-core Δ products: V (B × RP fp32, one per checkpoint
// at v_stride, or one for all when v_stride is 0) → kVTerms bf16 terms
// V ≈ hi + lo (relative error 2^-18 per element), stored transposed as
// vs[z][term][j][b] with rows of bp = B rounded up to 8 (zero padding), so
// that a B fragment is two adjacent b of one j and every row is 16-byte
// aligned.  A thread converts 8 consecutive b of one j and writes one
// 16-byte vector per term.
constexpr int kVTerms = 2;
__global__ void vsplit_kernel(const float* __restrict__ v_all, int64_t v_stride, int64_t B,
                              int64_t bp, int rp, uint16_t* __restrict__ out) {
  griddep_wait();
  const int64_t z = blockIdx.y;
  const float* __restrict__ v = v_all + z * v_stride;
  uint16_t* __restrict__ o = out + z * kVTerms * rp * bp;
  const int64_t nb8 = bp / 8;
  const int64_t n = nb8 * rp;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int j = static_cast<int>(i / nb8);
    const int64_t b0 = 8 * (i - static_cast<int64_t>(j) * nb8);
    uint32_t hw[4], lw[4];
#pragma unroll
    for (int e = 0; e < 8; e += 2) {
      float x[2];
#pragma unroll
      for (int u = 0; u < 2; ++u) x[u] = b0 + e + u < B ? __ldg(v + (b0 + e + u) * rp + j) : 0.f;
      const uint32_t h = pack_bf16x2_rn(x[0], x[1]);
      const float r0 = x[0] - __uint_as_float(h << 16);
      const float r1 = x[1] - __uint_as_float(h & 0xFFFF0000u);
      hw[e / 2] = h;
      lw[e / 2] = pack_bf16x2_rn(r0, r1);
    }
    *reinterpret_cast<uint4*>(o + static_cast<int64_t>(j) * bp + b0) =
        make_uint4(hw[0], hw[1], hw[2], hw[3]);
    *reinterpret_cast<uint4*>(o + static_cast<int64_t>(rp + j) * bp + b0) =
        make_uint4(lw[0], lw[1], lw[2], lw[3]);
  }
  // the next launch may start as this grid's last CTAs finish (a trigger at
  // the start let the next kernel's CTAs take the slots of this one's
  // later waves)
  griddep_launch_dependents();
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void cp16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

// Shared-memory geometry of one pipeline stage of the Δ-product kernel.
template <int RP, bool kT>
struct MulStage {
  // W tiles (W_i and W_base): !kT [64 a][32 b + 8], kT [32 b][64 a + 8] (bf16)
  static constexpr int kWRow = kT ? kTileA + 8 : kTileB + 8;
  static constexpr int kWRows = kT ? kTileB : kTileA;
  static constexpr int kWBytes = kWRows * kWRow * 2;
  // V terms: [kVTerms][RP j][32 b + 8] (bf16)
  static constexpr int kVRow = kTileB + 8;
  static constexpr int kVBytes = kVTerms * RP * kVRow * 2;
  static constexpr int kBytes = 2 * kWBytes + kVBytes;
};
constexpr int kMulStages = 3;

template <int RP, bool kT>
constexpr size_t mul_smem_bytes() {
  return static_cast<size_t>(kMulStages) * MulStage<RP, kT>::kBytes;
}

// out[a][j] = Σ_b Δ(a, b)·V[b][j] over b in this CTA's split, on the tensor
// cores (mma.sync m16n8k16, bf16 in, fp32 accumulate).
//   kT = false: a = row n of Δ, b = column c   (Y = Δ·V,  V: d_in × RP)
//   kT = true:  a = column c,   b = row n      (Z = Δᵀ·V, V: d_out × RP)
// Δ·V = W_i·Vhi − W_base·Vhi + Δ·Vlo with both weights as exact bf16
// operands, V as the sum of two bf16 terms (vsplit_kernel) and Δ rounded to
// bf16 for the low term only: three products per tile (four with W_i·Vlo −
// W_base·Vlo took 629 against 601 µs per 4096 x 4096, k = 4, rank-32 merge),
// the W_base one with the V fragments' sign bits flipped, all into one fp32
// accumulator.  With V's columns orthonormal (as in the iteration), the
// result stays within about 1e-6 of Δ·V relative to its largest entry
// (fp64 emulation of the four-product form: 5e-7; Δ's rounding adds at most
// 2^-17 of |Δ|·|V| per product), despite the cancellation.  Grid
// (ceil(A / 64), S, k); split s covers b in [s·b_chunk, (s+1)·b_chunk) and
// writes part[s][a][j] (or the output directly when S == 1); blockIdx.z picks
// the checkpoint.  128 threads; warp w owns rows a0 + 16w .. +15 and all RP
// columns.  Tiles arrive by cp.async through a kMulStages-deep ring; A
// fragments come from ldmatrix (.trans for Δᵀ).
template <int RP, bool kT>
__global__ void __launch_bounds__(kMulThreads) delta_mul_kernel(
    CkptTable tab, const uint16_t* __restrict__ wb, int64_t d_out, int64_t d_in,
    const uint16_t* __restrict__ vs_all, int64_t vs_stride, int64_t bp,
    float* __restrict__ dst_all, int64_t dst_stride, int64_t b_chunk) {
  griddep_wait();
  using G = MulStage<RP, kT>;
  constexpr int JT = RP / 8;
  extern __shared__ __align__(16) uint8_t sm[];
  const uint16_t* __restrict__ wft = tab.p[blockIdx.z];
  const int64_t A = kT ? d_in : d_out;
  const int64_t B = kT ? d_out : d_in;
  const uint16_t* __restrict__ vsz = vs_all + blockIdx.z * vs_stride;  // [kVTerms][RP][bp]
  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int64_t a0 = static_cast<int64_t>(blockIdx.x) * kTileA;
  const int64_t b_lo = static_cast<int64_t>(blockIdx.y) * b_chunk;
  const int64_t b_hi = b_lo + b_chunk < B ? b_lo + b_chunk : B;
  const uint32_t sm_sa = smem_addr(sm);
  const int n_steps = static_cast<int>((b_hi - b_lo + kTileB - 1) / kTileB);

  // One stage: W_i and W_base tiles (256 vectors of 16 bytes each, 2 per
  // thread per matrix) and the V-term tiles (kVTerms·RP rows of 64 bytes).
  // Elements past the matrix edge are zero-filled by plain stores.
  auto issue = [&](int stage, int step) {
    if (step < n_steps) {
      const int64_t b0 = b_lo + static_cast<int64_t>(step) * kTileB;
      const uint32_t st = sm_sa + stage * G::kBytes;
      uint8_t* stp = sm + stage * G::kBytes;
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int q = tid + kMulThreads * u;
        int row, col;
        int64_t n, c;
        bool ok;
        if (!kT) {
          row = q >> 2;
          col = 8 * (q & 3);
          n = a0 + row;
          c = b0 + col;
          ok = n < d_out && c < b_hi;
        } else {
          row = q >> 3;
          col = 8 * (q & 7);
          n = b0 + row;
          c = a0 + col;
          ok = n < b_hi && c < d_in;
        }
        const uint32_t off = static_cast<uint32_t>((row * G::kWRow + col) * 2);
        if (ok) {
          cp16(st + off, wft + n * d_in + c);
          cp16(st + G::kWBytes + off, wb + n * d_in + c);
        } else {
          *reinterpret_cast<uint4*>(stp + off) = make_uint4(0, 0, 0, 0);
          *reinterpret_cast<uint4*>(stp + G::kWBytes + off) = make_uint4(0, 0, 0, 0);
        }
      }
      // V terms: rows (term, j), 4 vectors of 8 b each
      for (int q = tid; q < kVTerms * RP * 4; q += kMulThreads) {
        const int row = q >> 2, col = 8 * (q & 3);
        const int64_t b = b0 + col;
        const uint32_t off = static_cast<uint32_t>(2 * G::kWBytes + (row * G::kVRow + col) * 2);
        if (b < b_hi)  // b_hi < B only at split boundaries (multiples of 32)
          cp16(st + off, vsz + static_cast<int64_t>(row) * bp + b);
        else
          *reinterpret_cast<uint4*>(stp + off) = make_uint4(0, 0, 0, 0);
      }
    }
    cp_async_commit();
  };

  float acc[JT][4];
#pragma unroll
  for (int jt = 0; jt < JT; ++jt)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[jt][e] = 0.f;

#pragma unroll
  for (int s = 0; s < kMulStages - 1; ++s) issue(s, s);
  for (int step = 0; step < n_steps; ++step) {
    cp_async_wait<kMulStages - 2>();
    __syncthreads();  // the stage is complete for every thread; the oldest slot is free
    issue((step + kMulStages - 1) % kMulStages, step + kMulStages - 1);
    const int stage = step % kMulStages;
    const uint32_t st = sm_sa + stage * G::kBytes;
#pragma unroll
    for (int kk = 0; kk < kTileB; kk += 16) {
      uint32_t af[2][4];  // [W_i, W_base] A fragments of rows 16w .. +15, k kk .. +15
#pragma unroll
      for (int mtx = 0; mtx < 2; ++mtx) {
        const uint32_t base = st + mtx * G::kWBytes;
        if (!kT) {
          const int m = 16 * warp + (lane & 7) + 8 * ((lane >> 3) & 1);
          const int k = kk + 8 * (lane >> 4);
          ldsm_x4(base + (m * G::kWRow + k) * 2, af[mtx][0], af[mtx][1], af[mtx][2], af[mtx][3]);
        } else {
          const int k = kk + (lane & 7) + 8 * (lane >> 4);
          const int m = 16 * warp + 8 * ((lane >> 3) & 1);
          ldsm_x4_t(base + (k * G::kWRow + m) * 2, af[mtx][0], af[mtx][1], af[mtx][2], af[mtx][3]);
        }
      }
      // Δ = W_i − W_base as one bf16 operand for V's low term: the difference
      // of two bf16 values is exact in fp32, and rounding it to bf16 (2^-9 of
      // Δ) multiplies a term 2^-8 of V, so three products per tile instead of
      // four (W_i·Vhi − W_base·Vhi + Δ·Vlo)
      uint32_t ad[4];
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const float dlo = __uint_as_float(af[0][r] << 16) - __uint_as_float(af[1][r] << 16);
        const float dhi = __uint_as_float(af[0][r] & 0xFFFF0000u) -
                          __uint_as_float(af[1][r] & 0xFFFF0000u);
        ad[r] = pack_bf16x2_rn(dlo, dhi);
      }
#pragma unroll
      for (int jp = 0; jp < JT; jp += 2) {
        // B fragments of tiles jp, jp+1 for each V term: [term][b0 jp, b1 jp, b0 jp+1, b1 jp+1]
        uint32_t bf[kVTerms][4];
#pragma unroll
        for (int term = 0; term < kVTerms; ++term) {
          const int j = 8 * (jp + (lane >> 4)) + (lane & 7);
          const int k = kk + 8 * ((lane >> 3) & 1);
          ldsm_x4(st + 2 * G::kWBytes + ((term * RP + j) * G::kVRow + k) * 2, bf[term][0],
                  bf[term][1], bf[term][2], bf[term][3]);
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          if (jp + h >= JT) break;
          float (&c)[4] = acc[jp + h];
          static_assert(kVTerms == 2, "V as a high and a low bf16 term");
          const uint32_t b0 = bf[0][2 * h], b1 = bf[0][2 * h + 1];
          mma_bf16_16816(c, af[0][0], af[0][1], af[0][2], af[0][3], b0, b1);
          mma_bf16_16816(c, af[1][0], af[1][1], af[1][2], af[1][3], b0 ^ 0x80008000u,
                         b1 ^ 0x80008000u);
          mma_bf16_16816(c, ad[0], ad[1], ad[2], ad[3], bf[1][2 * h], bf[1][2 * h + 1]);
        }
      }
    }
  }
  cp_async_wait<0>();
  float* dst = dst_all + blockIdx.z * dst_stride + static_cast<int64_t>(blockIdx.y) * A * RP;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int64_t a = a0 + 16 * warp + g + 8 * h;
    if (a >= A) continue;
#pragma unroll
    for (int jt = 0; jt < JT; ++jt)
      *reinterpret_cast<float2*>(dst + a * RP + 8 * jt + 2 * t) =
          make_float2(acc[jt][2 * h], acc[jt][2 * h + 1]);
  }
  // the next launch may start as this grid's last CTAs finish (a trigger at
  // the start let the next kernel's CTAs take the slots of this one's
  // later waves)
  griddep_launch_dependents();
}

// Checkpoint blockIdx.y, rows [r_lo, r_lo + kSlab) (1024 threads): A[row] = Σ_s part[s][row]
// (s in order; skipped when n_split == 0, A being complete already), then
// gpart[cta] = Σ_rows A[row]ᵀ·A[row] (RP × RP).
constexpr int kSlab = 128;
constexpr int kRgThreads = 1024;
template <int RP>
__global__ void __launch_bounds__(kRgThreads) reduce_gram_kernel(
    const float* __restrict__ part_all, int n_split, float* __restrict__ a_all,
    int64_t a_stride, int64_t m, float* __restrict__ gpart_all) {
  griddep_wait();
  __shared__ __align__(16) float rows[kSlab][RP];
  const int tid = threadIdx.x;
  const int64_t z = blockIdx.y;  // checkpoint
  const float* __restrict__ part = part_all + z * n_split * m * RP;
  float* __restrict__ a = a_all + z * a_stride;
  float* __restrict__ gpart = gpart_all + z * gridDim.x * RP * RP;
  const int64_t r_lo = static_cast<int64_t>(blockIdx.x) * kSlab;
  for (int q = tid; q < kSlab * RP / 4; q += kRgThreads) {
    const int rr = q / (RP / 4), j4 = q % (RP / 4);
    const int64_t row = r_lo + rr;
    float4 v4 = make_float4(0.f, 0.f, 0.f, 0.f);
    if (row < m) {
      if (n_split > 0) {
        for (int sp0 = 0; sp0 < n_split; sp0 += 8) {
          float4 t[8];
#pragma unroll
          for (int u = 0; u < 8; ++u)
            t[u] = sp0 + u < n_split
                       ? __ldg(reinterpret_cast<const float4*>(part + ((sp0 + u) * m + row) * RP) + j4)
                       : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            v4.x += t[u].x;
            v4.y += t[u].y;
            v4.z += t[u].z;
            v4.w += t[u].w;
          }
        }
        reinterpret_cast<float4*>(a + row * RP)[j4] = v4;
      } else {
        v4 = reinterpret_cast<const float4*>(a + row * RP)[j4];
      }
    }
    *reinterpret_cast<float4*>(&rows[rr][4 * j4]) = v4;
  }
  __syncthreads();
  float* gp = gpart + static_cast<int64_t>(blockIdx.x) * RP * RP;
  for (int q = tid; q < RP * RP; q += kRgThreads) {
    const int i = q / RP, j = q % RP;
    float s0 = 0.f, s1 = 0.f;
    for (int rr = 0; rr < kSlab; rr += 2) {
      s0 = fmaf(rows[rr][i], rows[rr][j], s0);
      s1 = fmaf(rows[rr + 1][i], rows[rr + 1][j], s1);
    }
    gp[q] = s0 + s1;
  }
  // the next launch may start as this grid's last CTAs finish (a trigger at
  // the start let the next kernel's CTAs take the slots of this one's
  // later waves)
  griddep_launch_dependents();
}

// One CTA: G = Σ gpart (in order), G = L·Lᵀ over the leading r × r block,
// and F (RP × RP, row-major): L below the diagonal, 1 / L[i][i] on it, zero
// outside r × r and for a dropped pivot (its row and column of L are zero
// too).  apply_right_kernel then solves against it, so no inverse is formed
// (the explicit triangular inverse here cost ~13 µs a launch: 672 against
// 620 µs per 4096 x 4096, k = 4, rank-32 merge).  Every thread takes part in
// the partial sums; warp 0 alone then factorises (rank <= 32: rows in the
// lanes' registers, exchanged by shuffles; else lane L owns rows L and L +
// 32 in shared memory, warp barriers only).
template <int RP>
__global__ void __launch_bounds__(kMsThreads) chol_factor_kernel(
    const float* __restrict__ gpart_all, int n_part, int r, float* __restrict__ t_all) {
  // one CTA per checkpoint, a single wave: the next launch may start at once
  // and waits for this grid before it reads
  griddep_launch_dependents();
  griddep_wait();
  constexpr int OWN = RP > 32 ? 2 : 1;  // rows / columns per lane
  // one CTA per checkpoint
  const float* __restrict__ gpart = gpart_all + static_cast<int64_t>(blockIdx.x) * n_part * RP * RP;
  float* __restrict__ t_out = t_all + static_cast<int64_t>(blockIdx.x) * RP * RP;
  __shared__ float g[RP][RP + 1];       // G (lower part), factorised in place into L
  __shared__ float x[RP][RP + 1];       // F, staged by the register form
  __shared__ float inv_d[RP];
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  // Σ_p gpart[p]: float4 columns, partials p ≡ u (mod 4) in chain u, the
  // chains added in order at the end
  for (int q4 = tid; q4 < RP * RP / 4; q4 += kMsThreads) {
    float4 cs[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) cs[u] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 2
    for (int p0 = 0; p0 < n_part; p0 += 4) {
      float4 t[4];
#pragma unroll
      for (int u = 0; u < 4; ++u)
        t[u] = p0 + u < n_part
                   ? __ldg(reinterpret_cast<const float4*>(gpart + static_cast<int64_t>(p0 + u) * RP * RP) + q4)
                   : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        cs[u].x += t[u].x;
        cs[u].y += t[u].y;
        cs[u].z += t[u].z;
        cs[u].w += t[u].w;
      }
    }
    const float sv[4] = {cs[0].x + cs[1].x + cs[2].x + cs[3].x, cs[0].y + cs[1].y + cs[2].y + cs[3].y,
                         cs[0].z + cs[1].z + cs[2].z + cs[3].z, cs[0].w + cs[1].w + cs[2].w + cs[3].w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int q = 4 * q4 + e;
      g[q / RP][q % RP] = sv[e];
      x[q / RP][q % RP] = 0.f;
    }
  }
  __syncthreads();
  if constexpr (RP <= 32) {
    // Register form (rank <= 32): lane i holds row i of G, then column i of
    // L⁻¹; pivots and multipliers travel by shuffles.
    if (tid < 32) {
      const unsigned full = 0xFFFFFFFFu;
      float gr[RP];
#pragma unroll
      for (int k = 0; k < RP; ++k) gr[k] = (lane < r && k < r) ? g[lane][k] : 0.f;
      float diag = 0.f;
#pragma unroll
      for (int k = 0; k < RP; ++k)
        if (k == lane) diag = gr[k];
      float mx = diag;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(full, mx, o));
      const float thr = 1e-6f * mx;
      float my_inv = 0.f;  // inv_d of this lane's row
#pragma unroll
      for (int j = 0; j < RP; ++j) {
        const float d = __shfl_sync(full, gr[j], j);  // G[j][j] after the updates
        const bool live = d > thr && thr > 0.f && j < r;
        const float sd = live ? sqrtf(d) : 0.f;
        const float id = live ? 1.f / sd : 0.f;
        const float lij = lane > j ? gr[j] * id : 0.f;  // L[lane][j]
        if (lane == j) {
          gr[j] = sd;
          my_inv = id;
        }
        if (lane > j) gr[j] = lij;
#pragma unroll
        for (int k = j + 1; k < RP; ++k) {
          const float lkj = __shfl_sync(full, lij, k);  // L[k][j]
          if (lane >= k) gr[k] = fmaf(-lij, lkj, gr[k]);
        }
      }
      // row `lane` of F: L[lane][i] below the diagonal, 1 / L[lane][lane] on
      // it (0 for a dropped pivot, and for rows and columns past r)
      if (lane < RP) {
#pragma unroll
        for (int i = 0; i < RP; ++i)
          x[lane][i] = (lane < r && i < r) ? (i < lane ? gr[i] : i == lane ? my_inv : 0.f) : 0.f;
      }
    }
    __syncthreads();
    for (int q = tid; q < RP * RP; q += kMsThreads) t_out[q] = x[q / RP][q % RP];
    return;
  }
  if (tid < 32) {
    float mx = 0.f;
#pragma unroll
    for (int o = 0; o < OWN; ++o)
      if (lane + 32 * o < r) mx = fmaxf(mx, g[lane + 32 * o][lane + 32 * o]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
    const float thr = 1e-6f * mx;
    // right-looking Cholesky: column j of L replaces column j of G
    for (int j = 0; j < r; ++j) {
      const float d = g[j][j];
      const bool live = d > thr && thr > 0.f;
      const float sd = live ? sqrtf(d) : 0.f;
      const float id = live ? 1.f / sd : 0.f;
      __syncwarp();
#pragma unroll
      for (int o = 0; o < OWN; ++o) {
        const int i = lane + 32 * o;
        if (i == j) g[j][j] = sd;
        if (i > j && i < r) g[i][j] *= id;
      }
      if (lane == 0) inv_d[j] = id;
      __syncwarp();
#pragma unroll
      for (int o = 0; o < OWN; ++o) {
        const int i = lane + 32 * o;
        if (i <= j || i >= r) continue;
        const float lij = g[i][j];
#pragma unroll 4
        for (int k = j + 1; k <= i; ++k) g[i][k] = fmaf(-lij, g[k][j], g[i][k]);
      }
      __syncwarp();
    }
  }
  __syncthreads();
  for (int q = tid; q < RP * RP; q += kMsThreads) {
    const int i = q / RP, j = q % RP;
    t_out[q] = (i < r && j < r) ? (j < i ? g[i][j] : j == i ? inv_d[i] : 0.f) : 0.f;
  }
}

// A[row] ← A[row]·L⁻ᵀ in place, one warp per row, for every checkpoint: the
// row q with q·Lᵀ = a by forward substitution against F (see
// chol_factor_kernel), q[c] = (a[c] − Σ_{m<c} L[c][m]·q[m]) / L[c][c]; lane
// L owns columns L (and L + 32), each q[m] is broadcast as it is finished.
template <int RP>
__global__ void __launch_bounds__(kMsThreads) apply_right_kernel(float* __restrict__ a_all,
                                                                 int64_t a_stride, int64_t m,
                                                                 const float* __restrict__ f_all) {
  griddep_wait();
  // checkpoint blockIdx.y: its rows and its F
  float* __restrict__ a = a_all + blockIdx.y * a_stride;
  const float* __restrict__ f = f_all + static_cast<int64_t>(blockIdx.y) * RP * RP;
  __shared__ float fs[RP][RP + 1];  // padded: the lanes read a column
  for (int q = threadIdx.x; q < RP * RP; q += kMsThreads) fs[q / RP][q % RP] = f[q];
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  constexpr int PER = (RP + 31) / 32;
  for (int64_t row = static_cast<int64_t>(blockIdx.x) * (kMsThreads / 32) + warp; row < m;
       row += static_cast<int64_t>(gridDim.x) * (kMsThreads / 32)) {
    float* ar = a + row * RP;
    float sv[PER], qv[PER];
#pragma unroll
    for (int p = 0; p < PER; ++p) {
      sv[p] = 32 * p + lane < RP ? ar[32 * p + lane] : 0.f;
      qv[p] = 0.f;
    }
#pragma unroll
    for (int mm = 0; mm < RP; ++mm) {
      const int pm = mm / 32, lm = mm % 32;
      const float qm = __shfl_sync(0xFFFFFFFFu, sv[pm] * fs[mm][mm], lm);
      if (lane == lm) qv[pm] = qm;
#pragma unroll
      for (int p = 0; p < PER; ++p) {
        const int c = 32 * p + lane;
        if (c > mm && c < RP) sv[p] = fmaf(-fs[c][mm], qm, sv[p]);
      }
    }
    __syncwarp();
#pragma unroll
    for (int p = 0; p < PER; ++p)
      if (32 * p + lane < RP) ar[32 * p + lane] = qv[p];
  }
  // the next launch may start as this grid's last CTAs finish (a trigger at
  // the start let the next kernel's CTAs take the slots of this one's
  // later waves)
  griddep_launch_dependents();
}

// Factor split for the tensor-core merge: the k checkpoints' factors
// F_i (rows × RP fp32, rows·RP apart), scaled by `scale`, side by side as
// two bf16 terms hi + lo of rows × kp (kp = k·RP; column i·RP + j holds
// F_i[row][j]).  A thread converts 8 consecutive columns of one row.
__global__ void fsplit_kernel(const float* __restrict__ f, int64_t rows, int rp, int k,
                              float scale, uint16_t* __restrict__ hi, uint16_t* __restrict__ lo) {
  griddep_wait();
  const int64_t kp = static_cast<int64_t>(k) * rp;
  const int64_t n8 = rows * (kp / 8);
  for (int64_t q = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; q < n8;
       q += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t row = q / (kp / 8);
    const int64_t col = 8 * (q - row * (kp / 8));
    const int64_t i = col / rp, j = col - i * rp;
    const float4* src = reinterpret_cast<const float4*>(f + (i * rows + row) * rp + j);
    const float4 x0 = __ldg(src), x1 = __ldg(src + 1);
    const float xv[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
    uint32_t hw[4], lw[4];
#pragma unroll
    for (int e = 0; e < 8; e += 2) {
      const float a = xv[e] * scale, b = xv[e + 1] * scale;
      const uint32_t h = pack_bf16x2_rn(a, b);
      hw[e / 2] = h;
      lw[e / 2] = pack_bf16x2_rn(a - __uint_as_float(h << 16), b - __uint_as_float(h & 0xFFFF0000u));
    }
    *reinterpret_cast<uint4*>(hi + row * kp + col) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
    *reinterpret_cast<uint4*>(lo + row * kp + col) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
  }
  // the next launch may start as this grid's last CTAs finish (a trigger at
  // the start let the next kernel's CTAs take the slots of this one's
  // later waves)
  griddep_launch_dependents();
}

constexpr int kMergeTile = 64;   // output rows and columns per CTA
constexpr int kMergeK = 64;      // K per stage
constexpr int kMergeRow = kMergeK + 8;  // bf16 per smem row (conflict-free ldmatrix)
constexpr int kMergeStageBytes = 4 * kMergeTile * kMergeRow * 2;  // P hi, P lo, R hi, R lo
constexpr size_t kMergeSmem = 2 * static_cast<size_t>(kMergeStageBytes);

// W_merged = bf16_rne(W_base + Σ_K P'[n][K]·R[c][K]) with P' = P/k, on the
// tensor cores: P' = Phi + Plo and R = Rhi + Rlo (bf16, fsplit_kernel), three
// products per tile (Phi·Rhi + Phi·Rlo + Plo·Rhi; the dropped Plo·Rlo is
// 2^-18 relative), fp32 accumulation.  CTA: 64 × 64 outputs, 4 warps of
// 16 rows × 64 columns; K in stages of 64 through a two-deep cp.async ring.
__global__ void __launch_bounds__(kMulThreads) merge_kernel(
    const uint16_t* __restrict__ wb, const uint16_t* __restrict__ phi,
    const uint16_t* __restrict__ plo, const uint16_t* __restrict__ rhi,
    const uint16_t* __restrict__ rlo, int64_t kp, int64_t d_out, int64_t d_in,
    uint16_t* __restrict__ out, float* __restrict__ corr) {
  // No early signal to dependents: this kernel writes the merged weights,
  // which a following bitdelta_linear may read before it waits.
  griddep_wait();
  constexpr int JT = kMergeTile / 8;
  extern __shared__ __align__(16) uint8_t sm[];
  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int64_t n0 = static_cast<int64_t>(blockIdx.y) * kMergeTile;
  const int64_t c0 = static_cast<int64_t>(blockIdx.x) * kMergeTile;
  const uint32_t sm_sa = smem_addr(sm);
  const int n_steps = static_cast<int>((kp + kMergeK - 1) / kMergeK);
  constexpr int kMat = kMergeTile * kMergeRow * 2;  // bytes of one matrix tile

  auto issue = [&](int stage, int step) {
    if (step < n_steps) {
      const int64_t k0 = static_cast<int64_t>(step) * kMergeK;
      const uint32_t st = sm_sa + stage * kMergeStageBytes;
      uint8_t* stp = sm + stage * kMergeStageBytes;
      // 4 matrices × 64 rows × 8 vectors of 8 bf16
      for (int q = tid; q < 4 * kMergeTile * (kMergeK / 8); q += kMulThreads) {
        const int mtx = q / (kMergeTile * (kMergeK / 8));
        const int rem = q - mtx * kMergeTile * (kMergeK / 8);
        const int row = rem >> 3, col = 8 * (rem & 7);
        const bool is_p = mtx < 2;
        const int64_t grow = (is_p ? n0 : c0) + row;
        const int64_t gk = k0 + col;
        const uint16_t* src = mtx == 0 ? phi : mtx == 1 ? plo : mtx == 2 ? rhi : rlo;
        const uint32_t off = static_cast<uint32_t>(mtx * kMat + (row * kMergeRow + col) * 2);
        if (grow < (is_p ? d_out : d_in) && gk < kp)
          cp16(st + off, src + grow * kp + gk);
        else
          *reinterpret_cast<uint4*>(stp + off) = make_uint4(0, 0, 0, 0);
      }
    }
    cp_async_commit();
  };

  float acc[JT][4];
#pragma unroll
  for (int jt = 0; jt < JT; ++jt)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[jt][e] = 0.f;

  issue(0, 0);
  for (int step = 0; step < n_steps; ++step) {
    cp_async_wait<0>();
    __syncthreads();  // stage `step` complete everywhere; the other slot is free
    issue((step + 1) & 1, step + 1);
    const uint32_t st = sm_sa + (step & 1) * kMergeStageBytes;
#pragma unroll
    for (int kk = 0; kk < kMergeK; kk += 16) {
      uint32_t ap[2][4];
#pragma unroll
      for (int term = 0; term < 2; ++term) {
        const int m = 16 * warp + (lane & 7) + 8 * ((lane >> 3) & 1);
        const int k = kk + 8 * (lane >> 4);
        ldsm_x4(st + term * kMat + (m * kMergeRow + k) * 2, ap[term][0], ap[term][1], ap[term][2],
                ap[term][3]);
      }
#pragma unroll
      for (int jp = 0; jp < JT; jp += 2) {
        uint32_t bq[2][4];
#pragma unroll
        for (int term = 0; term < 2; ++term) {
          const int j = 8 * (jp + (lane >> 4)) + (lane & 7);
          const int k = kk + 8 * ((lane >> 3) & 1);
          ldsm_x4(st + (2 + term) * kMat + (j * kMergeRow + k) * 2, bq[term][0], bq[term][1],
                  bq[term][2], bq[term][3]);
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          float (&c)[4] = acc[jp + h];
          const uint32_t bh0 = bq[0][2 * h], bh1 = bq[0][2 * h + 1];
          const uint32_t bl0 = bq[1][2 * h], bl1 = bq[1][2 * h + 1];
          mma_bf16_16816(c, ap[0][0], ap[0][1], ap[0][2], ap[0][3], bh0, bh1);
          mma_bf16_16816(c, ap[0][0], ap[0][1], ap[0][2], ap[0][3], bl0, bl1);
          mma_bf16_16816(c, ap[1][0], ap[1][1], ap[1][2], ap[1][3], bh0, bh1);
        }
      }
    }
  }
  cp_async_wait<0>();
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int64_t n = n0 + 16 * warp + g + 8 * h;
    if (n >= d_out) continue;
#pragma unroll
    for (int jt = 0; jt < JT; ++jt) {
      const int64_t c = c0 + 8 * jt + 2 * t;
      if (c >= d_in) continue;  // d_in % 8 == 0: c and c + 1 are inside together
      const uint32_t w = *reinterpret_cast<const uint32_t*>(wb + n * d_in + c);
      const float cv0 = acc[jt][2 * h], cv1 = acc[jt][2 * h + 1];
      const float m0 = __uint_as_float(w << 16) + cv0;
      const float m1 = __uint_as_float(w & 0xFFFF0000u) + cv1;
      *reinterpret_cast<uint32_t*>(out + n * d_in + c) = pack_bf16x2_rn(m0, m1);
      if (corr != nullptr)
        *reinterpret_cast<float2*>(corr + n * d_in + c) = make_float2(cv0, cv1);
    }
  }
}

// ------------------------------------------------------------------ host side

struct MsLayout {
  int rp = 0;
  size_t omega = 0, z = 0, part = 0, gpart = 0, t = 0, vsplit = 0, fsplit = 0, p = 0, r = 0,
         total = 0;
};

int padded_rank(int r) { return r <= 16 ? 16 : r <= 32 ? 32 : 64; }

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

// Workspace: Ω (d_in × RP), Z (k × d_in × RP), split partials (at most
// kMaxSplit outputs of the longer side, over all checkpoints), Gram partials
// (k × slabs × RP²), T (k × RP²), the bf16 terms of V (k × 2 × RP × the
// longer side rounded up to 8), the bf16 terms of the factors for the merge
// (2 × k·RP × (d_out + d_in)), factors Y_i = P (k × d_out × RP) and
// R_i (k × d_in × RP).
MsLayout ms_layout(int64_t d_out, int64_t d_in, int k, int r) {
  MsLayout L;
  L.rp = padded_rank(r);
  const size_t rp = static_cast<size_t>(L.rp);
  const size_t kk = static_cast<size_t>(k);
  const size_t a_max = static_cast<size_t>(d_out > d_in ? d_out : d_in);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off += align256(bytes);
    return o;
  };
  L.omega = take(static_cast<size_t>(d_in) * rp * 4);
  L.z = take(kk * d_in * rp * 4);
  L.part = take(kMaxSplit * a_max * rp * 4);
  L.gpart = take(kk * ((a_max + kSlab - 1) / kSlab) * rp * rp * 4);
  L.t = take(kk * rp * rp * 4);
  L.vsplit = take(kk * kVTerms * rp * ((a_max + 7) / 8 * 8) * 2);
  L.fsplit = take(2 * kk * rp * (static_cast<size_t>(d_out) + d_in) * 2);
  L.p = take(kk * d_out * rp * 4);
  L.r = take(kk * d_in * rp * 4);
  L.total = off;
  return L;
}

// Every step below processes all k checkpoints in one launch.
template <int RP>
struct MsRunner {
  const MonoSoupArgs& a;
  cudaStream_t s;
  uint8_t* ws;
  MsLayout L;
  int num_sms;
  CkptTable tab;

  float* f(size_t off) const { return reinterpret_cast<float*>(ws + off); }

  // CTAs of a Δ-product kernel that fit on one SM (queried once per kernel,
  // after its dynamic shared-memory limit is raised)
  template <bool kT>
  static int resident_ctas() {
    static int occ_dev[64] = {};  // per device: the attribute is per context
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return -1;
    std::lock_guard<std::mutex> lock(host_cache_mutex());
    int& occ = occ_dev[dev];
    if (occ == 0) {
      const size_t smem = mul_smem_bytes<RP, kT>();
      int n = 0;
      if (cudaFuncSetAttribute(delta_mul_kernel<RP, kT>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(smem)) == cudaSuccess &&
          cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, delta_mul_kernel<RP, kT>,
                                                        kMulThreads, smem) == cudaSuccess &&
          n > 0)
        occ = n;
      else
        occ = -1;
    }
    return occ;
  }

  // out_i = Δ_i·V_i (trans: Δ_iᵀ·V_i) for every checkpoint i; V_i at
  // v + i·v_stride (one V for all when v_stride is 0), out_i at
  // out + i·out_stride.  V is first split into three bf16 terms; the product
  // is split over the contracted side so that the grid is about two even
  // waves; *n_split = 0 when the outputs are complete, else the number of
  // partials left in L.part.
  cudaError_t delta_mul(bool trans, const float* v, int64_t v_stride, float* out,
                        int64_t out_stride, int* n_split) const {
    return trans ? delta_mul_t<true>(v, v_stride, out, out_stride, n_split)
                 : delta_mul_t<false>(v, v_stride, out, out_stride, n_split);
  }

  template <bool kT>
  cudaError_t delta_mul_t(const float* v, int64_t v_stride, float* out, int64_t out_stride,
                          int* n_split) const {
    const int64_t A = kT ? a.d_in : a.d_out;
    const int64_t B = kT ? a.d_out : a.d_in;
    const int64_t bp = (B + 7) / 8 * 8;
    const int nz = v_stride == 0 ? 1 : a.k;
    uint16_t* vs = reinterpret_cast<uint16_t*>(ws + L.vsplit);
    {
      const int64_t n = bp / 8 * RP;
      int64_t blocks = (n + 255) / 256;
      if (blocks > 2048) blocks = 2048;
      {
        const cudaError_t le =
            launch_pdl(vsplit_kernel,
                       dim3(static_cast<unsigned>(blocks), static_cast<unsigned>(nz)),
                       dim3(256), 0, s, v, v_stride, B, bp, RP, vs);
        if (le != cudaSuccess) return le;
      }
      const cudaError_t e = cudaGetLastError();
      if (e != cudaSuccess) return e;
    }
    const int occ = resident_ctas<kT>();
    if (occ < 0) return cudaErrorInvalidConfiguration;
    const int64_t a_blocks = (A + kTileA - 1) / kTileA;
    // two waves' worth of CTAs: the products are bound per SM (legacy tensor
    // path and its operand traffic), and 1024 CTAs over 608 slots leave each
    // SM within one CTA of the mean where one wave of 512 left 3 or 4 per SM
    // (716 -> 675 µs per 4096 x 4096, k = 4, rank-32 merge; three waves 680)
    const int64_t want = static_cast<int64_t>(occ) * num_sms * 2;
    int64_t split = want / (a_blocks * a.k);
    const int64_t split_max = kMaxSplit / a.k > 1 ? kMaxSplit / a.k : 1;
    if (split > split_max) split = split_max;
    if (split < 1) split = 1;
    int64_t b_chunk = (B + split - 1) / split;
    if (b_chunk < 2 * kTileB) b_chunk = 2 * kTileB;
    b_chunk = (b_chunk + kTileB - 1) / kTileB * kTileB;
    split = (B + b_chunk - 1) / b_chunk;
    float* dst = split == 1 ? out : f(L.part);
    const int64_t dst_stride = split == 1 ? out_stride : split * A * RP;
    const dim3 grid(static_cast<unsigned>(a_blocks), static_cast<unsigned>(split),
                    static_cast<unsigned>(a.k));
    {
      const cudaError_t le =
          launch_pdl(delta_mul_kernel<RP, kT>, dim3(grid), dim3(kMulThreads),
                     mul_smem_bytes<RP, kT>(), s, tab, a.w_base, a.d_out, a.d_in, vs,
                     v_stride == 0 ? 0 : kVTerms * RP * bp, bp, dst, dst_stride, b_chunk);
      if (le != cudaSuccess) return le;
    }
    *n_split = split == 1 ? 0 : static_cast<int>(split);
    return cudaGetLastError();
  }

  // Σ of the split partials into the outputs (and their Gram partials)
  cudaError_t reduce_gram(float* m_ptr, int64_t stride, int64_t m, int n_split) const {
    const int64_t parts = (m + kSlab - 1) / kSlab;
    {
      const cudaError_t le =
          launch_pdl(reduce_gram_kernel<RP>,
                     dim3(static_cast<unsigned>(parts), static_cast<unsigned>(a.k)),
                     dim3(kRgThreads), 0, s, f(L.part), n_split, m_ptr, stride, m, f(L.gpart));
      if (le != cudaSuccess) return le;
    }
    last_parts = static_cast<int>(parts);
    return cudaGetLastError();
  }
  mutable int last_parts = 0;

  cudaError_t finish(float* m_ptr, int64_t stride, int64_t m, int n_split) const {
    if (n_split == 0) return cudaSuccess;
    return reduce_gram(m_ptr, stride, m, n_split);
  }

  // orthonormalise the columns of every checkpoint's m × RP block
  cudaError_t orth(float* m_ptr, int64_t stride, int64_t m, int n_split) const {
    cudaError_t e = reduce_gram(m_ptr, stride, m, n_split);
    if (e != cudaSuccess) return e;
    {
      const cudaError_t le =
          launch_pdl(chol_factor_kernel<RP>, dim3(static_cast<unsigned>(a.k)), dim3(kMsThreads),
                     0, s, f(L.gpart), last_parts, a.rank, f(L.t));
      if (le != cudaSuccess) return le;
    }
    int64_t rows_blocks = (m + 7) / 8;
    if (rows_blocks > 1024) rows_blocks = 1024;
    {
      const cudaError_t le =
          launch_pdl(apply_right_kernel<RP>,
                     dim3(static_cast<unsigned>(rows_blocks), static_cast<unsigned>(a.k)),
                     dim3(kMsThreads), 0, s, m_ptr, stride, m, f(L.t));
      if (le != cudaSuccess) return le;
    }
    return cudaGetLastError();
  }

  cudaError_t run() const {
    cudaError_t e;
    if (a.rank > 0) {
      const int64_t n_om = a.d_in * RP;
      {
        const cudaError_t le =
            launch_pdl(sketch_fill_kernel,
                       dim3(static_cast<unsigned>((n_om + 255) / 256 < 4096 ? (n_om + 255) / 256
                                                                               : 4096)),
                       dim3(256), 0, s, f(L.omega), a.d_in, a.rank, RP, a.seed);
        if (le != cudaSuccess) return le;
      }
      if ((e = cudaGetLastError()) != cudaSuccess) return e;
      float* y = f(L.p);
      float* z = f(L.z);
      float* r = f(L.r);
      const int64_t ys = a.d_out * RP, zs = a.d_in * RP;
      int ns = 0;
      if ((e = delta_mul(false, f(L.omega), 0, y, ys, &ns)) != cudaSuccess) return e;
      if ((e = orth(y, ys, a.d_out, ns)) != cudaSuccess) return e;
      for (int it = 0; it < a.power_iters; ++it) {
        // Z = Δᵀ·Y needs no orthonormalisation of its own: only the span of
        // Y matters, and Y = Δ·Z is orthonormalised (its condition number
        // grows by at most (σ_1/σ_r)² per round)
        if ((e = delta_mul(true, y, ys, z, zs, &ns)) != cudaSuccess) return e;
        if ((e = finish(z, zs, a.d_in, ns)) != cudaSuccess) return e;
        if ((e = delta_mul(false, z, zs, y, ys, &ns)) != cudaSuccess) return e;
        if ((e = orth(y, ys, a.d_out, ns)) != cudaSuccess) return e;
      }
      if ((e = orth(y, ys, a.d_out, 0)) != cudaSuccess) return e;  // second Cholesky QR pass
      if ((e = delta_mul(true, y, ys, r, zs, &ns)) != cudaSuccess) return e;
      if ((e = finish(r, zs, a.d_in, ns)) != cudaSuccess) return e;
    }
    // merge: split the factors (P scaled by 1/k) into bf16 terms, then one
    // tensor-core pass over W_base
    const int64_t kp = a.rank > 0 ? static_cast<int64_t>(a.k) * RP : 0;
    uint16_t* fs = reinterpret_cast<uint16_t*>(ws + L.fsplit);
    uint16_t* phi = fs;
    uint16_t* plo = phi + a.d_out * kp;
    uint16_t* rhi = plo + a.d_out * kp;
    uint16_t* rlo = rhi + a.d_in * kp;
    if (kp > 0) {
      const int64_t np = a.d_out * (kp / 8), nr = a.d_in * (kp / 8);
      {
        const cudaError_t le =
            launch_pdl(fsplit_kernel,
                       dim3(static_cast<unsigned>((np + 255) / 256 < 4096 ? (np + 255) / 256
                                                                             : 4096)),
                       dim3(256), 0, s, f(L.p), a.d_out, RP, a.k, 1.0f / static_cast<float>(a.k),
                       phi, plo);
        if (le != cudaSuccess) return le;
      }
      {
        const cudaError_t le =
            launch_pdl(fsplit_kernel,
                       dim3(static_cast<unsigned>((nr + 255) / 256 < 4096 ? (nr + 255) / 256
                                                                             : 4096)),
                       dim3(256), 0, s, f(L.r), a.d_in, RP, a.k, 1.0f, rhi, rlo);
        if (le != cudaSuccess) return le;
      }
      if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    static bool merge_attr[64] = {};  // per device
    int dev = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    {
      std::lock_guard<std::mutex> lock(host_cache_mutex());
      if (!merge_attr[dev]) {
        if ((e = cudaFuncSetAttribute(merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      static_cast<int>(kMergeSmem))) != cudaSuccess)
          return e;
        merge_attr[dev] = true;
      }
    }
    const dim3 grid(static_cast<unsigned>((a.d_in + kMergeTile - 1) / kMergeTile),
                    static_cast<unsigned>((a.d_out + kMergeTile - 1) / kMergeTile));
    {
      const cudaError_t le =
          launch_pdl(merge_kernel, dim3(grid), dim3(kMulThreads), kMergeSmem, s, a.w_base, phi,
                     plo, rhi, rlo, kp, a.d_out, a.d_in, a.w_merged, a.correction);
      if (le != cudaSuccess) return le;
    }
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
  if (a.k < 1 || a.k > kMaxCkpt) return cudaErrorInvalidValue;
  CkptTable tab{};
  for (int i = 0; i < a.k; ++i) tab.p[i] = a.w_ft[i];
  switch (L.rp) {
    case 16:
      return MsRunner<16>{a, stream, ws, L, num_sms, tab}.run();
    case 32:
      return MsRunner<32>{a, stream, ws, L, num_sms, tab}.run();
    default:
      return MsRunner<64>{a, stream, ws, L, num_sms, tab}.run();
  }
}

}  // namespace bd
