// compress.cu — BitDelta compression in one pass over W_base and W_ft.
//
// Page "BitDelta: serving 14 Zen models from one GPU cluster", section
// "Mathematical foundation": Δ = W_ft − W_base; each Δ_ij reduced to one sign
// bit; α = (1/n)·‖Δ‖₁ = mean|Δ_ij| per matrix.  Section "Infrastructure
// details": the signs are stored 8 per byte, α as float32, one per output
// dimension.  Bit j of byte k holds column 8k+j, 1 = +1, sign(0) = +1.
//
// Layout of the work: one warp per row (grid-stride over rows).  Lane L owns
// the 8 adjacent columns of chunk L, L+32, ... (one 16-byte load from each
// matrix), so it forms its sign byte from its own 8 comparisons and stores it
// directly: the 32 lanes write 32 consecutive bytes.  (A warp ballot would
// need one column per lane, i.e. 2-byte loads; the register-local byte is
// cheaper and gives the same bits.)  |Δ| is summed per lane in fp32 (pairwise
// over the 8 values, then Neumaier-compensated across chunks), the lanes'
// (sum, compensation) pairs are combined with error-free TwoSum steps, and the
// row total is formed in fp64.  Per-matrix α adds the fp64 row totals in a
// fixed order in the last block to finish, so the result does not depend on
// scheduling.
#include <cstdint>
#include <mutex>

#include "bitdelta.h"
#include "common.cuh"
#include "kernels.h"

namespace bd {
namespace {

constexpr int kWarpsPerBlock = 8;
// 16-byte chunks in flight per lane and input: 4 measured fastest (6 and 8: 13% slower)
#ifndef BD_COMPRESS_UNROLL
#define BD_COMPRESS_UNROLL 4
#endif
constexpr int kUnroll = BD_COMPRESS_UNROLL;

struct FloatFloat {
  float s, c;
};

// Error-free combination of two compensated partial sums.
__device__ __forceinline__ FloatFloat ff_add(FloatFloat a, FloatFloat b) {
  const float s = __fadd_rn(a.s, b.s);
  const float bb = __fsub_rn(s, a.s);
  const float err = __fadd_rn(__fsub_rn(a.s, __fsub_rn(s, bb)), __fsub_rn(b.s, bb));
  return {s, __fadd_rn(__fadd_rn(a.c, b.c), err)};
}

// 8 columns: sign byte and the pairwise fp32 sum of |Δ|.
__device__ __forceinline__ uint32_t chunk_signs_abs(const uint4 wb, const uint4 wf, float& abs8) {
  const uint32_t b[4] = {wb.x, wb.y, wb.z, wb.w};
  const uint32_t f[4] = {wf.x, wf.y, wf.z, wf.w};
  uint32_t byte = 0;
  float pair[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float d0 = __fsub_rn(bf16lo_to_f32(f[j]), bf16lo_to_f32(b[j]));
    const float d1 = __fsub_rn(bf16hi_to_f32(f[j]), bf16hi_to_f32(b[j]));
    // bit 1 unless Δ < 0 (so ±0 deltas give +1)
    byte |= (d0 < 0.f ? 0u : 1u) << (2 * j);
    byte |= (d1 < 0.f ? 0u : 1u) << (2 * j + 1);
    pair[j] = __fadd_rn(fabsf(d0), fabsf(d1));
  }
  abs8 = __fadd_rn(__fadd_rn(pair[0], pair[1]), __fadd_rn(pair[2], pair[3]));
  return byte;
}

// Neumaier step for non-negative terms.
__device__ __forceinline__ void neumaier_add(FloatFloat& acc, float v) {
  const float t = __fadd_rn(acc.s, v);
  const float hi = fmaxf(acc.s, v);
  const float lo = fminf(acc.s, v);
  acc.c = __fadd_rn(acc.c, __fadd_rn(__fsub_rn(hi, t), lo));
  acc.s = t;
}

template <bool kPerRow>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
    compress_kernel(const uint16_t* __restrict__ w_base, const uint16_t* __restrict__ w_ft,
                    int64_t d_out, int64_t d_in, uint8_t* __restrict__ packed,
                    float* __restrict__ alpha, double* __restrict__ row_sums,
                    unsigned int* __restrict__ done_counter, DevCtx ctx) {
  (void)ctx;
  // No early signal to dependents: what this kernel writes can be a weight
  // operand of the next call, and bitdelta_linear reads weights before it
  // waits for the previous kernel, so a dependent starts only once this
  // grid has finished.  The wait covers inputs an earlier kernel writes.
  griddep_wait();
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int64_t chunks = d_in / 8;  // sign bytes per row
  const int64_t row_step = static_cast<int64_t>(gridDim.x) * kWarpsPerBlock;

  for (int64_t row = static_cast<int64_t>(blockIdx.x) * kWarpsPerBlock + warp; row < d_out;
       row += row_step) {
    const uint4* pb = reinterpret_cast<const uint4*>(w_base + row * d_in);
    const uint4* pf = reinterpret_cast<const uint4*>(w_ft + row * d_in);
    uint8_t* prow = packed + row * chunks;
    FloatFloat acc{0.f, 0.f};
    int64_t k = lane;
    for (; k + 32 * (kUnroll - 1) < chunks; k += 32 * kUnroll) {
      uint4 vb[kUnroll], vf[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        vb[u] = ldg_stream_v4(pb + k + 32 * u);
        vf[u] = ldg_stream_v4(pf + k + 32 * u);
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        float s8;
        prow[k + 32 * u] = static_cast<uint8_t>(chunk_signs_abs(vb[u], vf[u], s8));
        neumaier_add(acc, s8);
      }
    }
    for (; k < chunks; k += 32) {
      float s8;
      prow[k] = static_cast<uint8_t>(chunk_signs_abs(ldg_stream_v4(pb + k), ldg_stream_v4(pf + k), s8));
      neumaier_add(acc, s8);
    }
    // combine the 32 lanes' compensated sums (fixed butterfly order)
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      FloatFloat o{__shfl_xor_sync(0xFFFFFFFFu, acc.s, off), __shfl_xor_sync(0xFFFFFFFFu, acc.c, off)};
      acc = (lane & off) ? ff_add(o, acc) : ff_add(acc, o);
    }
    if (lane == 0) {
      const double total = static_cast<double>(acc.s) + static_cast<double>(acc.c);
      if (kPerRow)
        alpha[row] = static_cast<float>(total / static_cast<double>(d_in));
      else
        row_sums[row] = total;
    }
  }

  if (!kPerRow) {
    // Last block to finish adds the row totals in a fixed order.
    __shared__ unsigned int is_last;
    __shared__ double partial[kWarpsPerBlock * 32];
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) is_last = (atomicAdd(done_counter, 1u) == gridDim.x - 1) ? 1u : 0u;
    __syncthreads();
    if (is_last) {
      __threadfence();
      double s = 0.0;
      for (int64_t r = threadIdx.x; r < d_out; r += blockDim.x) s += __ldcg(row_sums + r);
      partial[threadIdx.x] = s;
      __syncthreads();
      for (int w = blockDim.x / 2; w > 0; w >>= 1) {
        if (threadIdx.x < w) partial[threadIdx.x] += partial[threadIdx.x + w];
        __syncthreads();
      }
      if (threadIdx.x == 0) {
        alpha[0] = static_cast<float>(partial[0] /
                                      (static_cast<double>(d_out) * static_cast<double>(d_in)));
        *done_counter = 0u;  // leave the counter reset for the next call
      }
    }
  }
}

}  // namespace

cudaError_t launch_compress(const uint16_t* w_base, const uint16_t* w_ft, int64_t d_out,
                            int64_t d_in, bool per_row, uint8_t* packed, float* alpha,
                            double* row_sums, unsigned int* done_counter, int num_sms,
                            cudaStream_t stream, DevCtx ctx) {
  const int64_t blocks_needed = (d_out + kWarpsPerBlock - 1) / kWarpsPerBlock;
  const int64_t max_blocks = static_cast<int64_t>(num_sms) * 8;
  const int grid = static_cast<int>(blocks_needed < max_blocks ? blocks_needed : max_blocks);
  const dim3 block(kWarpsPerBlock * 32);
  if (per_row)
    return launch_pdl(compress_kernel<true>, dim3(grid), block, 0, stream, w_base, w_ft, d_out,
                      d_in, packed, alpha, static_cast<double*>(nullptr),
                      static_cast<unsigned int*>(nullptr), ctx);
  return launch_pdl(compress_kernel<false>, dim3(grid), block, 0, stream, w_base, w_ft, d_out,
                    d_in, packed, alpha, row_sums, done_counter, ctx);
}

}  // namespace bd

// ------------------------------------------------------------------ no-alloc

// Fixed scratch for bitdelta_compress_noalloc: a 256-byte slot for the
// completion counter, then one fp64 row total per output row.  Every GPU that
// loads the library keeps this array for the life of the process.
namespace {

constexpr int64_t kNoAllocMaxRows = 65536;
constexpr size_t kNoAllocScratchBytes = 256 + 8 * static_cast<size_t>(kNoAllocMaxRows);
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of g_noalloc_scratch per device, looked up once per device
// with that device current (the host-side symbol is not a device address).
uint8_t* g_noalloc_ptr[64] = {};
std::mutex g_noalloc_mu;

bd_status noalloc_scratch(uint8_t** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return BD_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (g_noalloc_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
      return BD_ERR_CUDA;
    g_noalloc_ptr[dev] = static_cast<uint8_t*>(p);
  }
  *out = g_noalloc_ptr[dev];
  return BD_OK;
}

}  // namespace

extern "C" bd_status bitdelta_compress_noalloc(const uint16_t* w_base, const uint16_t* w_ft,
                                               int64_t d_out, int64_t d_in, bd_alpha_mode mode,
                                               uint8_t* packed_out, float* alpha_out,
                                               bd_stream_t stream) {
  if (!w_base || !w_ft || !packed_out || !alpha_out) return BD_ERR_INVALID_ARG;
  if (mode != BD_ALPHA_PER_MATRIX && mode != BD_ALPHA_PER_ROW) return BD_ERR_INVALID_ARG;
  if (d_out < 1 || d_in < 1) return BD_ERR_INVALID_ARG;
  if (d_in % 8 != 0 || d_in > (int64_t{1} << 40) || d_out > (int64_t{1} << 62) / d_in)
    return BD_ERR_UNSUPPORTED_SHAPE;
  if (mode == BD_ALPHA_PER_MATRIX && d_out > kNoAllocMaxRows) return BD_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(w_base) % 16 || reinterpret_cast<uintptr_t>(w_ft) % 16 ||
      reinterpret_cast<uintptr_t>(alpha_out) % 4)
    return BD_ERR_MISALIGNED;
  bd::DevCtx ctx;
  int num_sms = 0;
  bd_status st = static_cast<bd_status>(bd::current_device_context(&ctx, &num_sms));
  if (st != BD_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  unsigned int* counter = nullptr;
  double* row_sums = nullptr;
  if (mode == BD_ALPHA_PER_MATRIX) {
    uint8_t* scratch = nullptr;
    if ((st = noalloc_scratch(&scratch)) != BD_OK) return st;
    counter = reinterpret_cast<unsigned int*>(scratch);
    row_sums = reinterpret_cast<double*>(scratch + 256);
    // the counter must start at zero; the row totals are all overwritten
    if (cudaMemsetAsync(counter, 0, sizeof(unsigned int), s) != cudaSuccess) return BD_ERR_CUDA;
  }
  return bd::launch_compress(w_base, w_ft, d_out, d_in, mode == BD_ALPHA_PER_ROW, packed_out,
                             alpha_out, row_sums, counter, num_sms, s, ctx) == cudaSuccess
             ? BD_OK
             : BD_ERR_CUDA;
}
