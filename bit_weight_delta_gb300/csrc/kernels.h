// kernels.h — launchers of the BitDelta CUDA kernels (internal to the library;
// the public interface is include/bitdelta.h).
#pragma once

#include <cstddef>
#include <cstdint>
#include <mutex>
#include <utility>
#include <cuda.h>
#include <cuda_runtime.h>

#include "common.cuh"

namespace bd {

// Launch `kernel` with programmatic stream serialisation (see griddep_wait).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Row-major 2D tensor map [rows, cols] of elem_bytes-sized elements with a
// (box_cols x box_rows) box; out-of-range elements read as zero.  False when
// the driver rejects it (alignment, strides, box) or cannot be reached.
bool encode_tmap_2d(CUtensorMap* map, CUtensorMapDataType dtype, int elem_bytes, const void* base,
                    int64_t rows, int64_t cols, uint32_t box_cols, uint32_t box_rows,
                    CUtensorMapSwizzle swizzle);

// Current device's error word, wait limit and SM count (a bd_status code).
int current_device_context(DevCtx* ctx, int* num_sms);

// Guards the per-device launch caches (kernel attributes raised once per
// device, occupancy results): host threads may launch on one device at once.
std::mutex& host_cache_mutex();

cudaError_t launch_compress(const uint16_t* w_base, const uint16_t* w_ft, int64_t d_out,
                            int64_t d_in, bool per_row, uint8_t* packed, float* alpha,
                            double* row_sums, unsigned int* done_counter, int num_sms,
                            cudaStream_t stream, DevCtx ctx);

cudaError_t launch_reconstruct(const uint16_t* w_base, const uint8_t* packed, const float* alpha,
                               bool per_row, int64_t d_out, int64_t d_in, uint16_t* w_out,
                               int num_sms, cudaStream_t stream);

// Decode-size linear (mma.sync, bandwidth-bound).
struct GemvArgs {
  const uint16_t* x;
  int64_t M;  // rows of x (single) or M_total (grouped)
  const uint16_t* w;
  int64_t d_out, d_in;
  const uint8_t* packed;  // single-variant mode
  const float* alpha;
  int per_row;
  uint16_t* y;
  // multi-tenant mode
  const int32_t* seg_off;
  const int32_t* seg_var;
  int32_t n_seg, n_var, max_short;
  const uint8_t* const* packed_table;
  const float* const* alpha_table;
  DevCtx ctx;
};

cudaError_t launch_gemv(const GemvArgs& p, int num_sms, cudaStream_t stream);

size_t gemv_grouped_smem_bytes(int32_t n_var, int64_t max_rows);
cudaError_t launch_gemv_grouped(const GemvArgs& p, int64_t max_rows, int num_sms,
                                cudaStream_t stream);

// Prefill-size linear (tcgen05 + TMA).
struct GemmArgs {
  int64_t M, d_out, d_in;
  const uint8_t* packed;  // single-variant mode
  const float* alpha;
  int per_row;
  uint16_t* y;
  // multi-tenant mode (seg_off == nullptr for the single-variant call)
  const int32_t* seg_off;
  const int32_t* seg_var;
  int32_t n_seg, n_var, max_short;
  const uint8_t* const* packed_table;
  const float* const* alpha_table;
  DevCtx ctx;
  // single-variant mode: when tile_hi > 0, only flat tiles [tile_lo,
  // tile_hi) of the call's tile order (row tiles outer, token tiles inner)
  int64_t tile_lo, tile_hi;
  // single-variant mode, split region (sk_tiles > 0; needs tile_hi > 0):
  // flat tiles [sk_lo, sk_lo + sk_tiles), taken after each pair's whole tiles
  // of [tile_lo, tile_hi).  Their k-blocks, tile after tile, are cut into one
  // contiguous range per pair of the launch; a tile that several pairs share
  // is summed from fp32 partials in sk_part, in k order, by the last of its
  // contributors (sk_count), so the result does not depend on timing.
  int64_t sk_lo, sk_tiles;
  float* sk_part;          // [n_pairs][2][2 CTAs][BN tokens][128 rows] fp32
  unsigned int* sk_count;  // [sk_tiles][2 CTAs][4 epilogue warps], zero at launch
};

constexpr int kGemmMaxSegs = 1024;
int gemm_block_rows();    // d_out rows per CTA of a pair tile (128)

// Prefill-size linear on CTA pairs (tcgen05 cta_group::2): tiles of
// 2 * gemm_block_rows() output rows x gemm_pair_tokens(wide) tokens (256, or
// 512 for the wide tile); tmap_w's box has gemm_block_rows() rows, tmap_x's
// box gemm_pair_x_rows() (half of one MMA's 256 tokens), both
// gemm_pair_block_k() (narrow) or gemm_pair_wide_block_k() (wide) columns.
// pair_tiles_bound caps the pairs launched.
int gemm_pair_x_rows();
int gemm_pair_block_k();
int gemm_pair_wide_block_k();
int gemm_pair_tokens(bool wide);
// CTA pairs of that kernel the current device holds at once (0 if none fits;
// negative cudaError_t on a failed query).
int gemm_pair_capacity(bool wide);
// Split-region workspace of a launch of `pairs` pairs of the 512-token kernel
// over sk_tiles tiles: counters first (sk_count, 256-byte padded), then the
// partial slots (sk_part).
size_t gemm_split_count_bytes(int64_t sk_tiles);
size_t gemm_split_part_bytes(int64_t pairs);
cudaError_t launch_gemm_pair(const GemmArgs& p, const CUtensorMap& tmap_w,
                             const CUtensorMap& tmap_x, int64_t pair_tiles_bound, bool wide,
                             cudaStream_t stream);

// Cosine similarity of 1-bit task vectors (K-Merge).  sign_similarity_grid
// bounds the CTAs of a launch (the launch takes at most one wave of the
// device); workspace (sign_similarity_workspace_bytes): 256 bytes of
// counters, zeroed before the first call, then (2·n_b + 1) doubles per CTA
// of that bound and per group of 32 of them.
int sign_similarity_grid(int64_t d_out);
size_t sign_similarity_workspace_bytes(int64_t d_out, int32_t n_b);
cudaError_t launch_sign_similarity(const uint8_t* pa, const float* aa,
                                   const uint8_t* const* pb_table, const float* const* ab_table,
                                   int32_t n_b, bool per_row, int64_t d_out, int64_t d_in,
                                   double* cos_out, int32_t* best_out, void* workspace,
                                   bool vec, cudaStream_t stream);

// MonoSoup merge (monosoup.cu).  w_ft: host array of k device pointers.
struct MonoSoupArgs {
  const uint16_t* w_base;
  const uint16_t* const* w_ft;
  int k, rank, power_iters;
  uint64_t seed;
  int64_t d_out, d_in;
  uint16_t* w_merged;
  float* correction;  // nullable: fp32 (1/k)·Σ τ_i
};
size_t monosoup_workspace_bytes(int64_t d_out, int64_t d_in, int k, int rank);
cudaError_t launch_monosoup(const MonoSoupArgs& a, void* workspace, int num_sms,
                            cudaStream_t stream);

// Test hook: one CTA waiting on an mbarrier nothing completes.
cudaError_t launch_wait_timeout_probe(DevCtx ctx, cudaStream_t stream);

}  // namespace bd
