// abi.cu — the C ABI of include/bitdelta.h: host-side argument checks, the
// per-device error word, TMA descriptor encoding and kernel dispatch.
#include <atomic>
#include <climits>
#include <cstdint>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "bitdelta.h"
#include "kernels.h"
#include "split_schedule.h"

namespace {

// Sticky device error word; kernels receive its device address.
__device__ uint32_t g_error_word;

std::atomic<uint64_t> g_wait_limit_ns{2000000000ull};
std::atomic<int> g_prefill_tile{BD_PREFILL_TILE_AUTO};

constexpr int kMaxDevices = 64;
constexpr int64_t kDecodeMaxRows = 16;
// Shared memory the decode kernel's grouped pass may give to its bucket
// counts and short-row index list (the rest of the SM's shared memory is its
// cp.async ring).
constexpr size_t kGroupedListBytes = 200 * 1024;

struct DeviceState {
  bool ready = false;
  uint32_t* err = nullptr;
  int num_sms = 0;
};
DeviceState g_dev[kMaxDevices];
std::mutex g_dev_mu;

bd_status current_device(DeviceState** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return BD_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_dev_mu);
  DeviceState& s = g_dev[dev];
  if (!s.ready) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_error_word) != cudaSuccess) return BD_ERR_CUDA;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return BD_ERR_CUDA;
    if (cudaMemset(p, 0, sizeof(uint32_t)) != cudaSuccess) return BD_ERR_CUDA;
    s.err = static_cast<uint32_t*>(p);
    s.num_sms = sms;
    s.ready = true;
  }
  *out = &s;
  return BD_OK;
}

bd::DevCtx make_ctx(const DeviceState* s) {
  bd::DevCtx c;
  c.err = s->err;
  c.wait_limit_ns = g_wait_limit_ns.load();
  return c;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bd_status check_dims(int64_t d_out, int64_t d_in) {
  if (d_out < 1 || d_in < 1) return BD_ERR_INVALID_ARG;
  if (d_in % 8 != 0) return BD_ERR_UNSUPPORTED_SHAPE;
  if (d_out > (int64_t{1} << 40) || d_in > (int64_t{1} << 40) ||
      d_out > (int64_t{1} << 62) / d_in)
    return BD_ERR_UNSUPPORTED_SHAPE;
  return BD_OK;
}

bool mode_ok(bd_alpha_mode m) { return m == BD_ALPHA_PER_MATRIX || m == BD_ALPHA_PER_ROW; }

bd_status from_cuda(cudaError_t e) { return e == cudaSuccess ? BD_OK : BD_ERR_CUDA; }

// ------------------------------------------------------------------ TMA maps

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// Row-major bf16 [rows, cols] as a 2D tensor with a (box_cols x box_rows)
// box; box_cols = 64 (32) uses the 128-byte (64-byte) swizzle.  Out-of-range
// elements read as zero.
bool make_tmap_bf16(CUtensorMap* map, const void* base, int64_t rows, int64_t cols,
                    uint32_t box_cols, uint32_t box_rows) {
  return bd::encode_tmap_2d(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, rows, cols, box_cols,
                            box_rows,
                            box_cols == 64 ? CU_TENSOR_MAP_SWIZZLE_128B
                                           : CU_TENSOR_MAP_SWIZZLE_64B);
}

// Can the tensor-core kernel take this problem?
bool tc_shape_ok(int64_t rows_x, int64_t d_out, int64_t d_in) {
  return d_in % 128 == 0 && d_in < INT32_MAX && d_out < INT32_MAX && rows_x < INT32_MAX;
}

// Cost of one 512-token pair tile in 256-token pair tiles, in eighths: the
// steady state of the two kernels on 8192 x 57344 at M = 2048 measured 1454
// and 1266 TFLOP/s (2 x 1266 / 1454 = 1.74); on 8192 x 10240 three rounds of
// 512-token tiles took 300.6 µs against 308.0 for five rounds of 256-token
// tiles (1.64).  13/8 picks the 512-token tile there and leaves every other
// benchmark shape's choice as it was.
constexpr int64_t kWideTileCost8 = 13;

// 512-token pair tiles for this call?  Under BD_PREFILL_TILE_AUTO the width
// whose rounds of tiles over the device's pairs cost less, ceil(tiles /
// pairs) x the cost of one tile, with ceil(rows_x / width) token tiles per
// row tile (exact for one run of M rows; for a grouped batch, whose long
// segments the host cannot see, the same estimate over M_total); on a tie
// the 512-token tile (half the transform work).  long_tokens <= 256 (no
// segment fills half a wide tile) keeps 256.  Measured on the grouped
// workload (64 one-row and four 512-row segments over 4096 -> 14336): 0.462
// ms with 512-token tiles, 0.499 with 256.
bool use_wide_tiles(int64_t d_out, int64_t rows_x, int64_t long_tokens) {
  const int policy = g_prefill_tile.load();
  if (policy == BD_PREFILL_TILE_256) return false;
  if (policy == BD_PREFILL_TILE_512) return true;
  if (long_tokens <= bd::gemm_pair_tokens(false)) return false;
  const int pairs = bd::gemm_pair_capacity(true);
  if (pairs < 1) return false;  // the launch reports why
  const int64_t row_tiles = (d_out + 2 * bd::gemm_block_rows() - 1) / (2 * bd::gemm_block_rows());
  auto rounds = [&](bool wide) {
    const int64_t tok = bd::gemm_pair_tokens(wide);
    const int64_t tiles = row_tiles * ((rows_x + tok - 1) / tok);
    return (tiles + pairs - 1) / pairs;
  };
  return rounds(true) * kWideTileCost8 <= rounds(false) * 8;
}

// Launch the tensor-core kernel on g (x has rows_x rows, of which the
// longest run of one tile schedule — M, or the longest segment — has
// long_tokens; extra_tiles bounds the ragged token tiles beyond
// ceil(rows_x / tile tokens), one per segment in grouped mode): the pair
// kernel (cta_group::2, 256 output rows by 256 or 512 tokens per tile,
// use_wide_tiles).  Returns false, launching nothing, when a tensor map
// cannot be encoded or the device cannot place a cluster of two of its CTAs
// (every GB300 can); the caller then runs the rows on the decode kernel.
bool launch_tc(const bd::GemmArgs& g, const void* w_base, const void* x, int64_t rows_x,
               int64_t long_tokens, int64_t extra_tiles, void* ws, size_t ws_bytes,
               cudaStream_t s, cudaError_t* err) {
  CUtensorMap tw, tx;
  const bool wide = use_wide_tiles(g.d_out, rows_x, long_tokens);
  const int bk = wide ? bd::gemm_pair_wide_block_k() : bd::gemm_pair_block_k();
  const int64_t tok = bd::gemm_pair_tokens(wide);
  if (!make_tmap_bf16(&tw, w_base, g.d_out, g.d_in, bk, bd::gemm_block_rows()) ||
      !make_tmap_bf16(&tx, x, rows_x, g.d_in, bk, bd::gemm_pair_x_rows()))
    return false;
  const int64_t row_tiles = (g.d_out + 2 * bd::gemm_block_rows() - 1) / (2 * bd::gemm_block_rows());
  const int64_t pair_tiles = row_tiles * ((rows_x + tok - 1) / tok + extra_tiles);
  // With a split workspace, one run of M rows on 512-token tiles whose last
  // round is small (at most a quarter of the device's pairs): all rounds but
  // the last whole one run as whole tiles, and the k-blocks of the rest (that
  // round's tiles and the remainder) are cut evenly over the pairs, so every
  // pair ends at about the same time instead of a last round with idle
  // pairs.  Each pair's range spans more than one tile, so at most two pairs
  // share a tile; their fp32 partials are summed in k order (deterministic).
  // Measured on GB300, the split region runs ~20% slower per k-block than
  // rounds of whole tiles (its pairs no longer read the same x blocks at the
  // same time): 8192 -> 10240 at M = 2048 (160 tiles, a last round of 8)
  // 287 -> 261 µs, but 8192 -> 8192 (128 tiles, 52 in the last round)
  // 211 -> 218 µs, hence the quarter.
  if (ws != nullptr && wide && g.seg_off == nullptr) {
    const int pairs = bd::gemm_pair_capacity(true);
    const int64_t full = pairs > 0 ? pair_tiles / pairs : 0;
    const int64_t rem = pairs > 0 ? pair_tiles - full * pairs : 0;
    if (full >= 1 && rem > 0 && 4 * rem <= pairs) {
      const int64_t sk_tiles = rem + pairs;
      const size_t count_bytes = bd::gemm_split_count_bytes(sk_tiles);
      if (count_bytes + bd::gemm_split_part_bytes(pairs) <= ws_bytes) {
        *err = cudaMemsetAsync(ws, 0, count_bytes, s);
        if (*err != cudaSuccess) return true;
        bd::GemmArgs sg = g;
        sg.tile_lo = 0;
        sg.tile_hi = (full - 1) * pairs;
        sg.sk_lo = sg.tile_hi;
        sg.sk_tiles = sk_tiles;
        sg.sk_count = static_cast<unsigned int*>(ws);
        sg.sk_part = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + count_bytes);
        *err = bd::launch_gemm_pair(sg, tw, tx, pairs, true, s);
        if (*err != cudaErrorInvalidConfiguration) return true;
        (void)cudaGetLastError();  // no cluster of two fits: nothing was launched
        return false;
      }
    }
  }
  // One run of M rows on 512-token tiles (width chosen per shape) whose last
  // round is small (at most half the pairs): that round's tiles (a suffix of
  // the flat tile order) run instead as twice as many 256-token tiles in a
  // second launch, all at once, for ~0.6 of a 512-token round.  8192 ->
  // 10240 at M = 2048: 160 tiles over 76 pairs, the last 8 as 16; 300 -> 272
  // µs.  The two widths give bit-identical outputs.
  const bool auto_width = g_prefill_tile.load() == BD_PREFILL_TILE_AUTO;
  const int pairs = wide && auto_width && g.seg_off == nullptr ? bd::gemm_pair_capacity(true) : 0;
  const int64_t full = pairs > 0 ? pair_tiles / pairs : 0;
  const int64_t rem = pairs > 0 ? pair_tiles - full * pairs : 0;
  if (full >= 1 && rem > 0 && 2 * rem <= pairs) {
    bd::GemmArgs head = g;
    head.tile_lo = 0;
    head.tile_hi = full * pairs;
    *err = bd::launch_gemm_pair(head, tw, tx, full * pairs, true, s);
    if (*err == cudaErrorInvalidConfiguration) {
      (void)cudaGetLastError();  // no cluster of two fits: nothing was launched
      return false;
    }
    if (*err != cudaSuccess) return true;
    CUtensorMap tw_n, tx_n;
    const int bk_n = bd::gemm_pair_block_k();
    if (!make_tmap_bf16(&tw_n, w_base, g.d_out, g.d_in, bk_n, bd::gemm_block_rows()) ||
        !make_tmap_bf16(&tx_n, x, rows_x, g.d_in, bk_n, bd::gemm_pair_x_rows())) {
      *err = cudaErrorInvalidValue;  // the maps above were accepted: cannot happen
      return true;
    }
    // wide tile (nt, j) is narrow tiles (nt, 2j) and (nt, 2j + 1)
    const int64_t t_wide = (rows_x + tok - 1) / tok;
    const int64_t tok_n = bd::gemm_pair_tokens(false);
    const int64_t t_narrow = (rows_x + tok_n - 1) / tok_n;
    const int64_t first = full * pairs;
    bd::GemmArgs tail = g;
    tail.tile_lo = (first / t_wide) * t_narrow + 2 * (first % t_wide);
    tail.tile_hi = row_tiles * t_narrow;
    *err = bd::launch_gemm_pair(tail, tw_n, tx_n, tail.tile_hi - tail.tile_lo, false, s);
    return true;
  }
  *err = bd::launch_gemm_pair(g, tw, tx, pair_tiles, wide, s);
  if (*err != cudaErrorInvalidConfiguration) return true;
  (void)cudaGetLastError();  // no cluster of two fits: nothing was launched
  return false;
}

}  // namespace

namespace bd {
bool encode_tmap_2d(CUtensorMap* map, CUtensorMapDataType dtype, int elem_bytes, const void* base,
                    int64_t rows, int64_t cols, uint32_t box_cols, uint32_t box_rows,
                    CUtensorMapSwizzle swizzle) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * static_cast<cuuint64_t>(elem_bytes)};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  std::memset(map, 0, sizeof(*map));
  return fn(map, dtype, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

std::mutex& host_cache_mutex() {
  static std::mutex mu;
  return mu;
}

// Error word, wait limit and SM count of the current device, for entry points
// defined outside this file.  Returns a bd_status.
int current_device_context(DevCtx* ctx, int* num_sms) {
  DeviceState* dev = nullptr;
  const bd_status st = current_device(&dev);
  if (st != BD_OK) return st;
  *ctx = make_ctx(dev);
  *num_sms = dev->num_sms;
  return BD_OK;
}
}  // namespace bd

extern "C" {

size_t bitdelta_packed_bytes(int64_t d_out, int64_t d_in) {
  if (check_dims(d_out, d_in) != BD_OK) return 0;
  return static_cast<size_t>(d_out) * static_cast<size_t>(d_in / 8);
}

size_t bitdelta_compress_workspace_bytes(int64_t d_out, int64_t d_in, bd_alpha_mode mode) {
  if (check_dims(d_out, d_in) != BD_OK || !mode_ok(mode)) return 0;
  return mode == BD_ALPHA_PER_ROW ? 0 : static_cast<size_t>(d_out) * 8 + 256;
}

bd_status bitdelta_compress(const uint16_t* w_base, const uint16_t* w_ft, int64_t d_out,
                            int64_t d_in, bd_alpha_mode mode, uint8_t* packed_out,
                            float* alpha_out, void* workspace, size_t workspace_bytes,
                            bd_stream_t stream) {
  if (!w_base || !w_ft || !packed_out || !alpha_out || !mode_ok(mode)) return BD_ERR_INVALID_ARG;
  bd_status st = check_dims(d_out, d_in);
  if (st != BD_OK) return st;
  if (!aligned(w_base, 16) || !aligned(w_ft, 16) || !aligned(alpha_out, 4))
    return BD_ERR_MISALIGNED;
  const size_t need = bitdelta_compress_workspace_bytes(d_out, d_in, mode);
  if (need > 0 && (workspace == nullptr || workspace_bytes < need)) return BD_ERR_WORKSPACE;
  if (need > 0 && !aligned(workspace, 16)) return BD_ERR_MISALIGNED;
  DeviceState* dev = nullptr;
  if ((st = current_device(&dev)) != BD_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  unsigned int* counter = nullptr;
  double* row_sums = nullptr;
  if (mode == BD_ALPHA_PER_MATRIX) {
    counter = static_cast<unsigned int*>(workspace);
    row_sums = reinterpret_cast<double*>(static_cast<uint8_t*>(workspace) + 256);
    if (cudaMemsetAsync(counter, 0, sizeof(unsigned int), s) != cudaSuccess) return BD_ERR_CUDA;
  }
  return from_cuda(bd::launch_compress(w_base, w_ft, d_out, d_in, mode == BD_ALPHA_PER_ROW,
                                       packed_out, alpha_out, row_sums, counter, dev->num_sms, s,
                                       make_ctx(dev)));
}

bd_status bitdelta_reconstruct(const uint16_t* w_base, const uint8_t* packed, const float* alpha,
                               bd_alpha_mode mode, int64_t d_out, int64_t d_in, uint16_t* w_out,
                               bd_stream_t stream) {
  if (!w_base || !packed || !alpha || !w_out || !mode_ok(mode)) return BD_ERR_INVALID_ARG;
  bd_status st = check_dims(d_out, d_in);
  if (st != BD_OK) return st;
  if (!aligned(w_base, 16) || !aligned(w_out, 16) || !aligned(alpha, 4)) return BD_ERR_MISALIGNED;
  DeviceState* dev = nullptr;
  if ((st = current_device(&dev)) != BD_OK) return st;
  return from_cuda(bd::launch_reconstruct(w_base, packed, alpha, mode == BD_ALPHA_PER_ROW, d_out,
                                          d_in, w_out, dev->num_sms,
                                          reinterpret_cast<cudaStream_t>(stream)));
}

size_t bitdelta_linear_workspace_bytes(int64_t M, int64_t d_out, int64_t d_in) {
  if (check_dims(d_out, d_in) != BD_OK || M <= kDecodeMaxRows || M > INT32_MAX ||
      !tc_shape_ok(M, d_out, d_in))
    return 0;
  DeviceState* dev = nullptr;
  if (current_device(&dev) != BD_OK) return 0;
  const int pairs = bd::gemm_pair_capacity(true);
  if (pairs < 1) return 0;
  return bd::gemm_split_count_bytes(2 * static_cast<int64_t>(pairs)) +
         bd::gemm_split_part_bytes(pairs);
}

bd_status bitdelta_linear(const uint16_t* x, int64_t M, const uint16_t* w_base,
                          const uint8_t* packed, const float* alpha, bd_alpha_mode mode,
                          int64_t d_out, int64_t d_in, uint16_t* y, bd_stream_t stream) {
  return bitdelta_linear_ws(x, M, w_base, packed, alpha, mode, d_out, d_in, y, nullptr, 0,
                            stream);
}

bd_status bitdelta_linear_ws(const uint16_t* x, int64_t M, const uint16_t* w_base,
                             const uint8_t* packed, const float* alpha, bd_alpha_mode mode,
                             int64_t d_out, int64_t d_in, uint16_t* y, void* ws,
                             size_t ws_bytes, bd_stream_t stream) {
  if (M < 0 || !mode_ok(mode)) return BD_ERR_INVALID_ARG;
  if (ws != nullptr && !aligned(ws, 256)) return BD_ERR_MISALIGNED;
  if (M > 0 && (!x || !w_base || !packed || !alpha || !y)) return BD_ERR_INVALID_ARG;
  bd_status st = check_dims(d_out, d_in);
  if (st != BD_OK) return st;
  if (M == 0) return BD_OK;
  if (M > INT32_MAX) return BD_ERR_UNSUPPORTED_SHAPE;
  if (!aligned(x, 16) || !aligned(w_base, 16) || !aligned(y, 16) || !aligned(alpha, 4))
    return BD_ERR_MISALIGNED;
  if (ws != nullptr && ws_bytes < bitdelta_linear_workspace_bytes(M, d_out, d_in))
    return BD_ERR_WORKSPACE;
  DeviceState* dev = nullptr;
  if ((st = current_device(&dev)) != BD_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const bd::DevCtx ctx = make_ctx(dev);

  if (M > kDecodeMaxRows && tc_shape_ok(M, d_out, d_in) && aligned(packed, 16)) {
    bd::GemmArgs g{};
    g.M = M;
    g.d_out = d_out;
    g.d_in = d_in;
    g.packed = packed;
    g.alpha = alpha;
    g.per_row = mode == BD_ALPHA_PER_ROW;
    g.y = y;
    g.ctx = ctx;
    cudaError_t e = cudaSuccess;
    if (launch_tc(g, w_base, x, M, M, 0, ws, ws_bytes, s, &e)) return from_cuda(e);
  }
  bd::GemvArgs a{};
  a.x = x;
  a.M = M;
  a.w = w_base;
  a.d_out = d_out;
  a.d_in = d_in;
  a.packed = packed;
  a.alpha = alpha;
  a.per_row = mode == BD_ALPHA_PER_ROW;
  a.y = y;
  a.ctx = ctx;
  return from_cuda(bd::launch_gemv(a, dev->num_sms, s));
}

bd_status bitdelta_linear_grouped(const uint16_t* x, int64_t M_total, const int32_t* seg_offsets,
                                  const int32_t* seg_variant, int32_t n_seg, int32_t max_seg_len,
                                  const uint16_t* w_base, const uint8_t* const* packed_table,
                                  const float* const* alpha_table, int32_t n_var,
                                  bd_alpha_mode mode, int64_t d_out, int64_t d_in, uint16_t* y,
                                  bd_stream_t stream) {
  if (M_total < 0 || n_seg < 0 || n_var < 0 || max_seg_len < 0 || !mode_ok(mode))
    return BD_ERR_INVALID_ARG;
  bd_status st = check_dims(d_out, d_in);
  if (st != BD_OK) return st;
  if (M_total == 0 || n_seg == 0) return BD_OK;
  if (!x || !seg_offsets || !seg_variant || !w_base || !y) return BD_ERR_INVALID_ARG;
  if (n_var > 0 && (!packed_table || !alpha_table)) return BD_ERR_INVALID_ARG;
  if (M_total > INT32_MAX) return BD_ERR_UNSUPPORTED_SHAPE;
  if (!aligned(x, 16) || !aligned(w_base, 16) || !aligned(y, 16) || !aligned(seg_offsets, 4) ||
      !aligned(seg_variant, 4) || !aligned(packed_table, 8) || !aligned(alpha_table, 8))
    return BD_ERR_MISALIGNED;
  DeviceState* dev = nullptr;
  if ((st = current_device(&dev)) != BD_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const bd::DevCtx ctx = make_ctx(dev);

  // Long segments on the tensor cores when the shape allows it; the decode
  // kernel takes every segment the tensor-core kernel does not.  The pair
  // kernel holds at most kGemmMaxSegs segments in shared memory, so a longer
  // table is launched in consecutive slices of it (the offsets are absolute
  // row indices, so a slice is a pointer offset into both tables).
  bool use_tc = max_seg_len > kDecodeMaxRows && tc_shape_ok(M_total, d_out, d_in);
  // Every check before the first launch: the short rows' index list must fit
  // the decode kernel's shared memory whichever way the rows are split.
  const int64_t short_rows_bound =
      use_tc ? (M_total < int64_t{n_seg} * kDecodeMaxRows ? M_total
                                                          : int64_t{n_seg} * kDecodeMaxRows)
             : M_total;
  if (bd::gemv_grouped_smem_bytes(n_var, short_rows_bound) > kGroupedListBytes)
    return BD_ERR_UNSUPPORTED_SHAPE;
  if (use_tc) {
    bd::GemmArgs g{};
    g.M = M_total;
    g.d_out = d_out;
    g.d_in = d_in;
    g.per_row = mode == BD_ALPHA_PER_ROW;
    g.y = y;
    g.n_var = n_var;
    g.max_short = static_cast<int32_t>(kDecodeMaxRows);
    g.packed_table = packed_table;
    g.alpha_table = alpha_table;
    g.ctx = ctx;
    for (int32_t s0 = 0; s0 < n_seg; s0 += bd::kGemmMaxSegs) {
      g.seg_off = seg_offsets + s0;
      g.seg_var = seg_variant + s0;
      g.n_seg = n_seg - s0 < bd::kGemmMaxSegs ? n_seg - s0 : bd::kGemmMaxSegs;
      // token tiles over the slice's segments <= tiles of M_total + one
      // ragged tile per segment
      cudaError_t e = cudaSuccess;
      const bool launched =
          launch_tc(g, w_base, x, M_total, max_seg_len, g.n_seg, nullptr, 0, s, &e);
      if (launched && (st = from_cuda(e)) != BD_OK) return st;
      if (!launched) {
        if (s0 > 0) return BD_ERR_CUDA;  // the first slice launched: cannot happen
        use_tc = false;                  // no CTA pair fits: every row on the decode kernel
        break;
      }
    }
    // nothing launched yet when the first slice fell back
    if (!use_tc && bd::gemv_grouped_smem_bytes(n_var, M_total) > kGroupedListBytes)
      return BD_ERR_UNSUPPORTED_SHAPE;
  }
  const int32_t short_limit = use_tc ? static_cast<int32_t>(kDecodeMaxRows) : INT32_MAX;
  bd::GemvArgs a{};
  a.x = x;
  a.M = M_total;
  a.w = w_base;
  a.d_out = d_out;
  a.d_in = d_in;
  a.per_row = mode == BD_ALPHA_PER_ROW;
  a.y = y;
  a.seg_off = seg_offsets;
  a.seg_var = seg_variant;
  a.n_seg = n_seg;
  a.n_var = n_var;
  a.max_short = short_limit;
  a.packed_table = packed_table;
  a.alpha_table = alpha_table;
  a.ctx = ctx;
  return from_cuda(bd::launch_gemv_grouped(a, use_tc ? short_rows_bound : M_total, dev->num_sms, s));
}

bd_status bitdelta_check_error(bd_stream_t stream) {
  DeviceState* dev = nullptr;
  bd_status st = current_device(&dev);
  if (st != BD_OK) return st;
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return BD_ERR_CUDA;
  uint32_t word = 0;
  if (cudaMemcpy(&word, dev->err, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess)
    return BD_ERR_CUDA;
  if (word != 0 && cudaMemset(dev->err, 0, sizeof(word)) != cudaSuccess) return BD_ERR_CUDA;
  if (word & bd::kErrTimeout) return BD_ERR_DEVICE_TIMEOUT;
  if (word & bd::kErrBounds) return BD_ERR_DEVICE_BOUNDS;
  return BD_OK;
}

size_t bitdelta_sign_similarity_workspace_bytes(int64_t d_out, int32_t n_b) {
  if (d_out <= 0 || n_b < 1 || n_b > 256) return 0;
  return bd::sign_similarity_workspace_bytes(d_out, n_b);
}

bd_status bitdelta_sign_similarity(const uint8_t* packed_a, const float* alpha_a,
                                   const uint8_t* const* packed_table,
                                   const float* const* alpha_table, int32_t n_b,
                                   bd_alpha_mode mode, int64_t d_out, int64_t d_in,
                                   double* cos_out, int32_t* best_out, void* workspace,
                                   size_t ws_bytes, bd_stream_t stream) {
  if (!packed_a || !alpha_a || !packed_table || !alpha_table || !cos_out || !best_out ||
      !workspace || !mode_ok(mode))
    return BD_ERR_INVALID_ARG;
  bd_status st = check_dims(d_out, d_in);
  if (st != BD_OK) return st;
  if (n_b < 1 || n_b > 256) return BD_ERR_UNSUPPORTED_SHAPE;
  if (!aligned(alpha_a, 4) || !aligned(packed_table, 8) || !aligned(alpha_table, 8) ||
      !aligned(cos_out, 8) || !aligned(best_out, 4) || !aligned(workspace, 256))
    return BD_ERR_MISALIGNED;
  if (ws_bytes < bitdelta_sign_similarity_workspace_bytes(d_out, n_b)) return BD_ERR_WORKSPACE;
  DeviceState* dev = nullptr;
  if ((st = current_device(&dev)) != BD_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(workspace, 0, 256, s) != cudaSuccess) return BD_ERR_CUDA;  // counters
  const bool vec = d_in % 128 == 0 && aligned(packed_a, 16);
  return from_cuda(bd::launch_sign_similarity(packed_a, alpha_a, packed_table, alpha_table, n_b,
                                              mode == BD_ALPHA_PER_ROW, d_out, d_in, cos_out,
                                              best_out, workspace, vec, s));
}

size_t bitdelta_monosoup_workspace_bytes(int64_t d_out, int64_t d_in, int32_t k, int32_t rank) {
  if (check_dims(d_out, d_in) != BD_OK || k < 1 || k > 64 || rank < 0 || rank > 64) return 0;
  return bd::monosoup_workspace_bytes(d_out, d_in, k, rank);
}

bd_status bitdelta_monosoup(const uint16_t* w_base, const uint16_t* const* w_ft, int32_t k,
                            int32_t rank, int32_t power_iters, uint64_t seed, int64_t d_out,
                            int64_t d_in, uint16_t* w_merged, float* correction, void* workspace,
                            size_t ws_bytes, bd_stream_t stream) {
  if (!w_base || !w_ft || !w_merged || !workspace) return BD_ERR_INVALID_ARG;
  bd_status st = check_dims(d_out, d_in);
  if (st != BD_OK) return st;
  if (k < 1 || k > 64 || rank < 0 || rank > 64 || rank > d_out || rank > d_in ||
      power_iters < 0 || power_iters > 16)
    return BD_ERR_UNSUPPORTED_SHAPE;
  for (int32_t i = 0; i < k; ++i) {
    if (!w_ft[i]) return BD_ERR_INVALID_ARG;
    if (!aligned(w_ft[i], 16)) return BD_ERR_MISALIGNED;
  }
  if (!aligned(w_base, 16) || !aligned(w_merged, 16) || !aligned(correction, 16) ||
      !aligned(workspace, 256))
    return BD_ERR_MISALIGNED;
  if (ws_bytes < bd::monosoup_workspace_bytes(d_out, d_in, k, rank)) return BD_ERR_WORKSPACE;
  DeviceState* dev = nullptr;
  if ((st = current_device(&dev)) != BD_OK) return st;
  bd::MonoSoupArgs a{};
  a.w_base = w_base;
  a.w_ft = w_ft;
  a.k = k;
  a.rank = rank;
  a.power_iters = power_iters;
  a.seed = seed;
  a.d_out = d_out;
  a.d_in = d_in;
  a.w_merged = w_merged;
  a.correction = correction;
  return from_cuda(bd::launch_monosoup(a, workspace, dev->num_sms,
                                       reinterpret_cast<cudaStream_t>(stream)));
}

bd_status bitdelta_set_wait_limit_ns(uint64_t ns) {
  g_wait_limit_ns.store(ns < 1000 ? 1000 : ns);
  return BD_OK;
}

bd_status bitdelta_set_prefill_tile(bd_prefill_tile tile) {
  if (tile != BD_PREFILL_TILE_AUTO && tile != BD_PREFILL_TILE_256 && tile != BD_PREFILL_TILE_512)
    return BD_ERR_INVALID_ARG;
  g_prefill_tile.store(static_cast<int>(tile));
  return BD_OK;
}

bd_status bitdelta_debug_wait_timeout(bd_stream_t stream) {
  DeviceState* dev = nullptr;
  bd_status st = current_device(&dev);
  if (st != BD_OK) return st;
  return from_cuda(
      bd::launch_wait_timeout_probe(make_ctx(dev), reinterpret_cast<cudaStream_t>(stream)));
}

bd_status bitdelta_debug_split_schedule(int64_t n_pairs, int64_t t_total, int64_t sk_lo,
                                        int64_t sk_tiles, int64_t n_kb, int64_t* out,
                                        int64_t out_len, int64_t* n_records) {
  if (n_pairs <= 0 || t_total <= 0 || sk_lo < 0 || n_kb <= 0 || n_kb > INT32_MAX ||
      sk_tiles < n_pairs || n_records == nullptr || out_len < 0 || (out_len > 0 && !out))
    return BD_ERR_INVALID_ARG;
  int64_t n = 0;
  for (int64_t pair = 0; pair < n_pairs; ++pair) {
    const bd::SplitPair sp = bd::split_pair(pair, n_pairs, t_total, sk_lo, sk_tiles, n_kb);
    for (int64_t k = 0; k < sp.n_items; ++k, ++n) {
      if (n >= out_len) continue;
      const bd::SplitItem it = bd::split_item(sp, k, sk_lo, n_kb);
      int64_t* r = out + 10 * n;
      r[0] = pair;
      r[1] = it.tile;
      r[2] = it.kb0;
      r[3] = it.kb1;
      r[4] = it.j;
      r[5] = it.partial ? 1 : 0;
      r[6] = r[7] = r[8] = r[9] = -1;
      if (it.partial) {
        const bd::SplitShare sh = bd::split_share(sp, it.su, n_kb);
        r[6] = sh.pair_lo;
        r[7] = sh.pair_hi;
        r[8] = sh.j_lo;
        r[9] = sh.counter;
      }
    }
  }
  *n_records = n;
  return BD_OK;
}

const char* bitdelta_status_string(bd_status status) {
  switch (status) {
    case BD_OK:
      return "ok";
    case BD_ERR_INVALID_ARG:
      return "invalid argument";
    case BD_ERR_UNSUPPORTED_SHAPE:
      return "unsupported shape";
    case BD_ERR_MISALIGNED:
      return "misaligned pointer";
    case BD_ERR_WORKSPACE:
      return "workspace missing or too small";
    case BD_ERR_CUDA:
      return "CUDA runtime error";
    case BD_ERR_DEVICE_TIMEOUT:
      return "a bounded device wait ran out of time";
    case BD_ERR_DEVICE_BOUNDS:
      return "malformed segment table, variant id or table entry seen on the device";
    case BD_ERR_CACHE_FULL:
      return "delta cache full: every slot is held by a caller or pinned";
  }
  return "unknown status";
}

}  // extern "C"
