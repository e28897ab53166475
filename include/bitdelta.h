/*
 * bitdelta.h — C ABI of the GB300 (sm_103a) BitDelta hot path.
 *
 * The method: a fine-tuned weight W_ft is stored as the shared base weight
 * W_base plus a 1-bit delta, W_ft ≈ W_base + α·sign(Δ) with Δ = W_ft − W_base
 * and α = mean|Δ| (page "BitDelta: serving 14 Zen models from one GPU
 * cluster", hanzo blog 2026-02-28, section "Mathematical foundation").  At
 * serving time one fused kernel reads W_base and the packed sign bits and
 * multiplies by the effective weight without writing it to HBM (same page,
 * section "Serving architecture", the fused-kernel paragraph and the
 * conceptual fused_bitdelta_linear listing).
 *
 * Formats (all row-major, C order):
 *   bf16 tensors   uint16_t bit patterns (IEEE binary32 upper half).
 *   W_base, W_ft   bf16 [d_out, d_in]   (torch.nn.functional.linear layout).
 *   packed         uint8 [d_out, d_in/8]: bit j of byte k of row r is the sign
 *                  of Δ[r][8k+j]; bit 1 = +1, bit 0 = −1, and sign(0) = +1
 *                  (section "Infrastructure details": 8 bits per byte,
 *                  4096x4096 -> 4096x512).
 *   alpha          float32: one value (BD_ALPHA_PER_MATRIX, section
 *                  "Mathematical foundation") or one per output row
 *                  (BD_ALPHA_PER_ROW, section "Infrastructure details").
 *   x, y           bf16 [M, d_in] and [M, d_out]; M = batch·seq rows.
 *   W_eff          bf16_rne(fp32(W_base) + (bit ? α : −α)).
 *
 * Rules common to every call:
 *   - Pointers are device pointers (cudaMalloc / torch CUDA memory) owned by
 *     the caller, unless a parameter says "host".  The library keeps no
 *     pointer after a call returns and allocates no device memory.
 *   - Every compute call is asynchronous on `stream` (a cudaStream_t; NULL is
 *     the legacy default stream) and never synchronises the device.
 *   - Arguments are checked on the host before any launch; an invalid call
 *     returns an error status and launches nothing.  Nothing aborts or traps.
 *   - d_in must be a positive multiple of 8 (one whole sign byte per 8
 *     columns); d_out >= 1; M >= 0 (M == 0 is a no-op).
 *   - bf16 tensors must start on a 16-byte boundary (BD_ERR_MISALIGNED).
 *   - Device-side faults that cannot be seen on the host (a wait that ran out
 *     of time, a variant id out of range in device memory) set a sticky error
 *     word that bitdelta_check_error() reports.
 *   - The library caches, per device, the device addresses of its own
 *     device arrays (the error word, the scratch array of
 *     bitdelta_compress_noalloc) at the first call on that device.  Do not
 *     use it across a device reset (cudaDeviceReset, or a teardown of the
 *     primary context): those addresses would then be stale.
 */
#ifndef BITDELTA_H_
#define BITDELTA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t (struct CUstream_st*). */
typedef struct CUstream_st* bd_stream_t;

typedef enum {
  BD_OK = 0,
  BD_ERR_INVALID_ARG = 1,       /* null pointer, negative size, bad enum */
  BD_ERR_UNSUPPORTED_SHAPE = 2, /* d_in not a positive multiple of 8, size too large */
  BD_ERR_MISALIGNED = 3,        /* a bf16 tensor not 16-byte aligned */
  BD_ERR_WORKSPACE = 4,         /* workspace missing or smaller than required */
  BD_ERR_CUDA = 5,              /* a CUDA runtime call failed (launch, attribute) */
  BD_ERR_DEVICE_TIMEOUT = 6,    /* a bounded device wait ran out (check_error) */
  BD_ERR_DEVICE_BOUNDS = 7,     /* bad segment table / variant id seen on device */
  BD_ERR_CACHE_FULL = 8         /* delta cache: every slot held or pinned (bitdelta_cache.h) */
} bd_status;

typedef enum { BD_ALPHA_PER_MATRIX = 0, BD_ALPHA_PER_ROW = 1 } bd_alpha_mode;

/* Bytes of the packed sign matrix: d_out * d_in / 8 (0 on invalid sizes). */
size_t bitdelta_packed_bytes(int64_t d_out, int64_t d_in);

/* Workspace bytes bitdelta_compress needs: 0 for BD_ALPHA_PER_ROW,
 * 8*d_out + 256 for BD_ALPHA_PER_MATRIX (per-row fp64 partial sums and a
 * completion counter). */
size_t bitdelta_compress_workspace_bytes(int64_t d_out, int64_t d_in, bd_alpha_mode mode);

/*
 * Compression ("Mathematical foundation": Δ = W_ft − W_base, sign(Δ) to one
 * bit, α = (1/n)·‖Δ‖₁).  One pass over W_base and W_ft: writes packed_out
 * [d_out, d_in/8] and alpha_out (1 float for PER_MATRIX, d_out floats for
 * PER_ROW).  α is summed per row in compensated fp32 and fp64 across rows in
 * a fixed order, so the result is deterministic run to run.
 * workspace: device memory of at least bitdelta_compress_workspace_bytes()
 * (may be NULL when that is 0); its contents on entry do not matter.  Two
 * calls that share one workspace must not overlap on the GPU.
 */
bd_status bitdelta_compress(const uint16_t* w_base, const uint16_t* w_ft, int64_t d_out,
                            int64_t d_in, bd_alpha_mode mode, uint8_t* packed_out,
                            float* alpha_out, void* workspace, size_t workspace_bytes,
                            bd_stream_t stream);

/*
 * Reconstruction to memory ("Serving architecture", request step 3:
 * W_eff = W_base + α·sign(Δ)).  Writes w_out bf16 [d_out, d_in]; bit-exact
 * W_eff = bf16_rne(fp32(W_base) ± α).  w_out must not overlap the inputs.
 */
bd_status bitdelta_reconstruct(const uint16_t* w_base, const uint8_t* packed, const float* alpha,
                               bd_alpha_mode mode, int64_t d_out, int64_t d_in, uint16_t* w_out,
                               bd_stream_t stream);

/*
 * Fused delta linear ("Serving architecture", fused kernel paragraph and the
 * conceptual fused_bitdelta_linear listing): y = x · W_effᵀ with W_eff built
 * on chip and never written to memory.  x bf16 [M, d_in], y bf16 [M, d_out]
 * (fp32 accumulation, one RNE rounding at the end), no bias.
 * Dispatch: M <= 16 takes the bandwidth-bound decode kernel; larger M the
 * tcgen05 tensor-core kernel when d_in % 128 == 0 and every pointer allows
 * TMA, else the decode kernel over 16-row chunks.  The tensor-core kernel
 * runs on CTA pairs with tiles of 256 output rows by 256 or 512 tokens
 * (bitdelta_set_prefill_tile).
 * y must not overlap the inputs.
 * Stream order: the decode kernel is launched with programmatic dependent
 * launch and issues its first loads of w_base and packed before it waits for
 * the kernels ahead of it on the stream (x and alpha are read after the
 * wait, y written after it).  So w_base and packed must not be written by a
 * kernel that may still be running when this call's kernel starts, that is
 * by one that signals its dependents early (griddepcontrol.launch_dependents
 * or cudaTriggerProgrammaticLaunchCompletion).  This library's calls that
 * write such tensors (bitdelta_compress, bitdelta_compress_noalloc,
 * bitdelta_reconstruct, and the last kernel of bitdelta_monosoup, which
 * writes the merged weights) do not signal early; kernels that do not use
 * programmatic dependent launch never do.
 */
bd_status bitdelta_linear(const uint16_t* x, int64_t M, const uint16_t* w_base,
                          const uint8_t* packed, const float* alpha, bd_alpha_mode mode,
                          int64_t d_out, int64_t d_in, uint16_t* y, bd_stream_t stream);

/*
 * bitdelta_linear with a caller workspace for the tensor-core kernel's split
 * schedule.  (The page has no counterpart: this is a scheduling choice of
 * this library, not of the method.)  When the call's 512-token tiles leave
 * a small last round (at most a quarter of the device's CTA pairs busy), the
 * last whole round and that remainder are cut by k-blocks into one even
 * range per pair instead; a tile that two pairs share is the sum of their
 * two fp32 partials, formed by the pair that finishes its part last.  The
 * result is deterministic, but its fp32 sum order differs from
 * bitdelta_linear's for those tiles, so single bf16 outputs may differ by
 * the rounding of the split sum.  Other calls run exactly as
 * bitdelta_linear.
 *   workspace   device memory of at least bitdelta_linear_workspace_bytes
 *               (M, d_out, d_in) bytes on a 256-byte boundary, or NULL (the
 *               call is then exactly bitdelta_linear).  Its first bytes are
 *               cleared by the call (stream-ordered); nothing in it needs to
 *               survive between calls.  Calls that can overlap on the GPU
 *               need separate workspaces.
 *   Errors as bitdelta_linear; BD_ERR_WORKSPACE when workspace is not NULL
 *   and smaller than the size above, BD_ERR_MISALIGNED when it is not on a
 *   256-byte boundary.
 * bitdelta_linear_workspace_bytes returns 0 for calls that never split
 * (M <= 16, shapes the tensor-core kernel does not take) and when the
 * current device cannot be queried; the size depends on the device (about
 * 1 MiB per CTA pair that fits at once: 76 MiB on a 152-SM GB300).
 */
size_t bitdelta_linear_workspace_bytes(int64_t M, int64_t d_out, int64_t d_in);
bd_status bitdelta_linear_ws(const uint16_t* x, int64_t M, const uint16_t* w_base,
                             const uint8_t* packed, const float* alpha, bd_alpha_mode mode,
                             int64_t d_out, int64_t d_in, uint16_t* y, void* workspace,
                             size_t ws_bytes, bd_stream_t stream);

/*
 * Multi-tenant linear over one shared W_base ("Serving architecture": base
 * weights shared-read by every variant; a request's model id selects its
 * delta).  Rows [seg_offsets[s], seg_offsets[s+1]) of x use variant
 * seg_variant[s]; variant 0 is the base model (W_eff = W_base, no delta),
 * variant v in 1..n_var uses packed_table[v-1] and alpha_table[v-1].
 *   seg_offsets   device int32 [n_seg+1], non-decreasing, seg_offsets[0] = 0,
 *                 seg_offsets[n_seg] = M_total.
 *   seg_variant   device int32 [n_seg], values in [0, n_var].
 *   packed_table  device array of n_var device pointers (each [d_out, d_in/8]).
 *   alpha_table   device array of n_var device pointers (each 1 or d_out floats).
 *   max_seg_len   host upper bound on any segment's length (dispatch hint; a
 *                 segment longer than 16 rows takes the tensor-core kernel).
 * A malformed table found on the device sets BD_ERR_DEVICE_BOUNDS (see
 * bitdelta_check_error) and leaves the affected rows of y unspecified.
 * Limits: the rows that run on the decode kernel (segments of at most 16 rows
 * when max_seg_len > 16, else every row; the host bounds them by
 * min(M_total, 16·n_seg)) are listed in its shared memory, 4 bytes each next
 * to 8 bytes per variant slot, within 200 KB: a bound above
 * 51200 − 2·(n_var + 2) rows returns BD_ERR_UNSUPPORTED_SHAPE before any
 * launch.  A table of more than 1024 segments runs the tensor-core kernel
 * once per slice of 1024 segments.
 */
bd_status bitdelta_linear_grouped(const uint16_t* x, int64_t M_total, const int32_t* seg_offsets,
                                  const int32_t* seg_variant, int32_t n_seg, int32_t max_seg_len,
                                  const uint16_t* w_base, const uint8_t* const* packed_table,
                                  const float* const* alpha_table, int32_t n_var,
                                  bd_alpha_mode mode, int64_t d_out, int64_t d_in, uint16_t* y,
                                  bd_stream_t stream);

/*
 * bitdelta_compress without a caller workspace.  (The page has no counterpart:
 * this entry point exists for callers of this library, not for the method.)
 * It is meant for callers that cannot allocate device memory at the point
 * where they compress: for example a plug-in that only receives finished
 * device buffers from a host framework and has no allocator handle, or a
 * serving loop whose device memory is planned up front and where a
 * cudaMalloc could block on a device-wide synchronisation or fail under
 * memory pressure.  Same arguments and results as bitdelta_compress minus the
 * workspace; it allocates nothing.
 *   - Per-matrix α uses a fixed scratch array in the library's device memory
 *     (256 B + 8 B per output row), so d_out is limited to 65536 rows in
 *     BD_ALPHA_PER_MATRIX mode; larger d_out returns BD_ERR_WORKSPACE and
 *     launches nothing.  Per-row α needs no scratch and has no such limit.
 *   - The first call on a device looks up the array's device address with that
 *     device current and keeps it until the process exits; make that first
 *     call before any stream capture, and do not call it across a device
 *     reset (the kept address would be stale).
 *   - Every call on a device shares the one array and it keeps the last call's
 *     contents (the call clears its completion counter itself): calls that can
 *     overlap on the GPU (different streams without ordering) race and give
 *     wrong α.  Serialise them.
 */
bd_status bitdelta_compress_noalloc(const uint16_t* w_base, const uint16_t* w_ft, int64_t d_out,
                                    int64_t d_in, bd_alpha_mode mode, uint8_t* packed_out,
                                    float* alpha_out, bd_stream_t stream);

/*
 * Cosine similarity of task vectors in their 1-bit form (page section
 * "K-Merge": when an adapter outside the pool is requested, its pairwise
 * cosine similarity with every pool member on the task vectors decides the
 * most similar member).  The task vectors are the BitDelta deltas α ⊙ S, S = ±1
 * from the packed signs: for each pool member b
 *     cos[b] = <α_a⊙S_a, α_b⊙S_b> / (‖α_a⊙S_a‖·‖α_b⊙S_b‖)
 * computed as Σ_n α_a[n]·α_b[n]·(d_in − 2·popcount(S_a[n] xor S_b[n])) over
 * the rows (fp64; one α per matrix in BD_ALPHA_PER_MATRIX mode).
 *   packed_a, alpha_a      the candidate: packed [d_out, d_in/8], α [d_out] or [1]
 *   packed_table[b], alpha_table[b]   device arrays of n_b pool members' pointers
 *   n_b                    1 .. 256
 *   cos_out                device double [n_b]
 *   best_out               device int32 [1]: argmax of cos_out (ties: lowest b)
 *   workspace              device, bitdelta_sign_similarity_workspace_bytes()
 *                          bytes, 256-byte aligned; its first 256 bytes are
 *                          zeroed by the call (deterministic reduction in a fixed order;
 *                          the grid follows the device's SM count, so results
 *                          repeat bit for bit on the same device model)
 * Reads (1 + n_b) · d_out · d_in / 8 sign bytes.  Errors as bitdelta_linear
 * (BD_ERR_UNSUPPORTED_SHAPE for n_b outside 1 .. 256).
 */
size_t bitdelta_sign_similarity_workspace_bytes(int64_t d_out, int32_t n_b);
bd_status bitdelta_sign_similarity(const uint8_t* packed_a, const float* alpha_a,
                                   const uint8_t* const* packed_table,
                                   const float* const* alpha_table, int32_t n_b,
                                   bd_alpha_mode mode, int64_t d_out, int64_t d_in,
                                   double* cos_out, int32_t* best_out, void* workspace,
                                   size_t ws_bytes, bd_stream_t stream);

/*
 * MonoSoup merge of k fine-tuned checkpoints of one base (page section
 * "MonoSoup: complementing the single checkpoint with SVD"):
 *     W_merged = W_base + (1/k) · Σ_i τ_i,  τ_i = rank-r truncated SVD of
 *     Δ_i = W_i − W_base.
 * τ_i is computed by block subspace iteration on Δ_i (formed on the fly, never
 * stored): a ±1 sketch drawn from `seed`, power_iters rounds of Δᵀ/Δ products
 * each followed by a Cholesky-QR orthonormalisation, then τ_i = Y·Yᵀ·Δ_i.  It
 * reaches the truncated SVD when Δ_i has a gap after its r-th singular value
 * (error shrinking like (σ_{r+1}/σ_r)^(2·power_iters+1)); without a gap it
 * returns a rank-r approximation close to it, not the exact truncation.
 *   w_base       device bf16 [d_out, d_in].
 *   w_ft         HOST array of k device pointers, each bf16 [d_out, d_in].
 *   k            1..64 checkpoints;  rank 0..64 and <= min(d_out, d_in)
 *                (rank 0: W_merged = W_base);  power_iters 0..16.
 *   w_merged     device bf16 [d_out, d_in] (must not overlap the inputs):
 *                bf16_rne(fp32(W_base) + fp32 correction).
 *   correction   device fp32 [d_out, d_in] or NULL: the correction
 *                (1/k)·Σ τ_i before rounding.
 *   workspace    device, 256-byte aligned, >= bitdelta_monosoup_workspace_bytes.
 * Errors as bitdelta_linear; BD_ERR_UNSUPPORTED_SHAPE for k, rank or
 * power_iters out of range.
 */
size_t bitdelta_monosoup_workspace_bytes(int64_t d_out, int64_t d_in, int32_t k, int32_t rank);
bd_status bitdelta_monosoup(const uint16_t* w_base, const uint16_t* const* w_ft, int32_t k,
                            int32_t rank, int32_t power_iters, uint64_t seed, int64_t d_out,
                            int64_t d_in, uint16_t* w_merged, float* correction, void* workspace,
                            size_t ws_bytes, bd_stream_t stream);

/* Synchronises `stream`, then returns and clears the sticky device error word
 * of the current device (BD_OK, BD_ERR_DEVICE_TIMEOUT or BD_ERR_DEVICE_BOUNDS),
 * or BD_ERR_CUDA if the synchronisation itself failed. */
bd_status bitdelta_check_error(bd_stream_t stream);

/* Upper bound, in nanoseconds, on any single bounded wait inside a kernel
 * (default 2e9).  Values below 1000 are raised to 1000.  Host-side setting
 * read at each launch. */
bd_status bitdelta_set_wait_limit_ns(uint64_t ns);

/* Token width of the tensor-core kernel's CTA-pair tiles (bitdelta_linear
 * with M > 16 and the long segments of bitdelta_linear_grouped).  A 512-token
 * tile builds each W_eff tile once for twice the tokens of a 256-token tile
 * (half the transform work per FLOP) but makes half as many tiles.
 *   BD_PREFILL_TILE_AUTO  (default) per call, the width whose predicted time
 *                         is lower (512 on a tie): rounds of tiles over the
 *                         GPU's CTA pairs (ceil(tiles / pairs)) times the
 *                         measured cost of one tile, a 512-token tile costing
 *                         1.75 256-token tiles; grouped calls count tiles
 *                         over M_total and take 256 when max_seg_len <= 256.
 *   BD_PREFILL_TILE_256, BD_PREFILL_TILE_512  always that width.
 * Process-wide host setting read at each launch; BD_ERR_INVALID_ARG for any
 * other value. */
typedef enum {
  BD_PREFILL_TILE_AUTO = 0,
  BD_PREFILL_TILE_256 = 1,
  BD_PREFILL_TILE_512 = 2
} bd_prefill_tile;
bd_status bitdelta_set_prefill_tile(bd_prefill_tile tile);

/* Test hook: launches one CTA that waits on an mbarrier nothing will complete,
 * with the current wait limit.  The wait gives up, records
 * BD_ERR_DEVICE_TIMEOUT in the error word and the kernel returns normally. */
bd_status bitdelta_debug_wait_timeout(bd_stream_t stream);

/* Test hook (host only, no device needed): the split schedule of
 * bitdelta_linear_ws as the tensor-core kernel computes it, for a launch of
 * n_pairs CTA pairs over a split region of sk_tiles tiles starting at flat
 * tile sk_lo, t_total token tiles per row tile and n_kb k-blocks per tile
 * (sk_tiles >= n_pairs).  Writes one record of 10 int64 per split item of
 * every pair, pairs in order: pair, flat tile, kb0, kb1 (the item's k-blocks
 * [kb0, kb1)), partial slot j, shared (1 if the tile is shared with another
 * pair), and for a shared tile its first contributor, its second, the first
 * one's slot and the tile's counter index (else -1).  *n_records receives the
 * number of records; out_len (records) bounds what is written.
 * BD_ERR_INVALID_ARG for a non-positive size, sk_tiles < n_pairs or a NULL
 * n_records. */
bd_status bitdelta_debug_split_schedule(int64_t n_pairs, int64_t t_total, int64_t sk_lo,
                                        int64_t sk_tiles, int64_t n_kb, int64_t* out,
                                        int64_t out_len, int64_t* n_records);

/* Static string for a status code. */
const char* bitdelta_status_string(bd_status status);

#ifdef __cplusplus
}
#endif

#endif /* BITDELTA_H_ */
