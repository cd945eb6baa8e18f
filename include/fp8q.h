/*
 * fp8q.h -- C ABI of the GB300 (sm_103a) FP8 scaled-quantization library.
 *
 * The library computes the data-parallel hot path of FP8 tensor
 * quantization with scaling:
 *   amax reduction -> scale (current, or delayed from an amax history)
 *   -> round-to-nearest-even saturating cast of BF16/FP32 to E4M3FN or E5M2
 *   (rowwise, columnwise/transposed, 128x128 and 1x128 block-scaled)
 *   -> dequantize.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Memory.   Every tensor and scalar pointer is a DEVICE pointer owned by the
 *           caller (for example a PyTorch allocation).  The library never
 *           frees caller memory and never synchronises the device or a stream.
 *           The one allocation it makes is a 96 KB reduction workspace per
 *           (device, stream) pair, created on the first call that needs it
 *           and kept until process exit (see "Workspace" below).
 * Streams.  `stream` is a cudaStream_t passed as void*; NULL means the legacy
 *           default stream.  Every call only enqueues work on that stream and
 *           returns; results are ready when the stream reaches them.
 * Layout.   Row-major and contiguous.  BF16 is the 16-bit brain-float bit
 *           pattern; FP8 codes are bytes (E4M3FN or E5M2 encodings).
 * Scale.    The multiplier convention: q = encode(fl32(x * scale)),
 *           x ~= decode(q) * scale_inv, scale_inv = fl32(1 / scale).
 * Errors.   Arguments are checked on the host before anything is enqueued; a
 *           rejected call returns FP8_ERR_INVALID_ARG / FP8_ERR_UNSUPPORTED
 *           and touches no memory.  FP8_ERR_CUDA is returned when a CUDA
 *           runtime call or kernel launch fails; fp8_last_error_message()
 *           gives the text.  Kernels never trap or assert on the device.
 * Counters. Outputs named *_out (amax, saturation count, scales) are
 *           overwritten, never accumulated into.
 * Launches. Every kernel is launched with programmatic stream serialization:
 *           it may become resident while the previous kernel on the stream
 *           drains, and it waits for that kernel to complete before it touches
 *           memory, so stream order is kept.
 * Workspace. Calls that reduce (amax, a fused amax / saturation count, the
 *           delayed update) store one partial per CTA in a per-(device,
 *           stream) workspace; a one-CTA finalize kernel launched right after
 *           the main kernel reduces them.  Calls on the same stream are
 *           ordered and safe.  Calls on different streams use different
 *           workspaces and are safe.  A CUDA graph captured from a stream
 *           keeps that stream's workspace address: do not replay such a graph
 *           concurrently with other work on the capturing stream.  The first
 *           call on a new stream allocates (cudaMalloc) with the thread's
 *           capture mode relaxed, so it may happen during capture.
 *
 * Special values (the same in every cast):
 *   x NaN          -> code 0x7F (canonical NaN, sign dropped)
 *   x +-Inf        -> E5M2: +-Inf (0x7C / 0xFC); E4M3FN: +-448 (0x7E / 0xFE)
 *   x finite       -> fl32(x * scale) rounded to nearest-even onto the FP8
 *                     grid; magnitudes at or beyond the largest finite value
 *                     (448 / 57344) saturate to it; signed zeros keep sign.
 *
 * Scale rule (current and delayed):
 *   amax == 0, negative, NaN or Inf -> scale = scale_inv = 1
 *   else scale = fl32(fl32(FP8_MAX / amax) * 2^-margin), clamped to
 *        [FLT_MIN, FLT_MAX]; scale_inv = fl32(1 / scale).
 *
 * Page citations use the page title and section: "Megatron FP8" (a Megatron
 * / Transformer Engine FP8 training guide, sections §2 .. §28), "Low
 * Precision Training and Rollout" (vime documentation), "[Pytorch][Common]
 * Hybrid quantization #2817" (a Transformer Engine pull request).
 */
#ifndef FP8Q_H_
#define FP8Q_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define FP8Q_VERSION_MAJOR 0
#define FP8Q_VERSION_MINOR 1

/* "Megatron FP8" §2: E4M3 here is E4M3FN (bias 7, max 448, no Inf, NaN only
 * at S.1111.111); E5M2 is IEEE-like (bias 15, max 57344, Inf and NaN). */
typedef enum { FP8_E4M3 = 0, FP8_E5M2 = 1 } fp8_format_t;

/* Element type of high-precision tensors. */
typedef enum { FP8_DT_BF16 = 0, FP8_DT_FP32 = 1 } fp8_dtype_t;

/* "Megatron FP8" §5 / §7: amax_compute_algo of the delayed recipe. */
typedef enum { FP8_AMAX_MAX = 0, FP8_AMAX_MOST_RECENT = 1 } fp8_amax_algo_t;

/* "[Pytorch][Common] Hybrid quantization #2817", columnwise_source. */
typedef enum {
    FP8_COLUMNWISE_FROM_ORIGINAL = 0,            /* quantize x itself                            */
    FP8_COLUMNWISE_FROM_ROWWISE_DEQUANTIZED = 1  /* quantize the BF16 dequantized rowwise value */
} fp8_columnwise_source_t;

typedef enum {
    FP8_OK = 0,
    FP8_ERR_INVALID_ARG = 1, /* NULL pointer, negative size, bad enum or margin */
    FP8_ERR_UNSUPPORTED = 2, /* e.g. block shape other than 128x128 / 1x128     */
    FP8_ERR_CUDA = 3         /* a CUDA runtime call or launch failed            */
} fp8_status_t;

/* Static text for a status code. */
const char* fp8_status_string(fp8_status_t status);

/* Text of the last error raised on the calling thread ("" if none). */
const char* fp8_last_error_message(void);

/* Library version as (major << 16) | minor. */
int fp8_version(void);

/* Number of kernels this library has launched in this process (all devices,
 * all threads).  Lets a caller count launches inside a timed region. */
unsigned long long fp8_launch_count(void);

/* Number of waits inside the library's tile pipelines (a consumer waiting for
 * a tile's bulk copy to land, the copying warp waiting for a stage to be
 * released) that gave up after their limit of about two seconds, on the
 * current device, since the library was loaded.  Written to *count after the
 * device has finished all queued work (the call synchronises the device).  A
 * wait that gives up never hangs the kernel: the kernel finishes, but the
 * outputs of that launch are incomplete, so any nonzero change of the count
 * across a call means that call's outputs must not be used.  Correct inputs
 * never reach the limit: a stage is always filled and released by the same
 * launch.  FP8_ERR_INVALID_ARG if count is NULL. */
fp8_status_t fp8_wait_timeouts(unsigned long long* count);

/* Test hook for the bounded waits above: from the next launch on, the thread
 * that copies tiles in each CTA of the blockwise cast-transpose's tiled path
 * skips the copy of its tile number `tile` (counted from 0 per CTA; -1, the
 * default, skips none), so that every wait on that stage expires after its
 * limit: the kernel still ends, fp8_wait_timeouts grows, and the outputs of
 * those launches are garbage.  For tests of the error path only; it
 * synchronises with the device. */
fp8_status_t fp8_test_drop_tile_copy(int tile);

/* Frees the reduction workspace (96 KB) that the calls made on `stream` on the
 * current device, after waiting for the work queued on that stream.  A later
 * reducing call on the stream allocates a new one.  Returns FP8_OK when there
 * is none.  Call it before destroying a stream when many short-lived streams
 * are used, and not while the stream is being captured or while a captured
 * graph whose kernels used that workspace may still be launched (its nodes
 * hold the workspace's address). */
fp8_status_t fp8_release_stream_workspace(void* stream);

/* ------------------------------------------------------------------------ */
/* amax reduction with optional fused current-scaling finalize              */
/* ------------------------------------------------------------------------ */
/* "Megatron FP8" §4 (amax = max|x| by a dedicated reduction kernel, stored
 * as an fp32 scalar; scale_inv cached) and §10 (current scaling: scan the
 * tensor before the cast; margin headroom).
 *
 *   x           device, n elements of `dtype`, any alignment.
 *   n           element count, >= 0 (n == 0: amax 0, scale 1).
 *   amax_out    device float[1]: max_i |x_i|; NaN if any x_i is NaN
 *               (written as 0x7FC00000).
 *   fmt, margin used only when scale_out is given; -126 <= margin <= 126.
 *   scale_out, scale_inv_out
 *               device float[1] each, both NULL or both set: the current
 *               scale from this amax (scale rule above), computed by the
 *               finalize kernel.
 * Two launches: the reduction and the one-CTA finalize. */
fp8_status_t fp8_amax(const void* x, fp8_dtype_t dtype, int64_t n, float* amax_out,
                      fp8_format_t fmt, int margin, float* scale_out, float* scale_inv_out,
                      void* stream);

/* ------------------------------------------------------------------------ */
/* Delayed scaling: amax-history update and scale                           */
/* ------------------------------------------------------------------------ */
/* "Megatron FP8" §5 (amax history ring buffer; the slot step % history_len
 * takes the newest amax; eff = window max for algo max, the slot just
 * written for most_recent; scale 1 while the history is all zero) and §7
 * (amax_history_len, amax_compute_algo, margin).
 *
 *   amax_history  device float[history_len], caller-owned and caller
 *                 zero-initialised; updated in place.
 *   history_len   1 .. 65536.
 *   step          >= 0; the slot written is step % history_len.
 *   new_amax      device float[1] or NULL.  When set, it is stored into the
 *                 slot before the maximum is taken (typically the amax that
 *                 fp8_quantize recorded for the tensor of this step).
 *   algo, fmt, margin   as above.
 *   scale_out, scale_inv_out  device float[1] each (required): the scale for
 *                 the NEXT cast.
 * Per step k of the delayed recipe: fp8_quantize(x_k, scale) records amax_k,
 * then fp8_update_scale_delayed(.., step = k, new_amax = amax_k, ..) gives
 * the scale of step k + 1.  Before step 0, a call with new_amax = NULL on the
 * zero history gives scale 1.  history_len 1 with most_recent equals current
 * scaling.  One single-CTA launch. */
fp8_status_t fp8_update_scale_delayed(float* amax_history, int history_len, int64_t step,
                                      const float* new_amax, fp8_amax_algo_t algo,
                                      fp8_format_t fmt, int margin, float* scale_out,
                                      float* scale_inv_out, void* stream);

/* ------------------------------------------------------------------------ */
/* Per-tensor quantize                                                       */
/* ------------------------------------------------------------------------ */
/* "Megatron FP8" §4 (x scaled, clamped to +-FP8_MAX), §2 (E4M3FN saturates,
 * E5M2 keeps Inf), §6 (cast_to_fp8 before the FP8 GEMM), §24 (per-layer
 * overflow counts).
 *
 *   x              device, n elements of `dtype`, any alignment (16-byte
 *                  aligned x and q_out take the vector path).
 *   n              >= 0.
 *   scale          device float[1]: the multiplier.
 *   q_out          device uint8[n]: the codes.
 *   amax_out       device float[1] or NULL: max|x| of this tensor, fused
 *                  (the delayed recipe records it for the next update).
 *  sat_count_out  device uint64[1] or NULL: number of finite x_i with
 *                  |fl32(x_i * scale)| > FP8_MAX.
 * One kernel launch, plus the one-CTA finalize when amax_out or
 * sat_count_out is given. */
fp8_status_t fp8_quantize(const void* x, fp8_dtype_t dtype, int64_t n, fp8_format_t fmt,
                          const float* scale, uint8_t* q_out, float* amax_out,
                          unsigned long long* sat_count_out, void* stream);

/* ------------------------------------------------------------------------ */
/* Delayed scaling, fused: the cast of one step and the history update      */
/* ------------------------------------------------------------------------ */
/* "Megatron FP8" §5: per step, cast with the scale derived from the amax
 * history, record this step's amax into slot step % history_len, and derive
 * the scale of the next step -- here in one call: the cast (with fused amax
 * and saturation count) and a one-CTA finalize that performs the update of
 * fp8_update_scale_delayed.
 *
 * Equivalent, bit for bit, to
 *   fp8_quantize(x, .., scale, q_out, tmp_amax, sat_count_out)
 *   fp8_update_scale_delayed(amax_history, history_len, step, tmp_amax, algo,
 *                            fmt, margin, scale, scale_inv)
 *
 *   scale, scale_inv  device float[1] each, read and written: on entry the
 *                     scale of this step (scale_inv is not read), on return
 *                     the scale / scale_inv of the next step.
 *   amax_history      device float[history_len], updated in place.
 *   amax_out          device float[1] or NULL: this step's amax.
 *   sat_count_out     device uint64[1] or NULL: as in fp8_quantize.
 *   Other arguments as in fp8_quantize / fp8_update_scale_delayed.
 * Two launches: the cast (which records per-CTA amax / counts) and the
 * one-CTA finalize, which does the history update and writes the scales. */
fp8_status_t fp8_quantize_delayed(const void* x, fp8_dtype_t dtype, int64_t n, fp8_format_t fmt,
                                  float* scale, float* scale_inv, uint8_t* q_out, float* amax_history,
                                  int history_len, int64_t step, fp8_amax_algo_t algo, int margin,
                                  float* amax_out, unsigned long long* sat_count_out, void* stream);

/* ------------------------------------------------------------------------ */
/* Quantize with rowwise + columnwise (transposed) outputs                  */
/* ------------------------------------------------------------------------ */
/* "Megatron FP8" §6 (the weight-gradient GEMM consumes transpose(dy_fp8)) and
 * the columnwise storage of "[Pytorch][Common] Hybrid quantization #2817"
 * (a physically transposed FP8 copy for Hopper-style GEMMs;
 * columnwise_source = original).  Both copies use the one scale, so
 * q_col[c, r] == q_row[r, c] bit for bit.
 *
 *   x        device [rows, cols] of `dtype`, row-major.
 *   rows, cols  >= 0.
 *   scale    device float[1].
 *   q_row    device uint8[rows, cols] or NULL (columnwise only).
 *   q_col    device uint8[cols, rows] or NULL (rowwise only); not both NULL
 *            unless rows * cols == 0.
 *   amax_out device float[1] or NULL: max|x|, fused.
 * Current scaling is fp8_amax(.., scale_out, scale_inv_out) followed by this
 * call.  Interior 128x128 tiles take the vector path when cols % 16 == 0,
 * rows % 16 == 0 and the pointers are 16-byte aligned; edge tiles and other
 * shapes take a guarded element path.  One kernel launch (one CTA per tile;
 * with amax_out at most 8192 CTAs, each walking its share of the tiles), plus
 * the one-CTA finalize when amax_out is given. */
fp8_status_t fp8_quantize_cast_transpose(const void* x, fp8_dtype_t dtype, int64_t rows,
                                         int64_t cols, fp8_format_t fmt, const float* scale,
                                         uint8_t* q_row, uint8_t* q_col, float* amax_out,
                                         void* stream);

/* ------------------------------------------------------------------------ */
/* Current scaling: amax, scale and cast in one call                         */
/* ------------------------------------------------------------------------ */
/* "Megatron FP8" §10 (current scaling: the cast's scale comes from the amax
 * of the tensor being cast) and §4 (amax -> scale with margin -> saturating
 * cast).  Results are identical to fp8_amax(x, .., scale_out, scale_inv_out)
 * followed by fp8_quantize(x, .., scale_out, q_out):
 *   q_out[i] = encode(fl32(x[i] * scale)), scale by the scale rule above.
 *   amax_out, scale_out, scale_inv_out: device float[1] each, each nullable.
 * Aligned x and q_out, amax kernel leaving at most 256 partials (about 6M
 * BF16 elements): two launches, the amax kernel (one partial per CTA) and the
 * cast, whose CTAs reduce the partials themselves while their own loads of x
 * are in flight -- no separate finalize.  Larger tensors: the amax kernel,
 * the one-CTA finalize and the cast (faster there).  Unaligned pointers: the
 * fp8_amax + fp8_quantize kernels. */
fp8_status_t fp8_quantize_current(const void* x, fp8_dtype_t dtype, int64_t n, fp8_format_t fmt, int margin,
                                  uint8_t* q_out, float* amax_out, float* scale_out, float* scale_inv_out,
                                  void* stream);

/* ------------------------------------------------------------------------ */
/* Hybrid per-direction quantization                                         */
/* ------------------------------------------------------------------------ */
/* "[Pytorch][Common] Hybrid quantization #2817": the rowwise and columnwise
 * copies may use different per-tensor formats and scales, and the columnwise
 * copy may be quantized from the original tensor or from the dequantized
 * rowwise value (columnwise_source).  One read of x gives
 *   q_row [rows, cols] = codes of x in fmt_row with *scale_row,
 *   q_col [cols, rows] = codes, in fmt_col with *scale_col, of
 *     x^T                                       (FROM_ORIGINAL), or
 *     RNE_bf16(fl32(decode(q_row) * fl32(1 / *scale_row)))^T
 *                                               (FROM_ROWWISE_DEQUANTIZED:
 *                                                the value fp8_dequantize
 *                                                would produce).
 * With one format and one scale and FROM_ORIGINAL this is
 * fp8_quantize_cast_transpose.  Both outputs are required; same layouts and
 * alignment rules as fp8_quantize_cast_transpose.  One kernel launch. */
fp8_status_t fp8_quantize_hybrid(const void* x, fp8_dtype_t dtype, int64_t rows, int64_t cols,
                                 fp8_format_t fmt_row, const float* scale_row, uint8_t* q_row,
                                 fp8_format_t fmt_col, const float* scale_col, uint8_t* q_col,
                                 fp8_columnwise_source_t source, void* stream);

/* ------------------------------------------------------------------------ */
/* Block-scaled quantize (128x128 and 1x128)                                 */
/* ------------------------------------------------------------------------ */
/* "Low Precision Training and Rollout": block FP8 with 128x128 blocks
 * ("BF16 Training with FP8 Rollout", --block-size 128 128), FP32 block scales
 * ("FP8 Quick Start", NVTE_FP8_BLOCK_SCALING_FP32_SCALES=1), the stored block
 * factor being the inverse scale ("MXFP8 (Blackwell only)": weight_scale_inv);
 * the 1x128 tile is the activation-side Float8Blockwise shape named in
 * "[Pytorch][Common] Hybrid quantization #2817".
 *
 * For every block: amax over its elements (edge blocks: the elements that
 * exist), scale by the scale rule with margin 0, codes with that scale.
 *
 *   x              device [rows, cols] of `dtype`, row-major.
 *   block_rows, block_cols   (128, 128) or (1, 128); else FP8_ERR_UNSUPPORTED.
 *   q_out          device uint8[rows, cols].
 *   scale_inv_out  device float[ceil(rows/block_rows), ceil(cols/block_cols)],
 *                  row-major: the dequantization multiplier of each block.
 * One kernel launch. */
fp8_status_t fp8_quantize_block(const void* x, fp8_dtype_t dtype, int64_t rows, int64_t cols,
                                int block_rows, int block_cols, fp8_format_t fmt, uint8_t* q_out,
                                float* scale_inv_out, void* stream);

/* Blockwise cast + transpose: "[Pytorch][Common] Hybrid quantization #2817"
 * (Float8Blockwise sub-storage with a columnwise copy for the backward GEMM,
 * columnwise_source = original).  One read of x gives
 *   q_row [rows, cols] + scale_inv_row [rows, ceil(cols/128)]: the 1 x 128
 *       blockwise quantization of x (as fp8_quantize_block(1, 128));
 *   q_col [cols, rows] + scale_inv_col [cols, ceil(rows/128)]: the 1 x 128
 *       blockwise quantization of x^T, i.e. 128 x 1 blocks along the columns
 *       of x, written transposed.
 * Either direction may be NULL (codes and scales together).  BF16 inputs with
 * rows and cols multiples of 128 (each below 2^31) and 16-byte aligned x /
 * codes use one persistent kernel over 128 x 128 tiles, which reads x through
 * a tensor map (the driver's cuTensorMapEncodeTiled, reached through the
 * runtime; FP8_ERR_CUDA if it is unavailable or refuses the shape) and holds
 * 170 KB of shared memory per SM while it runs; its internal waits are
 * bounded and counted by fp8_wait_timeouts.  Other shapes use one guarded
 * kernel per direction. */
fp8_status_t fp8_quantize_block_cast_transpose(const void* x, fp8_dtype_t dtype, int64_t rows, int64_t cols,
                                               fp8_format_t fmt, uint8_t* q_row, float* scale_inv_row,
                                               uint8_t* q_col, float* scale_inv_col, void* stream);

/* ------------------------------------------------------------------------ */
/* Grouped (multi-tensor) current scaling                                    */
/* ------------------------------------------------------------------------ */
/* "Megatron FP8" §21: every expert of an MoE layer keeps its own per-tensor
 * FP8 scaling state; §24: the amax / scale overhead should stay a small share
 * of the step.  These two calls treat up to 128 tensors as one launch each
 * (plus one finalize), instead of two or three launches per tensor.
 *
 * fp8_amax_grouped: amax_out[i] = max |xs[i]| and, when scale_out /
 *   scale_inv_out are given, the current scale of tensor i by the scale rule
 *   with `margin`.  Outputs are device float arrays of `count` entries.
 * fp8_quantize_grouped: qs[i] = codes of xs[i] * scales[i] (scales: device
 *   float[count]).
 *   count      1 .. 128; xs, ns, qs are HOST arrays of `count` entries
 *              holding device pointers / element counts.
 *   xs[i], qs[i] must be 16-byte aligned when ns[i] > 0 (else
 *              FP8_ERR_UNSUPPORTED); all tensors share `dtype`. */
fp8_status_t fp8_amax_grouped(int count, const void* const* xs, const int64_t* ns, fp8_dtype_t dtype,
                              float* amax_out, fp8_format_t fmt, int margin, float* scale_out,
                              float* scale_inv_out, void* stream);
fp8_status_t fp8_quantize_grouped(int count, const void* const* xs, const int64_t* ns, fp8_dtype_t dtype,
                                  fp8_format_t fmt, const float* scales, uint8_t* const* qs, void* stream);

/* ------------------------------------------------------------------------ */
/* Dequantize                                                                */
/* ------------------------------------------------------------------------ */
/* "Megatron FP8" §4 (scale_inv cached so dequantize is one multiply) and §23
 * (reconstructed = fp8 value * scale); "Low Precision Training and Rollout",
 * "Implementation Notes" (FP8 weights dequantized to BF16).
 *
 * y = decode(q) * scale_inv in fp32 (one multiply), then rounded to nearest
 * even into BF16 (out_dtype FP8_DT_BF16) or kept as fp32 (FP8_DT_FP32).
 * NaN results are written as the canonical NaN (BF16 0x7FFF, fp32 0x7FFFFFFF).
 *
 *   q          device uint8[rows, cols].
 *   scale_inv  device float: one value when block_rows = block_cols = 0
 *              (per-tensor), else the [ceil(rows/br), ceil(cols/bc)] block
 *              grid of fp8_quantize_block with (br, bc) = (128,128) or (1,128).
 *   y          device [rows, cols] of out_dtype, written with evict-first
 *              (streaming) stores: the values leave L2 as they are written.
 * One kernel launch. */
fp8_status_t fp8_dequantize(const uint8_t* q, fp8_format_t fmt, int64_t rows, int64_t cols,
                            const float* scale_inv, int block_rows, int block_cols, void* y,
                            fp8_dtype_t out_dtype, void* stream);

/* ------------------------------------------------------------------------ */
/* MXFP8: E8M0 scale per 32 elements                                         */
/* ------------------------------------------------------------------------ */
/* "Megatron FP8" §10 / §16: every 32 consecutive elements share one E8M0
 * scale (8 exponent bits, no mantissa, no sign: 2^-127 .. 2^127; code 0xFF is
 * NaN) -- the OCP Microscaling format; "Low Precision Training and Rollout",
 * "MXFP8 (Blackwell only)": E4M3 values with UE8M0 scales per 32-element group.
 *
 * Scale of a block (the OCP MX rule): shared_exp = floor(log2(block amax))
 * - emax (8 for E4M3, 15 for E5M2), clamped to [-127, 127]; an all-zero
 * block takes -127; a block holding Inf or NaN gets scale 0xFF and NaN codes
 * (0x7F).  Codes: RNE-saturating encode of fl32(x * 2^-shared_exp).
 *
 *   x          device [rows, cols] of `dtype`, row-major.
 *   q_row      device uint8[rows, cols] or NULL: 1 x 32 blocks along rows.
 *   scale_row  device uint8[rows, ceil(cols/32)] (with q_row).
 *   q_col      device uint8[cols, rows] or NULL: 32 x 1 blocks along
 *              columns, written transposed (row c of q_col is column c of x).
 *   scale_col  device uint8[cols, ceil(rows/32)] (with q_col).
 * rows % 32 == 0, cols % 128 == 0, BF16 and 16-byte aligned pointers take
 * one tiled launch; other shapes take a guarded path (one launch per
 * direction). */
fp8_status_t fp8_quantize_mx(const void* x, fp8_dtype_t dtype, int64_t rows, int64_t cols, fp8_format_t fmt,
                             uint8_t* q_row, uint8_t* scale_row, uint8_t* q_col, uint8_t* scale_col,
                             void* stream);

/* y = decode(q) * 2^(scale - 127) in fp32 (one multiply), then BF16 (RNE) or
 * fp32; q [rows, cols] with scales [rows, ceil(cols/32)] (rowwise layout; a
 * columnwise copy is dequantized as its own [cols, rows] matrix).  A NaN scale
 * makes its block NaN (canonical NaN of the output type).  One launch. */
fp8_status_t fp8_dequantize_mx(const uint8_t* q, const uint8_t* scales, fp8_format_t fmt, int64_t rows,
                               int64_t cols, void* y, fp8_dtype_t out_dtype, void* stream);

/* "Low Precision Training and Rollout", "MXFP8 (Blackwell only)": block-FP8
 * [128,128] data re-blocked to [1,32] without dequantizing when its scales are
 * powers of two.  The codes stay as they are; this writes the E8M0 scale of
 * every 1 x 32 block from the fp32 scale_inv of its 128 x 128 block
 * (scale_inv [ceil(rows/128), ceil(cols/128)] as written by
 * fp8_quantize_block).  A scale_inv that is not a power of two in
 * [2^-127, 2^127] cannot be carried: its blocks get 0xFF and, when
 * bad_blocks_out (device uint64[1]) is given, it receives how many 128 x 128
 * blocks were like that (0 for an empty shape, which launches nothing
 * else).  One memset node (bad_blocks_out) + one launch. */
fp8_status_t fp8_block128_scales_to_mx(const float* scale_inv, int64_t rows, int64_t cols, uint8_t* mx_scales,
                                       unsigned long long* bad_blocks_out, void* stream);

/* ------------------------------------------------------------------------ */
/* amax without any device allocation                                       */
/* ------------------------------------------------------------------------ */
/* The pages have no counterpart to this entry point; it serves callers that
 * cannot let a library allocate device memory -- code running while a stream
 * is captured in the global capture mode (where cudaMalloc is an illegal
 * call), engines and plugins that work inside a fixed, pre-planned memory
 * budget, and frameworks whose allocator must own every device buffer.
 *
 * Same arguments, results and numerics as fp8_amax (bit-identical outputs).
 * Differences:
 *   - It allocates nothing (no cudaMalloc / cudaFree, no library allocator).
 *     Its scratch is a fixed 16.25 KB file-scope device array (one arrival
 *     counter and 4096 per-CTA partial maxima) that every GPU which loads
 *     the library holds until the process exits.
 *   - n must not exceed 2^28 (268,435,456) elements: each CTA reduces a fixed
 *     slice of 65,536 elements and the scratch has room for 4096 CTAs.
 *     Larger n returns FP8_ERR_UNSUPPORTED without touching the device.
 *   - The first call on each device looks up the scratch's device address
 *     (cudaGetSymbolAddress, which may load the library's GPU code); make that
 *     first call before any stream capture on that device.
 *   - Every call shares the one scratch array, which keeps the last call's
 *     contents.  Each call clears the counter on its stream before its kernel.
 *     Calls that overlap on the GPU (different streams, or graphs replayed
 *     concurrently) race on the scratch and give wrong results; serialise them.
 * One memset node plus one kernel launch. */
fp8_status_t fp8_amax_noalloc(const void* x, fp8_dtype_t dtype, int64_t n, float* amax_out,
                              fp8_format_t fmt, int margin, float* scale_out, float* scale_inv_out,
                              void* stream);

#ifdef __cplusplus
}
#endif

#endif /* FP8Q_H_ */
