/*
 * w4a16.h -- C ABI of the GB300 (sm_103a) W4A16 weight-only INT4 library.
 *
 * The library computes y = x * W^T for fp16 activations x [M, K] and weights
 * W [N, K] stored as symmetric INT4 in groups of 128 along K with one fp16
 * scale per group: the dequantize-on-the-fly product that dominates
 * memory-bound single-batch LLM decode ("W4A16 量化算子解码性能基准跑分与端侧大模型
 * 推理显存实测报告", mhpq.cn, §二 and §五), together with the group-wise
 * round-to-nearest quantizer that produces the packed weights ("LLM
 * quantization from IEEE 754 to GPTQ/AWQ/GGUF" tutorial, qaqbuyan.com
 * article 126, chapter "量化的数学基石" §2 formula and §3
 * per_group_symmetric_quantize / per_group_symmetric_dequantize).
 *
 * Conventions for every entry point
 *  - Pointers are DEVICE pointers owned by the caller (for example a torch
 *    tensor's data_ptr()); the library never allocates, frees or keeps them.
 *    Every pointer must be 16-byte aligned.  Tensors are dense and row-major.
 *  - `stream` is a cudaStream_t passed as void*; NULL means the legacy
 *    default stream.  Work is enqueued asynchronously on it; the call returns
 *    without synchronising.  Calls on one stream execute in order.
 *  - Argument errors are reported synchronously, before anything is
 *    launched, as a w4a16_status code; nothing is written in that case.
 *  - A device-side failure (a bounded wait inside a kernel that gave up) is
 *    recorded in a device status word, readable with w4a16_device_status().
 *  - All kernels are built for sm_103a only; on another device the calls
 *    return W4A16_ERR_DEVICE.
 *  - The library keeps no state across calls other than the device status
 *    word and per-device launch attributes set on first use (first use on a
 *    device should happen before any CUDA graph capture).
 */
#ifndef W4A16_H
#define W4A16_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum w4a16_status {
    W4A16_OK = 0,
    W4A16_ERR_NULL = 1,      /* a required pointer is NULL                    */
    W4A16_ERR_SHAPE = 2,     /* unsupported M, N, K or group size             */
    W4A16_ERR_ALIGN = 3,     /* a pointer is not 16-byte aligned              */
    W4A16_ERR_CUDA = 4,      /* a CUDA runtime call or launch failed          */
    W4A16_ERR_TIMEOUT = 5,   /* a kernel's bounded wait gave up (device)      */
    W4A16_ERR_DEVICE = 6     /* current device is not an sm_103 GPU           */
} w4a16_status;

/* Group size along K: one fp16 scale per 128 consecutive weights of a row. */
#define W4A16_GROUP 128

/* Human-readable name of a status code (static string, never NULL). */
const char *w4a16_status_string(int status);

/* Library ABI version (major * 100 + minor). */
int w4a16_version(void);

/*
 * w4a16_quantize -- group-wise symmetric round-to-nearest INT4 quantizer.
 *
 * Source: qaqbuyan.com tutorial, "量化的数学基石" §2 (x_q = clamp(round(x / s),
 * -8, 7), s = max|x| / 7) and §3 per_group_symmetric_quantize (groups along
 * in_features, clamp(min = 1e-8) on the scale, two nibbles per byte with the
 * even index in the low nibble, each stored as q + 8, scales cast to fp16).
 *
 * For each row n and group g of 128 weights, in IEEE binary32 on the exactly
 * upcast fp16 inputs:
 *     s32 = max(max_k |W[n,k]| / 7, 1e-8)             (correctly rounded /)
 *     q   = clamp(round_half_even(W[n,k] / s32), -8, 7)
 *     scales[n, g] = fp16_round_nearest_even(s32)
 *     qweight[n, k/2] = (q[k+1] + 8) << 4 | (q[k] + 8)   for even k
 *
 *   W_f16      [N, K] fp16, row-major (rows are output features).  Finite.
 *   N, K       N >= 1; K >= 128 and K % 128 == 0.
 *   group      must be 128 (W4A16_GROUP).
 *   qweight    [N, K/2] bytes, written (the canonical packed layout).
 *   scales_f16 [N, K/128] fp16, written.
 * The result is bit-identical to the library's CPU reference definition.
 * Errors: NULL -> W4A16_ERR_NULL; bad N, K or group -> W4A16_ERR_SHAPE;
 *         misaligned pointer -> W4A16_ERR_ALIGN.
 */
int w4a16_quantize(const void *W_f16, int64_t N, int64_t K, int32_t group, void *qweight,
                   void *scales_f16, void *stream);

/* group argument of the format variants: one group spanning each row. */
#define W4A16_GROUP_PER_CHANNEL (-1)

/*
 * w4a16_quantize_ex -- format variants of the quantizer: other group sizes
 * and asymmetric INT4 with a zero point per group.
 *
 * Source: the same tutorial chapter, §3 granularity (per-channel, per-group
 * 128 and 32) and §2 asymmetric formula x_q = clamp(round(x / s) + z, 0, 15),
 * s = (max - min) / 15, z = -round(min / s).
 *
 * Per row n and group g, in IEEE binary32 on the exactly upcast inputs:
 *   symmetric   as w4a16_quantize with the given group; the nibble holds q + 8.
 *   asymmetric  lo = min(0, min_k W), hi = max(0, max_k W) over the group
 *               (0 is kept in range so that z, the code of 0.0, is a 4-bit
 *               code); s32 = max((hi - lo) / 15, 1e-8);
 *               z = -round_half_even(lo / s32), in [0, 15];
 *               q = clamp(round_half_even(W / s32) + z, 0, 15);
 *               the nibble holds q; zeros_u8[n, g] = z.
 *   scales_f16[n, g] = fp16_round_nearest_even(s32).
 *
 *   group      32, 64, 128, or W4A16_GROUP_PER_CHANNEL (one group of K).
 *   asymmetric 0 (symmetric) or 1.
 *   qweight    [N, K/2] bytes (low nibble = even k), written.
 *   scales_f16 [N, K/group] fp16, written.
 *   zeros_u8   [N, K/group] bytes, written when asymmetric (may be NULL
 *              otherwise).
 * Group 128 symmetric is exactly w4a16_quantize.  The results are
 * bit-identical to the library's CPU reference definition.
 * Errors: as w4a16_quantize; a group other than the above -> W4A16_ERR_SHAPE.
 */
int w4a16_quantize_ex(const void *W_f16, int64_t N, int64_t K, int32_t group, int32_t asymmetric,
                      void *qweight, void *scales_f16, void *zeros_u8, void *stream);

/*
 * Bytes of the kernel layout produced by w4a16_repack for an [N, K] weight:
 * N rounded up to a multiple of 128, times K/2.  Returns -1 on a bad shape.
 */
int64_t w4a16_repacked_bytes(int64_t N, int64_t K);

/*
 * w4a16_repack -- one-time re-layout of canonical packed weights into the
 * kernel layout read by w4a16_gemm (a pure permutation of nibbles; rows
 * beyond N are padded with nibble 8, i.e. q = 0).
 *
 * The tutorial's packed layout is row-major [N, K/2]; its "block-major"
 * cache-friendly re-layout advice (qaqbuyan.com, llama.cpp tuning section)
 * motivates this step, but the exact layout is the library's own:
 *   block b = n / 128 (128 rows), chunk c = k / 64, tile i = (n % 128) / 16;
 *   512 bytes per (b, c, i), 16 bytes per lane L = 4 * g + t of a warp,
 *   holding rows 16 i + g and 16 i + g + 8 at k = 64 c + 16 t ... + 15.
 *   byte offset = ((b * (K/64) + c) * 8 + i) * 512 + 16 * L.
 *   Within the lane's 16 bytes, 32-bit word s covers k' = 64c + 16t + 4s
 *   .. k' + 3; its nibble positions 0..7 hold (row, k) =
 *   (r0,k'), (r1,k'), (r0,k'+2), (r1,k'+2), (r0,k'+1), (r1,k'+1),
 *   (r0,k'+3), (r1,k'+3) with r0 = 16 i + g and r1 = r0 + 8,
 *   so one lop3 per nibble pair yields the f16 MMA fragment directly.
 *
 *   qweight   [N, K/2] canonical bytes (from w4a16_quantize).
 *   repacked  w4a16_repacked_bytes(N, K) bytes, written.
 * Errors: as w4a16_quantize.  unrepack(repack(P)) == P byte for byte.
 */
int w4a16_repack(const void *qweight, int64_t N, int64_t K, void *repacked, void *stream);

/* Inverse of w4a16_repack: kernel layout -> canonical [N, K/2] bytes. */
int w4a16_unrepack(const void *repacked, int64_t N, int64_t K, void *qweight, void *stream);

/*
 * w4a16_gemm -- y[M, N] = x[M, K] * dequant(W)[N, K]^T.
 *
 * Source: mhpq.cn report §二/§五 (dequantize in registers on the fly, never
 * materialise the fp16 weights; the decode step is memory-bound) and the
 * qaqbuyan.com tutorial §3 dequantizer: W[n, k] = (nibble - 8) * scale[n, k/128].
 *
 *   x_f16      [M, K] fp16 activations.
 *   repacked   weights in the kernel layout (w4a16_repack).
 *   scales_f16 [N, K/128] fp16 scales (canonical layout, as quantized).
 *   y_f16      [M, N] fp16 output, written (FP32 accumulation, rounded to
 *              nearest-even fp16 once at the end).
 *   M          1..16 runs the decode GEMV (warp MMAs fed by a bulk-copy
 *              shared-memory ring); M > 16 runs the tcgen05 tensor-core GEMM
 *              (fp16 q*scale staged in shared memory, FP32 accumulators in
 *              tensor memory).
 *   N, K       N >= 1; K >= 128 and K % 128 == 0.
 * Accuracy against the exact result: max|y - y_ref| <= 2e-3 * max|y_ref|
 * and ||y - y_ref||_2 <= 1e-3 * ||y_ref||_2 for the library's test inputs.
 * The call is graph-capturable and uses programmatic dependent launch.
 * Weights and scales are read as constants of the call: their first tiles
 * may be loaded while the kernel enqueued before it on the stream is still
 * running (x is read and y written only after that kernel completes).  So
 * the weights and scales must not be written by work that is still pending
 * on the stream when w4a16_gemm is enqueued -- synchronise (or wait on an
 * event) after writing them -- except by w4a16_quantize and w4a16_repack,
 * which make their results visible before they finish.
 * Errors: NULL -> W4A16_ERR_NULL; bad M, N, K -> W4A16_ERR_SHAPE;
 *         misaligned pointer -> W4A16_ERR_ALIGN; launch failure ->
 *         W4A16_ERR_CUDA.
 */
int w4a16_gemm(const void *x_f16, const void *repacked, const void *scales_f16, void *y_f16,
               int64_t M, int64_t N, int64_t K, void *stream);

/*
 * w4a16_gemm_ex -- w4a16_gemm for the format variants of w4a16_quantize_ex,
 * with an optional AWQ activation scale:
 *   y[m, n] = sum_k x~[m, k] * (nib[n, k] - z[n, k/g]) * scale[n, k/g],
 * z = zeros_u8[n, k/g] for asymmetric codes, z = 8 for symmetric codes
 * (zeros_u8 NULL); x~ = x, or x~[m, k] = fp16_rne(x[m, k] * alpha[k]) when
 * alpha_f16 is given.  Source: tutorial §2 symmetric / asymmetric formulas,
 * §3 granularity and its AWQ section (x~_j = x_j alpha_j against weights
 * quantized from W_{:,j} / alpha_j; the alpha search is the caller's);
 * report §二/§五 for the decode product.
 *
 *   alpha_f16  [K] fp16 per-input-channel scale, or NULL.
 *   repacked   w4a16_repack of the variant's packed codes (the layout does
 *              not depend on the format).
 *   scales_f16 [N, K/g] fp16; zeros_u8 [N, K/g] bytes or NULL.
 *   group      32, 64, 128 or W4A16_GROUP_PER_CHANNEL (g = K).
 *   M          1 .. 2^22.  M <= 16 runs the variant decode GEMV while
 *              x[M, K] fits in its shared memory beside the weight ring
 *              (about 2 * M * K <= 200 KB: M = 1 any K up to 32768, M = 16
 *              K up to 6144); larger M, or a shape that does not fit, runs
 *              the tcgen05 tensor-core GEMM of w4a16_gemm with the variant's
 *              dequantisers.  There alpha multiplies the fp16 dequantised
 *              weight instead of x: y[m, n] = sum_k x[m, k] *
 *              fp16(fp16((nib - z) * scale) * alpha[k]), the same product
 *              with its rounding on the weight operand.
 * Group 128 with symmetric codes and no alpha runs w4a16_gemm's kernels
 * (exact q * x products, one FP32 rescale per group).  The other calls dequantise
 * (nib - z) * scale once to fp16 per weight (the tutorial's own fp16
 * dequantised weight) and accumulate in FP32; the accuracy bar is the same.
 * Errors: as w4a16_gemm; a group other than the above -> W4A16_ERR_SHAPE.
 */
int w4a16_gemm_ex(const void *x_f16, const void *alpha_f16, const void *repacked,
                  const void *scales_f16, const void *zeros_u8, void *y_f16, int64_t M,
                  int64_t N, int64_t K, int32_t group, void *stream);

/*
 * w4a16_quantize_q4_0 -- weights in GGUF Q4_0 blocks.
 *
 * Source: tutorial GGUF section (a Q4_0 block: 32 weights in 18 bytes, d as
 * little-endian fp16, then 16 bytes whose byte i holds element 2i in its low
 * nibble and 2i + 1 in its high nibble, decoded as (nibble - 8) * d); the
 * codes are the §2 / §3 symmetric quantizer with groups of 32 (the pages
 * give the block's decoder, not a separate quantizer), i.e. exactly
 * w4a16_quantize_ex(group 32, symmetric) laid out block after block.
 *
 *   W_f16      [N, K] fp16.  N >= 1; K >= 256, K % 256 == 0 (rows of whole
 *              16-byte lines for the GEMV's copies).
 *   blocks_u8  [N, K/32 * 18] bytes, written; block b of row n at byte
 *              (n * K/32 + b) * 18.
 * Bit-identical to the library's CPU reference definition.
 * Errors: NULL -> W4A16_ERR_NULL; bad N, K -> W4A16_ERR_SHAPE; misaligned
 *         pointer -> W4A16_ERR_ALIGN.
 */
int w4a16_quantize_q4_0(const void *W_f16, int64_t N, int64_t K, void *blocks_u8, void *stream);

/*
 * w4a16_gemm_q4_0 -- decode GEMV on Q4_0 blocks:
 *   y[m, n] = sum_b d[n, b] * sum_{i<32} x[m, 32 b + i] * (nib[n, 32 b + i] - 8),
 * exact q * x products, one FP32 rescale per block, y rounded once to fp16.
 * M = 1..16; K % 256 == 0; x[M, K] held in shared memory whole (as
 * w4a16_gemm_w8).  Errors: as w4a16_gemm_w8.
 */
int w4a16_gemm_q4_0(const void *x_f16, const void *blocks_u8, void *y_f16, int64_t M, int64_t N,
                    int64_t K, void *stream);

/*
 * w4a16_quantize_w8 -- W8A16 weights: per-channel symmetric INT8.
 *
 * Source: tutorial "量化的数学基石" §2 formula with b = 8 and its INT8
 * section ("per-channel, 对称").  Per row n, in IEEE binary32 on the exactly
 * upcast inputs:
 *     s32 = max(max_k |W[n, k]| / 127, 1e-8)          (correctly rounded /)
 *     q   = clamp(round_half_even(W[n, k] / s32), -128, 127)
 *     codes[n, k] = q + 128;  scales_f16[n] = fp16_round_nearest_even(s32)
 *
 *   W_f16      [N, K] fp16.  N >= 1; K >= 128, K % 128 == 0.
 *   codes_u8   [N, K] bytes, written (row-major; no repack step).
 *   scales_f16 [N] fp16, written.
 * Bit-identical to the library's CPU reference definition.
 * Errors: NULL -> W4A16_ERR_NULL; bad N, K -> W4A16_ERR_SHAPE; misaligned
 *         pointer -> W4A16_ERR_ALIGN.
 */
int w4a16_quantize_w8(const void *W_f16, int64_t N, int64_t K, void *codes_u8, void *scales_f16,
                      void *stream);

/*
 * w4a16_gemm_w8 -- W8A16 decode GEMV:
 *   y[m, n] = scale[n] * sum_k x[m, k] * (codes[n, k] - 128),
 * exact q * x products accumulated in FP32, the per-row scale applied once,
 * y rounded once to fp16.  M = 1..16; x[M, K] is held in shared memory whole
 * beside the ring (as w4a16_gemm_ex: about 2 * M * K <= 200 KB), a shape
 * that does not fit -> W4A16_ERR_SHAPE.  Graph-capturable, programmatic
 * dependent launch; codes and scales are constants of the call as in
 * w4a16_gemm.
 * Errors: as w4a16_gemm.
 */
int w4a16_gemm_w8(const void *x_f16, const void *codes_u8, const void *scales_f16, void *y_f16,
                  int64_t M, int64_t N, int64_t K, void *stream);

/* Paths reported by w4a16_gemm_plan. */
enum { W4A16_PATH_GEMV = 1, W4A16_PATH_TENSOR_CORE = 2 };

/*
 * w4a16_gemm_plan -- the launch w4a16_gemm makes for (M, N, K) on the current
 * device, without launching anything (introspection for tests and tuning).
 *
 *   *path            W4A16_PATH_GEMV (M <= 16) or W4A16_PATH_TENSOR_CORE.
 *   *splits          the thread-block cluster size: for the GEMV, the CTAs
 *                    sharing the K range of one 128-row block (1 = no
 *                    split); for the tensor-core GEMM, 1 (a CTA per
 *                    128 x 128 tile), 2 (CTA pairs with 2-CTA MMAs) or 4, 6, 8
 *                    (CTA pairs splitting K 2, 3, 4 ways, reduced through the
 *                    cluster's shared memory).
 *   *ctas            CTAs launched.
 *   *blocks_per_cta  most 128-row blocks one CTA walks (> 1: persistent).
 *   *rows_per_cta    weight rows one CTA computes of each block it handles:
 *                    128 (a whole block), or for the GEMV 16, 32 or 64 (1, 2
 *                    or 4 of a block's 16-row tiles over the whole K range,
 *                    the CTA's warps splitting K and reducing in its own
 *                    shared memory), or for the tensor-core GEMM's CTA pairs
 *                    with two x tiles 96 (six 16-row tiles; a pair covers 192
 *                    weight rows).
 * Errors: NULL output -> W4A16_ERR_NULL; bad M, N, K -> W4A16_ERR_SHAPE;
 *         no supported device -> W4A16_ERR_DEVICE / W4A16_ERR_CUDA.
 */
int w4a16_gemm_plan(int64_t M, int64_t N, int64_t K, int *path, int *splits, int *ctas,
                    int *blocks_per_cta, int *rows_per_cta);

/*
 * w4a16_gemm_plan_tail -- the last round of a persistent GEMV launch (more
 * 128-row blocks than CTAs, each CTA walking blocks y, y + ctas, ...).  When
 * the blocks do not divide evenly, the R blocks of the partial last round run
 * as R * 128 / tail_rows units of tail_rows weight rows (16, 32 or 64) over
 * the whole K range, one per CTA, so that round costs tail_rows / 128 of a
 * block instead of a whole one on a few CTAs.
 *
 *   *tail_rows   rows of each tail unit, 0 when the launch has no such round
 *                (not persistent, blocks divide evenly, or more than half a
 *                round left over) or M > 16.
 *   *tail_units  number of tail units (0 with tail_rows = 0).
 * Errors: as w4a16_gemm_plan.
 */
int w4a16_gemm_plan_tail(int64_t M, int64_t N, int64_t K, int *tail_rows, int *tail_units);

/*
 * w4a16_gemm_ex_plan -- the launch w4a16_gemm_ex makes for (M, N, K) with
 * the given group (32, 64, 128 or W4A16_GROUP_PER_CHANNEL), zero points
 * (nonzero: asymmetric codes) and AWQ scale (nonzero: alpha given), without
 * launching anything.
 *
 *   *path         W4A16_PATH_GEMV (M <= 16 with x[M, K] fitting in the
 *                 variant GEMV's shared memory) or W4A16_PATH_TENSOR_CORE.
 *   *splits       as w4a16_gemm_plan (1 for the variant GEMV).
 *   *ctas         CTAs launched.
 *   *rows_per_cta weight rows per CTA: 16, 32 or 64 for the variant GEMV,
 *                 128 for the tensor-core GEMM.
 * Group 128 with symmetric codes and no alpha reports w4a16_gemm_plan's
 * launch (the call runs w4a16_gemm).
 * Errors: NULL output -> W4A16_ERR_NULL; bad M, N, K or group ->
 *         W4A16_ERR_SHAPE; no supported device -> W4A16_ERR_DEVICE /
 *         W4A16_ERR_CUDA.
 */
int w4a16_gemm_ex_plan(int64_t M, int64_t N, int64_t K, int32_t group, int32_t zero_points,
                       int32_t alpha, int *path, int *splits, int *ctas, int *rows_per_cta);

/*
 * w4a16_device_status -- synchronises the current device, returns in
 * *status the OR of the W4A16_ERR_* conditions recorded by kernels since
 * the last call (W4A16_OK if none: W4A16_ERR_TIMEOUT when a bounded wait
 * gave up) and clears the record.  Returns W4A16_ERR_CUDA if the device
 * cannot be read.
 */
int w4a16_device_status(int *status);

/*
 * Upper bound, in nanoseconds, of every wait inside the library's kernels
 * (default 2e9, i.e. two seconds; 0 is taken as 1).  Applies to launches made
 * after the call.  A wait that gives up records W4A16_ERR_TIMEOUT (see
 * w4a16_device_status); the kernel then issues no more copies and waits for
 * those in flight before it exits.  That last wait is bounded by the larger
 * of this value and 100 ms, so a short limit cannot let a block exit while a
 * copy still writes into its shared memory.  Safe to call from any thread.
 */
void w4a16_set_wait_timeout_ns(uint64_t timeout_ns);

/*
 * w4a16_selftest_wait_timeout -- diagnostic: launches one block that waits
 * on an mbarrier nothing will ever arrive on, with a wait bound of
 * `timeout_ns`.  The kernel gives up after that time, records
 * W4A16_ERR_TIMEOUT in the device status word and exits normally, leaving
 * the context usable.  Used by the tests of the failure path.
 */
int w4a16_selftest_wait_timeout(uint64_t timeout_ns, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* W4A16_H */
