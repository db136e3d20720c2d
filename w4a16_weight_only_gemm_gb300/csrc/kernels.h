// kernels.h -- host-side launchers of the W4A16 kernels (internal to the
// library; the public C ABI is include/w4a16.h).
#pragma once

#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace w4a16 {

// Per-device facts and the device status word, resolved once per device.
struct DeviceCtx {
    unsigned* status;       // device address of the status word
    uint64_t timeout_ns;    // bound on every in-kernel wait
    int num_sms;
    int max_smem_optin;     // bytes of dynamic shared memory a block may opt into
};

// Rows per repacked block and chunk width of the kernel layout.
constexpr int kBlockRows = 128;
constexpr int kChunkK = 64;
constexpr int kGroup = 128;

// The driver's cuTensorMapEncodeTiled, resolved once (null if unavailable).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();

cudaError_t launch_quantize(const void* W, int64_t N, int64_t K, void* qweight, void* scales,
                            cudaStream_t stream, const DeviceCtx& ctx);
// Format variants of the quantizer: group = 32, 64, 128 or K (per-channel),
// symmetric or asymmetric (zeros: [N, K/group] bytes).
cudaError_t launch_quantize_fmt(const void* W, int64_t N, int64_t K, int group, bool asym,
                                void* qweight, void* scales, void* zeros, cudaStream_t stream,
                                const DeviceCtx& ctx);
// GGUF Q4_0 blocks (group-32 symmetric codes, 18 bytes per 32 weights) and the GEMV.
cudaError_t launch_quantize_q4_0(const void* W, int64_t N, int64_t K, void* blocks,
                                 cudaStream_t stream, const DeviceCtx& ctx);
cudaError_t launch_gemv_q4_0(const void* x, const void* blocks, void* y, int M, int64_t N,
                             int64_t K, cudaStream_t stream, const DeviceCtx& ctx);
// W8A16: per-channel symmetric INT8 codes (q + 128, [N, K] bytes) and the GEMV.
cudaError_t launch_quantize_w8(const void* W, int64_t N, int64_t K, void* q8, void* scales,
                               cudaStream_t stream, const DeviceCtx& ctx);
cudaError_t launch_gemv_w8(const void* x, const void* q8, const void* scales, void* y, int M,
                           int64_t N, int64_t K, cudaStream_t stream, const DeviceCtx& ctx);
cudaError_t launch_repack(const void* qweight, int64_t N, int64_t K, void* repacked,
                          cudaStream_t stream, const DeviceCtx& ctx);
cudaError_t launch_unrepack(const void* repacked, int64_t N, int64_t K, void* qweight,
                            cudaStream_t stream, const DeviceCtx& ctx);
// The cached tensor map of a GEMV unit launch: the kernel layout of an
// [N, K] weight as rows of 4 KB chunks, a box of T tiles x 32 / T chunks
// (T = 1, 2 or 4).
cudaError_t gemv_weight_map(const void* repacked, int64_t N, int64_t K, int T, CUtensorMap* out);
// Decode GEMV of the format variants (group = 32, 64, 128 or K; zeros NULL
// for symmetric codes; alpha [K] an AWQ activation scale or NULL).
cudaError_t launch_gemv_fmt(const void* x, const void* alpha, const void* repacked,
                            const void* scales, const void* zeros, void* y, int M, int64_t N,
                            int64_t K, int group, cudaStream_t stream, const DeviceCtx& ctx);
// Whether the decode GEMV of the format variants has a shared-memory layout
// for (M, K): x[M, K] and the smallest unit's scales beside a 3-stage ring.
bool gemv_fmt_fits(int M, int64_t N, int64_t K, int group, bool zp, const DeviceCtx& ctx);
// The launch the variant GEMV would make: CTAs and weight rows per CTA.
cudaError_t gemv_fmt_plan_info(int M, int64_t N, int64_t K, int group, bool zp, const DeviceCtx& ctx,
                               int* ctas, int* rows_per_cta);
// Tensor-core GEMM of the format variants (any M; same arguments as
// launch_gemv_fmt): fp16((nib - z) * s) weight tiles, times alpha[k] in the
// tile when an AWQ scale is given.
cudaError_t launch_gemm_tc_fmt(const void* x, const void* alpha, const void* repacked,
                               const void* scales, const void* zeros, void* y, int64_t M, int64_t N,
                               int64_t K, int group, cudaStream_t stream, const DeviceCtx& ctx);
cudaError_t launch_gemv(const void* x, const void* repacked, const void* scales, void* y, int M,
                        int64_t N, int64_t K, cudaStream_t stream, const DeviceCtx& ctx);
// The launch the decode GEMV would make: K split (cluster size), CTAs, the
// most 128-row blocks one CTA walks, the weight rows of one CTA's unit, and
// for a persistent launch with a partial last round the rows of each tail
// unit and their number (0, 0 without one).
cudaError_t gemv_plan_info(int M, int64_t N, int64_t K, const DeviceCtx& ctx, int* splits,
                           int* ctas, int* blocks_per_cta, int* rows_per_cta, int* tail_rows,
                           int* tail_units);
// The launch the tensor-core GEMM would make: cluster size (1: one CTA per
// 128 x 128 tile; 2: CTA pairs with 2-CTA MMAs; 4, 6 or 8: CTA pairs
// splitting K two, three or four ways, reduced over the cluster), CTAs and
// (if rows_per_cta) the weight rows of one CTA (128, or 96 for pairs with two
// x tiles).  fmt: the format variants' kernels (no scale slab).
void gemm_tc_plan_info(int64_t M, int64_t N, int64_t K, const DeviceCtx& ctx, int* cluster,
                       int* ctas, bool fmt = false, int* rows_per_cta = nullptr);
cudaError_t launch_gemm_tc(const void* x, const void* repacked, const void* scales, void* y,
                           int64_t M, int64_t N, int64_t K, cudaStream_t stream,
                           const DeviceCtx& ctx);
cudaError_t launch_selftest_wait(uint64_t timeout_ns, cudaStream_t stream, const DeviceCtx& ctx);

}  // namespace w4a16
