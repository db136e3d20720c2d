// api.cu -- the C ABI (include/w4a16.h): argument checks, per-device set-up,
// dispatch to the kernels, the device status word and its self-test.
#include <atomic>
#include <mutex>

#include "../../include/w4a16.h"
#include "common.cuh"
#include "kernels.h"

namespace w4a16 {
namespace {

// Status word written by kernels (atomicOr of kDev* bits); one per device.
__device__ unsigned g_device_status;

constexpr int kMaxDevices = 64;
std::atomic<uint64_t> g_timeout_ns{2000000000ull};  // read at every launch, set from any thread

struct DeviceSlot {
    std::once_flag once;
    cudaError_t init_error = cudaSuccess;
    bool supported = false;
    DeviceCtx ctx{};
};
DeviceSlot g_slots[kMaxDevices];

// Resolves the status word's device address (the symbol's host-side name is
// only a handle) and the SM count once per device, with that device current.
int device_ctx(DeviceCtx* out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return W4A16_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return W4A16_ERR_DEVICE;
    DeviceSlot& slot = g_slots[dev];
    std::call_once(slot.once, [&]() {
        cudaDeviceProp prop;
        slot.init_error = cudaGetDeviceProperties(&prop, dev);
        if (slot.init_error != cudaSuccess) return;
        slot.supported = (prop.major == 10 && prop.minor == 3);
        if (!slot.supported) return;
        void* p = nullptr;
        slot.init_error = cudaGetSymbolAddress(&p, g_device_status);
        if (slot.init_error != cudaSuccess) return;
        slot.ctx.status = static_cast<unsigned*>(p);
        slot.ctx.num_sms = prop.multiProcessorCount;
        slot.ctx.max_smem_optin = (int)prop.sharedMemPerBlockOptin;
    });
    if (slot.init_error != cudaSuccess) return W4A16_ERR_CUDA;
    if (!slot.supported) return W4A16_ERR_DEVICE;
    *out = slot.ctx;
    out->timeout_ns = g_timeout_ns.load(std::memory_order_relaxed);
    return W4A16_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool good_nk(int64_t N, int64_t K) {
    return N >= 1 && N <= (int64_t)1 << 30 && K >= kGroup && K % kGroup == 0 &&
           K <= (int64_t)1 << 20 && N * K <= (int64_t)1 << 40;
}

// Launchers report an unsupported configuration (no shared-memory layout
// fits) as cudaErrorInvalidValue before launching anything.
int from_cuda(cudaError_t e) {
    if (e == cudaSuccess) return W4A16_OK;
    return e == cudaErrorInvalidValue ? W4A16_ERR_SHAPE : W4A16_ERR_CUDA;
}

__global__ void selftest_wait_kernel(unsigned* status, uint64_t timeout_ns) {
    __shared__ __align__(8) uint64_t bar;
    const uint32_t b = smem_u32(&bar);
    if (threadIdx.x == 0) {
        mbar_init(b, 1);
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) (void)mbar_wait(b, 0, timeout_ns, status);  // nothing arrives
}

}  // namespace

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, []() {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

cudaError_t launch_selftest_wait(uint64_t timeout_ns, cudaStream_t stream, const DeviceCtx& ctx) {
    selftest_wait_kernel<<<1, 32, 0, stream>>>(ctx.status, timeout_ns);
    return cudaGetLastError();
}

}  // namespace w4a16

using namespace w4a16;

extern "C" {

const char* w4a16_status_string(int status) {
    switch (status) {
        case W4A16_OK: return "W4A16_OK";
        case W4A16_ERR_NULL: return "W4A16_ERR_NULL: a required pointer is NULL";
        case W4A16_ERR_SHAPE: return "W4A16_ERR_SHAPE: unsupported M, N, K or group size";
        case W4A16_ERR_ALIGN: return "W4A16_ERR_ALIGN: a pointer is not 16-byte aligned";
        case W4A16_ERR_CUDA: return "W4A16_ERR_CUDA: a CUDA runtime call or launch failed";
        case W4A16_ERR_TIMEOUT: return "W4A16_ERR_TIMEOUT: a kernel's bounded wait gave up";
        case W4A16_ERR_DEVICE: return "W4A16_ERR_DEVICE: the current device is not sm_103";
        default: return "W4A16: unknown status";
    }
}

int w4a16_version(void) { return 100; }

int w4a16_quantize(const void* W_f16, int64_t N, int64_t K, int32_t group, void* qweight,
                   void* scales_f16, void* stream) {
    if (!W_f16 || !qweight || !scales_f16) return W4A16_ERR_NULL;
    if (group != W4A16_GROUP || !good_nk(N, K)) return W4A16_ERR_SHAPE;
    if (!aligned16(W_f16) || !aligned16(qweight) || !aligned16(scales_f16)) return W4A16_ERR_ALIGN;
    DeviceCtx ctx;
    if (int rc = device_ctx(&ctx)) return rc;
    return from_cuda(launch_quantize(W_f16, N, K, qweight, scales_f16,
                                     static_cast<cudaStream_t>(stream), ctx));
}

int w4a16_quantize_ex(const void* W_f16, int64_t N, int64_t K, int32_t group, int32_t asymmetric,
                      void* qweight, void* scales_f16, void* zeros_u8, void* stream) {
    if (!W_f16 || !qweight || !scales_f16 || (asymmetric && !zeros_u8)) return W4A16_ERR_NULL;
    if (!good_nk(N, K) || (asymmetric != 0 && asymmetric != 1)) return W4A16_ERR_SHAPE;
    if (group == W4A16_GROUP_PER_CHANNEL) group = (int32_t)K;
    if (!(group == 32 || group == 64 || group == 128 || group == K)) return W4A16_ERR_SHAPE;
    if (!aligned16(W_f16) || !aligned16(qweight) || !aligned16(scales_f16) ||
        (asymmetric && !aligned16(zeros_u8)))
        return W4A16_ERR_ALIGN;
    DeviceCtx ctx;
    if (int rc = device_ctx(&ctx)) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (group == W4A16_GROUP && !asymmetric)
        return from_cuda(launch_quantize(W_f16, N, K, qweight, scales_f16, s, ctx));
    return from_cuda(launch_quantize_fmt(W_f16, N, K, group, asymmetric != 0, qweight, scales_f16,
                                         zeros_u8, s, ctx));
}

int64_t w4a16_repacked_bytes(int64_t N, int64_t K) {
    if (!good_nk(N, K)) return -1;
    return (N + kBlockRows - 1) / kBlockRows * kBlockRows * (K / 2);
}

int w4a16_repack(const void* qweight, int64_t N, int64_t K, void* repacked, void* stream) {
    if (!qweight || !repacked) return W4A16_ERR_NULL;
    if (!good_nk(N, K)) return W4A16_ERR_SHAPE;
    if (!aligned16(qweight) || !aligned16(repacked)) return W4A16_ERR_ALIGN;
    DeviceCtx ctx;
    if (int rc = device_ctx(&ctx)) return rc;
    return from_cuda(
        launch_repack(qweight, N, K, repacked, static_cast<cudaStream_t>(stream), ctx));
}

int w4a16_unrepack(const void* repacked, int64_t N, int64_t K, void* qweight, void* stream) {
    if (!qweight || !repacked) return W4A16_ERR_NULL;
    if (!good_nk(N, K)) return W4A16_ERR_SHAPE;
    if (!aligned16(qweight) || !aligned16(repacked)) return W4A16_ERR_ALIGN;
    DeviceCtx ctx;
    if (int rc = device_ctx(&ctx)) return rc;
    return from_cuda(
        launch_unrepack(repacked, N, K, qweight, static_cast<cudaStream_t>(stream), ctx));
}

int w4a16_gemm(const void* x_f16, const void* repacked, const void* scales_f16, void* y_f16,
               int64_t M, int64_t N, int64_t K, void* stream) {
    if (!x_f16 || !repacked || !scales_f16 || !y_f16) return W4A16_ERR_NULL;
    if (M < 1 || M > (int64_t)1 << 22 || !good_nk(N, K) || N > (int64_t)1 << 28 ||
        K > (int64_t)1 << 15)
        return W4A16_ERR_SHAPE;
    if (!aligned16(x_f16) || !aligned16(repacked) || !aligned16(scales_f16) || !aligned16(y_f16))
        return W4A16_ERR_ALIGN;
    DeviceCtx ctx;
    if (int rc = device_ctx(&ctx)) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (M <= 16) return from_cuda(launch_gemv(x_f16, repacked, scales_f16, y_f16, (int)M, N, K, s, ctx));
    return from_cuda(launch_gemm_tc(x_f16, repacked, scales_f16, y_f16, M, N, K, s, ctx));
}

int w4a16_gemm_ex(const void* x_f16, const void* alpha_f16, const void* repacked,
                  const void* scales_f16, const void* zeros_u8, void* y_f16, int64_t M,
                  int64_t N, int64_t K, int32_t group, void* stream) {
    if (!x_f16 || !repacked || !scales_f16 || !y_f16) return W4A16_ERR_NULL;
    if (M < 1 || M > (int64_t)1 << 22 || !good_nk(N, K) || N > (int64_t)1 << 28 ||
        K > (int64_t)1 << 15)
        return W4A16_ERR_SHAPE;
    if (group == W4A16_GROUP_PER_CHANNEL) group = (int32_t)K;
    if (!(group == 32 || group == 64 || group == 128 || group == K)) return W4A16_ERR_SHAPE;
    if (!aligned16(x_f16) || !aligned16(repacked) || !aligned16(scales_f16) || !aligned16(y_f16) ||
        (zeros_u8 && !aligned16(zeros_u8)) || (alpha_f16 && !aligned16(alpha_f16)))
        return W4A16_ERR_ALIGN;
    if (group == W4A16_GROUP && !zeros_u8 && !alpha_f16)
        return w4a16_gemm(x_f16, repacked, scales_f16, y_f16, M, N, K, stream);
    DeviceCtx ctx;
    if (int rc = device_ctx(&ctx)) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // Decode GEMV while x fits in its shared memory, else the tensor cores.
    if (M <= 16 && gemv_fmt_fits((int)M, N, K, group, zeros_u8 != nullptr, ctx))
        return from_cuda(launch_gemv_fmt(x_f16, alpha_f16, repacked, scales_f16, zeros_u8, y_f16,
                                         (int)M, N, K, group, s, ctx));
    return from_cuda(launch_gemm_tc_fmt(x_f16, alpha_f16, repacked, scales_f16, zeros_u8, y_f16, M,
                                        N, K, group, s, ctx));
}

int w4a16_quantize_q4_0(const void* W_f16, int64_t N, int64_t K, void* blocks_u8, void* stream) {
    if (!W_f16 || !blocks_u8) return W4A16_ERR_NULL;
    if (!good_nk(N, K) || K % 256 != 0) return W4A16_ERR_SHAPE;
    if (!aligned16(W_f16) || !aligned16(blocks_u8)) return W4A16_ERR_ALIGN;
    DeviceCtx ctx;
    if (int rc = device_ctx(&ctx)) return rc;
    return from_cuda(
        launch_quantize_q4_0(W_f16, N, K, blocks_u8, static_cast<cudaStream_t>(stream), ctx));
}

int w4a16_gemm_q4_0(const void* x_f16, const void* blocks_u8, void* y_f16, int64_t M, int64_t N,
                    int64_t K, void* stream) {
    if (!x_f16 || !blocks_u8 || !y_f16) return W4A16_ERR_NULL;
    if (M < 1 || M > 16 || !good_nk(N, K) || K % 256 != 0 || N > (int64_t)1 << 28 ||
        K > (int64_t)1 << 15)
        return W4A16_ERR_SHAPE;
    if (!aligned16(x_f16) || !aligned16(blocks_u8) || !aligned16(y_f16)) return W4A16_ERR_ALIGN;
    DeviceCtx ctx;
    if (int rc = device_ctx(&ctx)) return rc;
    return from_cuda(launch_gemv_q4_0(x_f16, blocks_u8, y_f16, (int)M, N, K,
                                      static_cast<cudaStream_t>(stream), ctx));
}

int w4a16_quantize_w8(const void* W_f16, int64_t N, int64_t K, void* codes_u8, void* scales_f16,
                      void* stream) {
    if (!W_f16 || !codes_u8 || !scales_f16) return W4A16_ERR_NULL;
    if (!good_nk(N, K)) return W4A16_ERR_SHAPE;
    if (!aligned16(W_f16) || !aligned16(codes_u8) || !aligned16(scales_f16)) return W4A16_ERR_ALIGN;
    DeviceCtx ctx;
    if (int rc = device_ctx(&ctx)) return rc;
    return from_cuda(launch_quantize_w8(W_f16, N, K, codes_u8, scales_f16,
                                        static_cast<cudaStream_t>(stream), ctx));
}

int w4a16_gemm_w8(const void* x_f16, const void* codes_u8, const void* scales_f16, void* y_f16,
                  int64_t M, int64_t N, int64_t K, void* stream) {
    if (!x_f16 || !codes_u8 || !scales_f16 || !y_f16) return W4A16_ERR_NULL;
    if (M < 1 || M > 16 || !good_nk(N, K) || N > (int64_t)1 << 28 || K > (int64_t)1 << 15)
        return W4A16_ERR_SHAPE;
    if (!aligned16(x_f16) || !aligned16(codes_u8) || !aligned16(scales_f16) || !aligned16(y_f16))
        return W4A16_ERR_ALIGN;
    DeviceCtx ctx;
    if (int rc = device_ctx(&ctx)) return rc;
    return from_cuda(launch_gemv_w8(x_f16, codes_u8, scales_f16, y_f16, (int)M, N, K,
                                    static_cast<cudaStream_t>(stream), ctx));
}

int w4a16_gemm_plan(int64_t M, int64_t N, int64_t K, int* path, int* splits, int* ctas,
                    int* blocks_per_cta, int* rows_per_cta) {
    if (!path || !splits || !ctas || !blocks_per_cta || !rows_per_cta) return W4A16_ERR_NULL;
    if (M < 1 || M > (int64_t)1 << 22 || !good_nk(N, K) || N > (int64_t)1 << 28 ||
        K > (int64_t)1 << 15)
        return W4A16_ERR_SHAPE;
    DeviceCtx ctx;
    if (int rc = device_ctx(&ctx)) return rc;
    if (M > 16) {
        *path = W4A16_PATH_TENSOR_CORE;
        gemm_tc_plan_info(M, N, K, ctx, splits, ctas, false, rows_per_cta);
        if (*splits == 0) return W4A16_ERR_CUDA;
        *blocks_per_cta = 1;
        return W4A16_OK;
    }
    int tail_rows = 0, tail_units = 0;
    if (int rc = from_cuda(gemv_plan_info((int)M, N, K, ctx, splits, ctas, blocks_per_cta,
                                          rows_per_cta, &tail_rows, &tail_units)))
        return rc;
    *path = W4A16_PATH_GEMV;
    return W4A16_OK;
}

int w4a16_gemm_plan_tail(int64_t M, int64_t N, int64_t K, int* tail_rows, int* tail_units) {
    if (!tail_rows || !tail_units) return W4A16_ERR_NULL;
    if (M < 1 || M > (int64_t)1 << 22 || !good_nk(N, K) || N > (int64_t)1 << 28 ||
        K > (int64_t)1 << 15)
        return W4A16_ERR_SHAPE;
    *tail_rows = 0;
    *tail_units = 0;
    if (M > 16) return W4A16_OK;
    DeviceCtx ctx;
    if (int rc = device_ctx(&ctx)) return rc;
    int splits = 0, ctas = 0, blocks = 0, rows = 0;
    return from_cuda(gemv_plan_info((int)M, N, K, ctx, &splits, &ctas, &blocks, &rows, tail_rows,
                                    tail_units));
}

int w4a16_gemm_ex_plan(int64_t M, int64_t N, int64_t K, int32_t group, int32_t zero_points,
                       int32_t alpha, int* path, int* splits, int* ctas, int* rows_per_cta) {
    if (!path || !splits || !ctas || !rows_per_cta) return W4A16_ERR_NULL;
    if (M < 1 || M > (int64_t)1 << 22 || !good_nk(N, K) || N > (int64_t)1 << 28 ||
        K > (int64_t)1 << 15)
        return W4A16_ERR_SHAPE;
    if (group == W4A16_GROUP_PER_CHANNEL) group = (int32_t)K;
    if (!(group == 32 || group == 64 || group == 128 || group == K)) return W4A16_ERR_SHAPE;
    if (group == W4A16_GROUP && !zero_points && !alpha) {
        int blocks_per_cta = 0;
        return w4a16_gemm_plan(M, N, K, path, splits, ctas, &blocks_per_cta, rows_per_cta);
    }
    DeviceCtx ctx;
    if (int rc = device_ctx(&ctx)) return rc;
    if (M <= 16 && gemv_fmt_fits((int)M, N, K, group, zero_points != 0, ctx)) {
        *path = W4A16_PATH_GEMV;
        *splits = 1;
        return from_cuda(
            gemv_fmt_plan_info((int)M, N, K, group, zero_points != 0, ctx, ctas, rows_per_cta));
    }
    *path = W4A16_PATH_TENSOR_CORE;
    gemm_tc_plan_info(M, N, K, ctx, splits, ctas, true);
    if (*splits == 0) return W4A16_ERR_CUDA;
    *rows_per_cta = 128;
    return W4A16_OK;
}

int w4a16_device_status(int* status) {
    if (!status) return W4A16_ERR_NULL;
    DeviceCtx ctx;
    if (int rc = device_ctx(&ctx)) return rc;
    if (cudaDeviceSynchronize() != cudaSuccess) return W4A16_ERR_CUDA;
    unsigned word = 0;
    if (cudaMemcpy(&word, ctx.status, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess)
        return W4A16_ERR_CUDA;
    const unsigned zero = 0;
    if (cudaMemcpy(ctx.status, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess)
        return W4A16_ERR_CUDA;
    *status = (word & kDevTimeout) ? W4A16_ERR_TIMEOUT
              : (word & kDevBadLaunch) ? W4A16_ERR_SHAPE
                                       : W4A16_OK;
    return W4A16_OK;
}

void w4a16_set_wait_timeout_ns(uint64_t timeout_ns) {
    g_timeout_ns.store(timeout_ns == 0 ? 1 : timeout_ns, std::memory_order_relaxed);
}

int w4a16_selftest_wait_timeout(uint64_t timeout_ns, void* stream) {
    DeviceCtx ctx;
    if (int rc = device_ctx(&ctx)) return rc;
    return from_cuda(launch_selftest_wait(timeout_ns, static_cast<cudaStream_t>(stream), ctx));
}

}  // extern "C"
