// gemm_tc.cu -- prefill path (M > 16): tcgen05 tensor-core GEMM.  Not built yet.
#include "kernels.h"

namespace w4a16 {

cudaError_t launch_gemm_tc(const void*, const void*, const void*, void*, int64_t, int64_t,
                           int64_t, cudaStream_t, const DeviceCtx&) {
    return cudaErrorNotSupported;
}

}  // namespace w4a16
