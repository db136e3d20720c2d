// quantize.cu -- group-wise symmetric round-to-nearest INT4 quantizer.
//
// Computes, per row and group of 128 weights along K (qaqbuyan.com tutorial
// "LLM quantization from IEEE 754 to GPTQ/AWQ/GGUF", chapter "量化的数学基石",
// §2 symmetric formula and §3 per_group_symmetric_quantize):
//   s32 = max(max|w| / 7, 1e-8) in binary32 with a correctly rounded divide,
//   q   = clamp(round_half_even(w / s32), -8, 7),
//   scale = fp16(s32) rounded to nearest even, byte = (q_odd+8)<<4 | (q_even+8).
//
// One half-warp per group: each of the 16 lanes loads 8 fp16 values with a
// single 16-byte load, the absmax is reduced with xor-shuffles inside the
// half-warp, and each lane writes its 4 packed bytes (the group's 64 bytes
// are one coalesced segment).  HBM-bound: 256 B read and 66 B written per
// group.
#include "common.cuh"
#include "kernels.h"

namespace w4a16 {
namespace {

constexpr int kQuantThreads = 256;

__global__ void __launch_bounds__(kQuantThreads)
    quantize_kernel(const uint4* __restrict__ W, int64_t groups_total,
                    uint32_t* __restrict__ qweight, __half* __restrict__ scales) {
    const int lane16 = threadIdx.x & 15;
    const int64_t step = (int64_t)gridDim.x * (kQuantThreads / 16);
    for (int64_t grp = (int64_t)blockIdx.x * (kQuantThreads / 16) + (threadIdx.x >> 4);
         grp < groups_total; grp += step) {
        // group `grp` = row grp / G, group grp % G; its 128 halves are
        // contiguous at element offset grp * 128 of the row-major matrix.
        const uint4 raw = __ldg(W + grp * 16 + lane16);
        const __half2* h2 = reinterpret_cast<const __half2*>(&raw);
        float w[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 f = __half22float2(h2[i]);
            w[2 * i] = f.x;
            w[2 * i + 1] = f.y;
        }
        float amax = 0.0f;
#pragma unroll
        for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(w[i]));
#pragma unroll
        for (int off = 8; off > 0; off >>= 1)
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));

        float s = __fdiv_rn(amax, 7.0f);
        if (s < 1e-8f) s = 1e-8f;

        uint32_t packed = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            int q = __float2int_rn(__fdiv_rn(w[i], s));
            q = q < -8 ? -8 : (q > 7 ? 7 : q);
            packed |= (uint32_t)(q + 8) << (4 * i);
        }
        qweight[grp * 16 + lane16] = packed;
        if (lane16 == 0) scales[grp] = __float2half_rn(s);
    }
    // Publish the packed weights and scales device-wide before this block
    // ends: a GEMM launched next on the stream may read them before the
    // grid-completion flush (it treats them as constants).
    __threadfence();
}

}  // namespace

cudaError_t launch_quantize(const void* W, int64_t N, int64_t K, void* qweight, void* scales,
                            cudaStream_t stream, const DeviceCtx& ctx) {
    const int G = (int)(K / kGroup);
    const int64_t groups = N * G;
    const int64_t per_block = kQuantThreads / 16;
    int64_t blocks = (groups + per_block - 1) / per_block;
    const int64_t cap = (int64_t)ctx.num_sms * 16;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    quantize_kernel<<<(unsigned)blocks, kQuantThreads, 0, stream>>>(
        static_cast<const uint4*>(W), groups, static_cast<uint32_t*>(qweight),
        static_cast<__half*>(scales));
    return cudaGetLastError();
}

}  // namespace w4a16
