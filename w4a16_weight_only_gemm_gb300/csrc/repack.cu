// repack.cu -- canonical packed INT4 weights <-> the kernel layout.
//
// Canonical layout (qaqbuyan.com tutorial, "量化的数学基石" §3): row-major
// [N, K/2] bytes, k even in the low nibble, k odd in the high nibble, each
// stored as q + 8.  Kernel layout (the library's own; the tutorial's
// llama.cpp tuning section motivates a block-major re-layout): for block
// b = n/128, chunk c = k/64 and 16-row tile i, 512 contiguous bytes of
// which lane L = 4g + t of a warp owns 16: rows r0 = 16i + g, r1 = r0 + 8 at
// k = 64c + 16t .. +15.  In the lane's 32-bit word s (k' = 64c + 16t + 4s)
// the nibble positions hold
//   0:(r0,k')  1:(r1,k')  2:(r0,k'+2)  3:(r1,k'+2)
//   4:(r0,k'+1) 5:(r1,k'+1) 6:(r0,k'+3) 7:(r1,k'+3)
// which is exactly the A fragment of mma.m16n8k16 once dequant8() splits
// the word into half2 pairs (0,4) (1,5) (2,6) (3,7).  The weights of one
// 128-row block for one 64-wide chunk are 4 KB contiguous, so a block's
// stream is one linear range.
#include "common.cuh"
#include "kernels.h"

namespace w4a16 {
namespace {

constexpr int kRepackThreads = 256;

// 16 nibbles of one row at k' .. k'+3 (low 16 bits of u) for rows r0 (u)
// and r1 (v) -> one kernel-layout word.
__device__ __forceinline__ uint32_t interleave_word(uint32_t u, uint32_t v) {
    return ((u >> 0) & 0xFu) | (((v >> 0) & 0xFu) << 4) | (((u >> 8) & 0xFu) << 8) |
           (((v >> 8) & 0xFu) << 12) | (((u >> 4) & 0xFu) << 16) | (((v >> 4) & 0xFu) << 20) |
           (((u >> 12) & 0xFu) << 24) | (((v >> 12) & 0xFu) << 28);
}

// Inverse: one kernel-layout word -> (u, v) 16-bit canonical nibble runs.
__device__ __forceinline__ void split_word(uint32_t w, uint32_t& u, uint32_t& v) {
    u = ((w >> 0) & 0xFu) | (((w >> 16) & 0xFu) << 4) | (((w >> 8) & 0xFu) << 8) |
        (((w >> 24) & 0xFu) << 12);
    v = ((w >> 4) & 0xFu) | (((w >> 20) & 0xFu) << 4) | (((w >> 12) & 0xFu) << 8) |
        (((w >> 28) & 0xFu) << 12);
}

struct LaneSite {
    int64_t r0, r1;   // global rows
    int64_t kbyte;    // canonical byte offset of k = 64c + 16t inside a row
};

__device__ __forceinline__ LaneSite lane_site(int64_t o, int64_t C) {
    // o = ((b * C + c) * 8 + i) * 32 + L
    const int L = (int)(o & 31);
    const int64_t tile = o >> 5;
    const int i = (int)(tile & 7);
    const int64_t bc = tile >> 3;
    const int64_t c = bc % C;
    const int64_t b = bc / C;
    const int g = L >> 2, t = L & 3;
    LaneSite s;
    s.r0 = b * kBlockRows + i * 16 + g;
    s.r1 = s.r0 + 8;
    s.kbyte = c * (kChunkK / 2) + t * 8;
    return s;
}

__global__ void __launch_bounds__(kRepackThreads)
    repack_kernel(const uint8_t* __restrict__ q, int64_t N, int64_t K, uint4* __restrict__ out,
                  int64_t total) {
    const int64_t C = K / kChunkK;
    for (int64_t o = (int64_t)blockIdx.x * kRepackThreads + threadIdx.x; o < total;
         o += (int64_t)gridDim.x * kRepackThreads) {
        const LaneSite s = lane_site(o, C);
        uint2 a = make_uint2(0x88888888u, 0x88888888u);  // padding rows: q = 0
        uint2 b = a;
        if (s.r0 < N) a = __ldg(reinterpret_cast<const uint2*>(q + s.r0 * (K / 2) + s.kbyte));
        if (s.r1 < N) b = __ldg(reinterpret_cast<const uint2*>(q + s.r1 * (K / 2) + s.kbyte));
        uint4 w;
        w.x = interleave_word(a.x & 0xFFFFu, b.x & 0xFFFFu);
        w.y = interleave_word(a.x >> 16, b.x >> 16);
        w.z = interleave_word(a.y & 0xFFFFu, b.y & 0xFFFFu);
        w.w = interleave_word(a.y >> 16, b.y >> 16);
        out[o] = w;
    }
    // Publish before the block ends: the GEMM that reads these weights may
    // start before the grid-completion flush (see w4a16_gemm).
    __threadfence();
}

__global__ void __launch_bounds__(kRepackThreads)
    unrepack_kernel(const uint4* __restrict__ in, int64_t N, int64_t K, uint8_t* __restrict__ q,
                    int64_t total) {
    const int64_t C = K / kChunkK;
    for (int64_t o = (int64_t)blockIdx.x * kRepackThreads + threadIdx.x; o < total;
         o += (int64_t)gridDim.x * kRepackThreads) {
        const LaneSite s = lane_site(o, C);
        const uint4 w = __ldg(in + o);
        uint32_t u[4], v[4];
        split_word(w.x, u[0], v[0]);
        split_word(w.y, u[1], v[1]);
        split_word(w.z, u[2], v[2]);
        split_word(w.w, u[3], v[3]);
        if (s.r0 < N)
            *reinterpret_cast<uint2*>(q + s.r0 * (K / 2) + s.kbyte) =
                make_uint2(u[0] | (u[1] << 16), u[2] | (u[3] << 16));
        if (s.r1 < N)
            *reinterpret_cast<uint2*>(q + s.r1 * (K / 2) + s.kbyte) =
                make_uint2(v[0] | (v[1] << 16), v[2] | (v[3] << 16));
    }
}

int64_t lane_chunks(int64_t N, int64_t K) {
    const int64_t blocks = (N + kBlockRows - 1) / kBlockRows;
    return blocks * (K / kChunkK) * 8 * 32;
}

unsigned grid_for(int64_t total, const DeviceCtx& ctx) {
    int64_t blocks = (total + kRepackThreads - 1) / kRepackThreads;
    const int64_t cap = (int64_t)ctx.num_sms * 32;
    if (blocks > cap) blocks = cap;
    return (unsigned)(blocks < 1 ? 1 : blocks);
}

}  // namespace

cudaError_t launch_repack(const void* qweight, int64_t N, int64_t K, void* repacked,
                          cudaStream_t stream, const DeviceCtx& ctx) {
    const int64_t total = lane_chunks(N, K);
    repack_kernel<<<grid_for(total, ctx), kRepackThreads, 0, stream>>>(
        static_cast<const uint8_t*>(qweight), N, K, static_cast<uint4*>(repacked), total);
    return cudaGetLastError();
}

cudaError_t launch_unrepack(const void* repacked, int64_t N, int64_t K, void* qweight,
                            cudaStream_t stream, const DeviceCtx& ctx) {
    const int64_t total = lane_chunks(N, K);
    unrepack_kernel<<<grid_for(total, ctx), kRepackThreads, 0, stream>>>(
        static_cast<const uint4*>(repacked), N, K, static_cast<uint8_t*>(qweight), total);
    return cudaGetLastError();
}

}  // namespace w4a16
