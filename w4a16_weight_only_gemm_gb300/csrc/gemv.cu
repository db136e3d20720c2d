// gemv.cu -- W4A16 decode GEMV/skinny GEMM for M = 1..16.
//
// y[m, n] = sum_k x[m, k] * (nib[n, k] - 8) * scale[n, k / 128]
// (mhpq.cn W4A16 report §二/§五: the packed weights stay packed in memory and
// are unpacked in registers; the qaqbuyan.com tutorial §3 dequantizer fixes
// the arithmetic).
//
// Design (one thread block = one 128-row block of W times a K range):
//  * a producer warp streams the block's weights -- 4 KB per 64-wide chunk,
//    contiguous in the kernel layout -- into a ring of shared-memory stages
//    with bulk async copies (TMA engine) completing on mbarriers, L2 policy
//    evict-first; the x slice of the K range arrives the same way;
//  * 8 consumer warps own 16 rows each.  Per 64-wide chunk a lane reads 16
//    bytes of its tile, expands each 32-bit word into an mma.m16n8k16 A
//    fragment with lop3 + one f16x2 op per nibble pair (exact q), and
//    multiplies it with x fragments read from shared memory.  M <= 8 uses
//    one n8 MMA per 16 k, M <= 16 two.  Each 128-wide group accumulates in a
//    fresh FP32 fragment that is scaled once by its fp16 scale and added to
//    the FP32 running sum -- products q * x are exact, only FP32 sums round;
//  * narrow N: the K range is split over the CTAs of a thread-block cluster
//    (up to 8), whose FP32 partials are reduced through distributed shared
//    memory in a fixed order -- no global workspace and no atomics;
//  * programmatic dependent launch: the block prefetches its first stages
//    into L2 before waiting on the previous kernel of the stream, and
//    releases its dependents once its main loop is done.
// Every wait is bounded (see common.cuh); on a time-out the block records it
// in the status word, stops issuing copies, drains the ones in flight and
// exits.
#include "common.cuh"
#include "kernels.h"

namespace w4a16 {
namespace {

constexpr int kConsumerWarps = 8;                      // 8 x 16 rows = one block
constexpr int kGemvThreads = (kConsumerWarps + 1) * 32;
constexpr int kChunkBytes = kBlockRows * kChunkK / 2;  // 4096 B per block-chunk
constexpr int kStages = 4;
constexpr int kChunksPerStage = 4;                     // even: whole groups
constexpr int kStageBytes = kChunksPerStage * kChunkBytes;
constexpr int kMaxSplits = 8;

struct GemvArgs {
    const uint8_t* wq;       // kernel-layout weights
    const __half* scales;    // [N, G]
    const __half* x;         // [M, K]
    __half* y;               // [M, N]
    unsigned* status;
    uint64_t timeout_ns;
    int M, N, K, G;
    int xs_stride;           // bytes between x rows in shared memory
    int ng_max;              // groups per split, rounded up
    uint32_t off_ring, off_x, off_s, off_red;
};

__device__ __forceinline__ int split_group_begin(int split, int S, int G) {
    return (int)(((long long)split * G) / S);
}

template <int MT>
__global__ void __launch_bounds__(kGemvThreads, 2) gemv_kernel(const __grid_constant__ GemvArgs a) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int S = (int)gridDim.x;  // cluster spans the whole x dimension
    const int split = (int)blockIdx.x;
    const int rb = (int)blockIdx.y;
    const int C = a.K / kChunkK;
    const int g0 = split_group_begin(split, S, a.G);
    const int g1 = split_group_begin(split + 1, S, a.G);
    const int ng = g1 - g0;
    const int nck = 2 * ng;
    const int iters = (nck + kChunksPerStage - 1) / kChunksPerStage;

    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar_full = sbase;
    const uint32_t bar_empty = sbase + 8 * kStages;
    const uint32_t bar_x = sbase + 16 * kStages;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + 16 * kStages + 8);
    const uint32_t ring = sbase + a.off_ring;
    const uint32_t xs = sbase + a.off_x;
    __half* ss = reinterpret_cast<__half*>(smem + a.off_s);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, kConsumerWarps);
        }
        mbar_init(bar_x, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();

    const uint8_t* wsrc = a.wq + ((size_t)rb * C + 2 * (size_t)g0) * kChunkBytes;

    if (warp == kConsumerWarps) {
        // ------------------------------ producer ------------------------------
        if (lane == 0) {
            const int pre = iters < kStages ? iters : kStages;
            for (int i = 0; i < pre; ++i) {
                const int nc = min(kChunksPerStage, nck - i * kChunksPerStage);
                bulk_prefetch_l2(wsrc + (size_t)i * kStageBytes, nc * kChunkBytes);
            }
            grid_dependency_wait();
            const uint64_t pol = l2_policy_evict_first();
            const uint32_t xbytes = (uint32_t)nck * (kChunkK * 2);
            mbar_arrive_expect_tx(bar_x, xbytes * a.M);
            for (int m = 0; m < a.M; ++m)
                bulk_g2s(xs + m * a.xs_stride, a.x + (size_t)m * a.K + (size_t)g0 * kGroup, xbytes,
                         bar_x);
            int issued = 0;
            for (int i = 0; i < iters; ++i) {
                const int slot = i % kStages;
                if (i >= kStages) {
                    if (!mbar_wait(bar_empty + 8 * slot, ((i / kStages) - 1) & 1, a.timeout_ns,
                                   a.status)) {
                        *abort_flag = 1;
                        break;
                    }
                }
                if (*abort_flag) break;
                const int nc = min(kChunksPerStage, nck - i * kChunksPerStage);
                mbar_arrive_expect_tx(bar_full + 8 * slot, nc * kChunkBytes);
                bulk_g2s_hint(ring + slot * kStageBytes, wsrc + (size_t)i * kStageBytes,
                              nc * kChunkBytes, bar_full + 8 * slot, pol);
                issued = i + 1;
            }
            // Drain: every issued copy must land before the block may exit.
            mbar_wait(bar_x, 0, a.timeout_ns, a.status);
            for (int i = (issued > kStages ? issued - kStages : 0); i < issued; ++i)
                mbar_wait(bar_full + 8 * (i % kStages), (i / kStages) & 1, a.timeout_ns, a.status);
        }
        __syncwarp();
    } else {
        // ------------------------------ consumers -----------------------------
        grid_dependency_wait();
        // Scales of this block's 128 rows and groups [g0, g1) -> smem [row][ng_max].
        {
            const int rows_here = min(kBlockRows, a.N - rb * kBlockRows);
            for (int idx = threadIdx.x; idx < kBlockRows * ng; idx += kConsumerWarps * 32) {
                const int r = idx / ng, gg = idx - r * ng;
                __half v = __ushort_as_half(0);
                if (r < rows_here) v = a.scales[(size_t)(rb * kBlockRows + r) * a.G + g0 + gg];
                ss[r * a.ng_max + gg] = v;
            }
            asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
        }

        const int g = lane >> 2, t = lane & 3;
        const int row0 = warp * 16 + g;  // local rows of this lane's fragments
        const int row1 = row0 + 8;
        const bool xl0 = g < a.M;
        const bool xl1 = (g + 8) < a.M;
        const uint32_t xa0 = xs + g * a.xs_stride + t * 32;
        const uint32_t xa1 = xs + (g + 8) * a.xs_stride + t * 32;
        const uint32_t wl = ring + warp * 512 + lane * 16;

        float acc[MT][4];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[mt][j] = 0.0f;

        bool ok = mbar_wait(bar_x, 0, a.timeout_ns, a.status);
        for (int i = 0; ok && i < iters; ++i) {
            const int slot = i % kStages;
            if (!mbar_wait(bar_full + 8 * slot, (i / kStages) & 1, a.timeout_ns, a.status)) {
                ok = false;
                break;
            }
            const int nc = min(kChunksPerStage, nck - i * kChunksPerStage);
#pragma unroll
            for (int j = 0; j < kChunksPerStage; j += 2) {
                if (j < nc) {
                    float gacc[MT][4];
#pragma unroll
                    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                        for (int e = 0; e < 4; ++e) gacc[mt][e] = 0.0f;
#pragma unroll
                    for (int jj = 0; jj < 2; ++jj) {
                        const int cl = i * kChunksPerStage + j + jj;  // local chunk
                        const uint4 wv = lds128(wl + slot * kStageBytes + (j + jj) * kChunkBytes);
                        uint4 xv0a = make_uint4(0, 0, 0, 0), xv0b = xv0a, xv1a = xv0a, xv1b = xv0a;
                        if (xl0) {
                            xv0a = lds128(xa0 + cl * 128);
                            xv0b = lds128(xa0 + cl * 128 + 16);
                        }
                        if (MT == 2 && xl1) {
                            xv1a = lds128(xa1 + cl * 128);
                            xv1b = lds128(xa1 + cl * 128 + 16);
                        }
                        const uint32_t wrd[4] = {wv.x, wv.y, wv.z, wv.w};
                        const uint32_t xb0[8] = {xv0a.x, xv0a.y, xv0a.z, xv0a.w,
                                                 xv0b.x, xv0b.y, xv0b.z, xv0b.w};
                        const uint32_t xb1[8] = {xv1a.x, xv1a.y, xv1a.z, xv1a.w,
                                                 xv1b.x, xv1b.y, xv1b.z, xv1b.w};
#pragma unroll
                        for (int s = 0; s < 4; ++s) {
                            uint32_t af[4];
                            dequant8(wrd[s], af);
                            mma_16816(gacc[0], af, xb0[2 * s], xb0[2 * s + 1], gacc[0]);
                            if (MT == 2)
                                mma_16816(gacc[MT - 1], af, xb1[2 * s], xb1[2 * s + 1],
                                          gacc[MT - 1]);
                        }
                    }
                    const int gl = (i * kChunksPerStage + j) >> 1;  // local group
                    const float s0 = __half2float(ss[row0 * a.ng_max + gl]);
                    const float s1 = __half2float(ss[row1 * a.ng_max + gl]);
#pragma unroll
                    for (int mt = 0; mt < MT; ++mt) {
                        acc[mt][0] = fmaf(s0, gacc[mt][0], acc[mt][0]);
                        acc[mt][1] = fmaf(s0, gacc[mt][1], acc[mt][1]);
                        acc[mt][2] = fmaf(s1, gacc[mt][2], acc[mt][2]);
                        acc[mt][3] = fmaf(s1, gacc[mt][3], acc[mt][3]);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_empty + 8 * slot);
        }
        if (!ok) *abort_flag = 1;

        grid_launch_dependents();

        const int R0 = rb * kBlockRows + row0;
        const int R1 = rb * kBlockRows + row1;
        if (S == 1) {
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
                const int m0 = mt * 8 + 2 * t, m1 = m0 + 1;
                if (m0 < a.M) {
                    if (R0 < a.N) a.y[(size_t)m0 * a.N + R0] = __float2half_rn(acc[mt][0]);
                    if (R1 < a.N) a.y[(size_t)m0 * a.N + R1] = __float2half_rn(acc[mt][2]);
                }
                if (m1 < a.M) {
                    if (R0 < a.N) a.y[(size_t)m1 * a.N + R0] = __float2half_rn(acc[mt][1]);
                    if (R1 < a.N) a.y[(size_t)m1 * a.N + R1] = __float2half_rn(acc[mt][3]);
                }
            }
        } else {
            float* red = reinterpret_cast<float*>(smem + a.off_red);  // [128][16]
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
                const int m0 = mt * 8 + 2 * t;
                red[row0 * 16 + m0] = acc[mt][0];
                red[row0 * 16 + m0 + 1] = acc[mt][1];
                red[row1 * 16 + m0] = acc[mt][2];
                red[row1 * 16 + m0 + 1] = acc[mt][3];
            }
        }
    }

    if (S > 1) {
        // Fixed-order reduction of the cluster's partials through DSMEM: CTA
        // `split` finalises rows split, split + S, ... of the block.
        cluster_sync_all();
        const uint32_t red_base = sbase + a.off_red;
        const int M = a.M;
        for (int idx = threadIdx.x; idx < kBlockRows * M; idx += kGemvThreads) {
            const int r = idx / M, m = idx - r * M;
            if (r % S != split) continue;
            const int R = rb * kBlockRows + r;
            if (R >= a.N) continue;
            float sum = 0.0f;
            for (int q = 0; q < S; ++q)
                sum += ld_cluster_f32(map_to_cta(red_base + (uint32_t)(r * 16 + m) * 4, q));
            a.y[(size_t)m * a.N + R] = __float2half_rn(sum);
        }
        cluster_sync_all();
    }
}

struct GemvPlan {
    int S;
    int xs_stride;
    int ng_max;
    uint32_t off_ring, off_x, off_s, off_red, smem;
};

GemvPlan plan_gemv(int M, int N, int K, const DeviceCtx& ctx) {
    const int G = K / kGroup;
    const int NB = (N + kBlockRows - 1) / kBlockRows;
    GemvPlan best{};
    best.S = 0;
    const int max_s = G < kMaxSplits ? G : kMaxSplits;
    for (int S = 1; S <= max_s; ++S) {
        GemvPlan p{};
        p.S = S;
        p.ng_max = (G + S - 1) / S;
        p.xs_stride = p.ng_max * kGroup * 2 + 16;  // +16 B: conflict-free x rows
        p.off_ring = 1024;
        p.off_x = p.off_ring + kStages * kStageBytes;
        p.off_s = p.off_x + ((M * p.xs_stride + 127) / 128) * 128;
        p.off_red = p.off_s + ((kBlockRows * p.ng_max * 2 + 127) / 128) * 128;
        p.smem = p.off_red + (S > 1 ? kBlockRows * 16 * 4 : 0);
        if ((int)p.smem > ctx.max_smem_optin) continue;
        if (best.S == 0) best = p;
        // Enough blocks to cover every SM at least once; stop at the first
        // split count that does, keeping clusters small.
        best = p;
        if ((long long)NB * S >= ctx.num_sms) break;
    }
    return best;
}

template <int MT>
cudaError_t launch_gemv_mt(const GemvArgs& args, const GemvPlan& p, int NB, cudaStream_t stream) {
    static bool attr_done[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 64 && !attr_done[dev]) {
        cudaError_t e = cudaFuncSetAttribute(gemv_kernel<MT>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             227 * 1024);
        if (e != cudaSuccess) return e;
        attr_done[dev] = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.S, (unsigned)NB, 1);
    cfg.blockDim = dim3(kGemvThreads, 1, 1);
    cfg.dynamicSmemBytes = p.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attrs[2];
    int na = 0;
    attrs[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
    if (p.S > 1) {
        attrs[na].id = cudaLaunchAttributeClusterDimension;
        attrs[na].val.clusterDim.x = (unsigned)p.S;
        attrs[na].val.clusterDim.y = 1;
        attrs[na].val.clusterDim.z = 1;
        ++na;
    }
    cfg.attrs = attrs;
    cfg.numAttrs = na;
    return cudaLaunchKernelEx(&cfg, gemv_kernel<MT>, args);
}

}  // namespace

cudaError_t launch_gemv(const void* x, const void* repacked, const void* scales, void* y, int M,
                        int64_t N, int64_t K, cudaStream_t stream, const DeviceCtx& ctx) {
    const GemvPlan p = plan_gemv(M, (int)N, (int)K, ctx);
    if (p.S == 0) return cudaErrorInvalidValue;
    GemvArgs a{};
    a.wq = static_cast<const uint8_t*>(repacked);
    a.scales = static_cast<const __half*>(scales);
    a.x = static_cast<const __half*>(x);
    a.y = static_cast<__half*>(y);
    a.status = ctx.status;
    a.timeout_ns = ctx.timeout_ns;
    a.M = M;
    a.N = (int)N;
    a.K = (int)K;
    a.G = (int)(K / kGroup);
    a.xs_stride = p.xs_stride;
    a.ng_max = p.ng_max;
    a.off_ring = p.off_ring;
    a.off_x = p.off_x;
    a.off_s = p.off_s;
    a.off_red = p.off_red;
    const int NB = (int)((N + kBlockRows - 1) / kBlockRows);
    if (M <= 8) return launch_gemv_mt<1>(a, p, NB, stream);
    return launch_gemv_mt<2>(a, p, NB, stream);
}

}  // namespace w4a16
