// gemm_tc.cu -- W4A16 prefill GEMM (M > 16) on the tcgen05 tensor cores.
//
// y[m, n] = sum_k x[m, k] * Wd[n, k],  Wd[n, k] = fp16((nib - 8) * scale[n, k/128])
// (qaqbuyan.com tutorial "量化的数学基石" §3 per_group_symmetric_dequantize:
// the fp16 dequantized weight is the fp32 product q * s rounded once to fp16;
// mhpq.cn W4A16 report §二 prefill column: the same packed format serves the
// prompt pass).  Unlike decode, the prompt pass is a dense contraction, so it
// runs on the tensor cores:
//
// One thread block computes a 128 (activation rows = MMA M) x 128 (weight
// rows = MMA N) tile of y with FP32 accumulators in tensor memory.
//  * warp 0 (one thread): TMA producer.  Per 64-wide k-block it loads the x
//    tile [128 x 64] fp16 (operand A) with a 2-D tensor-map copy in the
//    128-byte swizzled K-major layout and the block's 4 KB of packed weights
//    with a bulk copy, both completing on one mbarrier; the 128-row scale
//    slab arrives once.
//  * warps 4-19, two sets of 8 taking alternate k-blocks (one 16-byte lane
//    chunk of packed weights per thread): dequantise in registers (lop3
//    magic-number expansion, exact q), multiply by the fp16 group scale (one
//    RNE rounding, as the tutorial's dequantizer) and store the fp16 weight
//    tile [128 x 64] (operand B) in the same 128-byte swizzled K-major
//    layout; then fence the generic->async proxy and arrive.
//  * warp 1 (one thread): issues 4 tcgen05.mma (M=128, N=128, K=16) per
//    k-block from the shared-memory matrix descriptors and commits to the
//    stage's mbarrier, which frees the stage for the producer and the
//    dequantisers.  A last commit releases the epilogue.
//  * epilogue, warps 4-19: warp w reads TMEM lanes 32 (w % 4) .. +31 (rows
//    of y) and 32 accumulator columns (weight rows) with tcgen05.ld, rounds
//    to fp16 and writes 64 contiguous bytes of a y row per thread.
// Every wait is bounded; tensor memory is freed on every path.
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "tcgen05.cuh"

namespace w4a16 {
namespace {

constexpr int kTcThreads = 640;                 // 20 warps
constexpr int kDequantWarps = 16;               // warps 4 .. 19, two sets of 8
constexpr int kTileW = kBlockRows;              // weight rows per tile (MMA N)
constexpr int kTileX = 128;                     // activation rows per tile (MMA M)
constexpr int kBK = kChunkK;                    // 64: one kernel-layout chunk
constexpr int kStages = 4;                      // ring: x tile, packed and dequantised weights
constexpr int kAStageBytes = kTileW * kBK * 2;  // 16 KB fp16, 128B-swizzled
constexpr int kXStageBytes = kTileX * kBK * 2;  // 16 KB
constexpr int kWStageBytes = kTileW * kBK / 2;  // 4 KB packed
constexpr uint32_t kTmemCols = kTileW;          // fp32 accumulator columns

constexpr int kBarLoadFull = 0;                      // [stages] x + packed weights landed
constexpr int kBarAFull = kBarLoadFull + 8 * kStages;  // [stages] dequantised tile written
constexpr int kBarFree = kBarAFull + 8 * kStages;      // [stages] MMAs done: stage reusable
constexpr int kBarAcc = kBarFree + 8 * kStages;
constexpr int kBarSlab = kBarAcc + 8;
constexpr int kTmemSlot = kBarSlab + 8;
constexpr int kAbortFlag = kTmemSlot + 8;
constexpr int kOffA = 1024;                              // dequantised tiles
constexpr int kOffX = kOffA + kStages * kAStageBytes;    // x tiles
constexpr int kOffW = kOffX + kStages * kXStageBytes;    // packed weights
constexpr int kOffSlab = kOffW + kStages * kWStageBytes; // scale slab

struct TcArgs {
    const uint8_t* wq;
    const __half* scales;
    __half* y;
    unsigned* status;
    uint64_t timeout_ns;
    int M, N, K, G;
};

__device__ __forceinline__ void sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                       uint32_t d) {
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}

__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, __half2 s) {
    __half2 v = __hmul2(*reinterpret_cast<const __half2*>(&a), s);
    return *reinterpret_cast<uint32_t*>(&v);
}

// Byte offset of the 16-byte chunk `c` of row `r` in a 128-byte swizzled,
// K-major tile whose rows are 128 bytes (64 fp16) long.
__device__ __forceinline__ uint32_t swz128(int r, int c) {
    return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4));
}

__global__ void __launch_bounds__(kTcThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ TcArgs a) {
    extern __shared__ uint8_t smem_raw[];
    // Swizzled tiles need 1024-byte alignment: align the window by hand.
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* smem = smem_raw + (base - raw);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kAbortFlag);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int rb = (int)blockIdx.x;             // 128-row weight block
    const int m0 = (int)blockIdx.y * kTileX;    // first activation row
    const int nkb = a.K / kBK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(base + kBarLoadFull + 8 * s, 1);
            mbar_init(base + kBarAFull + 8 * s, kDequantWarps / 2 * 32);
            mbar_init(base + kBarFree + 8 * s, 1);
        }
        mbar_init(base + kBarAcc, 1);
        mbar_init(base + kBarSlab, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(base + kTmemSlot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + kTmemSlot);
    grid_launch_dependents();

    if (warp == 0) {
        // ============================ TMA producer ============================
        if (lane == 0) {
            tma_prefetch_map(&xmap);
            const uint8_t* w = a.wq + (size_t)rb * nkb * kWStageBytes;
            for (int i = 0; i < kStages && i < nkb; ++i)
                bulk_prefetch_l2(w + (size_t)i * kWStageBytes, kWStageBytes);
            grid_dependency_wait();
            {   // the block's scale slab (rows x G fp16, contiguous)
                const int rows = min(kTileW, a.N - rb * kTileW);
                const uint32_t bytes = (uint32_t)(rows * a.G * 2);
                const uint32_t bulk = bytes & ~15u;
                const __half* src = a.scales + (size_t)rb * kTileW * a.G;
                __half* dst = reinterpret_cast<__half*>(smem + kOffSlab);
                for (uint32_t e = bulk / 2; e < bytes / 2; ++e) dst[e] = src[e];
                mbar_arrive_expect_tx(base + kBarSlab, bulk);
                if (bulk) bulk_g2s(base + kOffSlab, src, bulk, base + kBarSlab);
            }
            int issued = 0;
            bool ok = true;
            for (int i = 0, ts = 0, round = 0; i < nkb; ++i) {
                if (i >= kStages &&
                    !mbar_wait(base + kBarFree + 8 * ts, (round - 1) & 1, a.timeout_ns,
                               a.status)) {
                    ok = false;
                    break;
                }
                if (*abort_flag) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(base + kBarLoadFull + 8 * ts, kXStageBytes + kWStageBytes);
                tma_load_2d(base + kOffX + ts * kXStageBytes, &xmap, i * kBK, m0,
                            base + kBarLoadFull + 8 * ts);
                bulk_g2s(base + kOffW + ts * kWStageBytes, w + (size_t)i * kWStageBytes,
                         kWStageBytes, base + kBarLoadFull + 8 * ts);
                issued = i + 1;
                if (++ts == kStages) {
                    ts = 0;
                    ++round;
                }
            }
            if (!ok) *abort_flag = 1;
            // Drain the copies in flight before the block may exit.
            mbar_wait(base + kBarSlab, 0, a.timeout_ns, a.status);
            for (int i = (issued > kStages ? issued - kStages : 0); i < issued; ++i)
                mbar_wait(base + kBarLoadFull + 8 * (i % kStages), (i / kStages) & 1, a.timeout_ns,
                          a.status);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ============================= MMA issuer =============================
        if (lane == 0) {
            const uint32_t idesc = umma_idesc_f16_f32(kTileX, kTileW);
            bool ok = true;
            for (int i = 0, ts = 0, tr = 0; i < nkb; ++i) {
                // the dequantisers waited for the stage's copies: A full implies x landed
                if (!mbar_wait(base + kBarAFull + 8 * ts, tr & 1, a.timeout_ns, a.status)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t xa = base + kOffX + ts * kXStageBytes;
                const uint32_t wa = base + kOffA + ts * kAStageBytes;
#pragma unroll
                for (int j = 0; j < kBK / 16; ++j)  // A = x rows, B = weight rows
                    tc_mma_f16(tmem, umma_desc_sw128(xa + 32 * j), umma_desc_sw128(wa + 32 * j),
                               idesc, (i | j) != 0);
                tc_commit(base + kBarFree + 8 * ts);  // stage reusable once these MMAs finish
                if (++ts == kStages) {
                    ts = 0;
                    ++tr;
                }
            }
            tc_commit(base + kBarAcc);  // completes once every issued MMA has
            if (!ok) *abort_flag = 1;
        }
        __syncwarp();
    } else if (warp >= 4) {
        // ===================== dequantisers, then epilogue ====================
        grid_dependency_wait();
        const int dw = (warp - 4) & 7;    // tile (16 weight rows) of this warp
        const int set = (warp - 4) >> 3;  // k-blocks set, set + 2, ...
        const int g = lane >> 2, tq = lane & 3;
        const int r0 = dw * 16 + g, r1 = r0 + 8;
        const __half* slab = reinterpret_cast<const __half*>(smem + kOffSlab);
        bool ok = mbar_wait(base + kBarSlab, 0, a.timeout_ns, a.status);
        for (int i = set; ok && i < nkb; i += 2) {
            // The stage's copies were issued after its previous MMAs finished,
            // so their arrival also means the dequantised slot is free.
            const int ts = i % kStages;
            if (!mbar_wait(base + kBarLoadFull + 8 * ts, (i / kStages) & 1, a.timeout_ns,
                           a.status)) {
                ok = false;
                break;
            }
            const int grp = i >> 1;  // two 64-wide k-blocks per scale group
            const uint32_t wst = base + kOffW + ts * kWStageBytes;
            const uint32_t ast = base + kOffA + ts * kAStageBytes;
            const uint4 pk = lds128(wst + (dw * 32 + lane) * 16);
            const __half2 s0 = __half2half2(slab[r0 * a.G + grp]);
            const __half2 s1 = __half2half2(slab[r1 * a.G + grp]);
            const uint32_t wrd[4] = {pk.x, pk.y, pk.z, pk.w};
            uint32_t o0[8], o1[8];  // rows r0 / r1, k = 16 tq .. 16 tq + 15
#pragma unroll
            for (int ws = 0; ws < 4; ++ws) {
                uint32_t af[4];
                dequant8(wrd[ws], af);
                o0[2 * ws] = hmul2_u32(af[0], s0);
                o0[2 * ws + 1] = hmul2_u32(af[2], s0);
                o1[2 * ws] = hmul2_u32(af[1], s1);
                o1[2 * ws + 1] = hmul2_u32(af[3], s1);
            }
            sts128(ast + swz128(r0, 2 * tq), o0[0], o0[1], o0[2], o0[3]);
            sts128(ast + swz128(r0, 2 * tq + 1), o0[4], o0[5], o0[6], o0[7]);
            sts128(ast + swz128(r1, 2 * tq), o1[0], o1[1], o1[2], o1[3]);
            sts128(ast + swz128(r1, 2 * tq + 1), o1[4], o1[5], o1[6], o1[7]);
            fence_proxy_async_smem();  // generic stores -> visible to the tensor core
            mbar_arrive(base + kBarAFull + 8 * ts);
        }
        if (!ok) *abort_flag = 1;

        // ------------------------------ epilogue ------------------------------
        if (mbar_wait(base + kBarAcc, 0, a.timeout_ns, a.status)) {
            tc_fence_after_sync();
            const int q = warp & 3;           // TMEM lane quarter = rows of y
            const int cc = (warp - 4) >> 2;   // 32-column chunk = weight rows
            const int m = m0 + q * 32 + lane;
            const int n = rb * kTileW + cc * 32;
            uint32_t v[32];
            tmem_ld_32x32b_x32(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(cc * 32), v);
            tmem_ld_wait();
            if (m < a.M) {
                __half* yrow = a.y + (size_t)m * a.N;
                if (n + 32 <= a.N && (a.N & 7) == 0) {
                    uint32_t h[16];
#pragma unroll
                    for (int c = 0; c < 16; ++c) {
                        __half2 p = __floats2half2_rn(__uint_as_float(v[2 * c]),
                                                      __uint_as_float(v[2 * c + 1]));
                        h[c] = *reinterpret_cast<uint32_t*>(&p);
                    }
                    uint4* dst = reinterpret_cast<uint4*>(yrow + n);
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        dst[c] = make_uint4(h[4 * c], h[4 * c + 1], h[4 * c + 2], h[4 * c + 3]);
                } else {
#pragma unroll
                    for (int c = 0; c < 32; ++c)
                        if (n + c < a.N) yrow[n + c] = __float2half_rn(__uint_as_float(v[c]));
                }
            }
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, kTmemCols);
    }
}

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

}  // namespace

cudaError_t launch_gemm_tc(const void* x, const void* repacked, const void* scales, void* y,
                           int64_t M, int64_t N, int64_t K, cudaStream_t stream,
                           const DeviceCtx& ctx) {
    const int G = (int)(K / kGroup);
    // +1 KB: slack for aligning the window to 1024 bytes
    const uint32_t smem = kOffSlab + ((kTileW * G * 2 + 127) / 128) * 128 + 1024;
    if ((int)smem > ctx.max_smem_optin) return cudaErrorInvalidValue;
    PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
    if (!encode) return cudaErrorNotSupported;
    CUtensorMap map;
    const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)M};
    const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    const cuuint32_t box[2] = {(cuuint32_t)kBK, (cuuint32_t)kTileX};
    const cuuint32_t estr[2] = {1, 1};
    if (encode(&map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(x), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;

    static bool attr_done[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !attr_done[dev]) {
        cudaError_t e = cudaFuncSetAttribute(gemm_tc_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             ctx.max_smem_optin);
        if (e != cudaSuccess) return e;
        attr_done[dev] = true;
    }
    TcArgs args{};
    args.wq = static_cast<const uint8_t*>(repacked);
    args.scales = static_cast<const __half*>(scales);
    args.y = static_cast<__half*>(y);
    args.status = ctx.status;
    args.timeout_ns = ctx.timeout_ns;
    args.M = (int)M;
    args.N = (int)N;
    args.K = (int)K;
    args.G = G;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((N + kTileW - 1) / kTileW), (unsigned)((M + kTileX - 1) / kTileX), 1);
    cfg.blockDim = dim3(kTcThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, gemm_tc_kernel, map, args);
}

}  // namespace w4a16
