// gemv_w8.cu -- W8A16 decode GEMV (M = 1..16): per-channel symmetric INT8
// weights, fp16 activations,
//   y[m, n] = scale[n] * sum_k x[m, k] * (code[n, k] - 128)
// (qaqbuyan.com tutorial "量化的数学基石": §2 formula with b = 8 and its INT8
// section, per-channel symmetric; the decode product as in the mhpq.cn report
// §二/§五).
//
// The codes are read in their canonical row-major [N, K] byte layout, with
// no repack: a 2-D tensor map over [N rows][K bytes] copies boxes of 128 k x
// the unit's 16 T rows into 16 KB ring stages with the 128-byte swizzle (the
// 16-byte pieces of row r permuted by r mod 8), so that the 8-byte reads of
// a warp's 8 row-pairs land in distinct banks; rows past N are zero-filled by
// the copy.  One CTA per unit of T 16-row tiles over the whole K range, 8
// consumer warps + 1 producer warp; warp (tile, ks) takes box ks of every
// stage.  A lane holds, per 32-wide k chunk, 8 consecutive bytes of rows
// g and g + 8: prmt with the fp16 exponent byte 0x64 and one subtraction of
// 1152 give the codes exactly as fp16, two mma.m16n8k16 (the k order inside
// the chunk permuted identically for the activations) accumulate the exact
// products in FP32, and the per-row scale multiplies the sum once at the end.
// Programmatic dependent launch as in gemv.cu.  Every wait is bounded.
#include <atomic>
#include <mutex>
#include <utility>
#include <vector>

#include "common.cuh"
#include "kernels.h"

namespace w4a16 {
namespace {

constexpr int kWWarps = 8;
constexpr int kWConsumers = kWWarps * 32;
constexpr int kWThreads = kWConsumers + 32;
constexpr int kWBoxK = 128;                 // k bytes per box row (one 128-byte swizzle line)
constexpr int kWStageBytes = 16384;
constexpr int kWMaxStages = 6;

constexpr int kWBarFull = 0;                              // [kWMaxStages]
constexpr int kWBarEmpty = kWBarFull + 8 * kWMaxStages;   // [kWMaxStages]
constexpr int kWBarX = kWBarEmpty + 8 * kWMaxStages;
constexpr int kWAbort = kWBarX + 8;
constexpr int kWBarArea = 1024;

struct W8Args {
    const __half* scales;  // [N]
    const __half* x;       // [M, K]
    __half* y;             // [M, N]
    unsigned* status;
    uint64_t timeout_ns;
    int M, N, K;
    int T;                 // 16-row tiles per CTA (1, 2, 4 or 8)
    int nstages;
    int xs_stride;
    uint32_t off_ring, off_x, off_red;
};

// Two int8 codes (bytes sel) of w as an fp16 pair q = code - 128, exact.
__device__ __forceinline__ uint32_t codes_to_half2(uint32_t w, uint32_t sel) {
    uint32_t r;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(w), "r"(0x64646464u), "r"(sel));
    const __half2 k1152 = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));
    __half2 v = __hsub2(*reinterpret_cast<const __half2*>(&r), k1152);  // (1024 + c) - 1152
    return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ uint2 lds64(uint32_t addr) {
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
    return v;
}

template <int MT>
__global__ void __launch_bounds__(kWThreads, MT == 1 ? 3 : 2)
    gemv_w8_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ W8Args a) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int T = a.T;
    const int W = kWWarps / T;                     // warps per tile = boxes per stage
    const int box_bytes = kWBoxK * 16 * T;
    const int kps = kWBoxK * W;                    // k per stage
    const int nstg = (a.K + kps - 1) / kps;
    const int r0 = (int)blockIdx.y * 16 * T;       // first weight row of the unit
    const int NS = a.nstages;
    const uint32_t sbase = smem_u32(smem);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kWAbort);
    const uint32_t ring = sbase + a.off_ring;

    grid_launch_dependents();

    if (warp == kWWarps) {
        // =============================== producer ===============================
        // The producer initialises the barriers and goes straight on to its
        // first copies; the consumers wait for that on named barrier 2.
        if (lane == 0) {
            for (int s = 0; s < NS; ++s) {
                mbar_init(sbase + kWBarFull + 8 * s, 1);
                mbar_init(sbase + kWBarEmpty + 8 * s, kWWarps);
            }
            mbar_init(sbase + kWBarX, 1);
            *abort_flag = 0;
            fence_barrier_init();
        }
        __syncwarp();
        asm volatile("bar.arrive 2, %0;" ::"n"(kWThreads) : "memory");
        if (lane == 0) {
            const uint64_t pol = l2_policy_evict_first();
            tma_prefetch_map(&qmap);
            bool x_issued = false;
            auto issue_x = [&]() {
                grid_dependency_wait();
                const uint32_t xbytes = (uint32_t)a.K * 2;
                mbar_arrive_expect_tx(sbase + kWBarX, xbytes * a.M);
                for (int m = 0; m < a.M; ++m)
                    bulk_g2s(sbase + a.off_x + m * a.xs_stride, a.x + (size_t)m * a.K, xbytes,
                             sbase + kWBarX);
                x_issued = true;
            };
            int it = 0, slot = 0, round = 0;
            bool ok = true;
            for (; it < nstg; ++it) {
                if (it >= NS && !x_issued) issue_x();
                if (it >= NS && !mbar_wait(sbase + kWBarEmpty + 8 * slot, (round - 1) & 1,
                                           a.timeout_ns, a.status)) {
                    ok = false;
                    break;
                }
                if (*abort_flag) {
                    ok = false;
                    break;
                }
                const int k0 = it * kps;
                const int nbox = min(W, (a.K - k0) / kWBoxK);  // K % 128 == 0
                const uint32_t bar = sbase + kWBarFull + 8 * slot;
                mbar_arrive_expect_tx(bar, nbox * box_bytes);
                for (int b = 0; b < nbox; ++b)
                    tma_load_2d_hint(ring + slot * kWStageBytes + b * box_bytes, &qmap,
                                     k0 + b * kWBoxK, r0, bar, pol);
                if (++slot == NS) {
                    slot = 0;
                    ++round;
                }
            }
            if (!x_issued) issue_x();
            if (!ok) *abort_flag = 1;
            const uint64_t dt = drain_bound(a.timeout_ns);
            mbar_wait(sbase + kWBarX, 0, dt, a.status);
            for (int i = (it > NS ? it - NS : 0); i < it; ++i)
                mbar_wait(sbase + kWBarFull + 8 * (i % NS), (i / NS) & 1, dt, a.status);
        }
        __syncwarp();
        return;
    }

    // ================================ consumers =================================
    asm volatile("bar.sync 2, %0;" ::"n"(kWThreads) : "memory");  // barriers initialised
    grid_dependency_wait();
    const int g = lane >> 2, t = lane & 3;
    const int ti = warp / W, ks = warp - ti * W;
    const int row0 = ti * 16 + g;                    // rows of this lane among the unit's rows
    const int xr0 = g < a.M ? g : a.M - 1;
    const int xr1 = g + 8 < a.M ? g + 8 : a.M - 1;
    const uint32_t x0 = sbase + a.off_x + xr0 * a.xs_stride + t * 16;
    const uint32_t x1 = sbase + a.off_x + xr1 * a.xs_stride + t * 16;
    bool ok = mbar_wait(sbase + kWBarX, 0, a.timeout_ns, a.status);
    ok = __all_sync(0xffffffffu, ok);
    float acc[2][MT][4];
#pragma unroll
    for (int c = 0; c < 2; ++c)
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[c][mt][e] = 0.0f;
    int slot = 0;
    uint32_t phase = 0;
    for (int st = 0; st < nstg; ++st) {
        if (ok) ok = mbar_wait(sbase + kWBarFull + 8 * slot, phase, a.timeout_ns, a.status);
        ok = __all_sync(0xffffffffu, ok);
        const int kb = st * kps + ks * kWBoxK;       // this warp's box
        if (ok && kb < a.K) {
            const uint32_t box = ring + slot * kWStageBytes + ks * box_bytes;
            const uint32_t rA = box + (uint32_t)row0 * kWBoxK;          // row r0 line
            const uint32_t rB = rA + 8 * kWBoxK;                         // row r0 + 8
#pragma unroll
            for (int c = 0; c < 4; ++c) {                 // 32-wide k chunks of the box
                const int piece = 2 * c + (t >> 1);       // 16-byte piece of k = 32 c + 8 t
                const uint32_t off = (uint32_t)(((piece ^ g) << 4) + 8 * (t & 1));  // r mod 8 == g
                const uint2 wa = lds64(rA + off);
                const uint2 wb = lds64(rB + off);
                const uint4 xa = lds128(x0 + (uint32_t)(kb + 32 * c) * 2);
                uint4 xb = xa;
                if (MT == 2) xb = lds128(x1 + (uint32_t)(kb + 32 * c) * 2);
                // MMA 0: k = 8t .. 8t + 3 (bytes 0-3); MMA 1: 8t + 4 .. 8t + 7
                uint32_t af[4];
                af[0] = codes_to_half2(wa.x, 0x4140);
                af[1] = codes_to_half2(wb.x, 0x4140);
                af[2] = codes_to_half2(wa.x, 0x4342);
                af[3] = codes_to_half2(wb.x, 0x4342);
                mma_16816(acc[0][0], af, xa.x, xa.y, acc[0][0]);
                if (MT == 2) mma_16816(acc[0][MT - 1], af, xb.x, xb.y, acc[0][MT - 1]);
                af[0] = codes_to_half2(wa.y, 0x4140);
                af[1] = codes_to_half2(wb.y, 0x4140);
                af[2] = codes_to_half2(wa.y, 0x4342);
                af[3] = codes_to_half2(wb.y, 0x4342);
                mma_16816(acc[1][0], af, xa.z, xa.w, acc[1][0]);
                if (MT == 2) mma_16816(acc[1][MT - 1], af, xb.z, xb.w, acc[1][MT - 1]);
            }
        }
        __syncwarp();
        if (ok && lane == 0) mbar_arrive(sbase + kWBarEmpty + 8 * slot);
        if (++slot == NS) {
            slot = 0;
            phase ^= 1u;
        }
    }
    float sum[MT][4];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int e = 0; e < 4; ++e) sum[mt][e] = acc[0][mt][e] + acc[1][mt][e];
    // the tile's W warps: the first adds the others' sums in warp order
    float4* red = reinterpret_cast<float4*>(smem + a.off_red);
    if (ks > 0) {
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
            red[(warp * MT + mt) * 32 + lane] = make_float4(sum[mt][0], sum[mt][1], sum[mt][2], sum[mt][3]);
    }
    asm volatile("bar.sync 1, %0;" ::"n"(kWConsumers) : "memory");
    if (ks == 0 && ok) {
        for (int w2 = 1; w2 < W; ++w2) {
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
                const float4 v = red[((warp + w2) * MT + mt) * 32 + lane];
                sum[mt][0] += v.x;
                sum[mt][1] += v.y;
                sum[mt][2] += v.z;
                sum[mt][3] += v.w;
            }
        }
        const int R0 = r0 + row0, R1 = R0 + 8;
        const float s0 = R0 < a.N ? __half2float(a.scales[R0]) : 0.0f;
        const float s1 = R1 < a.N ? __half2float(a.scales[R1]) : 0.0f;
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
            const int m0 = mt * 8 + 2 * t, m1 = m0 + 1;
            if (m0 < a.M) {
                if (R0 < a.N) a.y[(size_t)m0 * a.N + R0] = __float2half_rn(s0 * sum[mt][0]);
                if (R1 < a.N) a.y[(size_t)m0 * a.N + R1] = __float2half_rn(s1 * sum[mt][2]);
            }
            if (m1 < a.M) {
                if (R0 < a.N) a.y[(size_t)m1 * a.N + R0] = __float2half_rn(s0 * sum[mt][1]);
                if (R1 < a.N) a.y[(size_t)m1 * a.N + R1] = __float2half_rn(s1 * sum[mt][3]);
            }
        }
    }
    if (!ok) *abort_flag = 1;
}

struct W8Plan {
    int T = 0, nstages = 0, xs_stride = 0;
    uint32_t off_ring = 0, off_x = 0, off_red = 0, smem = 0;
};

template <int MT>
int w8_occupancy(uint32_t smem) {
    int blocks = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, gemv_w8_kernel<MT>, kWThreads,
                                                      smem) != cudaSuccess)
        return 0;
    return blocks;
}

template <int MT>
cudaError_t ensure_w8_attr() {
    static std::atomic<bool> done[64];  // per device; racing callers only repeat the set-up
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && done[dev].load(std::memory_order_acquire)) return cudaSuccess;
    const cudaError_t e = cudaFuncSetAttribute(
        gemv_w8_kernel<MT>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    if (e == cudaSuccess && dev >= 0 && dev < 64) done[dev].store(true, std::memory_order_release);
    return e;
}

template <int MT>
bool w8_layout(W8Plan& p, int M, int K, int T, int nst, const DeviceCtx& ctx) {
    p.T = T;
    const int kps = kWBoxK * (kWWarps / T);
    const int fill = (K + kps - 1) / kps;
    p.nstages = fill < nst ? fill : nst;
    p.xs_stride = K * 2 + 16;
    p.off_ring = kWBarArea;
    p.off_x = p.off_ring + p.nstages * kWStageBytes;
    p.off_red = p.off_x + ((M * p.xs_stride + 127) / 128) * 128;
    p.smem = p.off_red + kWWarps * MT * 32 * 16;
    return (int)p.smem <= ctx.max_smem_optin;
}

// The unit size: the fewest waves of CTAs, then the most CTAs per wave, with
// the deepest ring (up to 6 stages) that keeps the CTAs per SM it needs.
template <int MT>
W8Plan plan_w8(int M, int N, int K, const DeviceCtx& ctx) {
    W8Plan best;
    long long best_waves = 0, best_units = 0;
    for (int T = 1; T <= 8; T *= 2) {
        W8Plan p;
        if (!w8_layout<MT>(p, M, K, T, 3, ctx)) continue;
        const int occ = w8_occupancy<MT>(p.smem);
        const long long units = ((long long)N + 16 * T - 1) / (16 * T);
        if (occ == 0 || units > 65535) continue;
        const long long slots = (long long)ctx.num_sms * occ;
        const long long waves = (units + slots - 1) / slots;
        const int need = (int)(((units < slots ? units : slots) + ctx.num_sms - 1) / ctx.num_sms);
        for (int nst = kWMaxStages; nst > p.nstages; --nst) {
            W8Plan q;
            if (w8_layout<MT>(q, M, K, T, nst, ctx) && q.nstages == nst &&
                w8_occupancy<MT>(q.smem) >= need) {
                p = q;
                break;
            }
        }
        if (best.T == 0 || waves < best_waves || (waves == best_waves && units > best_units)) {
            best = p;
            best_waves = waves;
            best_units = units;
        }
    }
    return best;
}

// The codes' tensor map (encoded once per codes, shape and unit size).
cudaError_t codes_map(const uint8_t* q8, int N, int K, int T, CUtensorMap* out) {
    struct Entry {
        const uint8_t* q8;
        int N, K, T;
        CUtensorMap map;
    };
    static std::mutex mu;
    static std::vector<Entry> cache;
    {
        std::lock_guard<std::mutex> lock(mu);
        for (const Entry& e : cache)
            if (e.q8 == q8 && e.N == N && e.K == K && e.T == T) {
                *out = e.map;
                return cudaSuccess;
            }
    }
    PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
    if (!encode) return cudaErrorNotSupported;
    Entry e{q8, N, K, T, {}};
    const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)N};
    const cuuint64_t strides[1] = {(cuuint64_t)K};
    const cuuint32_t box[2] = {(cuuint32_t)kWBoxK, (cuuint32_t)(16 * T)};
    const cuuint32_t estr[2] = {1, 1};
    if (encode(&e.map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(q8), dims, strides,
               box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    *out = e.map;
    std::lock_guard<std::mutex> lock(mu);
    if (cache.size() >= 4096) cache.clear();
    cache.push_back(e);
    return cudaSuccess;
}

template <int MT>
cudaError_t launch_w8_mt(const uint8_t* q8, W8Args a, cudaStream_t stream, const DeviceCtx& ctx) {
    cudaError_t e = ensure_w8_attr<MT>();
    if (e != cudaSuccess) return e;
    struct Key {
        int dev, M, N, K;
    };
    static std::mutex mu;
    static std::vector<std::pair<Key, W8Plan>> cache;
    int dev = 0;
    cudaGetDevice(&dev);
    W8Plan p;
    {
        std::lock_guard<std::mutex> lock(mu);
        for (const auto& c : cache)
            if (c.first.dev == dev && c.first.M == a.M && c.first.N == a.N && c.first.K == a.K)
                p = c.second;
    }
    if (p.T == 0) {
        p = plan_w8<MT>(a.M, a.N, a.K, ctx);
        if (p.T == 0) return cudaErrorInvalidValue;
        std::lock_guard<std::mutex> lock(mu);
        if (cache.size() < 4096) cache.push_back({{dev, a.M, a.N, a.K}, p});
    }
    a.T = p.T;
    a.nstages = p.nstages;
    a.xs_stride = p.xs_stride;
    a.off_ring = p.off_ring;
    a.off_x = p.off_x;
    a.off_red = p.off_red;
    CUtensorMap qmap;
    e = codes_map(q8, a.N, a.K, p.T, &qmap);
    if (e != cudaSuccess) return e;
    const long long units = ((long long)a.N + 16 * p.T - 1) / (16 * p.T);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1, (unsigned)units, 1);
    cfg.blockDim = dim3(kWThreads, 1, 1);
    cfg.dynamicSmemBytes = p.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, gemv_w8_kernel<MT>, qmap, a);
}

}  // namespace

cudaError_t launch_gemv_w8(const void* x, const void* q8, const void* scales, void* y, int M,
                           int64_t N, int64_t K, cudaStream_t stream, const DeviceCtx& ctx) {
    W8Args a{};
    a.scales = static_cast<const __half*>(scales);
    a.x = static_cast<const __half*>(x);
    a.y = static_cast<__half*>(y);
    a.status = ctx.status;
    a.timeout_ns = ctx.timeout_ns;
    a.M = M;
    a.N = (int)N;
    a.K = (int)K;
    if (M <= 8) return launch_w8_mt<1>(static_cast<const uint8_t*>(q8), a, stream, ctx);
    return launch_w8_mt<2>(static_cast<const uint8_t*>(q8), a, stream, ctx);
}

}  // namespace w4a16
