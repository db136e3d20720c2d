// gemv_q40.cu -- decode GEMV (M = 1..16) on GGUF Q4_0 blocks:
//   y[m, n] = sum_b d[n, b] * sum_{i < 32} x[m, 32 b + i] * (nib[n, 32 b + i] - 8)
// (qaqbuyan.com tutorial, GGUF section: a Q4_0 block holds 32 weights in 18
// bytes -- d as fp16, then 16 bytes whose byte i carries element 2i in its
// low nibble and 2i + 1 in its high nibble; blocks follow one another along
// a row and rows one another.  The decode product as in the mhpq.cn report
// §二/§五.)
//
// The structure is gemv_w8.cu's: one CTA per unit of T 16-row tiles over the
// whole K range, 8 consumer warps + 1 producer warp, a ring of stages filled
// through a 2-D tensor map over the rows' bytes, one box per consumer warp
// per stage, rows past N zero-filled by the copy, PDL.  A box is 8 blocks
// (144 bytes, 256 k) of 16 T rows, copied unswizzled: a 144-byte row pitch
// already puts the 8 row-pairs of a warp in distinct banks.  Rows are 16-byte
// aligned when K % 256 == 0, which the path requires.  Per block a lane
// holds bytes 4 t .. 4 t + 3 of the quants of rows g and g + 8 (elements
// 8 t .. 8 t + 7, read as two 16-bit halves: blocks are 2-byte aligned);
// four lop3 with the fp16 magic 1024 and four fp16 subtractions or fmas
// turn those 8 nibbles into exact q - 8 pairs of elements (e, e + 4); two
// mma.m16n8k16 take them against x stored in the same pairing (permuted in
// shared memory once per CTA) into a fresh FP32 fragment, scaled once by
// each row's block scale into the sum.  Every wait is bounded.
#include <atomic>
#include <mutex>
#include <utility>
#include <vector>

#include "common.cuh"
#include "kernels.h"

namespace w4a16 {
namespace {

constexpr int kQWarps = 8;
constexpr int kQConsumers = kQWarps * 32;
constexpr int kQThreads = kQConsumers + 32;
constexpr int kQBlockBytes = 18;             // 32 weights
constexpr int kQBoxBlocks = 8;               // blocks per box row: 144 bytes, 256 k
constexpr int kQBoxBytesRow = kQBoxBlocks * kQBlockBytes;
constexpr int kQBoxK = kQBoxBlocks * 32;
constexpr int kQStageBytes = kQBoxBytesRow * 16 * kQWarps;  // 8 boxes of 16 T rows / T
constexpr int kQMaxStages = 6;

constexpr int kQBarFull = 0;                              // [kQMaxStages]
constexpr int kQBarEmpty = kQBarFull + 8 * kQMaxStages;   // [kQMaxStages]
constexpr int kQBarX = kQBarEmpty + 8 * kQMaxStages;
constexpr int kQAbort = kQBarX + 8;
constexpr int kQBarArea = 1024;

struct Q40Args {
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

// A lane's 4 quant bytes of one row (elements e0 .. e7 of the block, byte b
// holding e_2b low and e_2b+1 high) as four exact fp16 pairs of q - 8:
// r = {(e0, e4), (e1, e5), (e2, e6), (e3, e7)}.  lop3 ORs the low nibbles of
// bytes 0 and 2 (of w >> 8: 1 and 3) into the mantissa of 1024.0, the high
// nibbles as 16 n; one subtraction of 1032, or a multiply by 1/16 and
// subtraction of 72, leaves n - 8 exactly.  The activations are stored with
// the same pairing, (x0, x4, x1, x5, x2, x6, x3, x7) per 8 elements.
__device__ __forceinline__ void dequant8_q40(uint32_t w, uint32_t (&r)[4]) {
    constexpr uint32_t kMagic = 0x64006400u;         // (1024.0, 1024.0)
    constexpr uint32_t kLut = (0xF0 & 0xCC) | 0xAA;  // (a & b) | c
    const uint32_t w8 = w >> 8;
    const uint32_t lo0 = lop3<kLut>(w, 0x000F000Fu, kMagic);
    const uint32_t hi0 = lop3<kLut>(w, 0x00F000F0u, kMagic);
    const uint32_t lo1 = lop3<kLut>(w8, 0x000F000Fu, kMagic);
    const uint32_t hi1 = lop3<kLut>(w8, 0x00F000F0u, kMagic);
    const __half2 k1032 = __half2half2(__ushort_as_half(0x6408));
    const __half2 k16th = __half2half2(__ushort_as_half(0x2C00));
    const __half2 km72 = __half2half2(__ushort_as_half(0xD480));
    __half2 v;
    v = __hsub2(*reinterpret_cast<const __half2*>(&lo0), k1032);
    r[0] = *reinterpret_cast<uint32_t*>(&v);
    v = __hfma2(*reinterpret_cast<const __half2*>(&hi0), k16th, km72);
    r[1] = *reinterpret_cast<uint32_t*>(&v);
    v = __hsub2(*reinterpret_cast<const __half2*>(&lo1), k1032);
    r[2] = *reinterpret_cast<uint32_t*>(&v);
    v = __hfma2(*reinterpret_cast<const __half2*>(&hi1), k16th, km72);
    r[3] = *reinterpret_cast<uint32_t*>(&v);
}

// M1: a single activation row, so only output column 0 is ever stored and
// the odd columns' rescale is skipped.
template <int MT, bool M1>
__global__ void __launch_bounds__(kQThreads, MT == 1 ? 3 : 2)
    gemv_q40_kernel(const __grid_constant__ CUtensorMap bmap, const __grid_constant__ Q40Args a) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int T = a.T;
    const int W = kQWarps / T;                     // warps per tile = boxes per stage
    const int box_bytes = kQBoxBytesRow * 16 * T;
    const int kps = kQBoxK * W;                    // k per stage
    const int nstg = (a.K + kps - 1) / kps;
    const int r0 = (int)blockIdx.y * 16 * T;
    const int NS = a.nstages;
    const uint32_t sbase = smem_u32(smem);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kQAbort);
    const uint32_t ring = sbase + a.off_ring;

    grid_launch_dependents();

    if (warp == kQWarps) {
        // =============================== producer ===============================
        // The producer initialises the barriers and goes straight on to its
        // first copies; the consumers wait for that on named barrier 2.
        if (lane == 0) {
            for (int s = 0; s < NS; ++s) {
                mbar_init(sbase + kQBarFull + 8 * s, 1);
                mbar_init(sbase + kQBarEmpty + 8 * s, kQWarps);
            }
            mbar_init(sbase + kQBarX, 1);
            *abort_flag = 0;
            fence_barrier_init();
        }
        __syncwarp();
        asm volatile("bar.arrive 2, %0;" ::"n"(kQThreads) : "memory");
        if (lane == 0) {
            const uint64_t pol = l2_policy_evict_first();
            tma_prefetch_map(&bmap);
            bool x_issued = false;
            auto issue_x = [&]() {
                grid_dependency_wait();
                const uint32_t xbytes = (uint32_t)a.K * 2;
                mbar_arrive_expect_tx(sbase + kQBarX, xbytes * a.M);
                for (int m = 0; m < a.M; ++m)
                    bulk_g2s(sbase + a.off_x + m * a.xs_stride, a.x + (size_t)m * a.K, xbytes,
                             sbase + kQBarX);
                x_issued = true;
            };
            int it = 0, slot = 0, round = 0;
            bool ok = true;
            for (; it < nstg; ++it) {
                if (it >= NS && !x_issued) issue_x();
                if (it >= NS && !mbar_wait(sbase + kQBarEmpty + 8 * slot, (round - 1) & 1,
                                           a.timeout_ns, a.status)) {
                    ok = false;
                    break;
                }
                if (*abort_flag) {
                    ok = false;
                    break;
                }
                const int k0 = it * kps;
                const int nbox = min(W, (a.K - k0) / kQBoxK);  // K % 256 == 0
                const uint32_t bar = sbase + kQBarFull + 8 * slot;
                mbar_arrive_expect_tx(bar, nbox * box_bytes);
                for (int b = 0; b < nbox; ++b)
                    tma_load_2d_hint(ring + slot * kQStageBytes + b * box_bytes, &bmap,
                                     (k0 + b * kQBoxK) / 32 * kQBlockBytes, r0, bar, pol);
                if (++slot == NS) {
                    slot = 0;
                    ++round;
                }
            }
            if (!x_issued) issue_x();
            if (!ok) *abort_flag = 1;
            const uint64_t dt = drain_bound(a.timeout_ns);
            mbar_wait(sbase + kQBarX, 0, dt, a.status);
            for (int i = (it > NS ? it - NS : 0); i < it; ++i)
                mbar_wait(sbase + kQBarFull + 8 * (i % NS), (i / NS) & 1, dt, a.status);
        }
        __syncwarp();
        return;
    }

    // ================================ consumers =================================
    asm volatile("bar.sync 2, %0;" ::"n"(kQThreads) : "memory");  // barriers initialised
    grid_dependency_wait();
    const int g = lane >> 2, t = lane & 3;
    const int ti = warp / W, ks = warp - ti * W;
    const int row0 = ti * 16 + g;
    const int xr0 = g < a.M ? g : a.M - 1;
    const int xr1 = g + 8 < a.M ? g + 8 : a.M - 1;
    const uint32_t x0 = sbase + a.off_x + xr0 * a.xs_stride + t * 16;
    const uint32_t x1 = sbase + a.off_x + xr1 * a.xs_stride + t * 16;
    bool ok = mbar_wait(sbase + kQBarX, 0, a.timeout_ns, a.status);
    // x in the decode's pairing: (x0, x4, x1, x5, x2, x6, x3, x7) per 8
    // elements, in place, 16 bytes per thread per step; every consumer thread
    // takes part in the barrier below
    {
        const int per_row = a.K / 8;
        for (int q = (int)threadIdx.x; ok && q < a.M * per_row; q += kQConsumers) {
            const int m = q / per_row, off = q - m * per_row;
            uint4* xp = reinterpret_cast<uint4*>(smem + a.off_x + m * a.xs_stride + off * 16);
            const uint4 v = *xp;
            uint4 o;
            asm("prmt.b32 %0, %1, %2, 0x5410;" : "=r"(o.x) : "r"(v.x), "r"(v.z));
            asm("prmt.b32 %0, %1, %2, 0x7632;" : "=r"(o.y) : "r"(v.x), "r"(v.z));
            asm("prmt.b32 %0, %1, %2, 0x5410;" : "=r"(o.z) : "r"(v.y), "r"(v.w));
            asm("prmt.b32 %0, %1, %2, 0x7632;" : "=r"(o.w) : "r"(v.y), "r"(v.w));
            *xp = o;
        }
        asm volatile("bar.sync 1, %0;" ::"n"(kQConsumers) : "memory");
    }
    ok = __all_sync(0xffffffffu, ok);
    float acc[MT][4];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[mt][e] = 0.0f;
    int slot = 0;
    uint32_t phase = 0;
    for (int st = 0; st < nstg; ++st) {
        if (ok) ok = mbar_wait(sbase + kQBarFull + 8 * slot, phase, a.timeout_ns, a.status);
        ok = __all_sync(0xffffffffu, ok);
        const int kb = st * kps + ks * kQBoxK;       // this warp's box
        if (ok && kb < a.K) {
            // rows r0 and r0 + 8 of this warp's box (144-byte rows, 16-byte aligned)
            const uint8_t* bA = smem + a.off_ring + slot * kQStageBytes + ks * box_bytes +
                                row0 * kQBoxBytesRow;
            const uint8_t* bB = bA + 8 * kQBoxBytesRow;
#pragma unroll
            for (int j = 0; j < kQBoxBlocks; ++j) {
                const int bo = j * kQBlockBytes;
                const float d0 = __half2float(*reinterpret_cast<const __half*>(bA + bo));
                const float d1 = __half2float(*reinterpret_cast<const __half*>(bB + bo));
                // the lane's quant bytes 2 + 4 t .. 5 + 4 t of the block: one
                // aligned word in odd blocks (18 j = 2 mod 4), two aligned
                // words joined in even ones
                uint32_t q0, q1;
                if (j & 1) {
                    q0 = *reinterpret_cast<const uint32_t*>(bA + bo + 2 + 4 * t);
                    q1 = *reinterpret_cast<const uint32_t*>(bB + bo + 2 + 4 * t);
                } else {
                    const uint32_t* wA = reinterpret_cast<const uint32_t*>(bA + bo + 4 * t);
                    const uint32_t* wB = reinterpret_cast<const uint32_t*>(bB + bo + 4 * t);
                    q0 = __funnelshift_r(wA[0], wA[1], 16);
                    q1 = __funnelshift_r(wB[0], wB[1], 16);
                }
                const uint4 xa = lds128(x0 + (uint32_t)(kb + 32 * j) * 2);
                uint4 xb = xa;
                if (MT == 2) xb = lds128(x1 + (uint32_t)(kb + 32 * j) * 2);
                float f[MT][4];
#pragma unroll
                for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) f[mt][e] = 0.0f;
                // MMA 0: elements (8t, 8t + 4), (8t + 1, 8t + 5) of rows g and
                // g + 8; MMA 1: (8t + 2, 8t + 6), (8t + 3, 8t + 7)
                uint32_t p0[4], p1[4];
                dequant8_q40(q0, p0);
                dequant8_q40(q1, p1);
                uint32_t af[4] = {p0[0], p1[0], p0[1], p1[1]};
                mma_16816(f[0], af, xa.x, xa.y, f[0]);
                if (MT == 2) mma_16816(f[MT - 1], af, xb.x, xb.y, f[MT - 1]);
                af[0] = p0[2];
                af[1] = p1[2];
                af[2] = p0[3];
                af[3] = p1[3];
                mma_16816(f[0], af, xa.z, xa.w, f[0]);
                if (MT == 2) mma_16816(f[MT - 1], af, xb.z, xb.w, f[MT - 1]);
#pragma unroll
                for (int mt = 0; mt < MT; ++mt) {
                    acc[mt][0] = fmaf(d0, f[mt][0], acc[mt][0]);
                    acc[mt][2] = fmaf(d1, f[mt][2], acc[mt][2]);
                    if (!M1) {
                        acc[mt][1] = fmaf(d0, f[mt][1], acc[mt][1]);
                        acc[mt][3] = fmaf(d1, f[mt][3], acc[mt][3]);
                    }
                }
            }
        }
        __syncwarp();
        if (ok && lane == 0) mbar_arrive(sbase + kQBarEmpty + 8 * slot);
        if (++slot == NS) {
            slot = 0;
            phase ^= 1u;
        }
    }
    // the tile's W warps: the first adds the others' sums in warp order
    float4* red = reinterpret_cast<float4*>(smem + a.off_red);
    if (ks > 0) {
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
            red[(warp * MT + mt) * 32 + lane] = make_float4(acc[mt][0], acc[mt][1], acc[mt][2], acc[mt][3]);
    }
    asm volatile("bar.sync 1, %0;" ::"n"(kQConsumers) : "memory");
    if (ks == 0 && ok) {
        for (int w2 = 1; w2 < W; ++w2) {
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
                const float4 v = red[((warp + w2) * MT + mt) * 32 + lane];
                acc[mt][0] += v.x;
                acc[mt][1] += v.y;
                acc[mt][2] += v.z;
                acc[mt][3] += v.w;
            }
        }
        const int R0 = r0 + row0, R1 = R0 + 8;
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
    }
    if (!ok) *abort_flag = 1;
}

struct Q40Plan {
    int T = 0, nstages = 0, xs_stride = 0;
    uint32_t off_ring = 0, off_x = 0, off_red = 0, smem = 0;
};

template <int MT>
int q40_occupancy(uint32_t smem) {
    // at MT = 1 both column variants; the larger register count decides
    int b0 = 0, b1 = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b0, gemv_q40_kernel<MT, false>, kQThreads,
                                                      smem) != cudaSuccess)
        return 0;
    if (MT == 1 && cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                       &b1, gemv_q40_kernel<1, true>, kQThreads, smem) == cudaSuccess)
        return b1 < b0 ? b1 : b0;
    return b0;
}

template <int MT>
cudaError_t ensure_q40_attr() {
    static std::atomic<bool> done[64];  // per device; racing callers only repeat the set-up
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && done[dev].load(std::memory_order_acquire)) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(
        gemv_q40_kernel<MT, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    if (e == cudaSuccess && MT == 1)
        e = cudaFuncSetAttribute(gemv_q40_kernel<1, true>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    if (e == cudaSuccess && dev >= 0 && dev < 64) done[dev].store(true, std::memory_order_release);
    return e;
}

template <int MT>
bool q40_layout(Q40Plan& p, int M, int K, int T, int nst, const DeviceCtx& ctx) {
    p.T = T;
    const int kps = kQBoxK * (kQWarps / T);
    const int fill = (K + kps - 1) / kps;
    p.nstages = fill < nst ? fill : nst;
    p.xs_stride = K * 2 + 16;
    p.off_ring = kQBarArea;
    p.off_x = p.off_ring + p.nstages * kQStageBytes;
    p.off_red = p.off_x + ((M * p.xs_stride + 127) / 128) * 128;
    p.smem = p.off_red + kQWarps * MT * 32 * 16;
    return (int)p.smem <= ctx.max_smem_optin;
}

// The unit size: the fewest waves of CTAs, then the most CTAs per wave, with
// the deepest ring (up to 6 stages) that keeps the CTAs per SM it needs.
template <int MT>
Q40Plan plan_q40(int M, int N, int K, const DeviceCtx& ctx) {
    Q40Plan best;
    long long best_waves = 0, best_units = 0;
    for (int T = 1; T <= 8; T *= 2) {
        Q40Plan p;
        if (!q40_layout<MT>(p, M, K, T, 3, ctx)) continue;
        const int occ = q40_occupancy<MT>(p.smem);
        const long long units = ((long long)N + 16 * T - 1) / (16 * T);
        if (occ == 0 || units > 65535) continue;
        const long long slots = (long long)ctx.num_sms * occ;
        const long long waves = (units + slots - 1) / slots;
        const int need = (int)(((units < slots ? units : slots) + ctx.num_sms - 1) / ctx.num_sms);
        for (int nst = kQMaxStages; nst > p.nstages; --nst) {
            Q40Plan q;
            if (q40_layout<MT>(q, M, K, T, nst, ctx) && q.nstages == nst &&
                q40_occupancy<MT>(q.smem) >= need) {
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

// The blocks' tensor map: [N rows][K / 32 * 18 bytes], boxes of 144 bytes x
// 16 T rows (encoded once per buffer, shape and unit size).
cudaError_t blocks_map(const uint8_t* blocks, int N, int K, int T, CUtensorMap* out) {
    struct Entry {
        const uint8_t* p;
        int N, K, T;
        CUtensorMap map;
    };
    static std::mutex mu;
    static std::vector<Entry> cache;
    {
        std::lock_guard<std::mutex> lock(mu);
        for (const Entry& e : cache)
            if (e.p == blocks && e.N == N && e.K == K && e.T == T) {
                *out = e.map;
                return cudaSuccess;
            }
    }
    PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
    if (!encode) return cudaErrorNotSupported;
    Entry e{blocks, N, K, T, {}};
    const cuuint64_t row_bytes = (cuuint64_t)(K / 32) * kQBlockBytes;
    const cuuint64_t dims[2] = {row_bytes, (cuuint64_t)N};
    const cuuint64_t strides[1] = {row_bytes};
    const cuuint32_t box[2] = {(cuuint32_t)kQBoxBytesRow, (cuuint32_t)(16 * T)};
    const cuuint32_t estr[2] = {1, 1};
    if (encode(&e.map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(blocks), dims,
               strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    *out = e.map;
    std::lock_guard<std::mutex> lock(mu);
    if (cache.size() >= 4096) cache.clear();
    cache.push_back(e);
    return cudaSuccess;
}

template <int MT>
cudaError_t launch_q40_mt(const uint8_t* blocks, Q40Args a, cudaStream_t stream,
                          const DeviceCtx& ctx) {
    cudaError_t e = ensure_q40_attr<MT>();
    if (e != cudaSuccess) return e;
    struct Key {
        int dev, M, N, K;
    };
    static std::mutex mu;
    static std::vector<std::pair<Key, Q40Plan>> cache;
    int dev = 0;
    cudaGetDevice(&dev);
    Q40Plan p;
    {
        std::lock_guard<std::mutex> lock(mu);
        for (const auto& c : cache)
            if (c.first.dev == dev && c.first.M == a.M && c.first.N == a.N && c.first.K == a.K)
                p = c.second;
    }
    if (p.T == 0) {
        p = plan_q40<MT>(a.M, a.N, a.K, ctx);
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
    CUtensorMap bmap;
    e = blocks_map(blocks, a.N, a.K, p.T, &bmap);
    if (e != cudaSuccess) return e;
    const long long units = ((long long)a.N + 16 * p.T - 1) / (16 * p.T);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1, (unsigned)units, 1);
    cfg.blockDim = dim3(kQThreads, 1, 1);
    cfg.dynamicSmemBytes = p.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    if (MT == 1 && a.M == 1) return cudaLaunchKernelEx(&cfg, gemv_q40_kernel<1, true>, bmap, a);
    return cudaLaunchKernelEx(&cfg, gemv_q40_kernel<MT, false>, bmap, a);
}

}  // namespace

cudaError_t launch_gemv_q4_0(const void* x, const void* blocks, void* y, int M, int64_t N,
                             int64_t K, cudaStream_t stream, const DeviceCtx& ctx) {
    Q40Args a{};
    a.x = static_cast<const __half*>(x);
    a.y = static_cast<__half*>(y);
    a.status = ctx.status;
    a.timeout_ns = ctx.timeout_ns;
    a.M = M;
    a.N = (int)N;
    a.K = (int)K;
    if (M <= 8) return launch_q40_mt<1>(static_cast<const uint8_t*>(blocks), a, stream, ctx);
    return launch_q40_mt<2>(static_cast<const uint8_t*>(blocks), a, stream, ctx);
}

}  // namespace w4a16
