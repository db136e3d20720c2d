// gemv_fmt.cu -- decode GEMV (M = 1..16) for the format variants of the
// weights: groups of 32, 64 or 128 along K or one group per row
// (per-channel), symmetric codes (nibble = q + 8) or asymmetric codes with a
// zero point per group (nibble = q):
//   y[m, n] = sum_k x[m, k] * (nib[n, k] - z[n, k / g]) * scale[n, k / g],
// z = 8 for symmetric codes (qaqbuyan.com tutorial, "量化的数学基石" §2
// symmetric and asymmetric formulas, §3 granularity; mhpq.cn report §二/§五
// for the decode product from packed weights).  With an AWQ activation scale
// alpha [K] (tutorial AWQ section: x~_j = x_j alpha_j, the weights quantized
// from W_{:,j} / alpha_j), x is replaced by x~ = fp16(x * alpha) in shared
// memory before the products (one IEEE fp16 multiply per element).
//
// The structure is gemv_unit_kernel's (gemv.cu): one CTA per unit of T
// 16-row tiles over the whole K range, 8 consumer warps + 1 producer warp,
// a ring of 16 KB stages filled with one tensor-map box each (T tiles x
// 32 / T chunks), the tile's warps splitting every stage's groups and adding
// their sums in shared memory in warp order, programmatic dependent launch.
// What differs is the dequantisation.  Each lane decodes (nib - z) exactly in
// fp16 (magic 1024, then subtract the row's 1024 + z).  With groups of 64,
// 128 or per channel a whole 64-wide chunk lies in one group, so the chunk's
// four MMAs take the exact codes into a fresh FP32 fragment that the rows'
// scales multiply once (CHUNK_SCALE: exact products, FP32 sums).  With groups
// of 32 the two halves of a chunk differ in group, and one MMA spans both, so
// each lane multiplies its (nib - z) by the row's fp16 scale before the MMA:
// one fp16 rounding of (q - z) * s per weight -- the tutorial's own fp16
// dequantised weight.  No activation sums are needed.  The group size is a
// template parameter, so a lane's scale and zero-point offsets are a few
// shifts of its group index.  The unit's scale and zero-point slabs are
// copied group-blocked where the row length allows ([Gs / 8][16 T][8 scales],
// [Gs / 16][16 T][16 zero points], one 3-D tensor-map box each): with the
// row-major slab the 8 rows a warp reads at one group sit Gs * 2 bytes apart,
// in one bank when that is a multiple of 128.  The default format (groups of
// 128, symmetric) keeps the kernels of gemv.cu.
// Every wait is bounded; on a time-out the CTA records it in the status
// word, stops issuing copies, drains those in flight and exits.
#include <atomic>
#include <mutex>
#include <utility>
#include <vector>

#include "common.cuh"
#include "kernels.h"

namespace w4a16 {
namespace {

constexpr int kFWarps = 8;
constexpr int kFConsumers = kFWarps * 32;
constexpr int kFThreads = kFConsumers + 32;
constexpr int kFTileBytes = 16 * kChunkK / 2;           // 512 B: one 16-row tile, one chunk
constexpr int kFChunkBytes = kBlockRows * kChunkK / 2;  // 4096 B per block-chunk
constexpr int kFStageBytes = 16384;
constexpr int kFMaxStages = 6;

constexpr int kFBarFull = 0;                                // [kFMaxStages]
constexpr int kFBarEmpty = kFBarFull + 8 * kFMaxStages;     // [kFMaxStages]
constexpr int kFBarX = kFBarEmpty + 8 * kFMaxStages;
constexpr int kFBarS = kFBarX + 8;
constexpr int kFAbort = kFBarS + 8;
constexpr int kFBarArea = 1024;

struct FmtArgs {
    const uint8_t* wq;      // kernel-layout weights
    const __half* scales;   // [N, Gs]
    const uint8_t* zeros;   // [N, Gs] or null (symmetric: z = 8)
    const __half* alpha;    // [K] AWQ activation scale, or null
    const __half* x;        // [M, K]
    __half* y;              // [M, N]
    unsigned* status;
    uint64_t timeout_ns;
    int M, N, K;
    int Gs;                 // scale groups per row
    int gshift;             // group index of k = k >> gshift (31: one group per row)
    int T;                  // 16-row tiles per CTA (1, 2 or 4)
    int nstages;
    int xs_stride;
    uint32_t off_ring, off_x, off_s, off_z, off_red;
    // Slab addressing in shared memory: the scale of (unit row r, group gi)
    // sits at off_s + (gi >> 3) * s_blk + r * s_row + 2 (gi & 7), its zero
    // point at off_z + (gi >> 4) * z_blk + r * z_row + (gi & 15).  Row-major
    // ([16 T][Gs], one bulk copy): s_blk = 16, s_row = 2 Gs.  Group-blocked
    // ([Gs / 8][16 T][8], one 3-D tensor-map copy, s_blk = 256 T, s_row = 16):
    // the 8 rows a warp reads at one group then fill 8 distinct 16-byte bank
    // groups instead of one bank (rows 2 Gs bytes apart, a multiple of 128).
    int s_tma, z_tma;       // the slab (zero-point slab) comes group-blocked
    uint32_t s_blk, s_row, z_blk, z_row;
};

// (nib - z) * s for one lane's 32-bit word of a chunk: rows r0 in registers
// 0 and 2, rows r1 in 1 and 3 (the layout's nibble order, as dequant8).
// zc0 = 1024 + z0 and zc1 = 64 + z1 as half2, s0 / s1 the rows' scales.
__device__ __forceinline__ void dequant8_fmt(uint32_t w, __half2 zc0, __half2 zc1, __half2 s0,
                                             __half2 s1, uint32_t (&r)[4]) {
    constexpr uint32_t kMagic = 0x64006400u;  // (1024.0, 1024.0)
    constexpr uint32_t kLut = (0xF0 & 0xCC) | 0xAA;  // (a & b) | c
    const uint32_t lo0 = lop3<kLut>(w, 0x000F000Fu, kMagic);
    const uint32_t hi0 = lop3<kLut>(w, 0x00F000F0u, kMagic);
    const uint32_t w8 = w >> 8;
    const uint32_t lo1 = lop3<kLut>(w8, 0x000F000Fu, kMagic);
    const uint32_t hi1 = lop3<kLut>(w8, 0x00F000F0u, kMagic);
    const __half2 kSixteenth = __halves2half2(__ushort_as_half(0x2C00), __ushort_as_half(0x2C00));
    __half2 v;
    // low nibbles: (1024 + n) - (1024 + z0) = n - z0, exact
    v = __hmul2(__hsub2(*reinterpret_cast<const __half2*>(&lo0), zc0), s0);
    r[0] = *reinterpret_cast<uint32_t*>(&v);
    v = __hmul2(__hsub2(*reinterpret_cast<const __half2*>(&lo1), zc0), s0);
    r[2] = *reinterpret_cast<uint32_t*>(&v);
    // high nibbles: (1024 + 16 n) / 16 - (64 + z1) = n - z1, exact (one rounding of an exact value)
    v = __hmul2(__hfma2(*reinterpret_cast<const __half2*>(&hi0), kSixteenth, __hneg2(zc1)), s1);
    r[1] = *reinterpret_cast<uint32_t*>(&v);
    v = __hmul2(__hfma2(*reinterpret_cast<const __half2*>(&hi1), kSixteenth, __hneg2(zc1)), s1);
    r[3] = *reinterpret_cast<uint32_t*>(&v);
}

// (nib - z) for one lane's 32-bit word, exactly, in the same register order.
__device__ __forceinline__ void dequant8_zq(uint32_t w, __half2 zc0, __half2 nzc1,
                                            uint32_t (&r)[4]) {
    constexpr uint32_t kMagic = 0x64006400u;  // (1024.0, 1024.0)
    constexpr uint32_t kLut = (0xF0 & 0xCC) | 0xAA;  // (a & b) | c
    const uint32_t lo0 = lop3<kLut>(w, 0x000F000Fu, kMagic);
    const uint32_t hi0 = lop3<kLut>(w, 0x00F000F0u, kMagic);
    const uint32_t w8 = w >> 8;
    const uint32_t lo1 = lop3<kLut>(w8, 0x000F000Fu, kMagic);
    const uint32_t hi1 = lop3<kLut>(w8, 0x00F000F0u, kMagic);
    const __half2 kSixteenth = __halves2half2(__ushort_as_half(0x2C00), __ushort_as_half(0x2C00));
    __half2 v;
    v = __hsub2(*reinterpret_cast<const __half2*>(&lo0), zc0);
    r[0] = *reinterpret_cast<uint32_t*>(&v);
    v = __hsub2(*reinterpret_cast<const __half2*>(&lo1), zc0);
    r[2] = *reinterpret_cast<uint32_t*>(&v);
    v = __hfma2(*reinterpret_cast<const __half2*>(&hi0), kSixteenth, nzc1);
    r[1] = *reinterpret_cast<uint32_t*>(&v);
    v = __hfma2(*reinterpret_cast<const __half2*>(&hi1), kSixteenth, nzc1);
    r[3] = *reinterpret_cast<uint32_t*>(&v);
}

// One 128-wide group (two chunks) of one consumer lane, dequantised with
// the scale and zero point of the lane's group in each chunk, accumulated
// into acc (two MMA chains for M <= 8).  CHUNK_SCALE: the chunk's exact
// products summed in a fresh FP32 fragment, scaled once per row.
template <int MT, bool CHUNK_SCALE>
__device__ __forceinline__ void mma_group_fmt(uint32_t w_addr, uint32_t cs, uint32_t x0_addr,
                                              uint32_t x1_addr, const uint8_t* sr0,
                                              const uint8_t* sr1, const uint8_t* zr0,
                                              const uint8_t* zr1, uint32_t so0, uint32_t so1,
                                              uint32_t zo0, uint32_t zo1,
                                              float (&acc)[2][MT][4]) {
#pragma unroll
    for (int c = 0; c < 2; ++c) {
        const uint32_t so = c == 0 ? so0 : so1, zo = c == 0 ? zo0 : zo1;
        const __half2 s0 = __half2half2(*reinterpret_cast<const __half*>(sr0 + so));
        const __half2 s1 = __half2half2(*reinterpret_cast<const __half*>(sr1 + so));
        const uint32_t z0 = zr0 ? zr0[zo] : 8u;
        const uint32_t z1 = zr1 ? zr1[zo] : 8u;
        // 1024 + z0 is the fp16 bit pattern 0x6400 + z0 (exact for z0 < 1024);
        // 64 + z1 = (1024 + z1) - 960, an exact fp16 difference for z1 < 256
        const uint32_t zb0 = 0x64006400u + z0 * 0x10001u, zb1 = 0x64006400u + z1 * 0x10001u;
        const __half2 zc0 = *reinterpret_cast<const __half2*>(&zb0);
        const __half2 zc1 = __hsub2(*reinterpret_cast<const __half2*>(&zb1),
                                    __half2half2(__ushort_as_half(0x6380)));  // 960
        const uint4 wv = lds128(w_addr + c * cs);
        const uint4 xa = lds128(x0_addr + c * 128);
        const uint4 xb = lds128(x0_addr + c * 128 + 16);
        uint4 xa1 = xa, xb1 = xb;
        if (MT == 2) {
            xa1 = lds128(x1_addr + c * 128);
            xb1 = lds128(x1_addr + c * 128 + 16);
        }
        const uint32_t wrd[4] = {wv.x, wv.y, wv.z, wv.w};
        const uint32_t b0[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
        const uint32_t b1[8] = {xa1.x, xa1.y, xa1.z, xa1.w, xb1.x, xb1.y, xb1.z, xb1.w};
        if constexpr (CHUNK_SCALE) {
            float ch[MT][4];
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int e = 0; e < 4; ++e) ch[mt][e] = 0.0f;
            const __half2 nzc1 = __hneg2(zc1);
#pragma unroll
            for (int s = 0; s < 4; ++s) {
                uint32_t af[4];
                dequant8_zq(wrd[s], zc0, nzc1, af);
                mma_16816(ch[0], af, b0[2 * s], b0[2 * s + 1], ch[0]);
                if (MT == 2) mma_16816(ch[MT - 1], af, b1[2 * s], b1[2 * s + 1], ch[MT - 1]);
            }
            const float2 f0 = __half22float2(s0), f1 = __half22float2(s1);
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
                const float2 a01 = __ffma2_rn(f0, make_float2(ch[mt][0], ch[mt][1]),
                                              make_float2(acc[c][mt][0], acc[c][mt][1]));
                const float2 a23 = __ffma2_rn(f1, make_float2(ch[mt][2], ch[mt][3]),
                                              make_float2(acc[c][mt][2], acc[c][mt][3]));
                acc[c][mt][0] = a01.x;
                acc[c][mt][1] = a01.y;
                acc[c][mt][2] = a23.x;
                acc[c][mt][3] = a23.y;
            }
        } else {
#pragma unroll
            for (int s = 0; s < 4; ++s) {
                uint32_t af[4];
                dequant8_fmt(wrd[s], zc0, zc1, s0, s1, af);
                mma_16816(acc[c][0], af, b0[2 * s], b0[2 * s + 1], acc[c][0]);
                if (MT == 2)
                    mma_16816(acc[c][MT - 1], af, b1[2 * s], b1[2 * s + 1], acc[c][MT - 1]);
            }
        }
    }
}

// GSH: log2 of the group size (5, 6, 7), or 31 for one group per row.
template <int MT, int GSH>
__global__ void __launch_bounds__(kFThreads, MT == 1 ? 3 : 2)
    gemv_fmt_kernel(const __grid_constant__ CUtensorMap wmap, const __grid_constant__ CUtensorMap smap,
                    const __grid_constant__ CUtensorMap zmap, const __grid_constant__ FmtArgs a) {
    extern __shared__ __align__(1024) uint8_t smem[];
    constexpr bool CHUNK_SCALE = GSH >= 6;  // a whole 64-wide chunk in one group
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int T = a.T;
    const int W = kFWarps / T;                          // warps per tile
    const int CPS = kFStageBytes / (T * kFTileBytes);   // chunks per stage
    const int GPS = CPS / 2;                            // 128-groups per stage
    const int C = a.K / kChunkK, G = a.K / kGroup;
    const int nstg = (C + CPS - 1) / CPS;
    const int r0 = (int)blockIdx.y * 16 * T;            // first weight row of the unit
    const int rb = r0 / kBlockRows, t0 = (r0 % kBlockRows) / 16;
    const int rows = min(16 * T, a.N - r0);
    const int NS = a.nstages;
    const uint32_t sbase = smem_u32(smem);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kFAbort);
    const uint32_t ring = sbase + a.off_ring;

    grid_launch_dependents();

    if (warp == kFWarps) {
        // =============================== producer ===============================
        // The producer initialises the barriers and goes straight on to its
        // first copies; the consumers wait for that on named barrier 2.
        if (lane == 0) {
            for (int s = 0; s < NS; ++s) {
                mbar_init(sbase + kFBarFull + 8 * s, 1);
                mbar_init(sbase + kFBarEmpty + 8 * s, kFWarps);
            }
            mbar_init(sbase + kFBarX, 1);
            mbar_init(sbase + kFBarS, 1);
            *abort_flag = 0;
            fence_barrier_init();
        }
        __syncwarp();
        asm volatile("bar.arrive 2, %0;" ::"n"(kFThreads) : "memory");
        if (lane == 0) {
            const uint64_t pol = l2_policy_evict_first();
            const int box_x = t0 * (kFTileBytes / 8);
            const int cy0 = rb * C;
            tma_prefetch_map(&wmap);
            {   // scale slab (and zero-point slab) of the unit's rows: one
                // group-blocked tensor-map box (rows past N zero-filled), or
                // row-major by bulk copy with the unaligned tail by hand
                const int R = 16 * T;
                uint32_t sbulk = 0, zbulk = 0, tx = 0;
                const __half* ssrc = a.scales + (size_t)r0 * a.Gs;
                const uint8_t* zsrc = a.zeros ? a.zeros + (size_t)r0 * a.Gs : nullptr;
                if (a.s_tma) {
                    tx += (uint32_t)(R * a.Gs * 2);
                } else {
                    const uint32_t sbytes = (uint32_t)(rows * a.Gs * 2);
                    sbulk = sbytes & ~15u;
                    __half* sdst = reinterpret_cast<__half*>(smem + a.off_s);
                    for (uint32_t e = sbulk / 2; e < sbytes / 2; ++e) sdst[e] = ssrc[e];
                    tx += sbulk;
                }
                if (a.zeros) {
                    if (a.z_tma) {
                        tx += (uint32_t)(R * a.Gs);
                    } else {
                        const uint32_t zbytes = (uint32_t)(rows * a.Gs);
                        zbulk = zbytes & ~15u;
                        uint8_t* zdst = smem + a.off_z;
                        for (uint32_t e = zbulk; e < zbytes; ++e) zdst[e] = zsrc[e];
                        tx += zbulk;
                    }
                }
                mbar_arrive_expect_tx(sbase + kFBarS, tx);
                if (a.s_tma) tma_load_3d(sbase + a.off_s, &smap, 0, r0, 0, sbase + kFBarS);
                else if (sbulk) bulk_g2s(sbase + a.off_s, ssrc, sbulk, sbase + kFBarS);
                if (a.zeros && a.z_tma) tma_load_3d(sbase + a.off_z, &zmap, 0, r0, 0, sbase + kFBarS);
                else if (zbulk) bulk_g2s(sbase + a.off_z, zsrc, zbulk, sbase + kFBarS);
            }
            bool x_issued = false;
            auto issue_x = [&]() {
                grid_dependency_wait();
                const uint32_t xbytes = (uint32_t)a.K * 2;
                mbar_arrive_expect_tx(sbase + kFBarX, xbytes * a.M);
                for (int m = 0; m < a.M; ++m)
                    bulk_g2s(sbase + a.off_x + m * a.xs_stride, a.x + (size_t)m * a.K, xbytes,
                             sbase + kFBarX);
                x_issued = true;
            };
            int it = 0, slot = 0, round = 0;
            bool ok = true;
            for (; it < nstg; ++it) {
                if (it >= NS && !x_issued) issue_x();
                if (it >= NS && !mbar_wait(sbase + kFBarEmpty + 8 * slot, (round - 1) & 1,
                                           a.timeout_ns, a.status)) {
                    ok = false;
                    break;
                }
                if (*abort_flag) {
                    ok = false;
                    break;
                }
                const int nc = min(CPS, C - it * CPS);
                const uint32_t dst = ring + slot * kFStageBytes;
                const uint32_t bar = sbase + kFBarFull + 8 * slot;
                if (nc == CPS) {
                    mbar_arrive_expect_tx(bar, kFStageBytes);
                    tma_load_2d_hint(dst, &wmap, box_x, cy0 + it * CPS, bar, pol);
                } else {
                    const uint32_t rowb = (uint32_t)(T * kFTileBytes);
                    const uint8_t* src = a.wq + (size_t)(cy0 + it * CPS) * kFChunkBytes +
                                         (size_t)t0 * kFTileBytes;
                    mbar_arrive_expect_tx(bar, nc * rowb);
                    for (int c = 0; c < nc; ++c)
                        bulk_g2s_hint(dst + c * rowb, src + (size_t)c * kFChunkBytes, rowb, bar,
                                      pol);
                }
                if (++slot == NS) {
                    slot = 0;
                    ++round;
                }
            }
            if (!x_issued) issue_x();
            if (!ok) *abort_flag = 1;
            const uint64_t dt = drain_bound(a.timeout_ns);
            mbar_wait(sbase + kFBarX, 0, dt, a.status);
            for (int i = (it > NS ? it - NS : 0); i < it; ++i)
                mbar_wait(sbase + kFBarFull + 8 * (i % NS), (i / NS) & 1, dt, a.status);
            mbar_wait(sbase + kFBarS, 0, dt, a.status);
        }
        __syncwarp();
        return;
    }

    // ================================ consumers =================================
    asm volatile("bar.sync 2, %0;" ::"n"(kFThreads) : "memory");  // barriers initialised
    grid_dependency_wait();
    const int g = lane >> 2, t = lane & 3;
    const int ti = warp / W, ks = warp - ti * W;
    const int row0 = ti * 16 + g, row1 = row0 + 8;
    const int xr0 = g < a.M ? g : a.M - 1;
    const int xr1 = g + 8 < a.M ? g + 8 : a.M - 1;
    const uint32_t x0 = sbase + a.off_x + xr0 * a.xs_stride + t * 32;
    const uint32_t x1 = sbase + a.off_x + xr1 * a.xs_stride + t * 32;
    const uint32_t cs = (uint32_t)(T * kFTileBytes);
    const uint32_t wl = ring + ti * kFTileBytes + lane * 16;
    const uint8_t* sr0 = smem + a.off_s + row0 * a.s_row;
    const uint8_t* sr1 = sr0 + 8 * a.s_row;
    const uint8_t* zr0 = a.zeros ? smem + a.off_z + row0 * a.z_row : nullptr;
    const uint8_t* zr1 = a.zeros ? zr0 + 8 * a.z_row : nullptr;

    bool ok = mbar_wait(sbase + kFBarX, 0, a.timeout_ns, a.status);
    if (a.alpha) {
        // AWQ: x~ = fp16(x * alpha) in place, 16 bytes per thread per step;
        // every consumer thread takes part in the barrier below.
        const int per_row = a.K / 8;
        for (int q = (int)threadIdx.x; ok && q < a.M * per_row; q += kFConsumers) {
            const int m = q / per_row, off = q - m * per_row;
            const uint4 av = __ldg(reinterpret_cast<const uint4*>(a.alpha) + off);
            uint4* xp = reinterpret_cast<uint4*>(smem + a.off_x + m * a.xs_stride + off * 16);
            uint4 xv = *xp;
            __half2* xh = reinterpret_cast<__half2*>(&xv);
            const __half2* ah = reinterpret_cast<const __half2*>(&av);
#pragma unroll
            for (int i = 0; i < 4; ++i) xh[i] = __hmul2(xh[i], ah[i]);
            *xp = xv;
        }
        asm volatile("bar.sync 1, %0;" ::"n"(kFConsumers) : "memory");
    }
    if (ok) ok = mbar_wait(sbase + kFBarS, 0, a.timeout_ns, a.status);
    ok = __all_sync(0xffffffffu, ok);  // warp-uniform before the warp MMAs
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
        if (ok) ok = mbar_wait(sbase + kFBarFull + 8 * slot, phase, a.timeout_ns, a.status);
        ok = __all_sync(0xffffffffu, ok);
        if (ok) {
            const int gs = min(GPS, G - st * GPS);  // 128-groups in this stage
            // the warp's two groups of the stage; at MT = 1 both unguarded
            // unless the last stage is short, so that the common case is
            // straight-line code (at MT = 2 that code spills)
            auto group = [&](int gi) __attribute__((always_inline)) {
                const int gsl = ks * 2 + gi;        // this warp's group within the stage
                const int gl = st * GPS + gsl;  // 128-group index along the row
                // The scale group of this lane's k (16 t .. 16 t + 15 of
                // each chunk) in chunks 2 gl and 2 gl + 1: gi0 and gi1.
                // They share a run of 8 scales and of 16 zero points, so
                // the second chunk's offsets are the first's plus
                // 2 (gi1 - gi0) and gi1 - gi0 in either slab layout.
                uint32_t so = 0, zo = 0;
                constexpr uint32_t dg = GSH == 5 ? 2 : GSH == 6 ? 1 : 0;  // gi1 - gi0
                if constexpr (GSH < 31) {
                    const uint32_t gi0 = GSH == 5 ? 4 * gl + (t >> 1) : GSH == 6 ? 2 * gl : gl;
                    so = (gi0 >> 3) * a.s_blk + ((gi0 & 7) << 1);
                    zo = (gi0 >> 4) * a.z_blk + (gi0 & 15);
                }
                mma_group_fmt<MT, CHUNK_SCALE>(wl + slot * kFStageBytes + gsl * 2 * cs, cs,
                                               x0 + gl * 256, x1 + gl * 256, sr0, sr1, zr0, zr1,
                                               so, so + 2 * dg, zo, zo + dg, acc);
            };
            if (MT == 1 && ks * 2 + 1 < gs) {
                group(0);
                group(1);
            } else {
                if (ks * 2 < gs) group(0);
                if (ks * 2 + 1 < gs) group(1);
            }
        }
        __syncwarp();
        if (ok && lane == 0) mbar_arrive(sbase + kFBarEmpty + 8 * slot);
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
    asm volatile("bar.sync 1, %0;" ::"n"(kFConsumers) : "memory");
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
        const int R0 = r0 + row0, R1 = r0 + row1;
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
            const int m0 = mt * 8 + 2 * t, m1 = m0 + 1;
            if (m0 < a.M) {
                if (R0 < a.N) a.y[(size_t)m0 * a.N + R0] = __float2half_rn(sum[mt][0]);
                if (R1 < a.N) a.y[(size_t)m0 * a.N + R1] = __float2half_rn(sum[mt][2]);
            }
            if (m1 < a.M) {
                if (R0 < a.N) a.y[(size_t)m1 * a.N + R0] = __float2half_rn(sum[mt][1]);
                if (R1 < a.N) a.y[(size_t)m1 * a.N + R1] = __float2half_rn(sum[mt][3]);
            }
        }
    }
    if (!ok) *abort_flag = 1;
}

struct FmtPlan {
    int T = 0, nstages = 0, xs_stride = 0;
    uint32_t off_ring = 0, off_x = 0, off_s = 0, off_z = 0, off_red = 0, smem = 0;
};

template <int MT>
int fmt_occupancy(uint32_t smem) {
    // every group size has the same launch bounds; the largest register count decides
    const void* fns[4] = {reinterpret_cast<const void*>(gemv_fmt_kernel<MT, 5>),
                          reinterpret_cast<const void*>(gemv_fmt_kernel<MT, 6>),
                          reinterpret_cast<const void*>(gemv_fmt_kernel<MT, 7>),
                          reinterpret_cast<const void*>(gemv_fmt_kernel<MT, 31>)};
    int occ = 0;
    for (int i = 0; i < 4; ++i) {
        int b = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, fns[i], kFThreads, smem) != cudaSuccess)
            return 0;
        occ = i == 0 || b < occ ? b : occ;
    }
    return occ;
}

template <int MT>
cudaError_t ensure_fmt_attr() {
    static std::atomic<bool> done[64];  // per device; racing callers only repeat the set-up
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && done[dev].load(std::memory_order_acquire)) return cudaSuccess;
    const void* fns[4] = {reinterpret_cast<const void*>(gemv_fmt_kernel<MT, 5>),
                          reinterpret_cast<const void*>(gemv_fmt_kernel<MT, 6>),
                          reinterpret_cast<const void*>(gemv_fmt_kernel<MT, 7>),
                          reinterpret_cast<const void*>(gemv_fmt_kernel<MT, 31>)};
    cudaError_t e = cudaSuccess;
    for (int i = 0; i < 4 && e == cudaSuccess; ++i)
        e = cudaFuncSetAttribute(fns[i], cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    if (e == cudaSuccess && dev >= 0 && dev < 64) done[dev].store(true, std::memory_order_release);
    return e;
}

template <int MT>
bool fmt_layout(FmtPlan& p, int M, int K, int Gs, bool zp, int T, int nst, const DeviceCtx& ctx) {
    p.T = T;
    const int chunks = K / kChunkK;
    const int fill = (chunks * T * kFTileBytes + kFStageBytes - 1) / kFStageBytes;
    p.nstages = fill < nst ? fill : nst;
    p.xs_stride = K * 2 + 16;
    p.off_ring = kFBarArea;
    p.off_x = p.off_ring + p.nstages * kFStageBytes;
    p.off_s = p.off_x + ((M * p.xs_stride + 127) / 128) * 128;
    p.off_z = p.off_s + ((16 * T * Gs * 2 + 127) / 128) * 128;
    p.off_red = p.off_z + (zp ? ((16 * T * Gs + 127) / 128) * 128 : 0);
    p.smem = p.off_red + kFWarps * MT * 32 * 16;
    return (int)p.smem <= ctx.max_smem_optin;
}

// The unit size: the fewest waves of CTAs, then the most CTAs per wave,
// with the deepest ring (2 to 6 stages) that keeps the CTAs per SM.
template <int MT>
FmtPlan plan_fmt(int M, int N, int K, int Gs, bool zp, const DeviceCtx& ctx) {
    FmtPlan best;
    long long best_waves = 0, best_units = 0;
    for (int T = 1; T <= 4; T *= 2) {
        FmtPlan p;
        if (!fmt_layout<MT>(p, M, K, Gs, zp, T, 3, ctx)) continue;
        {   // a 2-stage ring when that fits more CTAs per SM (the large
            // slabs of groups of 32: 64-row units at K = 4096 go from 2 to 3)
            FmtPlan q2;
            if (fmt_layout<MT>(q2, M, K, Gs, zp, T, 2, ctx) &&
                fmt_occupancy<MT>(q2.smem) > fmt_occupancy<MT>(p.smem))
                p = q2;
        }
        const int occ = fmt_occupancy<MT>(p.smem);
        const long long units = ((long long)N + 16 * T - 1) / (16 * T);
        if (occ == 0 || units > 65535) continue;
        const long long slots = (long long)ctx.num_sms * occ;
        const long long waves = (units + slots - 1) / slots;
        const int need = (int)((units < slots ? units : slots) + ctx.num_sms - 1) / ctx.num_sms;
        for (int nst = kFMaxStages; nst > p.nstages; --nst) {
            FmtPlan q;
            if (fmt_layout<MT>(q, M, K, Gs, zp, T, nst, ctx) && q.nstages == nst &&
                fmt_occupancy<MT>(q.smem) >= need) {
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

// The group-blocked view of a [N, Gs] slab of `eb`-byte elements (fp16
// scales or byte zero points): dimension 0 is one 16-byte run of groups,
// dimension 1 the rows (stride Gs * eb), dimension 2 the runs of a row
// (stride 16 bytes); a box of R rows lands in shared memory as
// [Gs * eb / 16][R][16 bytes].  Encoded once per (slab, shape, R).  Returns
// false when the slab does not fit the view (rows not a whole number of
// 16-byte runs, more than 256 runs, or an unaligned base); the launch then
// copies the slab row-major.
bool slab_map(const void* base, int eb, int N, int Gs, int R, CUtensorMap* out) {
    const int runs = Gs * eb / 16;
    if ((Gs * eb) % 16 != 0 || runs < 1 || runs > 256 || R > 256 ||
        (reinterpret_cast<uintptr_t>(base) & 15) != 0)
        return false;
    struct Entry {
        const void* base;
        int eb, N, Gs, R;
        CUtensorMap map;
    };
    static std::mutex mu;
    static std::vector<Entry> cache;
    {
        std::lock_guard<std::mutex> lock(mu);
        for (const Entry& e : cache)
            if (e.base == base && e.eb == eb && e.N == N && e.Gs == Gs && e.R == R) {
                *out = e.map;
                return true;
            }
    }
    PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
    if (!encode) return false;
    Entry e{base, eb, N, Gs, R, {}};
    const cuuint64_t dims[3] = {(cuuint64_t)(16 / eb), (cuuint64_t)N, (cuuint64_t)runs};
    const cuuint64_t strides[2] = {(cuuint64_t)Gs * eb, 16};
    const cuuint32_t box[3] = {(cuuint32_t)(16 / eb), (cuuint32_t)R, (cuuint32_t)runs};
    const cuuint32_t estr[3] = {1, 1, 1};
    if (encode(&e.map, eb == 2 ? CU_TENSOR_MAP_DATA_TYPE_UINT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 3,
               const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return false;
    *out = e.map;
    std::lock_guard<std::mutex> lock(mu);
    if (cache.size() < 4096) cache.push_back(e);
    return true;
}

template <int MT>
cudaError_t launch_fmt_mt(FmtArgs a, cudaStream_t stream, const DeviceCtx& ctx) {
    cudaError_t e = ensure_fmt_attr<MT>();
    if (e != cudaSuccess) return e;
    struct Key {
        int dev, M, N, K, Gs;
        bool zp;
    };
    static std::mutex mu;
    static std::vector<std::pair<Key, FmtPlan>> cache;
    int dev = 0;
    cudaGetDevice(&dev);
    FmtPlan p;
    {
        std::lock_guard<std::mutex> lock(mu);
        for (const auto& c : cache)
            if (c.first.dev == dev && c.first.M == a.M && c.first.N == a.N && c.first.K == a.K &&
                c.first.Gs == a.Gs && c.first.zp == (a.zeros != nullptr))
                p = c.second;
    }
    if (p.T == 0) {
        p = plan_fmt<MT>(a.M, a.N, a.K, a.Gs, a.zeros != nullptr, ctx);
        if (p.T == 0) return cudaErrorInvalidValue;
        std::lock_guard<std::mutex> lock(mu);
        if (cache.size() < 4096) cache.push_back({{dev, a.M, a.N, a.K, a.Gs, a.zeros != nullptr}, p});
    }
    a.T = p.T;
    a.nstages = p.nstages;
    a.xs_stride = p.xs_stride;
    a.off_ring = p.off_ring;
    a.off_x = p.off_x;
    a.off_s = p.off_s;
    a.off_z = p.off_z;
    a.off_red = p.off_red;
    CUtensorMap wmap;
    e = gemv_weight_map(a.wq, a.N, a.K, p.T, &wmap);
    if (e != cudaSuccess) return e;
    const int R = 16 * p.T;
    CUtensorMap smap{}, zmap{};
    a.s_tma = slab_map(a.scales, 2, a.N, a.Gs, R, &smap) ? 1 : 0;
    a.z_tma = a.zeros && slab_map(a.zeros, 1, a.N, a.Gs, R, &zmap) ? 1 : 0;
    a.s_blk = a.s_tma ? (uint32_t)R * 16 : 16;
    a.s_row = a.s_tma ? 16 : (uint32_t)a.Gs * 2;
    a.z_blk = a.z_tma ? (uint32_t)R * 16 : 16;
    a.z_row = a.z_tma ? 16 : (uint32_t)a.Gs;
    const long long units = ((long long)a.N + 16 * p.T - 1) / (16 * p.T);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1, (unsigned)units, 1);
    cfg.blockDim = dim3(kFThreads, 1, 1);
    cfg.dynamicSmemBytes = p.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    // groups of 64 and more: a whole chunk in one group, scaled in FP32
    switch (a.gshift) {
    case 5: return cudaLaunchKernelEx(&cfg, gemv_fmt_kernel<MT, 5>, wmap, smap, zmap, a);
    case 6: return cudaLaunchKernelEx(&cfg, gemv_fmt_kernel<MT, 6>, wmap, smap, zmap, a);
    case 7: return cudaLaunchKernelEx(&cfg, gemv_fmt_kernel<MT, 7>, wmap, smap, zmap, a);
    default: return cudaLaunchKernelEx(&cfg, gemv_fmt_kernel<MT, 31>, wmap, smap, zmap, a);
    }
}

}  // namespace

cudaError_t launch_gemv_fmt(const void* x, const void* alpha, const void* repacked,
                            const void* scales, const void* zeros, void* y, int M, int64_t N,
                            int64_t K, int group, cudaStream_t stream, const DeviceCtx& ctx) {
    FmtArgs a{};
    a.alpha = static_cast<const __half*>(alpha);
    a.wq = static_cast<const uint8_t*>(repacked);
    a.scales = static_cast<const __half*>(scales);
    a.zeros = static_cast<const uint8_t*>(zeros);
    a.x = static_cast<const __half*>(x);
    a.y = static_cast<__half*>(y);
    a.status = ctx.status;
    a.timeout_ns = ctx.timeout_ns;
    a.M = M;
    a.N = (int)N;
    a.K = (int)K;
    a.Gs = (int)(K / group);
    a.gshift = group == 32 ? 5 : group == 64 ? 6 : group == 128 ? 7 : 31;
    if (M <= 8) return launch_fmt_mt<1>(a, stream, ctx);
    return launch_fmt_mt<2>(a, stream, ctx);
}

cudaError_t gemv_fmt_plan_info(int M, int64_t N, int64_t K, int group, bool zp, const DeviceCtx& ctx,
                               int* ctas, int* rows_per_cta) {
    cudaError_t e = M <= 8 ? ensure_fmt_attr<1>() : ensure_fmt_attr<2>();
    if (e != cudaSuccess) return e;
    const int Gs = (int)(K / group);
    const FmtPlan p = M <= 8 ? plan_fmt<1>(M, (int)N, (int)K, Gs, zp, ctx)
                             : plan_fmt<2>(M, (int)N, (int)K, Gs, zp, ctx);
    if (p.T == 0) return cudaErrorInvalidValue;
    *rows_per_cta = 16 * p.T;
    *ctas = (int)((N + 16 * p.T - 1) / (16 * p.T));
    return cudaSuccess;
}

bool gemv_fmt_fits(int M, int64_t N, int64_t K, int group, bool zp, const DeviceCtx& ctx) {
    FmtPlan p;
    const int Gs = (int)(K / group);
    if ((N + 63) / 64 > 65535) return false;
    return M <= 8 ? fmt_layout<1>(p, M, (int)K, Gs, zp, 1, 3, ctx)
                  : fmt_layout<2>(p, M, (int)K, Gs, zp, 1, 3, ctx);
}

}  // namespace w4a16
