// gemm_tc.cu -- W4A16 prefill GEMM (M > 16) on the tcgen05 tensor cores.
//
// y[m, n] = sum_k x[m, k] * Wd[n, k],  Wd[n, k] = fp16((nib - 8) * scale[n, k/128])
// (qaqbuyan.com tutorial "量化的数学基石" §3 per_group_symmetric_dequantize:
// the fp16 dequantized weight is the fp32 product q * s rounded once to fp16;
// mhpq.cn W4A16 report §二 prefill column: the same packed format serves the
// prompt pass).  Unlike decode, the prompt pass is a dense contraction, so it
// runs on the tensor cores:
//
// A thread block computes a 128 (activation rows = MMA M) x 128 (weight rows
// = MMA N) tile of y with FP32 accumulators in tensor memory; once M > 128 a
// cluster of two blocks computes a 256 x 256 tile with 2-CTA MMAs (see
// gemm_tc_kernel<true, XT>), which cuts the shared-memory operand traffic per
// FLOP and puts more MMA work behind every stage hand-off.
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

#include <algorithm>
#include <atomic>
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
constexpr int kMaxStages = 6;                   // ring: x tile, packed and dequantised weights
constexpr int kSingleStages = 4;                // ring of the single-CTA tile
constexpr int kXStageBytes = kTileX * kBK * 2;  // 16 KB

constexpr int kBarLoadFull = 0;                      // [stages] x + packed weights landed
constexpr int kBarAFull = kBarLoadFull + 8 * kMaxStages;  // [stages] dequantised tile written
constexpr int kBarFree = kBarAFull + 8 * kMaxStages;      // [stages] MMAs done: stage reusable
constexpr int kBarAcc = kBarFree + 8 * kMaxStages;
constexpr int kBarSlab = kBarAcc + 8;
constexpr int kTmemSlot = kBarSlab + 8;
constexpr int kAbortFlag = kTmemSlot + 8;
// Split-K reduction: per source split, 128 rows of 64 FP32 columns padded to
// 68 (16-byte accesses of 8 consecutive rows hit distinct banks).
constexpr int kRedRow = 68;
constexpr int kRedSlotFloats = 128 * kRedRow;
constexpr int kOffA = 1024;                              // dequantised tiles
// then x tiles, packed weights and the scale slab at offsets set per launch

struct TcArgs {
    const uint8_t* wq;
    const __half* scales;
    __half* y;
    unsigned* status;
    uint64_t timeout_ns;
    int M, N, K, G;
    int nst;                           // ring stages (<= kMaxStages)
    uint32_t off_x, off_w, off_slab;   // shared-memory offsets after the window base
    // Split K (pairs only, splits > 1): blockIdx.z takes k-blocks
    // [z nkb / splits, (z + 1) nkb / splits); the splits of a tile form one
    // thread-block cluster (2 x splits CTAs) and reduce their accumulators
    // through distributed shared memory.
    int splits;
    // Scale slab: slab_ld groups per row.  slab_tma = 1: a 2-D tensor-map copy
    // of the 128 rows x slab_ld groups starting at this CTA's first group
    // rounded down to 8 (a split's own groups only); else the whole
    // [128][G] slab by bulk copy (slab_ld = G).
    int slab_ld, slab_tma;
    // Format variants (FMT kernels; G = 0, no slab): the scale of weight row
    // n for k is scales[n * gcount + (k >> gshift)] (gshift 5, 6, 7 for
    // groups of 32, 64, 128; 31 per channel), its zero point
    // zeros[n * gcount + (k >> gshift)] (NULL: symmetric, z = 8), and an
    // optional AWQ activation scale alpha[k] (NULL: none).
    const uint8_t* zeros;
    const __half* alpha;
    int gshift, gcount;
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

// The format coefficients one dequantising thread needs for one k-block:
// the scales and zero points of its rows r0 / r0 + 8 for its 16 k (one group
// at every group size) and alpha at those 16 k.
struct FmtCoef {
    __half s0, s1;
    int z0, z1;
    uint4 al0, al1;
};

__device__ __forceinline__ FmtCoef fmt_coef(const TcArgs& a, int kblock, int n0, int tq) {
    FmtCoef c;
    c.s0 = c.s1 = __ushort_as_half(0);
    c.z0 = c.z1 = 8;
    c.al0 = c.al1 = make_uint4(0u, 0u, 0u, 0u);
    const int kk = kblock * kBK;
    const int gi = (kk + 16 * tq) >> a.gshift;
    const int n1 = n0 + 8;
    if (n0 < a.N) {
        c.s0 = __ldg(a.scales + (size_t)n0 * a.gcount + gi);
        if (a.zeros) c.z0 = __ldg(a.zeros + (size_t)n0 * a.gcount + gi);
    }
    if (n1 < a.N) {
        c.s1 = __ldg(a.scales + (size_t)n1 * a.gcount + gi);
        if (a.zeros) c.z1 = __ldg(a.zeros + (size_t)n1 * a.gcount + gi);
    }
    if (a.alpha) {
        const uint4* p = reinterpret_cast<const uint4*>(a.alpha + kk + 16 * tq);
        c.al0 = __ldg(p);
        c.al1 = __ldg(p + 1);
    }
    return c;
}

// (nib - z) for the 8 nibbles of a kernel-layout word, exactly: the low
// nibbles (rows r0, zero point z0) OR-ed into the mantissa of 1024.0 minus
// (1024 + z0); the high nibbles (rows r1, z1) give 1024 + 16 nib, times 1/16
// minus (64 + z1).  r[0] / r[2]: rows r0, r[1] / r[3]: rows r1, as dequant8
// (which is this with z = 8).
__device__ __forceinline__ void dequant8_z(uint32_t w, __half2 lo_off, __half2 hi_off,
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
    v = __hsub2(*reinterpret_cast<const __half2*>(&lo0), lo_off);
    r[0] = *reinterpret_cast<uint32_t*>(&v);
    v = __hfma2(*reinterpret_cast<const __half2*>(&hi0), kSixteenth, hi_off);
    r[1] = *reinterpret_cast<uint32_t*>(&v);
    v = __hsub2(*reinterpret_cast<const __half2*>(&lo1), lo_off);
    r[2] = *reinterpret_cast<uint32_t*>(&v);
    v = __hfma2(*reinterpret_cast<const __half2*>(&hi1), kSixteenth, hi_off);
    r[3] = *reinterpret_cast<uint32_t*>(&v);
}

// Rounds 32 FP32 accumulators to fp16 and stores them at y[m, n .. n + 31]
// (64 contiguous bytes when N allows, else element by element up to N).
__device__ __forceinline__ void store_y32(const TcArgs& a, int m, int n, const uint32_t (&v)[32]) {
    if (m >= a.M) return;
    __half* yrow = a.y + (size_t)m * a.N;
    if (n + 32 <= a.N && (a.N & 7) == 0) {
        uint32_t h[16];
#pragma unroll
        for (int c = 0; c < 16; ++c) {
            __half2 p2 = __floats2half2_rn(__uint_as_float(v[2 * c]), __uint_as_float(v[2 * c + 1]));
            h[c] = *reinterpret_cast<uint32_t*>(&p2);
        }
        uint4* dst = reinterpret_cast<uint4*>(yrow + n);
#pragma unroll
        for (int c = 0; c < 4; ++c) dst[c] = make_uint4(h[4 * c], h[4 * c + 1], h[4 * c + 2], h[4 * c + 3]);
    } else {
#pragma unroll
        for (int c = 0; c < 32; ++c)
            if (n + c < a.N) yrow[n + c] = __float2half_rn(__uint_as_float(v[c]));
    }
}

// Byte offset of the 16-byte chunk `c` of row `r` in a 128-byte swizzled,
// K-major tile whose rows are 128 bytes (64 fp16) long.
__device__ __forceinline__ uint32_t swz128(int r, int c) {
    return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4));
}

// PAIR = false: one CTA computes a 128 x 128 tile of y with its own MMAs.
// PAIR = true: a cluster of two CTAs computes a (256 XT) (x rows) x 256
// (weight rows) tile with 2-CTA MMAs (tcgen05 cta_group::2): CTA r of the
// pair dequantises weight rows n0 + 128 r (its half of B) and stages XT x
// tiles, rows m0 + 256 t + 128 r (its half of A for MMA t); the even CTA
// issues XT MMAs per 16-wide k-step, which read both CTAs' shared memory and
// leave in each CTA's tensor memory its 128 rows of the 256 XT x 256 D
// (MMA t in columns 256 t ..).  Each SM reads (16 XT + 16) KB of operands per
// 64-wide k-block for 2 XT times the FLOPs of the single-CTA tile, and every
// stage hand-off covers XT times more MMA work.
// FMT = true: the format variants.  The dequantisers read each k-block's
// group scales and zero points from global memory (one k-block of their set
// ahead) and form fp16((nib - z) * s) from the exact difference nib - z.
// With an AWQ scale they multiply it into the weight tile as well,
// fp16(fp16((nib - z) * s) * alpha[k]): the product x * alpha * Wd with its
// rounding on the weight operand.  Scaling this CTA's x tiles in shared memory
// instead (the decode kernel's placement) re-scaled every x tile once per
// weight-block column and added half again to the shared-memory traffic of a
// k-block: 30 % slower at M = 512.
// TW: weight rows per CTA, 128 (a kernel-layout block) or, for CTA pairs with
// two x tiles, 96 (six 16-row tiles: a pair covers 192 weight rows with
// N = 192 MMAs, so N = 14336 fills 150 CTAs instead of 112).  A CTA's tiles
// are tiles TW x / 16 .. + TW / 16 - 1 of the layout, at most two contiguous
// runs of each 64-wide chunk (one per 128-row block they touch).
template <bool PAIR, int XT, bool FMT = false, int TW = kTileW>
__global__ void __launch_bounds__(kTcThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap smap,
                   const __grid_constant__ TcArgs a) {
    extern __shared__ uint8_t smem_raw[];
    // Swizzled tiles need 1024-byte alignment: align the window by hand.
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* smem = smem_raw + (base - raw);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kAbortFlag);

    static_assert(XT == 1 || (PAIR && XT == 2), "two x tiles per stage need CTA pairs");
    static_assert(TW == kTileW || (PAIR && XT == 2 && TW == 96), "96-row CTAs: pairs, two x tiles");
    constexpr int kAStg = TW * kBK * 2;   // dequantised weight tile of a stage
    constexpr int kWStg = TW * kBK / 2;   // packed weights of a stage
    constexpr int kTilesW = TW / 16;      // 16-row tiles of this CTA
    constexpr uint32_t kCols = PAIR ? 2 * TW * XT : TW;  // accumulator columns
    // tensor memory is allocated in powers of two
    constexpr uint32_t kAlloc = kCols <= 128 ? 128 : kCols <= 256 ? 256 : 512;
    constexpr int kXBytes = XT * kXStageBytes;                     // x bytes per stage
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // Cluster rank: CTA pairs are ranks (2 j, 2 j + 1); with split K the
    // cluster holds the pairs of all splits of one tile (split = rank / 2).
    const uint32_t crank = PAIR ? cluster_cta_rank() : 0u;
    const int rank = (int)(crank & 1u);
    const uint32_t lead = crank & ~1u;  // the pair's even CTA: issues its MMAs
    const bool leader = rank == 0;
    const uint16_t pair_mask = (uint16_t)(3u << lead);
    // This CTA's 128-row weight block and first x row; y columns start at n_out.
    const int r_start = (int)blockIdx.x * TW;  // first weight row of this CTA
    const int n_out = PAIR ? ((int)blockIdx.x >> 1) * 2 * TW : (int)blockIdx.x * TW;
    const int m0 = PAIR ? (int)blockIdx.y * 2 * kTileX * XT + rank * kTileX : (int)blockIdx.y * kTileX;
    const int NB = (a.N + kTileW - 1) / kTileW;
    const bool wvalid = r_start < a.N;  // the odd CTA of the last pair may hold no weights
    // its tiles in the layout (padded to NB blocks): run 1 = tiles wt0 .. wt0 + wn1 - 1
    // of block wb, run 2 = tiles 0 .. wn2 - 1 of block wb + 1
    const int wtile = r_start / 16;
    const int wvalid_tiles = wvalid ? min(kTilesW, NB * 8 - wtile) : 0;
    const int wb = wtile >> 3, wt0 = wtile & 7;
    const int wn1 = min(wvalid_tiles, 8 - wt0), wn2 = wvalid_tiles - wn1;
    // this CTA's k-blocks: kb0 .. kb0 + nkb - 1 (all of K unless split)
    const int kb0 = (int)(((long long)blockIdx.z * (a.K / kBK)) / a.splits);
    const int nkb = (int)((((long long)blockIdx.z + 1) * (a.K / kBK)) / a.splits) - kb0;
    const int slab_g0 = a.slab_tma ? ((kb0 >> 1) & ~7) : 0;  // first group held in the slab
    // The single-CTA tile always runs kSingleStages stages at fixed offsets
    // (compile-time constants there); pairs size their ring per launch.
    const int NS = PAIR ? a.nst : kSingleStages;
    const uint32_t kOffX = PAIR ? a.off_x : kOffA + kSingleStages * kAStg;
    const uint32_t kOffW = PAIR ? a.off_w : kOffX + kSingleStages * kXStageBytes;
    const uint32_t kOffSlab = PAIR ? a.off_slab : kOffW + kSingleStages * kWStg;

    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(base + kBarLoadFull + 8 * s, 1);
            // pair: one elected arrival per dequantising warp of a set in
            // both CTAs (the peer's are remote); single: every dequantiser
            mbar_init(base + kBarAFull + 8 * s, PAIR ? kDequantWarps : kDequantWarps / 2 * 32);
            mbar_init(base + kBarFree + 8 * s, 1);
        }
        mbar_init(base + kBarAcc, 1);
        mbar_init(base + kBarSlab, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        if (PAIR) {
            tmem_alloc_pair(base + kTmemSlot, kAlloc);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(base + kTmemSlot, kAlloc);
            tmem_relinquish();
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + kTmemSlot);
    // Pair: the peer's barriers must be initialised before the first remote
    // arrival or multicast commit.  Every thread arrives now and waits once,
    // before its first remote operation or at the end.
    bool cl_waited = !PAIR;
    if (PAIR) cluster_arrive();
    grid_launch_dependents();

    if (warp == 0) {
        // ============================ TMA producer ============================
        if (lane == 0) {
            tma_prefetch_map(&xmap);
            // chunk kb of block b starts at (b C + kb) 4 KB; tile t at + 512 t
            const size_t C = (size_t)(a.K / kBK);
            const uint8_t* w1 = a.wq + ((size_t)wb * C + kb0) * 4096 + (size_t)wt0 * 512;
            const uint8_t* w2 = a.wq + ((size_t)(wb + 1) * C + kb0) * 4096;
            // Weights and scales are constants of the call: the scale slab and
            // the first ring pass's packed weights load while the previous
            // kernel may still run; x (its output, possibly) after the wait.
            if (a.slab_tma) {  // this split's groups of the CTA's TW rows
                mbar_arrive_expect_tx(base + kBarSlab, (uint32_t)(TW * a.slab_ld * 2));
                tma_load_2d(base + kOffSlab, &smap, slab_g0, r_start, base + kBarSlab);
            } else {  // the CTA's scale slab (rows x G fp16, contiguous)
                const int rows = max(0, min(TW, a.N - r_start));
                const uint32_t bytes = (uint32_t)(rows * a.G * 2);
                const uint32_t bulk = bytes & ~15u;
                const __half* src = a.scales + (size_t)r_start * a.G;
                __half* dst = reinterpret_cast<__half*>(smem + kOffSlab);
                for (uint32_t e = bulk / 2; e < bytes / 2; ++e) dst[e] = src[e];
                mbar_arrive_expect_tx(base + kBarSlab, bulk);
                if (bulk) bulk_g2s(base + kOffSlab, src, bulk, base + kBarSlab);
            }
            const int first = NS < nkb ? NS : nkb;  // the first ring pass
            for (int i = 0; i < first; ++i) {
                mbar_arrive_expect_tx(base + kBarLoadFull + 8 * i,
                                      kXBytes + (uint32_t)wvalid_tiles * 512);
                if (wn1)
                    bulk_g2s(base + kOffW + i * kWStg, w1 + (size_t)i * 4096, (uint32_t)wn1 * 512,
                             base + kBarLoadFull + 8 * i);
                if (wn2)
                    bulk_g2s(base + kOffW + i * kWStg + (uint32_t)wn1 * 512, w2 + (size_t)i * 4096,
                             (uint32_t)wn2 * 512, base + kBarLoadFull + 8 * i);
            }
            grid_dependency_wait();
            for (int i = 0; i < first; ++i)
#pragma unroll
                for (int xt = 0; xt < XT; ++xt)
                    tma_load_2d(base + kOffX + i * kXBytes + xt * kXStageBytes, &xmap, (kb0 + i) * kBK,
                                m0 + xt * 2 * kTileX, base + kBarLoadFull + 8 * i);
            int issued = first;
            bool ok = true;
            for (int i = first, ts = first % NS, round = first / NS; i < nkb; ++i) {
                if (i >= NS &&
                    !mbar_wait(base + kBarFree + 8 * ts, (round - 1) & 1, a.timeout_ns,
                               a.status)) {
                    ok = false;
                    break;
                }
                if (*abort_flag) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(base + kBarLoadFull + 8 * ts,
                                      kXBytes + (uint32_t)wvalid_tiles * 512);
#pragma unroll
                for (int xt = 0; xt < XT; ++xt)
                    tma_load_2d(base + kOffX + ts * kXBytes + xt * kXStageBytes, &xmap, (kb0 + i) * kBK,
                                m0 + xt * 2 * kTileX, base + kBarLoadFull + 8 * ts);
                if (wn1)
                    bulk_g2s(base + kOffW + ts * kWStg, w1 + (size_t)i * 4096, (uint32_t)wn1 * 512,
                             base + kBarLoadFull + 8 * ts);
                if (wn2)
                    bulk_g2s(base + kOffW + ts * kWStg + (uint32_t)wn1 * 512, w2 + (size_t)i * 4096,
                             (uint32_t)wn2 * 512, base + kBarLoadFull + 8 * ts);
                issued = i + 1;
                if (++ts == NS) {
                    ts = 0;
                    ++round;
                }
            }
            if (!ok) *abort_flag = 1;
            // Drain the copies in flight before the block may exit.
            const uint64_t dt = drain_bound(a.timeout_ns);
            mbar_wait(base + kBarSlab, 0, dt, a.status);
            for (int i = (issued > NS ? issued - NS : 0); i < issued; ++i)
                mbar_wait(base + kBarLoadFull + 8 * (i % NS), (i / NS) & 1, dt, a.status);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ============================= MMA issuer =============================
        if (lane == 0 && leader) {
            // A = x rows (M), B = weight rows (N), both K-major.
            const uint32_t idesc = umma_idesc_f16_f32(PAIR ? 2 * kTileX : kTileX, PAIR ? 2 * TW : TW);
            bool ok = true;
            for (int i = 0, ts = 0, tr = 0; i < nkb; ++i) {
                // the dequantisers waited for the stage's copies: A full implies x landed
                const bool got = PAIR ? mbar_wait_cluster(base + kBarAFull + 8 * ts, tr & 1,
                                                          a.timeout_ns, a.status)
                                      : mbar_wait(base + kBarAFull + 8 * ts, tr & 1, a.timeout_ns,
                                                  a.status);
                if (!got) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t xa = base + kOffX + ts * kXBytes;
                const uint32_t wa = base + kOffA + ts * kAStg;
#pragma unroll
                for (int j = 0; j < kBK / 16; ++j) {
                    if (PAIR) {
#pragma unroll
                        for (int xt = 0; xt < XT; ++xt)
                            tc_mma_f16_pair(tmem + (uint32_t)(xt * 2 * TW),
                                            umma_desc_sw128(xa + xt * kXStageBytes + 32 * j),
                                            umma_desc_sw128(wa + 32 * j), idesc, (i | j) != 0);
                    } else
                        tc_mma_f16(tmem, umma_desc_sw128(xa + 32 * j), umma_desc_sw128(wa + 32 * j),
                                   idesc, (i | j) != 0);
                }
                // stage reusable (in both CTAs of a pair) once these MMAs finish
                if (PAIR)
                    tc_commit_pair_multicast(base + kBarFree + 8 * ts, pair_mask);
                else
                    tc_commit(base + kBarFree + 8 * ts);
                if (++ts == NS) {
                    ts = 0;
                    ++tr;
                }
            }
            // completes once every issued MMA has
            if (PAIR)
                tc_commit_pair_multicast(base + kBarAcc, pair_mask);
            else
                tc_commit(base + kBarAcc);
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
        // the stage barrier lives in the even CTA of a pair
        const uint32_t afull0 = PAIR ? map_to_cta(base + kBarAFull, lead) : base + kBarAFull;
        if (PAIR && !leader) {
            cluster_wait();
            cl_waited = true;
        }
        bool ok = mbar_wait(base + kBarSlab, 0, a.timeout_ns, a.status);
        // stage ts = i % NS and its pass parity, advanced by two k-blocks a step
        int ts = set % NS;
        uint32_t tph = (uint32_t)((set / NS) & 1);
        // FMT: coefficients of this set's k-blocks, loaded one k-block of the
        // set ahead (the dequantisers are rarely kept waiting on a stage, so a
        // load issued just before the wait would stall them)
        [[maybe_unused]] FmtCoef cf;
        if constexpr (FMT) {
            if (set < nkb) cf = fmt_coef(a, kb0 + set, r_start + r0, tq);
        }
        for (int i = set; ok && i < nkb; i += 2) {
            [[maybe_unused]] FmtCoef nx;
            if constexpr (FMT) {
                if (i + 2 < nkb) nx = fmt_coef(a, kb0 + i + 2, r_start + r0, tq);
            }
            // The stage's copies were issued after its previous MMAs finished,
            // so their arrival also means the dequantised slot is free.
            if (!mbar_wait(base + kBarLoadFull + 8 * ts, tph, a.timeout_ns, a.status)) {
                ok = false;
                break;
            }
            if (wvalid && dw < kTilesW) {
                const uint32_t wst = base + kOffW + ts * kWStg;
                const uint32_t ast = base + kOffA + ts * kAStg;
                const uint4 pk = lds128(wst + (dw * 32 + lane) * 16);
                __half2 s0, s1;
                [[maybe_unused]] __half2 lo_off, hi_off;  // 1024 + z0, -(64 + z1): exact
                if constexpr (FMT) {
                    s0 = __half2half2(cf.s0);
                    s1 = __half2half2(cf.s1);
                    lo_off = __half2half2(__int2half_rn(1024 + cf.z0));
                    hi_off = __half2half2(__int2half_rn(-64 - cf.z1));
                } else {
                    const int grp = (kb0 + i) >> 1;  // two 64-wide k-blocks per scale group
                    s0 = __half2half2(slab[r0 * a.slab_ld + grp - slab_g0]);
                    s1 = __half2half2(slab[r1 * a.slab_ld + grp - slab_g0]);
                }
                const uint32_t wrd[4] = {pk.x, pk.y, pk.z, pk.w};
                uint32_t o0[8], o1[8];  // rows r0 / r1, k = 16 tq .. 16 tq + 15
#pragma unroll
                for (int ws = 0; ws < 4; ++ws) {
                    uint32_t af[4];
                    if constexpr (FMT)
                        dequant8_z(wrd[ws], lo_off, hi_off, af);
                    else
                        dequant8(wrd[ws], af);
                    o0[2 * ws] = hmul2_u32(af[0], s0);
                    o0[2 * ws + 1] = hmul2_u32(af[2], s0);
                    o1[2 * ws] = hmul2_u32(af[1], s1);
                    o1[2 * ws + 1] = hmul2_u32(af[3], s1);
                }
                if constexpr (FMT) {
                    if (a.alpha) {
                        // AWQ: o[j] holds k = 16 tq + 2 j, + 1 of rows r0 / r1;
                        // fp16(Wd * alpha), alpha on the weight operand
                        const uint32_t alw[8] = {cf.al0.x, cf.al0.y, cf.al0.z, cf.al0.w,
                                                 cf.al1.x, cf.al1.y, cf.al1.z, cf.al1.w};
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            const __half2 aj = *reinterpret_cast<const __half2*>(&alw[j]);
                            o0[j] = hmul2_u32(o0[j], aj);
                            o1[j] = hmul2_u32(o1[j], aj);
                        }
                    }
                }
                sts128(ast + swz128(r0, 2 * tq), o0[0], o0[1], o0[2], o0[3]);
                sts128(ast + swz128(r0, 2 * tq + 1), o0[4], o0[5], o0[6], o0[7]);
                sts128(ast + swz128(r1, 2 * tq), o1[0], o1[1], o1[2], o1[3]);
                sts128(ast + swz128(r1, 2 * tq + 1), o1[4], o1[5], o1[6], o1[7]);
                fence_proxy_async_smem();  // generic stores -> visible to the tensor core
            }
            if (PAIR) {
                __syncwarp();
                if (lane == 0) {
                    if (leader)
                        mbar_arrive(base + kBarAFull + 8 * ts);
                    else
                        mbar_arrive_remote(afull0 + 8 * ts);
                }
            } else {
                mbar_arrive(base + kBarAFull + 8 * ts);
            }
            if constexpr (FMT) cf = nx;
            ts += 2;
            if (ts >= NS) {
                ts -= NS;
                tph ^= 1u;
            }
        }
        if (!ok) *abort_flag = 1;

        // ------------------------------ epilogue ------------------------------
        const bool acc_ok = mbar_wait(base + kBarAcc, 0, a.timeout_ns, a.status);
        if (acc_ok) tc_fence_after_sync();
        const int q = warp & 3;           // TMEM lane quarter = rows of y
        const int cc = (warp - 4) >> 2;   // column chunk = weight rows
        constexpr int kChunkCols = (int)kCols / 4;  // 32 (single), 64, 128 or 96 (pair)
        const int row = q * 32 + lane;    // accumulator row (TMEM lane)
        if (a.splits == 1) {  // split K: reduced over the cluster below
            if (acc_ok) {
#pragma unroll
                for (int half = 0; half < kChunkCols / 32; ++half) {
                    const int col = cc * kChunkCols + half * 32;
                    // pair: columns 256 t .. belong to MMA t, i.e. x rows m0 + 256 t
                    const int xt = PAIR ? col / (2 * TW) : 0;
                    uint32_t v[32];
                    tmem_ld_32x32b_x32(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)col, v);
                    tmem_ld_wait();
                    store_y32(a, m0 + xt * 2 * kTileX + row, n_out + (PAIR ? col % (2 * TW) : col),
                              v);
                }
            }
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    if (PAIR) {
        if (!cl_waited) cluster_wait();
        if (a.splits > 1) {
            // Split-K reduction over the cluster.  Split z owns columns
            // [z part, (z + 1) part) of the tile; in rounds of 64 columns every
            // CTA pushes its partial of each split's columns (its own
            // included) into slot z of that split's ring memory (free now:
            // all MMAs of the cluster are done), and each owner sums its S
            // slots in split order and writes y.  Every thread joins the
            // cluster barriers; warps 4..19 move the data, each reading only
            // its own TMEM lane quarter.
            tc_fence_after_sync();
            const int S = a.splits, z = (int)blockIdx.z;
            // owner z: columns [z part, min((z + 1) part, kCols)), part a
            // multiple of 64 (S = 3 owns 192 / 192 / 128 of 512)
            const int part = (((int)kCols / S + 63) / 64) * 64;
            float* recv = reinterpret_cast<float*>(smem + kOffA);
            const uint32_t recv_u32 = base + kOffA;
            const int q = warp & 3, wq = (warp - 4) >> 2;  // quarter; warp index within it
            const int row = q * 32 + lane;
#pragma unroll 1
            for (int r = 0; r < part / 64; ++r) {
                cluster_sync_all();  // mainloops done / previous round's slices read
                if (warp >= 4) {
#pragma unroll 1
                    for (int task = wq; task < 2 * S; task += 4) {
                        const int d = task >> 1, c = task & 1;  // destination split, 32-column half
                        const int col = d * part + r * 64 + c * 32;
                        if (col >= (int)kCols) continue;  // d owns fewer rounds
                        uint32_t v[32];
                        tmem_ld_32x32b_x32(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)col, v);
                        tmem_ld_wait();
                        const uint32_t dst = map_to_cta(
                            recv_u32 + (uint32_t)((z * kRedSlotFloats + row * kRedRow + c * 32) * 4),
                            (uint32_t)(2 * d + rank));
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            st_cluster_v4(dst + 16 * e, v[4 * e], v[4 * e + 1], v[4 * e + 2], v[4 * e + 3]);
                    }
                }
                cluster_sync_all();  // every slice of this round has landed
                if (warp >= 4 && wq < 2 && z * part + r * 64 + wq * 32 < (int)kCols) {
                    const int col = z * part + r * 64 + wq * 32;
                    float sum[32];
#pragma unroll
                    for (int e = 0; e < 32; ++e) sum[e] = 0.0f;
#pragma unroll 1
                    for (int zz = 0; zz < S; ++zz) {
                        const float4* src = reinterpret_cast<const float4*>(
                            recv + zz * kRedSlotFloats + row * kRedRow + wq * 32);
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            const float4 f = src[e];
                            sum[4 * e] += f.x;
                            sum[4 * e + 1] += f.y;
                            sum[4 * e + 2] += f.z;
                            sum[4 * e + 3] += f.w;
                        }
                    }
                    uint32_t v[32];
#pragma unroll
                    for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(sum[e]);
                    const int xt = col / (2 * TW);
                    store_y32(a, m0 + xt * 2 * kTileX + row, n_out + col % (2 * TW), v);
                }
            }
            tc_fence_before_sync();
        }
        // Neither CTA frees its tensor memory or leaves while the pair's
        // MMAs, the peer's arrivals or the cluster's pushes may still touch it.
        cluster_sync_all();
    }
    if (warp == 1) {
        tc_fence_after_sync();
        if (PAIR)
            tmem_dealloc_pair(tmem, kAlloc);
        else
            tmem_dealloc(tmem, kAlloc);
    }
}

// Launch shape of the tensor-core GEMM for (M, N):
//  * xt = 2: CTA pairs with two x tiles per CTA, 512 x rows x 256 weight rows
//    per pair -- the most MMA work per stage hand-off -- when M > 256 and the
//    pairs still occupy at least half of the SMs;
//  * xt = 1: CTA pairs with 256 x 256 tiles when M > 128 and they cover
//    every SM;
//  * otherwise one CTA per 128 x 128 tile (cluster 1).
struct TcPlan {
    int cluster = 1, xt = 1, splits = 1;
    int tw = kTileW;  // weight rows per CTA: 128, or 96 for pairs with two x tiles
    int slab_ld = 0;  // > 0: split slab of this many groups per row (tensor-map copy)
    unsigned gx = 0, gy = 0;
    long long ctas = 0;
};

int max_active_clusters(const void* fn, int cluster_z, uint32_t smem) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2, 1, (unsigned)cluster_z);
    cfg.blockDim = dim3(kTcThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = 2;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = (unsigned)cluster_z;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess) return 0;
    return n;
}

// Shared memory of a launch: `nst` ring stages with xt x tiles each, next to
// a scale slab of `ld` groups per row, +1 KB slack for aligning the window to
// 1024 bytes.
uint32_t tc_smem(int nst, int xt, int ld, int tw = kTileW) {
    const uint32_t slab = ((tw * ld * 2 + 127) / 128) * 128;
    const uint32_t stage = (uint32_t)(tw * kBK * 2 + xt * kXStageBytes + tw * kBK / 2);
    return kOffA + (uint32_t)nst * stage + slab + 1024;
}

// Groups per slab row when K is split S ways: the widest span from a
// split's first group rounded down to 8 to its last group, rounded up to 8
// (the tensor-map copy needs 16-byte rows and a 16-byte aligned start).
// 0 when G is not a multiple of 8 or the span exceeds a copy's 256 limit.
int split_slab_ld(long long nkb, int S, int G) {
    if (G % 8 != 0) return 0;
    int w = 0;
    for (int z = 0; z < S; ++z) {
        const long long kb0 = z * nkb / S, kb1 = (z + 1) * nkb / S;
        const int g0 = (int)(kb0 >> 1) & ~7, g1 = (int)((kb1 - 1) >> 1);
        w = std::max(w, ((g1 - g0 + 1 + 7) / 8) * 8);
    }
    return w <= 256 ? w : 0;
}

// Pairs take as many ring stages as fit: a deeper ring hides more of the
// copy -> dequantise -> MMA -> release round trip.  The single-CTA tile keeps
// kSingleStages (deeper measured slower there).
int tc_stages(const TcPlan& p, int ld, const DeviceCtx& ctx) {
    if (p.cluster == 1) return kSingleStages;
    int nst = kMaxStages;
    while (nst > 2 && tc_smem(nst, p.xt, ld, p.tw) > (uint32_t)ctx.max_smem_optin) --nst;
    return nst;
}

// Launch shape of the tensor-core GEMM for (M, N, K), the cheapest of:
//  * one CTA per 128 x 128 tile (cluster 1);
//  * CTA pairs with 256 x 256 tiles (xt = 1, cluster 2), M > 128;
//  * CTA pairs with 512 x-row x 256 weight-row tiles (xt = 2), M > 256 --
//    the most MMA work per stage hand-off;
//  * the latter splitting K two to four ways (every k-range >= 8 k-blocks),
//    the splits of a tile forming one cluster (4, 6 or 8 CTAs) that reduces
//    through distributed shared memory; only when the whole grid is
//    co-resident.
// Cost = waves x k-blocks per CTA x the measured time of one k-block of the
// tile on a busy GPU (about 0.36, 0.63 and 0.84 us at M = 512), plus about a
// microsecond per 64-column round of a split reduction.  fmt: the format
// variants' kernels, which hold no scale slab.
TcPlan tc_plan(int64_t M, int64_t N, int64_t K, const DeviceCtx& ctx, bool fmt = false) {
    constexpr double kSingleKb = 0.36, kPairKb = 0.63, kPair2Kb = 0.84, kPair2Kb96 = 0.66,
                     kRound = 1.0;
    const int NB = (int)((N + kTileW - 1) / kTileW);
    const long long pairs = (NB + 1) / 2;
    const long long nkb = K / kBK;
    const int G = fmt ? 0 : (int)(K / kGroup);
    auto waves = [&](long long ctas) { return (double)((ctas + ctx.num_sms - 1) / ctx.num_sms); };

    TcPlan best;  // single-CTA tiles
    best.gx = (unsigned)NB;
    best.gy = (unsigned)((M + kTileX - 1) / kTileX);
    best.ctas = (long long)best.gx * best.gy;
    double t_best = waves(best.ctas) * nkb * kSingleKb;
    if (NB < 2) return best;

    if (M > kTileX) {
        TcPlan p;
        p.cluster = 2;
        p.gx = (unsigned)(2 * pairs);
        p.gy = (unsigned)((M + 2 * kTileX - 1) / (2 * kTileX));
        p.ctas = (long long)p.gx * p.gy;
        const double t = waves(p.ctas) * nkb * kPairKb;
        if (t < t_best) {
            t_best = t;
            best = p;
        }
    }
    // CTA pairs with two x tiles, 128 or 96 weight rows per CTA (one kernel-
    // layout block, or six of its 16-row tiles: 192 rows per pair, which
    // spreads N = 14336 over 150 CTAs instead of 112), each optionally
    // splitting K.
    for (int tw : {kTileW, 96}) {
        if (M <= 2 * kTileX) break;
        const double per_kb = tw == kTileW ? kPair2Kb : kPair2Kb96;
        TcPlan p;
        p.cluster = 2;
        p.xt = 2;
        p.tw = tw;
        const long long tiles = (N + tw - 1) / tw;
        const long long tw_pairs = (tiles + 1) / 2;
        p.gx = (unsigned)(2 * tw_pairs);
        p.gy = (unsigned)((M + 4 * kTileX - 1) / (4 * kTileX));
        p.ctas = (long long)p.gx * p.gy;
        double t = waves(p.ctas) * nkb * per_kb * (tc_stages(p, G, ctx) >= 4 ? 1.0 : 1.25);
        if (t < t_best) {
            t_best = t;
            best = p;
        }
        for (int S = 2; S <= 4; ++S) {
            const long long ctas = p.ctas * S;
            if (ctas > ctx.num_sms || nkb < 8 * S) continue;
            // a split holds only its own groups' scales, leaving room for a
            // deeper ring (3 stages run a k-block about 25 % slower than 4)
            const int ld = fmt ? 0 : split_slab_ld(nkb, S, G);
            const int nst = tc_stages(p, ld ? ld : G, ctx);
            const uint32_t smem = tc_smem(nst, 2, ld ? ld : G, tw);
            const uint32_t ring = (uint32_t)nst * (tw * kBK * 2 + 2 * kXStageBytes + tw * kBK / 2);
            // the S receive slots of the reduction live in the ring
            if ((uint32_t)S * kRedSlotFloats * 4 > ring) continue;
            const void* fn = tw == kTileW ? (fmt ? (const void*)gemm_tc_kernel<true, 2, true>
                                                 : (const void*)gemm_tc_kernel<true, 2>)
                                          : (fmt ? (const void*)gemm_tc_kernel<true, 2, true, 96>
                                                 : (const void*)gemm_tc_kernel<true, 2, false, 96>);
            const long long fit = (long long)max_active_clusters(fn, S, smem);
            if (fit * 2 * S < ctas) continue;  // not one co-resident wave
            t = (double)((nkb + S - 1) / S) * per_kb * (nst >= 4 ? 1.0 : 1.25) +
                kRound * ((4 * tw / S + 63) / 64 + 1);
            if (t < t_best) {
                t_best = t;
                best = p;
                best.splits = S;
                best.cluster = 2 * S;
                best.ctas = ctas;
                best.slab_ld = ld;
            }
        }
    }
    return best;
}

cudaError_t ensure_tc_attrs(const DeviceCtx& ctx) {
    static std::atomic<bool> attr_done[64];  // per device; racing callers only repeat the set-up
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && attr_done[dev].load(std::memory_order_acquire)) return cudaSuccess;
    for (auto fn : {gemm_tc_kernel<false, 1>, gemm_tc_kernel<true, 1>, gemm_tc_kernel<true, 2>,
                    gemm_tc_kernel<false, 1, true>, gemm_tc_kernel<true, 1, true>,
                    gemm_tc_kernel<true, 2, true>, gemm_tc_kernel<true, 2, false, 96>,
                    gemm_tc_kernel<true, 2, true, 96>}) {
        cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             ctx.max_smem_optin);
        if (e != cudaSuccess) return e;
    }
    if (dev >= 0 && dev < 64) attr_done[dev].store(true, std::memory_order_release);
    return cudaSuccess;
}

}  // namespace

void gemm_tc_plan_info(int64_t M, int64_t N, int64_t K, const DeviceCtx& ctx, int* cluster,
                       int* ctas, bool fmt, int* rows_per_cta) {
    if (ensure_tc_attrs(ctx) != cudaSuccess) {
        *cluster = 0;
        *ctas = 0;
        return;
    }
    const TcPlan p = tc_plan(M, N, K, ctx, fmt);
    *cluster = p.cluster;
    *ctas = (int)p.ctas;
    if (rows_per_cta) *rows_per_cta = p.tw;
}

namespace {

// Encodes the maps, sizes the ring and launches the plan's kernel; `a`
// carries the operands (and the format fields when FMT).
template <bool FMT>
cudaError_t launch_tc(TcArgs a, const void* x, int64_t M, int64_t N, int64_t K, cudaStream_t stream,
                      const DeviceCtx& ctx) {
    const int G = FMT ? 0 : (int)(K / kGroup);
    cudaError_t e = ensure_tc_attrs(ctx);
    if (e != cudaSuccess) return e;
    const TcPlan plan = tc_plan(M, N, K, ctx, FMT);
    const int ld = plan.slab_ld ? plan.slab_ld : G;
    const int nst = tc_stages(plan, ld, ctx);
    const uint32_t smem = tc_smem(nst, plan.xt, ld, plan.tw);
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
    CUtensorMap smap = map;  // unused unless the slab is copied per split
    if (plan.slab_ld) {
        const cuuint64_t sdims[2] = {(cuuint64_t)G, (cuuint64_t)N};
        const cuuint64_t sstrides[1] = {(cuuint64_t)G * 2};
        const cuuint32_t sbox[2] = {(cuuint32_t)plan.slab_ld, (cuuint32_t)plan.tw};
        if (encode(&smap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<__half*>(a.scales), sdims,
                   sstrides, sbox, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }

    a.status = ctx.status;
    a.timeout_ns = ctx.timeout_ns;
    a.M = (int)M;
    a.N = (int)N;
    a.K = (int)K;
    a.G = G;
    a.nst = nst;
    a.off_x = kOffA + (uint32_t)nst * (uint32_t)(plan.tw * kBK * 2);
    a.off_w = a.off_x + (uint32_t)nst * plan.xt * kXStageBytes;
    a.off_slab = a.off_w + (uint32_t)nst * (uint32_t)(plan.tw * kBK / 2);
    a.splits = plan.splits;
    a.slab_ld = ld;
    a.slab_tma = plan.slab_ld ? 1 : 0;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(plan.gx, plan.gy, (unsigned)plan.splits);
    cfg.blockDim = dim3(kTcThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attrs[2];
    attrs[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[0].val.programmaticStreamSerializationAllowed = 1;
    attrs[1].id = cudaLaunchAttributeClusterDimension;
    attrs[1].val.clusterDim.x = 2;
    attrs[1].val.clusterDim.y = 1;
    attrs[1].val.clusterDim.z = (unsigned)plan.splits;
    cfg.attrs = attrs;
    cfg.numAttrs = plan.cluster > 1 ? 2 : 1;
    if (plan.cluster == 1) return cudaLaunchKernelEx(&cfg, gemm_tc_kernel<false, 1, FMT>, map, smap, a);
    if (plan.xt == 1) return cudaLaunchKernelEx(&cfg, gemm_tc_kernel<true, 1, FMT>, map, smap, a);
    if (plan.tw == 96) return cudaLaunchKernelEx(&cfg, gemm_tc_kernel<true, 2, FMT, 96>, map, smap, a);
    return cudaLaunchKernelEx(&cfg, gemm_tc_kernel<true, 2, FMT>, map, smap, a);
}

}  // namespace

cudaError_t launch_gemm_tc(const void* x, const void* repacked, const void* scales, void* y,
                           int64_t M, int64_t N, int64_t K, cudaStream_t stream,
                           const DeviceCtx& ctx) {
    TcArgs a{};
    a.wq = static_cast<const uint8_t*>(repacked);
    a.scales = static_cast<const __half*>(scales);
    a.y = static_cast<__half*>(y);
    return launch_tc<false>(a, x, M, N, K, stream, ctx);
}

cudaError_t launch_gemm_tc_fmt(const void* x, const void* alpha, const void* repacked,
                               const void* scales, const void* zeros, void* y, int64_t M, int64_t N,
                               int64_t K, int group, cudaStream_t stream, const DeviceCtx& ctx) {
    if (!(group == 32 || group == 64 || group == 128 || group == K)) return cudaErrorInvalidValue;
    TcArgs a{};
    a.wq = static_cast<const uint8_t*>(repacked);
    a.scales = static_cast<const __half*>(scales);
    a.y = static_cast<__half*>(y);
    a.zeros = static_cast<const uint8_t*>(zeros);
    a.alpha = static_cast<const __half*>(alpha);
    a.gshift = group == K ? 31 : (group == 32 ? 5 : group == 64 ? 6 : 7);
    a.gcount = (int)(K / group);
    return launch_tc<true>(a, x, M, N, K, stream, ctx);
}

}  // namespace w4a16
