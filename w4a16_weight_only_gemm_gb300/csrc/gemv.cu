// gemv.cu -- W4A16 decode GEMV / skinny GEMM for M = 1..16.
//
// y[m, n] = sum_k x[m, k] * (nib[n, k] - 8) * scale[n, k / 128]
// (mhpq.cn W4A16 report §二/§五: the packed weights stay packed in memory and
// are unpacked in registers; the qaqbuyan.com tutorial §3 dequantizer fixes
// the arithmetic).
//
// One thread block = 8 consumer warps + 1 producer warp.  A CTA computes
// either whole 128-row blocks of the kernel layout (one 16-row tile per
// warp) or a sub-block unit of T = 1, 2 or 4 tiles over the whole K range,
// the 8 / T warps of a tile sharing out the groups of every stage.
//  * The producer streams weights into a ring of 16 KB shared-memory stages
//    with async copies (TMA engine) that complete on mbarriers, L2 policy
//    evict-first: a whole block's 64-wide chunks are 4 KB contiguous (one
//    bulk copy per stage); a unit's T tiles of 32 / T consecutive chunks are
//    one tensor-map box.  The fp16 scale slab of the CTA's rows (contiguous
//    in the canonical layout) arrives the same way into one of two buffers,
//    and the x slice of the CTA's K range once per thread block -- or, for
//    whole blocks with M > 4, each stage's 4 chunks of x for all M rows in
//    the stage itself (one swizzled tensor-map box), so that the CTA's
//    shared memory no longer grows with M x K.
//  * Consumers: per 64-wide chunk a lane reads 16 bytes of its tile, turns
//    each 32-bit word into an mma.m16n8k16 A fragment of exact codes
//    q = n - 8 in fp16 (one lop3 per nibble pair OR-ing it into the mantissa
//    of 1024.0, then one subtraction or fma per register), and multiplies it
//    with x fragments read from shared memory.  M <= 8 uses one n8 MMA per
//    16 k, M <= 16 two.  Every 128-wide group accumulates in fresh FP32
//    fragments and is scaled once by its fp16 scale: the products are exact
//    and only FP32 sums round.  Persistent launches and long units with
//    M <= 4 feed the unbiased codes n instead, as fp16 subnormals that the
//    masks alone produce (n 2^-24, n 2^-20), and take the zero point off in
//    the FP32 rescale with per-group x sums computed once per CTA: 5 instead
//    of 9 instructions per 8 weights, products still exact.
//  * Work split, chosen per shape by a launch-time model: sub-block units
//    (the warps of a tile add their partial sums in shared memory, in a
//    fixed order); or whole blocks with the K range split over the S CTAs of
//    a thread-block cluster (up to 8), each CTA pushing its FP32 partials
//    into the shared memory of the CTA that owns the row (distributed shared
//    memory) and the owner summing them in a fixed order one cluster barrier
//    later (no global workspace, no atomics); or, with more blocks than CTA
//    slots, a persistent grid where each CTA walks blocks y, y + gridDim.y,
//    ... while the producer keeps the ring full across block boundaries.
//  * Programmatic dependent launch: the CTA releases its dependents at once
//    and loads its first ring stages and scale slab -- constants of the call
//    -- while the previous kernel on the stream is still running; x (which
//    that kernel may produce) is copied, and y written, only after the
//    grid-dependency wait.
// Every wait is bounded (common.cuh); on a time-out the CTA records it in the
// status word, stops issuing copies, drains those in flight and exits.
#include <atomic>
#include <mutex>
#include <utility>
#include <vector>

#include "common.cuh"
#include "kernels.h"

namespace w4a16 {
namespace {

constexpr int kConsumerWarps = 8;                      // 8 x 16 rows = one block
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kGemvThreads = kConsumers + 32;
constexpr int kTileBytes = 16 * kChunkK / 2;           // 512 B: one 16-row tile, one chunk
constexpr int kChunkBytes = kBlockRows * kChunkK / 2;  // 4096 B per block-chunk
constexpr int kStages = 3;                             // ring depth of non-persistent launches
constexpr int kMaxStages = 6;                          // deepest ring (persistent launches)
constexpr int kStageBytes = 16384;                     // every ring stage
constexpr int kGroupsPerWarpStage = 2;                 // groups a warp takes from one stage
constexpr int kMaxSplits = 8;

// Barrier area at the start of shared memory.
constexpr int kBarFull = 0;                    // [kMaxStages]
constexpr int kBarEmpty = kBarFull + 8 * kMaxStages;
constexpr int kBarX = kBarEmpty + 8 * kMaxStages;
constexpr int kBarSFull = kBarX + 8;           // [2]
constexpr int kBarSEmpty = kBarSFull + 16;     // [2]
constexpr int kAbortFlag = kBarSEmpty + 16;
constexpr int kBarAreaBytes = 1024;

struct GemvArgs {
    const uint8_t* wq;       // kernel-layout weights
    const __half* scales;    // [N, G]
    const __half* x;         // [M, K]
    __half* y;               // [M, N]
    unsigned* status;
    uint64_t timeout_ns;
    int M, N, K, G;
    int NB;                  // 128-row blocks
    int T;                   // 16-row tiles per CTA: 8 = whole blocks; 1, 2, 4 = sub-block units
    int xs_stride;           // bytes between x rows in shared memory
    int slab_bytes;          // bytes of one scale buffer (16 T rows x G, rounded)
    int n_sbuf;              // scale buffers: 2 when a CTA walks several blocks, else 1
    int nstages;             // ring stages (<= kMaxStages)
    int rpo;                 // rows owned per CTA in the split reduction
    // Launch constants computed on the host, so that a CTA's producer gets
    // to its first copy with few instructions (it shares the SM's issue slots
    // with the previous kernel's CTAs): for units, chunks and groups per
    // stage, warps per tile and stages per unit; for persistent launches the
    // blocks per CTA (nb_q, plus one on the first nb_r CTAs); for a K split
    // the first group of every split (g0s[S] = G).
    int cps, gps, wpt, nstg_u;
    int nb_q, nb_r;
    int g0s[kMaxSplits + 1];
    // Persistent whole-block launches whose last round is partial: the
    // blocks from tail_base on run as tail_units sub-block units of tail_T
    // tiles (tail_T = 0: no tail), unit u on CTA u after its whole blocks.
    int tail_T, tail_base, tail_units;
    // Whole-block launches with M > 4 stream x through the ring: every stage
    // holds, after its 16 KB of weights, the stage's 4 chunks of x for all M
    // rows (one 3-D tensor-map box, 128-byte swizzled, 1024-aligned inside
    // xs_stage bytes); xs_stage = 0: x is one CTA-wide slice instead.
    int xs_stage;
    int stage_stride;        // bytes between ring stages (16 KB + xs_stage)
    // off_sx: the x sums of the subnormal-code decode, [group][16] floats
    uint32_t off_ring, off_x, off_s, off_red, off_sx;
};

__device__ __forceinline__ uint32_t align1024(uint32_t a) { return (a + 1023u) & ~1023u; }

// The first group of split `split` of S over G groups (host side).
inline int split_group_begin(int split, int S, int G) { return (split * G) / S; }

// One 128-wide group (two chunks) of one consumer lane: 8 MMAs into fresh
// FP32 fragments, then scaled into acc.  The A fragments hold the exact codes
// q = n - 8 in fp16 (dequant8), so every product q * x is exact and the FP32
// sums carry only the group's own dot product.  (Feeding 64 + n and removing
// 64 * sum(x) afterwards is cheaper by 4 instructions per 8 weights, but the
// MMA adds its products at the precision of the running sum: activations with
// a large common offset make that sum ~64 sum(x) and lose the dot product's
// low bits, beyond the accuracy bar for x = 4 + N(0, 1).)
// x addresses: xa[c][h] the h-th 16 bytes of this lane's activations (row
// min(g, M - 1)) in chunk c of the group, xb[c][h] the same for row
// min(g + 8, M - 1) (read only when M > 8).
struct XAddr {
    uint32_t a[2][2], b[2][2];
};

// The x of a CTA-wide slice: rows xs_stride bytes apart, chunks 128 bytes.
__device__ __forceinline__ XAddr x_slice(uint32_t x0_addr, uint32_t x1_addr) {
    XAddr x;
#pragma unroll
    for (int c = 0; c < 2; ++c)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            x.a[c][h] = x0_addr + c * 128 + h * 16;
            x.b[c][h] = x1_addr + c * 128 + h * 16;
        }
    return x;
}

// x in a ring stage (whole-block launches with M > 4): the stage's box is
// [4 chunks][M rows][128 bytes], the 16-byte unit u of 128-byte row q stored
// at unit u ^ (q & 7); rows r0 / r1 of chunks cc0, cc0 + 1.
__device__ __forceinline__ XAddr x_stage(uint32_t xbase, int M, int cc0, int r0, int r1, int t) {
    XAddr x;
#pragma unroll
    for (int c = 0; c < 2; ++c) {
        const int q0 = (cc0 + c) * M + r0, q1 = (cc0 + c) * M + r1;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            x.a[c][h] = xbase + (uint32_t)q0 * 128u + ((uint32_t)((2 * t + h) ^ (q0 & 7)) << 4);
            x.b[c][h] = xbase + (uint32_t)q1 * 128u + ((uint32_t)((2 * t + h) ^ (q1 & 7)) << 4);
        }
    }
    return x;
}

// SUB: the A fragments hold the unbiased codes n as fp16 subnormals
// (dequant8_subnormal, no arithmetic): the MMAs give 2^-24 sum(n x) for rows
// r0 and 2^-20 sum(n x) for rows r1, and the rescale takes off 8 sum(x) with
// the group's x sums (sx_addr: this lane's columns 2t, 2t + 1, FP32).  The
// MMA's running sums then reach ~sum(n x) rather than the result, within a
// small factor of it for offset activations (the bias of 64 + n was not).
template <int MT, bool SUB = false>
__device__ __forceinline__ void mma_group(uint32_t w_addr, uint32_t cs, const XAddr& xad, float s0,
                                          float s1, uint32_t sx_addr, float (&acc)[MT][4]) {
    // M <= 8: one FP32 fragment per chunk -- two independent MMA chains per
    // group halve the dependent-latency path of a lane (M <= 16 has two
    // chains already, one per n8 tile, and no registers to spare).
    constexpr int NCH = MT == 1 ? 2 : 1;
    float g[NCH][MT][4];
#pragma unroll
    for (int c = 0; c < NCH; ++c)
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int e = 0; e < 4; ++e) g[c][mt][e] = 0.0f;
#pragma unroll
    for (int c = 0; c < 2; ++c) {
        const uint4 wv = lds128(w_addr + c * cs);
        const uint4 xa = lds128(xad.a[c][0]);
        const uint4 xb = lds128(xad.a[c][1]);
        uint4 xa1 = xa, xb1 = xb;
        if (MT == 2) {
            xa1 = lds128(xad.b[c][0]);
            xb1 = lds128(xad.b[c][1]);
        }
        const uint32_t wrd[4] = {wv.x, wv.y, wv.z, wv.w};
        const uint32_t b0[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
        const uint32_t b1[8] = {xa1.x, xa1.y, xa1.z, xa1.w, xb1.x, xb1.y, xb1.z, xb1.w};
#pragma unroll
        for (int s = 0; s < 4; ++s) {
            uint32_t af[4];
            if (SUB)
                dequant8_subnormal(wrd[s], af);
            else
                dequant8(wrd[s], af);
            mma_16816(g[c % NCH][0], af, b0[2 * s], b0[2 * s + 1], g[c % NCH][0]);
            if (MT == 2)
                mma_16816(g[c % NCH][MT - 1], af, b1[2 * s], b1[2 * s + 1], g[c % NCH][MT - 1]);
        }
    }
    // The rescale runs on (column 2t, 2t + 1) pairs through the packed binary32
    // instructions; each component rounds as the scalar fma.
    // SUB: s (2^24 or 2^20) G - 8 s Sx, in two fmas.
    const float f0 = SUB ? 16777216.0f * s0 : s0, f1 = SUB ? 1048576.0f * s1 : s1;
    const float2 s00 = make_float2(f0, f0), s11 = make_float2(f1, f1);
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
        float2 v01 = make_float2(g[0][mt][0], g[0][mt][1]);
        float2 v23 = make_float2(g[0][mt][2], g[0][mt][3]);
        if (NCH == 2) {
            v01 = __fadd2_rn(v01, make_float2(g[NCH - 1][mt][0], g[NCH - 1][mt][1]));
            v23 = __fadd2_rn(v23, make_float2(g[NCH - 1][mt][2], g[NCH - 1][mt][3]));
        }
        float2 c01 = make_float2(acc[mt][0], acc[mt][1]);
        float2 c23 = make_float2(acc[mt][2], acc[mt][3]);
        if (SUB) {
            const float2 sx = lds64f(sx_addr + mt * 32);
            c01 = __ffma2_rn(make_float2(-8.0f * s0, -8.0f * s0), sx, c01);
            c23 = __ffma2_rn(make_float2(-8.0f * s1, -8.0f * s1), sx, c23);
        }
        const float2 a01 = __ffma2_rn(s00, v01, c01);
        const float2 a23 = __ffma2_rn(s11, v23, c23);
        acc[mt][0] = a01.x;
        acc[mt][1] = a01.y;
        acc[mt][2] = a23.x;
        acc[mt][3] = a23.y;
    }
}

// Stores the FP32 results of a lane's fragments (rows R0, R1; columns
// 2t, 2t + 1 of each n8 tile) as fp16.
template <int MT>
__device__ __forceinline__ void store_y(const GemvArgs& a, int R0, int R1, int t,
                                        const float (&acc)[MT][4]) {
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

// The consumer side of a sub-block unit of T tiles over the K range of the
// CTA: a stage holds GPS = 8 / T groups of the unit's T tiles (chunk c of
// tile i at c * cs + i * 512 bytes); the W = 8 / T warps of a tile take
// groups 2 ks, 2 ks + 1 of every stage.  Returns false on a time-out.
template <int MT, bool SUB = false>
__device__ __forceinline__ bool unit_stages(const GemvArgs& a, uint32_t sbase, int nstg, int ng,
                                            int GPS, int ks, uint32_t wl, uint32_t cs, uint32_t x0,
                                            uint32_t x1, uint32_t sxl, const __half* sc0,
                                            const __half* sc1, int lane, int& slot, uint32_t& phase,
                                            float (&acc)[MT][4]) {
    const int NS = a.nstages;
    for (int st = 0; st < nstg; ++st) {
        if (!mbar_wait(sbase + kBarFull + 8 * slot, phase, a.timeout_ns, a.status)) return false;
        const int gs = min(GPS, ng - st * GPS);     // groups in this stage
        const int gsl0 = ks * kGroupsPerWarpStage;  // this warp's first group in it
        const int gl0 = st * GPS + gsl0;
        const uint32_t wa = wl + slot * a.stage_stride + gsl0 * 2 * cs;
        if (gs == GPS) {
#pragma unroll
            for (int gi = 0; gi < kGroupsPerWarpStage; ++gi)
                mma_group<MT, SUB>(wa + gi * 2 * cs, cs,
                                   x_slice(x0 + (gl0 + gi) * 256, x1 + (gl0 + gi) * 256),
                                   __half2float(sc0[gl0 + gi]), __half2float(sc1[gl0 + gi]),
                                   sxl + (gl0 + gi) * 64, acc);
        } else {
            for (int gi = 0; gi < kGroupsPerWarpStage && gsl0 + gi < gs; ++gi)
                mma_group<MT, SUB>(wa + gi * 2 * cs, cs,
                                   x_slice(x0 + (gl0 + gi) * 256, x1 + (gl0 + gi) * 256),
                                   __half2float(sc0[gl0 + gi]), __half2float(sc1[gl0 + gi]),
                                   sxl + (gl0 + gi) * 64, acc);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(sbase + kBarEmpty + 8 * slot);
        if (++slot == NS) {
            slot = 0;
            phase ^= 1u;
        }
    }
    return true;
}

// The W warps of a unit's tile hold sums over disjoint groups of its rows:
// the first adds the others' in warp order (fixed, so repeated calls agree
// bit for bit) and writes rows rbase + R0 and rbase + R1.  All consumer
// warps of the CTA take part (named barrier 1).
template <int MT>
__device__ __forceinline__ void unit_reduce_store(const GemvArgs& a, uint8_t* smem, int warp, int lane,
                                                  int ks, int W, bool ok, float (&part)[MT][4],
                                                  int rbase, int R0, int R1, int t) {
    float4* red = reinterpret_cast<float4*>(smem + a.off_red);  // [warp][MT][lane]
    if (ks > 0) {
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
            red[(warp * MT + mt) * 32 + lane] =
                make_float4(part[mt][0], part[mt][1], part[mt][2], part[mt][3]);
    }
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
    if (ks == 0 && ok) {
        // every partial's load issued before the first add; the adds keep
        // warp order
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
            float4 v[kConsumerWarps - 1];
#pragma unroll
            for (int w2 = 1; w2 < kConsumerWarps; ++w2)
                if (w2 < W) v[w2 - 1] = red[((warp + w2) * MT + mt) * 32 + lane];
#pragma unroll
            for (int w2 = 1; w2 < kConsumerWarps; ++w2) {
                if (w2 < W) {
                    part[mt][0] += v[w2 - 1].x;
                    part[mt][1] += v[w2 - 1].y;
                    part[mt][2] += v[w2 - 1].z;
                    part[mt][3] += v[w2 - 1].w;
                }
            }
        }
        store_y<MT>(a, rbase + R0, rbase + R1, t, part);
    }
}

// The consumer side of a CTA's tail unit after its whole blocks (persistent
// launches with a partial last round): tT tiles of block t_rb from tile t_t0,
// W2 = 8 / tT warps per tile over the K range.  Every consumer warp reaches
// the reduction's barrier, whatever `ok` says.  Kept out of line so that the
// whole-block loop keeps its registers.
template <int MT, bool SUB>
__device__ __noinline__ bool tail_unit_consume(const GemvArgs& a, uint8_t* smem, uint32_t sbase,
                                               uint32_t ring, int nblk, int nck, int ng, int g0,
                                               uint32_t x0, uint32_t x1, uint32_t sxl, int slot,
                                               uint32_t phase, bool ok) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    const int tT = a.tail_T;
    const int t_rb = a.tail_base + (int)blockIdx.y / (kConsumerWarps / tT);
    const int t_t0 = ((int)blockIdx.y % (kConsumerWarps / tT)) * tT;
    const int sbuf = nblk & (a.n_sbuf - 1);
    const int W2 = kConsumerWarps / tT;
    const int ti2 = warp / W2, ks2 = warp - ti2 * W2;
    const int tr0 = ti2 * 16 + g, tr1 = tr0 + 8;
    const uint32_t tcs = (uint32_t)(tT * kTileBytes);
    const uint32_t twl = ring + ti2 * kTileBytes + lane * 16;
    const int tCPS = kStageBytes / (tT * kTileBytes);
    const int tnstg = (nck + tCPS - 1) / tCPS;
    float tacc[MT][4];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int e = 0; e < 4; ++e) tacc[mt][e] = 0.0f;
    if (ok && !mbar_wait(sbase + kBarSFull + 8 * sbuf, (nblk >> (a.n_sbuf - 1)) & 1, a.timeout_ns,
                         a.status))
        ok = false;
    if (ok) {
        const __half* tsc0 =
            reinterpret_cast<const __half*>(smem + a.off_s + sbuf * a.slab_bytes) + tr0 * a.G + g0;
        if (!unit_stages<MT, SUB>(a, sbase, tnstg, ng, tCPS / 2, ks2, twl, tcs, x0, x1, sxl, tsc0,
                             tsc0 + 8 * a.G, lane, slot, phase, tacc))
            ok = false;
    }
    unit_reduce_store<MT>(a, smem, warp, lane, ks2, W2, ok, tacc, t_rb * kBlockRows + t_t0 * 16, tr0,
                          tr1, t);
    return ok;
}

// WHOLE: the CTA computes whole 128-row blocks (T = 8, stage geometry fixed
// at compile time); otherwise sub-block units of a.T tiles.  The weight map
// (`wmap`) views the kernel layout as rows of 4 KB chunks (512 eight-byte
// elements, one row per block-chunk); sub-block launches copy a box of T
// tiles x 32 / T chunks per ring stage through it.
// XS: x streamed through the ring (whole blocks, M > 4; a.xs_stage > 0).
// SUB: the subnormal-code decode (persistent whole-block launches, M <= 4).
template <int MT, bool WHOLE, bool XS = false, bool SUB = false>
__device__ __forceinline__ void gemv_body(const CUtensorMap* wmap, const CUtensorMap* xmap,
                                          const GemvArgs& a) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int S = (int)gridDim.x;  // the cluster spans the whole x dimension
    const int split = (int)blockIdx.x;
    const int C = a.K / kChunkK;
    const int T = WHOLE ? kConsumerWarps : a.T;
    constexpr bool whole = WHOLE;
    // warps per tile (sharing out its groups), chunks and groups per stage
    const int W = WHOLE ? 1 : a.wpt;
    const int CPS = WHOLE ? kStageBytes / (kConsumerWarps * kTileBytes) : a.cps;
    const int GPS = WHOLE ? CPS / 2 : a.gps;
    const int g0 = a.g0s[split];
    const int ng = a.g0s[split + 1] - g0;
    const int nck = 2 * ng;
    const int nstg = WHOLE ? (nck + CPS - 1) / CPS : a.nstg_u;
    // Whole blocks: the CTA walks blocks y, y + gridDim.y, ...  Sub-block
    // units: CTA y owns rows [16 T y, 16 T (y + 1)), tiles t0 .. t0 + T - 1
    // of block 16 T y / 128.
    const int nblk = !whole ? 1 : a.nb_q + ((int)blockIdx.y < a.nb_r ? 1 : 0);
    // The tail unit of this CTA (persistent launches with a partial last
    // round): tT tiles from tile t_t0 of block t_rb.  Evaluated where used.
    auto has_tail = [&]() { return whole && !XS && a.tail_T > 0 && (int)blockIdx.y < a.tail_units; };
#define W4A16_TAIL_GEOMETRY                                                         \
    const int tT = a.tail_T;                                                        \
    const int t_rb = a.tail_base + (int)blockIdx.y / (kConsumerWarps / tT);         \
    const int t_t0 = ((int)blockIdx.y % (kConsumerWarps / tT)) * tT;
    const int t0 = whole ? 0 : ((int)blockIdx.y * T) & (kConsumerWarps - 1);
    auto block_of = [&](int j) {
        return whole ? (int)blockIdx.y + j * (int)gridDim.y : ((int)blockIdx.y * T) / kConsumerWarps;
    };

    const uint32_t sbase = smem_u32(smem);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kAbortFlag);
    const uint32_t ring = sbase + a.off_ring;

    // K split over a cluster: the partial sums go into peer CTAs' shared
    // memory, which must not be written before those CTAs run.  Every thread
    // arrives here and waits (cluster_wait) once before the exchange.
    if (S > 1) cluster_arrive_relaxed();
    // Dependents may start their own prologue (and first copies) right away;
    // their griddepcontrol.wait still waits for this grid to complete.
    grid_launch_dependents();

    if (warp == kConsumerWarps) {
        // =============================== producer ===============================
        // The producer initialises the barriers and goes straight on to its
        // first copies; the consumer warps wait for the initialisation on
        // named barrier 2 (the producer warp arrives, the consumers sync), so
        // the copies do not wait for the slowest consumer warp to start.
        if (lane == 0) {
            for (int s = 0; s < a.nstages; ++s) {
                mbar_init(sbase + kBarFull + 8 * s, 1);
                mbar_init(sbase + kBarEmpty + 8 * s, kConsumerWarps);
            }
            mbar_init(sbase + kBarX, 1);
            for (int b = 0; b < 2; ++b) {
                mbar_init(sbase + kBarSFull + 8 * b, 1);
                mbar_init(sbase + kBarSEmpty + 8 * b, kConsumerWarps);
            }
            *abort_flag = 0;
            fence_barrier_init();
        }
        __syncwarp();
        asm volatile("bar.arrive 2, %0;" ::"n"(kGemvThreads) : "memory");
        if constexpr (WHOLE) {
            // Whole blocks: one bulk copy of CPS contiguous 4 KB chunks per stage.
            if (lane == 0) {
                const uint64_t pol = l2_policy_evict_first();
                const size_t block_stride = (size_t)C * kChunkBytes;
                // Weights and scales are constants of the call: the first ring
                // stages and scale slab load while the previous kernel is still
                // running.  x (its output, possibly) loads only after the wait.
                bool x_issued = false;
                const int NS = a.nstages;
                const uint32_t stride = (uint32_t)a.stage_stride;
                constexpr bool xs = XS;
                const uint32_t xbox = 512u * (uint32_t)a.M;  // one stage's x: 4 chunks x M rows x 128 B
                int it = 0, slot = 0, round = 0;  // slot = it % NS, round = it / NS
                auto issue_x = [&]() {
                    grid_dependency_wait();
                    if (xs) {
                        // the x of the stages issued so far (at most the first ring pass;
                        // their barriers already expect these bytes)
                        for (int i = 0; i < it; ++i)
                            tma_load_3d(align1024(ring + (uint32_t)(i % NS) * stride + kStageBytes), xmap,
                                        0, 0, 2 * g0 + 4 * (i % nstg), sbase + kBarFull + 8 * (i % NS));
                    } else {
                        const uint32_t xbytes = (uint32_t)nck * (kChunkK * 2);
                        mbar_arrive_expect_tx(sbase + kBarX, xbytes * a.M);
                        for (int m = 0; m < a.M; ++m)
                            bulk_g2s(sbase + a.off_x + m * a.xs_stride,
                                     a.x + (size_t)m * a.K + (size_t)g0 * kGroup, xbytes, sbase + kBarX);
                    }
                    x_issued = true;
                };
                bool ok = true;
                int sb_issued = 0;
                for (int j = 0; ok && j < nblk; ++j) {
                    const int rb = (int)blockIdx.y + j * (int)gridDim.y;
                    // --- scale slab of block rb ---
                    const int sbuf = j & (a.n_sbuf - 1);
                    // a slab buffer frees only after the consumers, who need
                    // x first, finish a block with it
                    if (j >= a.n_sbuf && !x_issued) issue_x();
                    if (j >= a.n_sbuf &&
                        !mbar_wait(sbase + kBarSEmpty + 8 * sbuf, ((j >> (a.n_sbuf - 1)) - 1) & 1,
                                   a.timeout_ns, a.status)) {
                        ok = false;
                        break;
                    }
                    {
                        const int rows = min(kBlockRows, a.N - rb * kBlockRows);
                        const uint32_t bytes = (uint32_t)(rows * a.G * 2);
                        const uint32_t bulk = bytes & ~15u;
                        const __half* src = a.scales + (size_t)rb * kBlockRows * a.G;
                        __half* dst = reinterpret_cast<__half*>(smem + a.off_s + sbuf * a.slab_bytes);
                        for (uint32_t e = bulk / 2; e < bytes / 2; ++e) dst[e] = src[e];  // ragged tail
                        mbar_arrive_expect_tx(sbase + kBarSFull + 8 * sbuf, bulk);
                        if (bulk)
                            bulk_g2s(sbase + a.off_s + sbuf * a.slab_bytes, src, bulk,
                                     sbase + kBarSFull + 8 * sbuf);
                        sb_issued = j + 1;
                    }
                    // --- weight stages of block rb ---
                    const uint8_t* w = a.wq + (size_t)rb * block_stride + 2 * (size_t)g0 * kChunkBytes;
                    for (int st = 0; st < nstg; ++st) {
                        if (it >= NS && !x_issued) issue_x();
                        if (it >= NS &&
                            !mbar_wait(sbase + kBarEmpty + 8 * slot, (round - 1) & 1, a.timeout_ns,
                                       a.status)) {
                            ok = false;
                            break;
                        }
                        if (*abort_flag) {
                            ok = false;
                            break;
                        }
                        const int nc = min(CPS, nck - st * CPS);
                        mbar_arrive_expect_tx(sbase + kBarFull + 8 * slot,
                                              nc * kChunkBytes + (xs ? xbox : 0u));
                        bulk_g2s_hint(ring + slot * stride, w + (size_t)st * kStageBytes,
                                      nc * kChunkBytes, sbase + kBarFull + 8 * slot, pol);
                        if (xs && x_issued)
                            tma_load_3d(align1024(ring + slot * stride + kStageBytes), xmap, 0, 0,
                                        2 * g0 + 4 * st, sbase + kBarFull + 8 * slot);
                        ++it;
                        if (++slot == NS) {
                            slot = 0;
                            ++round;
                        }
                    }
                }
                if (ok && has_tail()) {
                    // The tail unit: scale slab of its 16 tT rows, then boxes of
                    // tT tiles x 32 / tT chunks through the tensor map.
                    W4A16_TAIL_GEOMETRY
                    const int sbuf = nblk & (a.n_sbuf - 1);
                    if (nblk >= a.n_sbuf && !x_issued) issue_x();
                    if (nblk >= a.n_sbuf &&
                        !mbar_wait(sbase + kBarSEmpty + 8 * sbuf, ((nblk >> (a.n_sbuf - 1)) - 1) & 1,
                                   a.timeout_ns, a.status))
                        ok = false;
                    const int r0 = t_rb * kBlockRows + t_t0 * 16;
                    if (ok) {
                        const int rows = max(0, min(16 * tT, a.N - r0));
                        const uint32_t bytes = (uint32_t)(rows * a.G * 2);
                        const uint32_t bulk = bytes & ~15u;
                        const __half* src = a.scales + (size_t)r0 * a.G;
                        __half* dst = reinterpret_cast<__half*>(smem + a.off_s + sbuf * a.slab_bytes);
                        for (uint32_t e = bulk / 2; e < bytes / 2; ++e) dst[e] = src[e];  // ragged tail
                        mbar_arrive_expect_tx(sbase + kBarSFull + 8 * sbuf, bulk);
                        if (bulk)
                            bulk_g2s(sbase + a.off_s + sbuf * a.slab_bytes, src, bulk,
                                     sbase + kBarSFull + 8 * sbuf);
                        sb_issued = nblk + 1;
                    }
                    const int tCPS = kStageBytes / (tT * kTileBytes);
                    const int tnstg = (C + tCPS - 1) / tCPS;
                    const int box_x = t_t0 * (kTileBytes / 8);
                    const int cy0 = t_rb * C;
                    for (int st = 0; ok && st < tnstg; ++st) {
                        if (it >= NS && !x_issued) issue_x();
                        if (it >= NS &&
                            !mbar_wait(sbase + kBarEmpty + 8 * slot, (round - 1) & 1, a.timeout_ns,
                                       a.status)) {
                            ok = false;
                            break;
                        }
                        if (*abort_flag) {
                            ok = false;
                            break;
                        }
                        const int nc = min(tCPS, C - st * tCPS);
                        const uint32_t dst = ring + slot * stride;
                        const uint32_t bar = sbase + kBarFull + 8 * slot;
                        if (nc == tCPS) {
                            mbar_arrive_expect_tx(bar, kStageBytes);
                            tma_load_2d_hint(dst, wmap, box_x, cy0 + st * tCPS, bar, pol);
                        } else {
                            const uint32_t rowb = (uint32_t)(tT * kTileBytes);
                            const uint8_t* src = a.wq + (size_t)(cy0 + st * tCPS) * kChunkBytes +
                                                 (size_t)t_t0 * kTileBytes;
                            mbar_arrive_expect_tx(bar, nc * rowb);
                            for (int c = 0; c < nc; ++c)
                                bulk_g2s_hint(dst + c * rowb, src + (size_t)c * kChunkBytes, rowb, bar,
                                              pol);
                        }
                        ++it;
                        if (++slot == NS) {
                            slot = 0;
                            ++round;
                        }
                    }
                }
                if (!x_issued) issue_x();
                if (!ok) *abort_flag = 1;
                // Drain: every issued copy must land before the CTA may exit.
                const uint64_t dt = drain_bound(a.timeout_ns);
                if (!xs) mbar_wait(sbase + kBarX, 0, dt, a.status);
                for (int i = (it > NS ? it - NS : 0); i < it; ++i)
                    mbar_wait(sbase + kBarFull + 8 * (i % NS), (i / NS) & 1, dt, a.status);
                for (int j = (sb_issued > a.n_sbuf ? sb_issued - a.n_sbuf : 0); j < sb_issued; ++j)
                    mbar_wait(sbase + kBarSFull + 8 * (j & (a.n_sbuf - 1)), (j >> (a.n_sbuf - 1)) & 1, dt,
                              a.status);
            }
        } else {
            // Sub-block units (one block, one scale buffer): a tensor-map box of
            // T tiles x CPS chunks per stage, the K tail chunk by chunk.
            if (lane == 0) {
                const uint64_t pol = l2_policy_evict_first();
                const int NS = a.nstages;
                const int rb = block_of(0);
                const int r0 = rb * kBlockRows + t0 * 16;    // first weight row of the unit
                const int box_x = t0 * (kTileBytes / 8);     // map x coordinate of its tiles
                const int cy0 = rb * C + 2 * g0;             // map row of its first chunk
                tma_prefetch_map(wmap);
                {   // scale slab of the unit's rows
                    const int rows = min(16 * T, a.N - r0);
                    const uint32_t bytes = (uint32_t)(rows * a.G * 2);
                    const uint32_t bulk = bytes & ~15u;
                    const __half* src = a.scales + (size_t)r0 * a.G;
                    __half* dst = reinterpret_cast<__half*>(smem + a.off_s);
                    for (uint32_t e = bulk / 2; e < bytes / 2; ++e) dst[e] = src[e];  // ragged tail
                    mbar_arrive_expect_tx(sbase + kBarSFull, bulk);
                    if (bulk) bulk_g2s(sbase + a.off_s, src, bulk, sbase + kBarSFull);
                }
                // Weights and scales are constants of the call and load before
                // the grid-dependency wait; x loads after it.
                bool x_issued = false;
                auto issue_x = [&]() {
                    grid_dependency_wait();
                    const uint32_t xbytes = (uint32_t)nck * (kChunkK * 2);
                    mbar_arrive_expect_tx(sbase + kBarX, xbytes * a.M);
                    for (int m = 0; m < a.M; ++m)
                        bulk_g2s(sbase + a.off_x + m * a.xs_stride,
                                 a.x + (size_t)m * a.K + (size_t)g0 * kGroup, xbytes, sbase + kBarX);
                    x_issued = true;
                };
                int it = 0, slot = 0, round = 0;  // slot = it % NS, round = it / NS
                bool ok = true;
                for (; it < nstg; ++it) {
                    if (it >= NS && !x_issued) issue_x();
                    if (it >= NS && !mbar_wait(sbase + kBarEmpty + 8 * slot, (round - 1) & 1,
                                               a.timeout_ns, a.status)) {
                        ok = false;
                        break;
                    }
                    if (*abort_flag) {
                        ok = false;
                        break;
                    }
                    const int nc = min(CPS, nck - it * CPS);
                    const uint32_t dst = ring + slot * (uint32_t)a.stage_stride;
                    const uint32_t bar = sbase + kBarFull + 8 * slot;
                    if (nc == CPS) {
                        mbar_arrive_expect_tx(bar, kStageBytes);
                        tma_load_2d_hint(dst, wmap, box_x, cy0 + it * CPS, bar, pol);
                    } else {
                        // the K tail: one copy of T tiles per chunk
                        const uint32_t rowb = (uint32_t)(T * kTileBytes);
                        const uint8_t* src = a.wq + (size_t)(cy0 + it * CPS) * kChunkBytes +
                                             (size_t)t0 * kTileBytes;
                        mbar_arrive_expect_tx(bar, nc * rowb);
                        for (int c = 0; c < nc; ++c)
                            bulk_g2s_hint(dst + c * rowb, src + (size_t)c * kChunkBytes, rowb, bar,
                                          pol);
                    }
                    if (++slot == NS) {
                        slot = 0;
                        ++round;
                    }
                }
                if (!x_issued) issue_x();
                if (!ok) *abort_flag = 1;
                // Drain: every issued copy must land before the CTA may exit.
                const uint64_t dt = drain_bound(a.timeout_ns);
                mbar_wait(sbase + kBarX, 0, dt, a.status);
                for (int i = (it > NS ? it - NS : 0); i < it; ++i)
                    mbar_wait(sbase + kBarFull + 8 * (i % NS), (i / NS) & 1, dt, a.status);
                mbar_wait(sbase + kBarSFull, 0, dt, a.status);
            }
        }
        __syncwarp();
        if (S > 1) cluster_wait();
    } else {
        // =============================== consumers ==============================
        asm volatile("bar.sync 2, %0;" ::"n"(kGemvThreads) : "memory");  // barriers initialised
        grid_dependency_wait();
        if (S > 1) cluster_wait();  // every peer runs: their reduction slots exist
        const int g = lane >> 2, t = lane & 3;
        const int ti = warp / W;         // tile of this warp within the CTA's rows
        const int ks = warp - ti * W;    // its share of every stage's groups
        const int row0 = ti * 16 + g;    // rows of this lane's fragments among the CTA's rows
        const int row1 = row0 + 8;
        // x rows: lanes beyond M read row M-1; their MMA columns are discarded.
        const int xr0 = g < a.M ? g : a.M - 1;
        const int xr1 = g + 8 < a.M ? g + 8 : a.M - 1;
        const uint32_t x0 = sbase + a.off_x + xr0 * a.xs_stride + t * 32;
        const uint32_t x1 = sbase + a.off_x + xr1 * a.xs_stride + t * 32;
        const uint32_t cs = (uint32_t)(T * kTileBytes);  // bytes between chunks in a stage
        const uint32_t wl = ring + ti * kTileBytes + lane * 16;

        // x arrives once per CTA, or (whole blocks, M > 4) with every stage
        bool ok = XS ? true : mbar_wait(sbase + kBarX, 0, a.timeout_ns, a.status);
        if constexpr (SUB) {
            // x sums per group and row, Sx[gl][m] in FP32 (rows m >= M zero):
            // 8 threads per (group, row), 16 values each as 8 pairs summed by
            // a tree of packed adds, then xor-shuffles in a fixed order.
            float* sxw = reinterpret_cast<float*>(smem + a.off_sx);
            const int total = ng * a.M * 8;
            for (int base = 0; base < total; base += kConsumers) {
                const int task = base + (int)threadIdx.x;
                const int e = task >> 3, gl = e / a.M, m = e - gl * a.M;
                float sum = 0.0f;
                if (ok && task < total) {
                    uint4 p[2];
                    if (XS) {
                        // x rides in the ring: read the CTA's K range from global memory
                        // (after the grid-dependency wait, so the previous kernel's x is there)
                        const uint4* src = reinterpret_cast<const uint4*>(
                            a.x + (size_t)m * a.K + (size_t)(g0 + gl) * kGroup + (task & 7) * 16);
                        p[0] = src[0];
                        p[1] = src[1];
                    } else {
                        const uint32_t src =
                            sbase + a.off_x + m * a.xs_stride + gl * 256 + (task & 7) * 32;
                        p[0] = lds128(src);
                        p[1] = lds128(src + 16);
                    }
                    const uint32_t wv[8] = {p[0].x, p[0].y, p[0].z, p[0].w,
                                            p[1].x, p[1].y, p[1].z, p[1].w};
                    float2 f[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        f[i] = __half22float2(*reinterpret_cast<const __half2*>(&wv[i]));
#pragma unroll
                    for (int w2 = 4; w2 >= 1; w2 >>= 1)
#pragma unroll
                        for (int i = 0; i < w2; ++i) f[i] = __fadd2_rn(f[i], f[i + w2]);
                    sum = f[0].x + f[0].y;
                }
                sum += __shfl_xor_sync(0xffffffffu, sum, 4);
                sum += __shfl_xor_sync(0xffffffffu, sum, 2);
                sum += __shfl_xor_sync(0xffffffffu, sum, 1);
                if (task < total && (task & 7) == 0) sxw[gl * 16 + m] = sum;
            }
            for (int i = (int)threadIdx.x; i < ng * 16; i += kConsumers)
                if ((i & 15) >= a.M) sxw[i] = 0.0f;
            asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
        }
        const uint32_t sxl = sbase + a.off_sx + t * 8;  // Sx of this lane's columns 2t, 2t + 1
        const int NS = a.nstages;
        int slot = 0;
        uint32_t phase = 0;  // parity of the ring's current pass
        float part[MT][4] = {};  // sub-block units: this warp's sums, for the in-CTA reduction
        for (int j = 0; ok && j < nblk; ++j) {
            const int rb = block_of(j);
            const int sbuf = j & (a.n_sbuf - 1);
            if (!mbar_wait(sbase + kBarSFull + 8 * sbuf, (j >> (a.n_sbuf - 1)) & 1, a.timeout_ns,
                           a.status)) {
                ok = false;
                break;
            }
            const __half* sc0 = reinterpret_cast<const __half*>(smem + a.off_s + sbuf * a.slab_bytes) +
                                row0 * a.G + g0;
            const __half* sc1 = sc0 + 8 * a.G;
            float acc[MT][4];
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[mt][e] = 0.0f;

            if constexpr (WHOLE) {
                // Whole blocks: every stage holds two groups of the warp's
                // tile, except a one-group tail when the K range has an odd
                // number of groups.
                const int nfull = nck / 4;
                uint32_t xs_off = 0;
                for (int st = 0; st < nfull; ++st, xs_off += 4 * 128) {
                    if (!mbar_wait(sbase + kBarFull + 8 * slot, phase, a.timeout_ns, a.status)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sa = ring + slot * (uint32_t)a.stage_stride;
                    const uint32_t wa = wl + slot * (uint32_t)a.stage_stride;
#pragma unroll
                    for (int gi = 0; gi < 2; ++gi) {
                        const int gl = st * 2 + gi;
                        const XAddr xad =
                            XS ? x_stage(align1024(sa + kStageBytes), a.M, 2 * gi, xr0, xr1, t)
                               : x_slice(x0 + xs_off + gi * 256, x1 + xs_off + gi * 256);
                        mma_group<MT, SUB>(wa + gi * 2 * kChunkBytes, kChunkBytes, xad,
                                           __half2float(sc0[gl]), __half2float(sc1[gl]),
                                           sxl + gl * 64, acc);
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(sbase + kBarEmpty + 8 * slot);
                    if (++slot == NS) {
                        slot = 0;
                        phase ^= 1u;
                    }
                }
                if (ok && (nck & 3)) {
                    if (!mbar_wait(sbase + kBarFull + 8 * slot, phase, a.timeout_ns, a.status)) {
                        ok = false;
                    } else {
                        const int gl = nfull * 2;
                        const uint32_t sa = ring + slot * (uint32_t)a.stage_stride;
                        const XAddr xad = XS ? x_stage(align1024(sa + kStageBytes), a.M, 0, xr0, xr1, t)
                                             : x_slice(x0 + xs_off, x1 + xs_off);
                        mma_group<MT, SUB>(wl + slot * (uint32_t)a.stage_stride, kChunkBytes, xad,
                                           __half2float(sc0[gl]), __half2float(sc1[gl]),
                                           sxl + gl * 64, acc);
                        __syncwarp();
                        if (lane == 0) mbar_arrive(sbase + kBarEmpty + 8 * slot);
                    }
                    if (++slot == NS) {
                        slot = 0;
                        phase ^= 1u;
                    }
                }
            } else {
                // Sub-block units: a stage holds GPS groups of T tiles; the W
                // warps of a tile take two groups each.
                if (!unit_stages<MT, SUB>(a, sbase, nstg, ng, GPS, ks, wl, cs, x0, x1, sxl, sc0, sc1,
                                          lane, slot, phase, acc))
                    ok = false;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(sbase + kBarSEmpty + 8 * sbuf);
            if constexpr (!WHOLE) {
#pragma unroll
                for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) part[mt][e] = acc[mt][e];
                break;  // one unit per CTA
            }
            if (!ok) break;

            const int R0 = rb * kBlockRows + row0;
            const int R1 = rb * kBlockRows + row1;
            if (S == 1) {
                store_y<MT>(a, R0, R1, t, acc);
            } else {
                // One block per CTA in split mode: push the partials straight
                // into the owner of each row (CTA row % S), slot [split][row / S].
                const uint32_t red = sbase + a.off_red;  // [S][rpo][16] floats
                const uint32_t d0 = red + (uint32_t)((split * a.rpo + row0 / S) * 64);
                const uint32_t d1 = red + (uint32_t)((split * a.rpo + row1 / S) * 64);
#pragma unroll
                for (int mt = 0; mt < MT; ++mt) {
                    const uint32_t c = (uint32_t)((mt * 8 + 2 * t) * 4);
                    st_cluster_v2f(map_to_cta(d0 + c, (uint32_t)(row0 % S)), acc[mt][0], acc[mt][1]);
                    st_cluster_v2f(map_to_cta(d1 + c, (uint32_t)(row1 % S)), acc[mt][2], acc[mt][3]);
                }
            }
        }
        if constexpr (!WHOLE) {
            unit_reduce_store<MT>(a, smem, warp, lane, ks, W, ok, part,
                                  block_of(0) * kBlockRows + t0 * 16, row0, row1, t);
        } else {
            if (has_tail())
                ok = tail_unit_consume<MT, SUB>(a, smem, sbase, ring, nblk, nck, ng, g0, x0, x1, sxl,
                                                slot, phase, ok);
        }
        if (!ok) *abort_flag = 1;
    }

    if (S > 1) {
        // One cluster barrier: every CTA has pushed its partials into the
        // owners' shared memory (release/acquire), and nobody touches a
        // peer's shared memory afterwards.  CTA `split` then sums, in a
        // fixed order, the S slices of the rows split, split + S, ...
        cluster_sync_all();
        const int rb = (int)blockIdx.y;
        const float* red = reinterpret_cast<const float*>(smem + a.off_red);
        const int M = a.M;
        const int rows_owned = (kBlockRows - split + S - 1) / S;
        for (int idx = threadIdx.x; idx < rows_owned * M; idx += kGemvThreads) {
            const int li = idx / M, m = idx - li * M;
            const int R = rb * kBlockRows + split + li * S;
            if (R >= a.N) continue;
            float sum = 0.0f;
            for (int q = 0; q < S; ++q) sum += red[(q * a.rpo + li) * 16 + m];
            a.y[(size_t)m * a.N + R] = __float2half_rn(sum);
        }
    }
}

#undef W4A16_TAIL_GEOMETRY

// Whole 128-row blocks per CTA (split or persistent launches).
// (The tensor map is used only by the tail units of a persistent launch.)
// Variants of the whole-block kernel: x as a CTA-wide slice, x through the
// ring (M > 4), or the subnormal-code decode (persistent launches, M <= 4).
enum GemvVariant { kVarSlice = 0, kVarXRing = 1, kVarSubnormal = 2, kVarXRingSubnormal = 3 };

template <int MT, int VAR>
__global__ void __launch_bounds__(kGemvThreads, MT == 1 ? 3 : 2)
    gemv_kernel(const __grid_constant__ CUtensorMap wmap, const __grid_constant__ CUtensorMap xmap,
                const __grid_constant__ GemvArgs a) {
    gemv_body<MT, true, VAR == kVarXRing || VAR == kVarXRingSubnormal,
              VAR == kVarSubnormal || VAR == kVarXRingSubnormal>(&wmap, &xmap, a);
}

// (The subnormal-code variant with x as a CTA-wide slice exists for M <= 8
// only: above that x always rides in the ring.)
template <int MT>
const void* gemv_kernel_ptr(int var) {
    if constexpr (MT == 1)
        if (var == kVarSubnormal) return reinterpret_cast<const void*>(gemv_kernel<1, kVarSubnormal>);
    if (var == kVarXRingSubnormal)
        return reinterpret_cast<const void*>(gemv_kernel<MT, kVarXRingSubnormal>);
    return var == kVarXRing ? reinterpret_cast<const void*>(gemv_kernel<MT, kVarXRing>)
                            : reinterpret_cast<const void*>(gemv_kernel<MT, kVarSlice>);
}

// Sub-block units of a.T tiles, weights copied through the tensor map.
template <int MT, int VAR>
__global__ void __launch_bounds__(kGemvThreads, MT == 1 ? 3 : 2)
    gemv_unit_kernel(const __grid_constant__ CUtensorMap wmap, const __grid_constant__ GemvArgs a) {
    gemv_body<MT, false, false, VAR == kVarSubnormal>(&wmap, nullptr, a);
}

template <int MT>
const void* gemv_unit_kernel_ptr(int var) {
    if constexpr (MT == 1)
        if (var == kVarSubnormal)
            return reinterpret_cast<const void*>(gemv_unit_kernel<1, kVarSubnormal>);
    return reinterpret_cast<const void*>(gemv_unit_kernel<MT, kVarSlice>);
}

struct GemvPlan {
    int S = 0;
    int T = kConsumerWarps;
    int grid_y = 0;
    int n_sbuf = 1;
    int nstages = kStages;
    int xs_stride = 0;
    int slab_bytes = 0;
    int rpo = 0;
    int tail_T = 0, tail_base = 0, tail_units = 0;  // persistent launches: last-round units
    int xs_stage = 0, stage_stride = kStageBytes;    // x in the ring (whole blocks, M > 4)
    int var = kVarSlice;                              // whole-block kernel variant
    uint32_t off_ring = 0, off_x = 0, off_s = 0, off_red = 0, off_sx = 0, smem = 0;
    double cost = 0.0;
};

template <int MT, bool WHOLE = true>
int occupancy(uint32_t smem, int var = kVarSlice) {
    int blocks = 0;
    const cudaError_t e =
        WHOLE ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, gemv_kernel_ptr<MT>(var),
                                                              kGemvThreads, smem)
              : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, gemv_unit_kernel_ptr<MT>(var),
                                                              kGemvThreads, smem);
    return e == cudaSuccess ? blocks : 0;
}

template <int MT>
int max_active_clusters(int S, uint32_t smem, int var) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)S, 1, 1);
    cfg.blockDim = dim3(kGemvThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = (unsigned)S;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, gemv_kernel_ptr<MT>(var), &cfg) != cudaSuccess) return 0;
    return n;
}

template <int MT>
cudaError_t ensure_smem_attr() {
    static std::atomic<bool> done[64];  // per device; racing callers only repeat the set-up
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && done[dev].load(std::memory_order_acquire)) return cudaSuccess;
    cudaError_t e = cudaSuccess;
    for (int var : {kVarSlice, kVarXRing, kVarSubnormal, kVarXRingSubnormal})
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(gemv_kernel_ptr<MT>(var),
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    if (e == cudaSuccess)
        for (int var : {kVarSlice, kVarSubnormal})
            if (e == cudaSuccess)
                e = cudaFuncSetAttribute(gemv_unit_kernel_ptr<MT>(var),
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    if (e == cudaSuccess && dev >= 0 && dev < 64) done[dev].store(true, std::memory_order_release);
    return e;
}

// Shared-memory layout of a launch with K split S, T tiles per CTA and
// `nsb` scale buffers (a persistent launch always reserves the in-CTA
// reduction buffer of its tail units).
template <int MT>
bool layout(GemvPlan& p, int M, int G, int S, int T, int nsb, const DeviceCtx& ctx,
            int nst = kStages, bool subnormal = false) {
    p.S = S;
    p.T = T;
    p.n_sbuf = nsb;
    // whole blocks with M > 4: x rides in the ring (4 chunks x M rows per
    // stage, 1024-aligned in a slot with 1 KB of slack) instead of a CTA-wide
    // M x K slice, which at M = 16, K = 4096 alone takes 128 KB
    const bool xs = T == kConsumerWarps && M > 4;
    p.xs_stage = xs ? ((512 * M + 1023) / 1024) * 1024 + 1024 : 0;
    p.stage_stride = kStageBytes + p.xs_stage;
    p.var = xs ? (subnormal ? kVarXRingSubnormal : kVarXRing) : subnormal ? kVarSubnormal : kVarSlice;
    const int ng_max = (G + S - 1) / S;
    // a CTA that sees only one block needs no more stages than it fills
    const int fill = (2 * ng_max * T * kTileBytes + kStageBytes - 1) / kStageBytes;
    p.nstages = nsb == 1 && fill < nst ? fill : nst;
    p.xs_stride = ng_max * kGroup * 2 + 16;  // +16 B keeps x rows conflict-free
    p.slab_bytes = ((16 * T * G * 2 + 127) / 128) * 128;
    p.off_ring = kBarAreaBytes;
    p.off_x = p.off_ring + p.nstages * p.stage_stride;
    p.off_s = p.off_x + (xs ? 0 : ((M * p.xs_stride + 127) / 128) * 128);
    p.off_red = p.off_s + nsb * p.slab_bytes;
    p.rpo = (kBlockRows + S - 1) / S;
    const int red_bytes = S > 1 ? S * p.rpo * 16 * 4
                          : T < kConsumerWarps || nsb == 2 ? kConsumerWarps * MT * 32 * 16
                                                           : 0;
    p.off_sx = p.off_red + red_bytes;
    p.smem = p.off_sx + (subnormal ? ng_max * 16 * 4 : 0);
    return (int)p.smem <= ctx.max_smem_optin;
}

// Launch-time model (microseconds) used to rank the candidate launches,
// fitted to GB300 timings of every candidate on the Llama-3-8B and
// Qwen2.5-7B decode shapes at M = 1..16.  A CTA wave costs a fixed start-up
// plus the longer of (a) the heaviest SM streaming its CTAs' weights at the
// per-SM rate seen when every SM streams, and (b) one CTA streaming its own
// weights, which its 8 consumer warps cap (at half the rate with two n8
// tiles, M > 8); copying and summing the CTA's activation slice (M x its K
// range) adds to both.  A K split adds the cluster barrier and the exchange
// of partial sums through distributed shared memory.
constexpr double kWaveUs = 1.5;
constexpr int kSubnormalMinGroups = 16;  // groups per warp and x-sum round
constexpr double kSmBytesPerUs = 36.0e3;
constexpr double kCtaBytesPerUs = 14.0e3;
constexpr double kXBytesPerUs = 32.0e3;
constexpr double kSplitReduceUs = 3.5;

template <int MT>
double launch_cost(long long units, long long slots, double w_bytes, double x_bytes, int S,
                   const DeviceCtx& ctx) {
    const long long waves = (units + slots - 1) / slots;
    const long long per_wave = units < slots ? units : slots;
    const long long heaviest = (per_wave + ctx.num_sms - 1) / ctx.num_sms;
    const double x_us = x_bytes / kXBytesPerUs;
    const double sm_us = (double)heaviest * (w_bytes / kSmBytesPerUs + x_us);
    const double cta_us = w_bytes * MT / kCtaBytesPerUs + x_us;
    return (double)waves * (kWaveUs + (sm_us > cta_us ? sm_us : cta_us)) +
           (S > 1 ? kSplitReduceUs : 0.0);
}

// Chooses the launch.  With more 128-row blocks than CTA slots the grid is
// persistent (whole blocks, one CTA per slot walking blocks).  Otherwise the
// cheapest under launch_cost of
//  * whole blocks with K split S ways over a cluster of S CTAs (S = 1..8),
//  * sub-block units of T = 1, 2 or 4 tiles (16 T rows) over the whole K
//    range, the 8 warps splitting K and reducing inside the CTA, each with
//    the deepest ring that keeps the CTAs per SM its units need.
template <int MT>
GemvPlan plan_gemv(int M, int N, int K, const DeviceCtx& ctx) {
    const int G = K / kGroup;
    const int NB = (N + kBlockRows - 1) / kBlockRows;
    {
        GemvPlan p;
        // Persistent launches take the subnormal-code decode: its x-sum pass
        // (~0.3 us once per CTA; from global memory when x rides in the ring)
        // is paid back over many blocks.
        const bool sn = true;
        if (layout<MT>(p, M, G, 1, kConsumerWarps, 2, ctx, kStages, sn)) {
            const int occ = occupancy<MT>(p.smem, p.var);
            if (occ > 0 && NB > ctx.num_sms * occ) {
                // The deepest ring that keeps the same CTAs per SM: more bytes
                // in flight per CTA, for the same number of streams.
                for (int nst = kMaxStages; nst > kStages; --nst) {
                    GemvPlan q;
                    if (layout<MT>(q, M, G, 1, kConsumerWarps, 2, ctx, nst, sn) &&
                        occupancy<MT>(q.smem, q.var) == occ) {
                        p = q;
                        break;
                    }
                }
                p.grid_y = ctx.num_sms * occ;
                // A partial last round of R blocks runs as units of T tiles,
                // the smallest T that gives each of the first CTAs at most one
                // (T / 8 of a block-time instead of a whole one).
                const int rem = NB % p.grid_y;
                for (int tt = 1; rem > 0 && p.xs_stage == 0 && tt < kConsumerWarps; tt *= 2) {
                    if (rem * (kConsumerWarps / tt) <= p.grid_y) {
                        p.tail_T = tt;
                        p.tail_base = NB - rem;
                        p.tail_units = rem * (kConsumerWarps / tt);
                        break;
                    }
                }
                p.cost = 0.0;
                return p;
            }
        }
    }
    GemvPlan best;
    const int max_s = G < kMaxSplits ? G : kMaxSplits;
    for (int S = 1; S <= max_s; ++S) {
        // Clusters live inside one GPC: count co-resident clusters, not SM slots.
        auto slots_of = [&](const GemvPlan& q) -> long long {
            const int occ = occupancy<MT>(q.smem, q.var);
            if (occ == 0) return 0;
            return S == 1 ? (long long)ctx.num_sms * occ
                          : (long long)max_active_clusters<MT>(S, q.smem, q.var) * S;
        };
        GemvPlan p;
        if (!layout<MT>(p, M, G, S, kConsumerWarps, 1, ctx)) continue;
        long long slots = slots_of(p);
        if (slots == 0) continue;
        // Unsplit: the deepest ring that needs no more waves -- more bytes in
        // flight per CTA, and no SM given more CTAs than the grid needs (a grid
        // of 2 per SM on 3 slots per SM leaves some SMs 3 CTAs and others 1).
        // (Clusters of 5 to 8 with fewer CTAs per SM measured slower.)
        const long long units = (long long)NB * S;
        const long long waves = (units + slots - 1) / slots;
        for (int nst = kMaxStages; S == 1 && nst > p.nstages; --nst) {
            GemvPlan q;
            if (!layout<MT>(q, M, G, S, kConsumerWarps, 1, ctx, nst) || q.nstages != nst) continue;
            const long long qs = slots_of(q);
            if (qs > 0 && (units + qs - 1) / qs <= waves) {
                p = q;
                slots = qs;
                break;
            }
        }
        const int ng = (G + S - 1) / S;
        p.grid_y = NB;
        p.cost = launch_cost<MT>((long long)NB * S, slots, (double)ng * kBlockRows * kGroup / 2,
                                 (double)M * ng * kGroup * 2, S, ctx);
        if (best.S == 0 || p.cost < best.cost) best = p;
    }
    for (int T = 1; T < kConsumerWarps; T *= 2) {
        GemvPlan p;
        // The subnormal-code decode saves 4 instructions per 8 weights; its
        // x-sum pass (ceil(8 G M / 256) rounds, on the path before the first
        // MMA) pays off only with >= 16 groups per warp and round (units of
        // 64 rows at K = 4096 and M = 1: yes; 16 rows at K = 14336: no).
        const int sx_rounds = (G * M * 8 + kConsumers - 1) / kConsumers;
        const bool sn = MT == 1 && M <= 4 && G * T / kConsumerWarps >= kSubnormalMinGroups * sx_rounds;
        if (!layout<MT>(p, M, G, 1, T, 1, ctx, kStages, sn)) continue;
        const int occ = occupancy<MT, false>(p.smem, p.var);
        if (occ == 0) continue;
        const long long units = ((long long)N + 16 * T - 1) / (16 * T);
        const long long fit = (units + ctx.num_sms - 1) / ctx.num_sms;
        const int need = fit < occ ? (int)fit : occ;
        for (int nst = kMaxStages; nst > p.nstages; --nst) {
            GemvPlan q;
            if (layout<MT>(q, M, G, 1, T, 1, ctx, nst, sn) && q.nstages == nst &&
                occupancy<MT, false>(q.smem, q.var) >= need) {
                p = q;
                break;
            }
        }
        p.grid_y = (int)units;
        p.cost = launch_cost<MT>(units, (long long)ctx.num_sms * occ,
                                 (double)G * 16 * T * kGroup / 2, (double)M * G * kGroup * 2, 1, ctx);
        if (best.S == 0 || p.cost < best.cost) best = p;
    }
    return best;
}

struct PlanKey {
    int dev, M, N, K;
    bool operator==(const PlanKey& o) const {
        return dev == o.dev && M == o.M && N == o.N && K == o.K;
    }
};

template <int MT>
GemvPlan cached_plan(int M, int N, int K, const DeviceCtx& ctx) {
    static std::mutex mu;
    static std::vector<std::pair<PlanKey, GemvPlan>> cache;
    int dev = 0;
    cudaGetDevice(&dev);
    const PlanKey key{dev, M, N, K};
    {
        std::lock_guard<std::mutex> lock(mu);
        for (const auto& e : cache)
            if (e.first == key) return e.second;
    }
    const GemvPlan p = plan_gemv<MT>(M, N, K, ctx);
    std::lock_guard<std::mutex> lock(mu);
    if (cache.size() < 4096) cache.emplace_back(key, p);
    return p;
}

// The tensor map of a sub-block launch: the kernel layout as [NB * C chunk
// rows] x [512 eight-byte words]; a box is T tiles (64 T words) of 32 / T
// consecutive chunks, 16 KB.  Encoded once per (weights, shape, T) and
// reused: a decode step calls the same weights every token.
cudaError_t weight_map(const uint8_t* wq, int NB, int K, int T, CUtensorMap* out) {
    struct Entry {
        const uint8_t* wq;
        int NB, K, T;
        CUtensorMap map;
    };
    static std::mutex mu;
    static std::vector<Entry> cache;
    {
        std::lock_guard<std::mutex> lock(mu);
        for (const Entry& e : cache)
            if (e.wq == wq && e.NB == NB && e.K == K && e.T == T) {
                *out = e.map;
                return cudaSuccess;
            }
    }
    PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
    if (!encode) return cudaErrorNotSupported;
    Entry e{wq, NB, K, T, {}};
    const cuuint64_t dims[2] = {(cuuint64_t)(kChunkBytes / 8),
                                (cuuint64_t)NB * (cuuint64_t)(K / kChunkK)};
    const cuuint64_t strides[1] = {(cuuint64_t)kChunkBytes};
    const cuuint32_t box[2] = {(cuuint32_t)(T * kTileBytes / 8),
                               (cuuint32_t)(kStageBytes / (T * kTileBytes))};
    const cuuint32_t estr[2] = {1, 1};
    if (encode(&e.map, CU_TENSOR_MAP_DATA_TYPE_UINT64, 2, const_cast<uint8_t*>(wq), dims, strides,
               box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    *out = e.map;
    std::lock_guard<std::mutex> lock(mu);
    if (cache.size() >= 4096) cache.clear();
    cache.push_back(e);
    return cudaSuccess;
}

// The tensor map of x for launches that stream it through the ring: x[M, K]
// as [K / 64 chunks][M rows][64 halves], a box of 4 chunks x M rows (one
// stage), 128-byte swizzled.  Cached per (x, M, K): a decode loop reuses its
// activation buffers.
cudaError_t x_map(const void* x, int M, int K, CUtensorMap* out) {
    struct Entry {
        const void* x;
        int M, K;
        CUtensorMap map;
    };
    static std::mutex mu;
    static std::vector<Entry> cache;
    {
        std::lock_guard<std::mutex> lock(mu);
        for (const Entry& e : cache)
            if (e.x == x && e.M == M && e.K == K) {
                *out = e.map;
                return cudaSuccess;
            }
    }
    PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
    if (!encode) return cudaErrorNotSupported;
    Entry e{x, M, K, {}};
    const cuuint64_t dims[3] = {(cuuint64_t)kChunkK, (cuuint64_t)M, (cuuint64_t)(K / kChunkK)};
    const cuuint64_t strides[2] = {(cuuint64_t)K * 2, (cuuint64_t)kChunkK * 2};
    const cuuint32_t box[3] = {(cuuint32_t)kChunkK, (cuuint32_t)M, 4};
    const cuuint32_t estr[3] = {1, 1, 1};
    if (encode(&e.map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void*>(x), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    *out = e.map;
    std::lock_guard<std::mutex> lock(mu);
    if (cache.size() >= 4096) cache.clear();
    cache.push_back(e);
    return cudaSuccess;
}

template <int MT>
cudaError_t launch_gemv_mt(GemvArgs args, int M, cudaStream_t stream, const DeviceCtx& ctx) {
    cudaError_t e = ensure_smem_attr<MT>();
    if (e != cudaSuccess) return e;
    const GemvPlan p = cached_plan<MT>(M, args.N, args.K, ctx);
    if (p.S == 0) return cudaErrorInvalidValue;
    args.xs_stride = p.xs_stride;
    args.slab_bytes = p.slab_bytes;
    args.n_sbuf = p.n_sbuf;
    args.nstages = p.nstages;
    args.off_ring = p.off_ring;
    args.off_x = p.off_x;
    args.off_s = p.off_s;
    args.off_red = p.off_red;
    args.rpo = p.rpo;
    args.T = p.T;
    args.tail_T = p.tail_T;
    args.tail_base = p.tail_base;
    args.tail_units = p.tail_units;
    args.cps = kStageBytes / (p.T * kTileBytes);
    args.gps = args.cps / 2;
    args.wpt = kConsumerWarps / p.T;
    args.nstg_u = (2 * args.G + args.cps - 1) / args.cps;
    if (p.tail_T > 0) {
        args.nb_q = p.tail_base / p.grid_y;  // every CTA: its whole blocks, then its tail unit
        args.nb_r = 0;
    } else {
        args.nb_q = args.NB / p.grid_y;
        args.nb_r = args.NB % p.grid_y;
    }
    for (int i = 0; i <= p.S; ++i) args.g0s[i] = split_group_begin(i, p.S, args.G);
    args.xs_stage = p.xs_stage;
    args.stage_stride = p.stage_stride;
    args.off_sx = p.off_sx;
    CUtensorMap xmap = {};
    if (p.xs_stage) {
        const cudaError_t xe = x_map(args.x, M, args.K, &xmap);
        if (xe != cudaSuccess) return xe;
    }
    CUtensorMap wmap = {};
    if (p.T < kConsumerWarps || p.tail_T > 0) {
        const cudaError_t me =
            weight_map(args.wq, args.NB, args.K, p.T < kConsumerWarps ? p.T : p.tail_T, &wmap);
        if (me != cudaSuccess) return me;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.S, (unsigned)p.grid_y, 1);
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
    if (p.T < kConsumerWarps) {
        void* kargs[] = {&wmap, &args};
        return cudaLaunchKernelExC(&cfg, gemv_unit_kernel_ptr<MT>(p.var), kargs);
    }
    void* kargs[] = {&wmap, &xmap, &args};
    return cudaLaunchKernelExC(&cfg, gemv_kernel_ptr<MT>(p.var), kargs);
}

}  // namespace

cudaError_t gemv_weight_map(const void* repacked, int64_t N, int64_t K, int T, CUtensorMap* out) {
    return weight_map(static_cast<const uint8_t*>(repacked),
                      (int)((N + kBlockRows - 1) / kBlockRows), (int)K, T, out);
}

cudaError_t gemv_plan_info(int M, int64_t N, int64_t K, const DeviceCtx& ctx, int* splits,
                           int* ctas, int* blocks_per_cta, int* rows_per_cta, int* tail_rows,
                           int* tail_units) {
    cudaError_t e = M <= 8 ? ensure_smem_attr<1>() : ensure_smem_attr<2>();
    if (e != cudaSuccess) return e;
    const GemvPlan p = M <= 8 ? cached_plan<1>(M, (int)N, (int)K, ctx)
                              : cached_plan<2>(M, (int)N, (int)K, ctx);
    if (p.S == 0) return cudaErrorInvalidValue;
    const int NB = (int)((N + kBlockRows - 1) / kBlockRows);
    *splits = p.S;
    *ctas = p.S * p.grid_y;
    *blocks_per_cta = p.T == kConsumerWarps ? (NB + p.grid_y - 1) / p.grid_y : 1;
    *rows_per_cta = 16 * p.T;
    *tail_rows = 16 * p.tail_T;
    *tail_units = p.tail_units;
    return cudaSuccess;
}

cudaError_t launch_gemv(const void* x, const void* repacked, const void* scales, void* y, int M,
                        int64_t N, int64_t K, cudaStream_t stream, const DeviceCtx& ctx) {
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
    a.NB = (int)((N + kBlockRows - 1) / kBlockRows);
    if (M <= 8) return launch_gemv_mt<1>(a, M, stream, ctx);
    return launch_gemv_mt<2>(a, M, stream, ctx);
}

}  // namespace w4a16
