// quantize.cu -- group-wise symmetric round-to-nearest INT4 quantizer.
//
// Computes, per row and group of 128 weights along K (qaqbuyan.com tutorial
// "LLM quantization from IEEE 754 to GPTQ/AWQ/GGUF", chapter "量化的数学基石",
// §2 symmetric formula and §3 per_group_symmetric_quantize):
//   s32 = max(max|w| / 7, 1e-8) in binary32 with a correctly rounded divide,
//   q   = clamp(round_half_even(fl(w / s32)), -8, 7)  (fl: IEEE division),
//   scale = fp16(s32) rounded to nearest even, byte = (q_odd+8)<<4 | (q_even+8).
//
// One team of 8 lanes per group: each lane loads 16 fp16 values with two
// 16-byte loads, the absmax is reduced with three xor-shuffles inside the
// team, and each lane writes its 8 packed bytes (the group's 64 bytes are one
// coalesced segment).  The per-group scalar work (reduction, scale, its
// reciprocal) is shared by 16 elements a lane.  A team issues the loads of
// its next group before quantizing the current one (software pipelining in
// registers: 30.5 -> 28.7 us on [14336, 4096]; more groups per iteration raise
// register pressure and were slower), and the grid is one resident wave.
// 256 B are read and 66 B written per group; the per-element work
// (fma-rounding, its residual, the tie test) runs on pairs through the packed
// binary32 instructions, about two instructions per element.
#include <atomic>

#include "common.cuh"
#include "kernels.h"

namespace w4a16 {
namespace {

constexpr int kQuantThreads = 256;
constexpr int kQuantTeam = 8;    // lanes per group, 16 weights each
constexpr int kQuantUnroll = 1;  // groups per team per iteration (the next ones' loads are in flight)

// s32 = RN(a / 7) for an fp16 absmax a, by Markstein's theorem on FMA
// division (P. Markstein, IBM J. Res. Dev. 34(1), 1990): with y = RN(1/7)
// and q = RN(a * y) within an ulp of a / 7, the residual a - 7q is exact and
// RN(q + (a - 7q) y) = RN(a / 7).  a is never subnormal in binary32 here; the
// identity was also checked for every finite fp16 a against IEEE division.
__device__ __forceinline__ float div7_rn(float a) {
    constexpr float y = 1.0f / 7.0f;
    const float q = __fmul_rn(a, y);
    const float r = __fmaf_rn(-q, 7.0f, a);
    return __fmaf_rn(r, y, q);
}

// 1/s to within 2^-23 relative: hardware approximation plus one
// Newton-Raphson step (e = 1 - s y0, y = y0 + y0 e).  s >= 1e-8 is normal.
__device__ __forceinline__ float rcp_nr(float s) {
    float y0;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y0) : "f"(s));
    return __fmaf_rn(y0, __fmaf_rn(-s, y0, 1.0f), y0);
}

// Adding kRound = 1.5 * 2^23 + 8 to a binary32 |r| < 8 rounds r to the
// nearest integer, ties to even (kRound is even and the sum's ulp is 1), and
// leaves q + 8 in the low 4 bits of the sum.
constexpr float kRound = 12582920.0f;

// Quantizes one group held as 16 fp16 values per lane of an 8-lane team.
//
// q = round_half_even(fl(w / s)) is formed from the exact product w * y of
// the refined reciprocal, rounded by the fma with kRound: |w y - w / s| <=
// 7 * 2^-23 and |fl(w / s) - w / s| <= 7 * 2^-24, so the two sit within
// 1.3e-6 of each other and round to the same integer unless the product's
// distance to its integer exceeds 1/2 - 1e-5.  When any lane of the warp
// sees that (exact ties included) the warp takes the correctly rounded
// divide for all its elements.  No clamp is needed: s >= (max|w| / 7)(1 -
// 2^-24) bounds |w / s| below 7.5, so q already lies in [-7, 7].
// packed[0] holds the lane's elements 0..7 (element 2j in the low nibble of
// byte j), packed[1] elements 8..15.
__device__ __forceinline__ void quantize_group(const uint4 (&raw)[2], uint32_t (&packed)[2],
                                               float& scale) {
    const __half2* h2 = reinterpret_cast<const __half2*>(&raw[0]);  // 8 pairs (raw is contiguous)
    __half2 m2 = __habs2(h2[0]);
#pragma unroll
    for (int i = 1; i < 8; ++i) m2 = __hmax2(m2, __habs2(h2[i]));
    float amax = fmaxf(__low2float(m2), __high2float(m2));
#pragma unroll
    for (int off = kQuantTeam / 2; off > 0; off >>= 1)
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));

    float s = div7_rn(amax);
    if (s < 1e-8f) s = 1e-8f;
    const float y = rcp_nr(s);

    float w[16], t[16];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float2 f = __half22float2(h2[i]);
        w[2 * i] = f.x;
        w[2 * i + 1] = f.y;
    }
    // Pairs of elements go through the packed binary32 instructions, each
    // component rounded exactly as the scalar form: t = RN(w y + kRound),
    // d = RN(q - w y) with q = t - kRound, and e = RN(d^2 - kTieSq), which is
    // negative exactly when |d| < sqrt(kTieSq) ~ 1/2 - 1e-5 (the fma rounds
    // once, so its sign is exact).  AND-ing the sign bits leaves bit 31 clear
    // when some element is a near tie (e = +0 counts as one: the exact
    // fallback below is always correct).
    constexpr float kTieSq = 0.25f - 1.0e-5f;
    const float2 y2 = make_float2(y, y), ny2 = make_float2(-y, -y);
    const float2 kr2 = make_float2(kRound, kRound), nkr2 = make_float2(-kRound, -kRound);
    const float2 ntie2 = make_float2(-kTieSq, -kTieSq);
    uint32_t clear_bits = 0xffffffffu;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float2 wv = make_float2(w[2 * i], w[2 * i + 1]);
        const float2 tv = __ffma2_rn(wv, y2, kr2);
        const float2 d = __ffma2_rn(wv, ny2, __fadd2_rn(tv, nkr2));  // q - w y
        const float2 e = __ffma2_rn(d, d, ntie2);
        clear_bits &= __float_as_uint(e.x) & __float_as_uint(e.y);
        t[2 * i] = tv.x;
        t[2 * i + 1] = tv.y;
    }
    if (__any_sync(0xffffffffu, (clear_bits >> 31) == 0)) {
#pragma unroll
        for (int i = 0; i < 16; ++i) t[i] = __fadd_rn(__fdiv_rn(w[i], s), kRound);
    }
    // Each t holds 0x4B400000 + (q + 8): sum t_i 16^i (Horner, integer
    // multiply-adds) and remove the constant part once; the nibbles q + 8
    // occupy disjoint bits, so no carries cross between them.
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        uint32_t acc = __float_as_uint(t[8 * h + 7]);
#pragma unroll
        for (int i = 6; i >= 0; --i) acc = acc * 16u + __float_as_uint(t[8 * h + i]);
        packed[h] = acc - 0x4B400000u * 0x11111111u;
    }
    scale = s;
}

__global__ void __launch_bounds__(kQuantThreads)
    quantize_kernel(const uint4* __restrict__ W, int64_t groups_total,
                    uint2* __restrict__ qweight, __half* __restrict__ scales) {
    constexpr int kTeams = kQuantThreads / kQuantTeam;
    const int tl = threadIdx.x & (kQuantTeam - 1);
    const int64_t stride = (int64_t)gridDim.x * kTeams;
    // group `grp` = row grp / G, group grp % G; its 128 halves are contiguous
    // at element offset grp * 128 of the row-major matrix (16 uint4; lane tl
    // takes 2 tl and 2 tl + 1).  The four teams of a warp differ only in the
    // low two bits of g0 (stride is a multiple of 4), so the loop test on g0
    // with those bits cleared is warp-uniform and the full-warp shuffles always
    // see every lane; groups past the end load nothing and store nothing.
    int64_t g0 = (int64_t)blockIdx.x * kTeams + (threadIdx.x / kQuantTeam);
    uint4 raw[kQuantUnroll][2];
#pragma unroll
    for (int u = 0; u < kQuantUnroll; ++u) {
        const int64_t grp = g0 + u * stride;
        const bool live = grp < groups_total;
        raw[u][0] = live ? __ldcs(W + grp * 16 + 2 * tl) : make_uint4(0, 0, 0, 0);
        raw[u][1] = live ? __ldcs(W + grp * 16 + 2 * tl + 1) : make_uint4(0, 0, 0, 0);
    }
    for (; (g0 & ~(int64_t)3) < groups_total; g0 += kQuantUnroll * stride) {
        uint4 nxt[kQuantUnroll][2];  // the next iteration's groups, loading meanwhile
#pragma unroll
        for (int u = 0; u < kQuantUnroll; ++u) {
            const int64_t grp = g0 + (kQuantUnroll + u) * stride;
            const bool live = grp < groups_total;
            nxt[u][0] = live ? __ldcs(W + grp * 16 + 2 * tl) : make_uint4(0, 0, 0, 0);
            nxt[u][1] = live ? __ldcs(W + grp * 16 + 2 * tl + 1) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < kQuantUnroll; ++u) {
            const int64_t grp = g0 + u * stride;
            uint32_t packed[2];
            float sc;
            quantize_group(raw[u], packed, sc);
            if (grp < groups_total) {
                qweight[grp * kQuantTeam + tl] = make_uint2(packed[0], packed[1]);
                if (tl == 0) scales[grp] = __float2half_rn(sc);
            }
        }
#pragma unroll
        for (int u = 0; u < kQuantUnroll; ++u) {
            raw[u][0] = nxt[u][0];
            raw[u][1] = nxt[u][1];
        }
    }
    // Publish the packed weights and scales device-wide before this block
    // ends: a GEMM launched next on the stream may read them before the
    // grid-completion flush (it treats them as constants).
    __threadfence();
}

// ---------------------------------------------------------------------------
// Format variants: groups of 32, 64 or 128 weights or one group per row
// (per-channel), symmetric as above or asymmetric (tutorial §2 asymmetric
// formula: s = (max - min) / 15 with min and max taken over the group and 0,
// z = -round(min / s), q = clamp(round(w / s) + z, 0, 15); the nibble holds
// q, the zero point one byte per group).  Every step is the binary32
// operation of the formula with a correctly rounded divide, so the codes,
// scales and zero points match the plain statement bit for bit.
//
// A team of L = min(32, group / 8) lanes owns a group; each lane loads 8
// weights (16 bytes) per pass and packs their 8 nibbles into one 32-bit word.
// Groups wider than 256 (per-channel) take several passes, reading the row
// twice (reduce, then quantize).
// ---------------------------------------------------------------------------
constexpr int kFmtThreads = 256;

// Q40: the GGUF Q4_0 block layout (tutorial GGUF section) instead of
// separate codes and scales -- group 32, symmetric; group g's block is the 18
// bytes at g * 18: the fp16 scale, then the 16 code bytes (lane tl's 4 bytes
// at offset 2 + 4 tl, stored as two 16-bit halves: blocks are 2-byte aligned).
template <bool ASYM, bool Q40>
__global__ void __launch_bounds__(kFmtThreads)
    quantize_fmt_kernel(const uint4* __restrict__ W, int64_t groups_total, int group, int L,
                        uint32_t* __restrict__ qweight, __half* __restrict__ scales,
                        uint8_t* __restrict__ zeros) {
    const int lane = threadIdx.x & 31;
    const int tl = lane % L;                 // lane within the team
    const unsigned team_mask = L == 32 ? 0xffffffffu : (((1u << L) - 1u) << (lane - tl));
    const int teams_per_block = kFmtThreads / L;
    const int64_t stride = (int64_t)gridDim.x * teams_per_block;
    const int passes = group / (8 * L);
    // Whole warps iterate together (a warp's teams share the loop test), so
    // every team's shuffles see all of its lanes.
    const int64_t warp_first =
        (int64_t)blockIdx.x * teams_per_block + (threadIdx.x / 32) * (32 / L);
    for (int64_t base = warp_first; base < groups_total; base += stride) {
        const int64_t grp = base + lane / L;
        const bool live = grp < groups_total;
        const uint4* src = W + (live ? grp : 0) * (group / 8);
        // --- pass 1: max |w| (symmetric) or min / max with 0 (asymmetric) ---
        float lo = 0.0f, hi = 0.0f;
        for (int p = 0; p < passes; ++p) {
            const uint4 raw = live ? __ldg(src + p * L + tl) : make_uint4(0, 0, 0, 0);
            const __half2* h2 = reinterpret_cast<const __half2*>(&raw);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float2 f = __half22float2(h2[i]);
                if (ASYM) {
                    lo = fminf(lo, fminf(f.x, f.y));
                    hi = fmaxf(hi, fmaxf(f.x, f.y));
                } else {
                    hi = fmaxf(hi, fmaxf(fabsf(f.x), fabsf(f.y)));
                }
            }
        }
        for (int off = L / 2; off > 0; off >>= 1) {
            hi = fmaxf(hi, __shfl_xor_sync(team_mask, hi, off));
            if (ASYM) lo = fminf(lo, __shfl_xor_sync(team_mask, lo, off));
        }
        float s = ASYM ? __fdiv_rn(__fsub_rn(hi, lo), 15.0f) : __fdiv_rn(hi, 7.0f);
        if (s < 1e-8f) s = 1e-8f;
        const float z = ASYM ? -rintf(__fdiv_rn(lo, s)) : 8.0f;  // nibble offset
        // --- pass 2: codes ---
        for (int p = 0; p < passes && live; ++p) {
            const uint4 raw = __ldg(src + p * L + tl);
            const __half2* h2 = reinterpret_cast<const __half2*>(&raw);
            uint32_t word = 0;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float2 f = __half22float2(h2[i]);
                const float qa = fminf(fmaxf(rintf(__fdiv_rn(f.x, s)) + (ASYM ? z : 0.0f),
                                             ASYM ? 0.0f : -8.0f), ASYM ? 15.0f : 7.0f);
                const float qb = fminf(fmaxf(rintf(__fdiv_rn(f.y, s)) + (ASYM ? z : 0.0f),
                                             ASYM ? 0.0f : -8.0f), ASYM ? 15.0f : 7.0f);
                const uint32_t na = (uint32_t)(int)(ASYM ? qa : qa + 8.0f);
                const uint32_t nb = (uint32_t)(int)(ASYM ? qb : qb + 8.0f);
                word |= (na | (nb << 4)) << (8 * i);
            }
            if (Q40) {
                uint16_t* b = reinterpret_cast<uint16_t*>(reinterpret_cast<uint8_t*>(qweight) +
                                                          grp * 18 + 2 + 4 * tl);
                b[0] = (uint16_t)(word & 0xffffu);
                b[1] = (uint16_t)(word >> 16);
            } else {
                qweight[grp * (group / 8) + p * L + tl] = word;
            }
        }
        if (live && tl == 0) {
            if (Q40)
                *reinterpret_cast<__half*>(reinterpret_cast<uint8_t*>(qweight) + grp * 18) =
                    __float2half_rn(s);
            else
                scales[grp] = __float2half_rn(s);
            if (ASYM) zeros[grp] = (uint8_t)(int)z;
        }
    }
    // as quantize_kernel: publish before a following GEMM reads them
    __threadfence();
}

// ---------------------------------------------------------------------------
// W8A16: per-channel symmetric INT8 (tutorial §2 formula with b = 8):
// s = max(max_k |w| / 127, 1e-8), q = clamp(round(w / s), -128, 127), code =
// q + 128, one warp per row, the row read twice (absmax, then codes), every
// step the binary32 operation of the formula (correctly rounded divides).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kFmtThreads)
    quantize_w8_kernel(const uint4* __restrict__ W, int64_t N, int K,
                       uint2* __restrict__ q8, __half* __restrict__ scales) {
    const int lane = threadIdx.x & 31;
    const int64_t warps = (int64_t)gridDim.x * (kFmtThreads / 32);
    const int pieces = K / 8;  // 16-byte pieces per row
    for (int64_t n = (int64_t)blockIdx.x * (kFmtThreads / 32) + threadIdx.x / 32; n < N;
         n += warps) {
        const uint4* row = W + n * pieces;
        float amax = 0.0f;
        for (int p = lane; p < pieces; p += 32) {
            const uint4 raw = __ldg(row + p);
            const __half2* h2 = reinterpret_cast<const __half2*>(&raw);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float2 f = __half22float2(h2[i]);
                amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
            }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
        float s = __fdiv_rn(amax, 127.0f);
        if (s < 1e-8f) s = 1e-8f;
        for (int p = lane; p < pieces; p += 32) {
            const uint4 raw = __ldg(row + p);
            const __half2* h2 = reinterpret_cast<const __half2*>(&raw);
            uint32_t b[2] = {0, 0};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float2 f = __half22float2(h2[i]);
                const float qa = fminf(fmaxf(rintf(__fdiv_rn(f.x, s)), -128.0f), 127.0f);
                const float qb = fminf(fmaxf(rintf(__fdiv_rn(f.y, s)), -128.0f), 127.0f);
                const uint32_t pair = (uint32_t)((int)qa + 128) | ((uint32_t)((int)qb + 128) << 8);
                b[i / 2] |= pair << (16 * (i & 1));
            }
            q8[n * pieces + p] = make_uint2(b[0], b[1]);
        }
        if (lane == 0) scales[n] = __float2half_rn(s);
    }
    __threadfence();
}

}  // namespace

cudaError_t launch_quantize(const void* W, int64_t N, int64_t K, void* qweight, void* scales,
                            cudaStream_t stream, const DeviceCtx& ctx) {
    const int G = (int)(K / kGroup);
    const int64_t groups = N * G;
    const int64_t per_block = kQuantThreads / kQuantTeam;
    int64_t blocks = (groups + per_block - 1) / per_block;
    static std::atomic<int> occ[64];  // resident blocks per SM, per device (one resident wave)
    int dev = 0;
    cudaGetDevice(&dev);
    int per_sm = (dev >= 0 && dev < 64) ? occ[dev].load(std::memory_order_relaxed) : 0;
    if (per_sm == 0) {
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, quantize_kernel, kQuantThreads,
                                                          0) != cudaSuccess ||
            per_sm < 1)
            per_sm = 1;
        if (dev >= 0 && dev < 64) occ[dev].store(per_sm, std::memory_order_relaxed);
    }
    const int64_t cap = (int64_t)ctx.num_sms * per_sm;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    quantize_kernel<<<(unsigned)blocks, kQuantThreads, 0, stream>>>(
        static_cast<const uint4*>(W), groups, static_cast<uint2*>(qweight),
        static_cast<__half*>(scales));
    return cudaGetLastError();
}

}  // namespace w4a16

namespace w4a16 {

cudaError_t launch_quantize_q4_0(const void* W, int64_t N, int64_t K, void* blocks_out,
                                 cudaStream_t stream, const DeviceCtx& ctx) {
    const int L = 4;  // group 32: 8 weights per lane
    const int64_t groups = N * (K / 32);
    const int64_t per_block = kFmtThreads / L;
    int64_t blocks = (groups + per_block - 1) / per_block;
    const int64_t cap = (int64_t)ctx.num_sms * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    quantize_fmt_kernel<false, true><<<(unsigned)blocks, kFmtThreads, 0, stream>>>(
        static_cast<const uint4*>(W), groups, 32, L, static_cast<uint32_t*>(blocks_out), nullptr,
        nullptr);
    return cudaGetLastError();
}

cudaError_t launch_quantize_w8(const void* W, int64_t N, int64_t K, void* q8, void* scales,
                               cudaStream_t stream, const DeviceCtx& ctx) {
    int64_t blocks = (N + kFmtThreads / 32 - 1) / (kFmtThreads / 32);
    const int64_t cap = (int64_t)ctx.num_sms * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    quantize_w8_kernel<<<(unsigned)blocks, kFmtThreads, 0, stream>>>(
        static_cast<const uint4*>(W), N, (int)K, static_cast<uint2*>(q8),
        static_cast<__half*>(scales));
    return cudaGetLastError();
}

cudaError_t launch_quantize_fmt(const void* W, int64_t N, int64_t K, int group, bool asym,
                                void* qweight, void* scales, void* zeros, cudaStream_t stream,
                                const DeviceCtx& ctx) {
    // team width: 8 weights per lane per pass, a power of two dividing the
    // group's 16-byte pieces (groups are multiples of 32; per-channel rows of
    // K % 256 == 128 take teams of 16)
    const int L = group / 8 < 32 ? group / 8 : ((group / 8) % 32 == 0 ? 32 : 16);
    const int64_t groups = N * (K / group);
    const int64_t per_block = kFmtThreads / L;
    int64_t blocks = (groups + per_block - 1) / per_block;
    const int64_t cap = (int64_t)ctx.num_sms * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    if (asym)
        quantize_fmt_kernel<true, false><<<(unsigned)blocks, kFmtThreads, 0, stream>>>(
            static_cast<const uint4*>(W), groups, group, L, static_cast<uint32_t*>(qweight),
            static_cast<__half*>(scales), static_cast<uint8_t*>(zeros));
    else
        quantize_fmt_kernel<false, false><<<(unsigned)blocks, kFmtThreads, 0, stream>>>(
            static_cast<const uint4*>(W), groups, group, L, static_cast<uint32_t*>(qweight),
            static_cast<__half*>(scales), nullptr);
    return cudaGetLastError();
}

}  // namespace w4a16
