// common.cuh -- device helpers shared by the W4A16 kernels (sm_103a only).
//
// Inline PTX wrappers for mbarriers, bulk async copies (TMA engine), L2
// cache policies, thread-block-cluster shared memory, programmatic dependent
// launch and the warp-level f16 MMA, plus the bounded wait every kernel uses
// so that no wait can spin forever: after `timeout_ns` a wait records
// W4A16_DEV_TIMEOUT in the library's device status word and returns false.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace w4a16 {

// Bits of the device status word (read back by w4a16_device_status()).
enum : unsigned {
    kDevTimeout = 1u << 0,   // a bounded wait gave up
    kDevBadLaunch = 1u << 1  // a kernel saw a launch shape it does not support
};

// ---------------------------------------------------------------------------
// Shared-memory addresses and mbarriers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Makes mbarrier initialisation visible to the async proxy and the cluster.
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Same wait with cluster-scope acquire: for barriers completed by remote
// CTAs (remote arrivals) after which this thread reads their data.
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait for the phase of parity `parity` to complete, giving up after
// `timeout_ns` nanoseconds.  On time-out the status word gets kDevTimeout.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint64_t timeout_ns,
                                          unsigned* status) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 31u) == 0 && global_timer_ns() - t0 > timeout_ns) {
            atomicOr(status, kDevTimeout);
            return false;
        }
    }
}

// Bound of a drain wait: before a CTA exits, every copy it issued must have
// landed in its shared memory, so the wait for those copies never gives up
// sooner than this, however short the caller's wait limit (still bounded).
constexpr uint64_t kDrainFloorNs = 100000000ull;  // 100 ms

__device__ __forceinline__ uint64_t drain_bound(uint64_t timeout_ns) {
    return timeout_ns > kDrainFloorNs ? timeout_ns : kDrainFloorNs;
}

__device__ __forceinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity,
                                                  uint64_t timeout_ns, unsigned* status) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait_cluster(bar, parity)) return true;
        if ((i & 31u) == 0 && global_timer_ns() - t0 > timeout_ns) {
            atomicOr(status, kDevTimeout);
            return false;
        }
    }
}

// ---------------------------------------------------------------------------
// Bulk async copies (global -> shared) completing on an mbarrier
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// `bytes` and both addresses must be multiples of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void bulk_g2s_hint(uint32_t dst, const void* src, uint32_t bytes,
                                              uint32_t bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1], %2, [%3], %4;" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}

// Prefetch `bytes` (multiple of 16) of global memory into L2.  L2 is the
// coherence point, so this is safe before a grid-dependency wait.
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// ---------------------------------------------------------------------------
// Tensor-map (tiled) async copies
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tma_prefetch_map(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 2-D tiled load; c0 is the innermost coordinate (elements).
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void tma_load_2d_hint(uint32_t dst, const CUtensorMap* map, int c0,
                                                 int c1, uint32_t bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar), "l"(policy)
        : "memory");
}

// 3-D tiled load; c0 is the innermost coordinate (elements).
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                            int c2, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
        : "memory");
}

// L2 prefetch of one 2-D box.
__device__ __forceinline__ void tma_prefetch_2d(const CUtensorMap* map, int c0, int c1) {
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(c0), "r"(c1)
                 : "memory");
}

// ---------------------------------------------------------------------------
// Programmatic dependent launch
// ---------------------------------------------------------------------------
__device__ __forceinline__ void grid_dependency_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void grid_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------------------
// Thread-block clusters
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_cta_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void cluster_sync_all() {
    asm volatile(
        "barrier.cluster.arrive.release.aligned;\n\t"
        "barrier.cluster.wait.acquire.aligned;" ::
            : "memory");
}

__device__ __forceinline__ uint32_t map_to_cta(uint32_t smem_addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr), "r"(rank));
    return r;
}

// Store two floats into another CTA's shared memory (cluster window address).
__device__ __forceinline__ void st_cluster_v2f(uint32_t addr, float a, float b) {
    asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};" ::"r"(addr), "f"(a), "f"(b)
                 : "memory");
}

// Store four 32-bit words into another CTA's shared memory (16-byte aligned
// cluster window address).
__device__ __forceinline__ void st_cluster_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                              uint32_t d) {
    asm volatile("st.shared::cluster.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b),
                 "r"(c), "r"(d)
                 : "memory");
}

// Split cluster barrier: every thread of every CTA arrives, later waits.
__device__ __forceinline__ void cluster_arrive() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}

// Arrival with no memory ordering: used once at the start, so that a later
// cluster_wait() guarantees every CTA of the cluster is running (its shared
// memory may then be written remotely).
__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_wait() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Arrive (release, cluster scope) on an mbarrier of another CTA.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t remote_bar) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(remote_bar)
                 : "memory");
}

// ---------------------------------------------------------------------------
// Loads
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr));
    return v;
}

// ---------------------------------------------------------------------------
// Nibble dequantisation and the warp-level MMA
// ---------------------------------------------------------------------------
template <uint32_t LUT>
__device__ __forceinline__ uint32_t lop3(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, %4;" : "=r"(d) : "r"(a), "r"(b), "r"(c), "n"(LUT));
    return d;
}

// Expands a 32-bit word of eight stored nibbles (value q + 8) into four
// half2 registers holding exact q in [-8, 7].  OR-ing a nibble into the
// mantissa of 1024.0 (0x6400) gives 1024 + n (low position) or 1024 + 16 n
// (position 4..7 of a half); subtracting 1032, or scaling by 1/16 and
// subtracting 72, leaves n - 8 exactly.  Output order (nibble positions):
// r[0] = (0, 4), r[1] = (1, 5), r[2] = (2, 6), r[3] = (3, 7).
__device__ __forceinline__ void dequant8(uint32_t w, uint32_t (&r)[4]) {
    constexpr uint32_t kMagic = 0x64006400u;  // (1024.0, 1024.0)
    constexpr uint32_t kLut = (0xF0 & 0xCC) | 0xAA;  // (a & b) | c
    const uint32_t lo0 = lop3<kLut>(w, 0x000F000Fu, kMagic);
    const uint32_t hi0 = lop3<kLut>(w, 0x00F000F0u, kMagic);
    const uint32_t w8 = w >> 8;
    const uint32_t lo1 = lop3<kLut>(w8, 0x000F000Fu, kMagic);
    const uint32_t hi1 = lop3<kLut>(w8, 0x00F000F0u, kMagic);
    const __half2 k1032 = __halves2half2(__ushort_as_half(0x6408), __ushort_as_half(0x6408));
    const __half2 kSixteenth = __halves2half2(__ushort_as_half(0x2C00), __ushort_as_half(0x2C00));
    const __half2 kMinus72 = __halves2half2(__ushort_as_half(0xD480), __ushort_as_half(0xD480));
    __half2 v;
    v = __hsub2(*reinterpret_cast<const __half2*>(&lo0), k1032);
    r[0] = *reinterpret_cast<uint32_t*>(&v);
    v = __hfma2(*reinterpret_cast<const __half2*>(&hi0), kSixteenth, kMinus72);
    r[1] = *reinterpret_cast<uint32_t*>(&v);
    v = __hsub2(*reinterpret_cast<const __half2*>(&lo1), k1032);
    r[2] = *reinterpret_cast<uint32_t*>(&v);
    v = __hfma2(*reinterpret_cast<const __half2*>(&hi1), kSixteenth, kMinus72);
    r[3] = *reinterpret_cast<uint32_t*>(&v);
}

// The same word as unbiased codes n in fp16 subnormals, with no arithmetic:
// a nibble masked into bits 0..3 of a half is n * 2^-24 exactly, into bits
// 4..7 it is n * 2^-20.  r[0] / r[2] (positions 0, 4 and 2, 6) carry 2^-24,
// r[1] / r[3] (positions 1, 5 and 3, 7) carry 2^-20; in the layout's
// fragment order that is one factor per weight row (rows r0: 2^-24, rows
// r1: 2^-20), removed with the zero point 8 in the FP32 group rescale.
__device__ __forceinline__ void dequant8_subnormal(uint32_t w, uint32_t (&r)[4]) {
    r[0] = w & 0x000F000Fu;
    r[1] = w & 0x00F000F0u;
    const uint32_t w8 = w >> 8;
    r[2] = w8 & 0x000F000Fu;
    r[3] = w8 & 0x00F000F0u;
}

__device__ __forceinline__ float2 lds64f(uint32_t addr) {
    float2 v;
    asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(addr));
    return v;
}

// D = A(16x16, row) * B(16x8, col) + C, f16 inputs, f32 accumulate.
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                          uint32_t b1, const float (&c)[4]) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%10, %11, %12, %13};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]),
          "f"(c[2]), "f"(c[3]));
}

}  // namespace w4a16
