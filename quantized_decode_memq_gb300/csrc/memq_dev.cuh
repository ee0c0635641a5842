// memq_dev.cuh -- inline-PTX building blocks shared by the memq kernels (sm_103a).
//
// Bulk asynchronous copies (cp.async.bulk, the 1-D form of the Tensor Memory Accelerator)
// completing on shared-memory mbarriers, bounded barrier waits, programmatic dependent launch
// controls, and the small numeric conversions the GEMV inner loops use.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace memq {

constexpr unsigned kFullMask = 0xffffffffu;

// ---------------------------------------------------------------------------------------------
// Programmatic dependent launch.  `griddep_wait` returns once every grid this launch depends on
// has completed and its writes are visible (a no-op when the launch carried no programmatic
// dependency).  `griddep_launch_dependents` lets the next launch in the stream begin its
// prologue early; that launch still waits for this grid before reading what it wrote.
//
// Because the kernels here release their successor at entry, a launch's lifetime overlaps the
// end of its predecessor's.  Data the predecessor writes (the activation x, the q8_1 qs / d) is
// therefore NOT constant over the reader's lifetime and must not go through the non-coherent
// read-only path (ld.global.nc / __ldg): it is read after griddep_wait with L2-coherent loads
// (__ldcg).  __ldg stays for true constants (weights, scale grids, the RMSNorm weight).
// ---------------------------------------------------------------------------------------------
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------------------------------------
// mbarrier + bulk copy
// ---------------------------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

// Make barrier initialisation visible to the async proxy before any bulk copy uses it.
__device__ __forceinline__ void mbar_init_fence() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// One arrival that also announces `bytes` of incoming transaction count.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

// Waits for phase `parity` of `bar` to complete; the thread is suspended (not spinning) until
// the phase completes or about 1 ms passes, whichever comes first.  Returns whether it completed.
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(1000000u)
        : "memory");
    return ok != 0;
}

// About one second at GB300 clocks.  No correct launch comes anywhere near it; it only turns a
// would-be hang (a transaction count that never completes) into a recorded fault.
constexpr long long kWaitCycles = 2000000000LL;

// Warp-uniform bounded wait for phase `parity` of `bar`: every lane performs its own acquire,
// and all lanes return the same verdict (true = phase complete, false = gave up).
__device__ __forceinline__ bool warp_wait_bounded(uint64_t *bar, uint32_t parity) {
    bool ok = mbar_try_wait(bar, parity);
    if (__all_sync(kFullMask, ok)) return true;
    const long long t0 = clock64();
    for (;;) {
        ok = mbar_try_wait(bar, parity);
        if (__all_sync(kFullMask, ok)) return true;
        const bool late = (clock64() - t0) > kWaitCycles;
        if (__any_sync(kFullMask, late)) return false;
    }
}

// L2 policy for the weight stream: every weight byte is read once per call, so it is marked
// evict-first and does not push the activation or other tensors out of L2.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// Global -> shared bulk copy of `bytes` (multiple of 16; both addresses 16-byte aligned),
// completing `bytes` of transaction count on `bar`.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar,
                                         uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// Tiled 2-D tensor copy global -> shared (TMA): the box of the tensor map `map` (a generic
// address of a __grid_constant__ kernel parameter) at element coordinates (x, y), completing
// on `bar`.  The destination must be 128-byte aligned and x * element size a multiple of 16.
__device__ __forceinline__ void tma_load_2d(void *dst, const void *map, int x, int y,
                                            uint64_t *bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// As tma_load_2d, with the default L2 policy.
__device__ __forceinline__ void tma_load_2d_plain(void *dst, const void *map, int x, int y,
                                                  uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void tma_prefetch_map(const void *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// As bulk_g2s, with the default L2 policy.
__device__ __forceinline__ void bulk_g2s_plain(void *dst, const void *src, uint32_t bytes,
                                               uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// ---------------------------------------------------------------------------------------------
// Shared-memory loads.  Plain C++ loads (not volatile asm), so the compiler can interleave
// independent blocks while still ordering them after the barrier waits, which clobber memory.
// ---------------------------------------------------------------------------------------------
__device__ __forceinline__ uint4 lds128(const void *p) { return *static_cast<const uint4 *>(p); }
__device__ __forceinline__ uint2 lds64(const void *p) { return *static_cast<const uint2 *>(p); }
__device__ __forceinline__ uint32_t lds32(const void *p) { return *static_cast<const uint32_t *>(p); }
__device__ __forceinline__ uint32_t lds16(const void *p) { return *static_cast<const uint16_t *>(p); }

// ---------------------------------------------------------------------------------------------
// Numeric helpers
// ---------------------------------------------------------------------------------------------

// Two E4M3 codes (low byte = first element) -> f16x2 (low half = first element).  Every E4M3
// value is exact in f16.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_codes) {
    uint32_t out;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(out) : "h"(static_cast<unsigned short>(two_codes)));
    return out;
}

// Four E4M3 codes (one 32-bit word, low byte first) -> f16x2 {c0,c1} and {c2,c3}; the word is
// split into its two 16-bit halves inside PTX so no shift or mask is needed.
__device__ __forceinline__ void e4m3x4_to_f16x2x2(uint32_t w4, uint32_t &lo, uint32_t &hi) {
    asm("{\n\t.reg .b16 l, h;\n\t"
        "mov.b32 {l, h}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, l;\n\t"
        "cvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
        : "=r"(lo), "=r"(hi)
        : "r"(w4));
}

// Four int8 (one 32-bit word, low byte first) -> two f16x2 {q0,q1}, {q2,q3}, exactly: each byte
// biased to u = q + 128 is placed under the f16 exponent of 1024 (0x64uu = 1024 + u), and 1152
// is subtracted in f16 (both steps exact for integers below 2048).
__device__ __forceinline__ void s8x4_to_f16x2x2(uint32_t q4, uint32_t &lo, uint32_t &hi) {
    const uint32_t u = q4 ^ 0x80808080u;
    uint32_t a, b;
    asm("prmt.b32 %0, %1, %2, 0x4140;" : "=r"(a) : "r"(u), "r"(0x64646464u));
    asm("prmt.b32 %0, %1, %2, 0x4342;" : "=r"(b) : "r"(u), "r"(0x64646464u));
    const uint32_t bias = 0x64806480u;  // f16x2 {1152, 1152}
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(lo) : "r"(a), "r"(bias));
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(hi) : "r"(b), "r"(bias));
}

// D = A(16x16, f16, row) * B(16x8, f16, col) + C with f32 accumulation.
__device__ __forceinline__ void mma_f16_16816(float (&c)[4], uint32_t a0, uint32_t a1,
                                              uint32_t a2, uint32_t a3, uint32_t b0,
                                              uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFullMask, v, o);
    return v;
}
__device__ __forceinline__ double warp_sum(double v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFullMask, v, o);
    return v;
}

}  // namespace memq
