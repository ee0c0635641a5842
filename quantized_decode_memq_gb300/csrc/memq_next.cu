// memq_next.cu -- the silu(gate) * up -> q8_1 activation producer and the load-time repack of
// E4M3 weights into a Q8_0 slab.
//
// Operations: q8_fuse_gate.rs (memra-engine 0.125.0), `main` -- the expert-ff site's
// "silu/gate*up -> q8_1" producer (width 1536); gemv_e4m3_bench.rs, module doc "QUESTION" --
// the shipping path converts FP8 weights into a Q8_0 copy once, when the model loads (ARM B').
//
// silu_mul_q8_1_kernel: elementwise, one thread per float4 of a row; a 32-element block is 8
// adjacent threads, so its amax is a 3-step xor shuffle (as in the RMSNorm producer).  In the
// decode chain it follows the gate / up GEMVs, so it takes part in programmatic dependent
// launch and reads its inputs with L2-coherent loads after the dependency wait.
//
// repack_kernel: the slab is a flat array of 34-byte blocks whose inputs are the flat array of
// 32-byte E4M3 blocks (rows are contiguous in both), so a warp converts 32 consecutive blocks
// -- 1 KB in, 1088 B out -- assembles the output in shared memory and writes it with 16-byte
// stores.  Per block: W = e4m3 * s (f32), d = amax / 127, f16(d), qs = round(W / d), every
// step an IEEE f32 operation, so the bytes match a plain C evaluation of the same formulas.
#include <cmath>
#include <cstdint>
#include <cuda_fp16.h>

#include "memq.h"
#include "memq_dev.cuh"

namespace memq {
namespace {

constexpr int kNextThreads = 256;

__device__ __forceinline__ int8_t round_code(float v, float dd) {
    return dd != 0.0f ? static_cast<int8_t>(roundf(__fdiv_rn(v, dd))) : static_cast<int8_t>(0);
}

__device__ __forceinline__ float silu_mul1(float g, float u) {
    return __fmul_rn(__fdiv_rn(g, __fadd_rn(1.0f, expf(-g))), u);
}

__global__ void __launch_bounds__(kNextThreads)
    silu_mul_q8_1_kernel(const float *__restrict__ gate, const float *__restrict__ up,
                         float *__restrict__ z, int8_t *__restrict__ qs, float *__restrict__ d,
                         int64_t n4) {
    griddep_launch_dependents();
    griddep_wait();
    const float4 *g4 = reinterpret_cast<const float4 *>(gate);
    const float4 *u4 = reinterpret_cast<const float4 *>(up);
    // n4 is a multiple of 8 (ncols % 32 == 0), and the stride a multiple of 256, so every
    // 8-thread block group is wholly in range or wholly out; all lanes join the shuffles.
    for (int64_t base = static_cast<int64_t>(blockIdx.x) * kNextThreads; base < n4;
         base += static_cast<int64_t>(gridDim.x) * kNextThreads) {
        const int64_t f = base + threadIdx.x;
        const bool act = f < n4;
        float4 gv = make_float4(0.f, 0.f, 0.f, 0.f), uv = gv;
        if (act) {
            gv = __ldcg(g4 + f);
            uv = __ldcg(u4 + f);
        }
        float4 zz;
        zz.x = silu_mul1(gv.x, uv.x);
        zz.y = silu_mul1(gv.y, uv.y);
        zz.z = silu_mul1(gv.z, uv.z);
        zz.w = silu_mul1(gv.w, uv.w);
        float am = fmaxf(fmaxf(fabsf(zz.x), fabsf(zz.y)), fmaxf(fabsf(zz.z), fabsf(zz.w)));
        am = fmaxf(am, __shfl_xor_sync(kFullMask, am, 1));
        am = fmaxf(am, __shfl_xor_sync(kFullMask, am, 2));
        am = fmaxf(am, __shfl_xor_sync(kFullMask, am, 4));
        const float dd = __fdiv_rn(am, 127.0f);
        if (act) {
            const uint32_t packed =
                static_cast<uint32_t>(static_cast<uint8_t>(round_code(zz.x, dd))) |
                static_cast<uint32_t>(static_cast<uint8_t>(round_code(zz.y, dd))) << 8 |
                static_cast<uint32_t>(static_cast<uint8_t>(round_code(zz.z, dd))) << 16 |
                static_cast<uint32_t>(static_cast<uint8_t>(round_code(zz.w, dd))) << 24;
            reinterpret_cast<uint32_t *>(qs)[f] = packed;
            if ((threadIdx.x & 7) == 0) d[f >> 3] = dd;
            if (z) reinterpret_cast<float4 *>(z)[f] = zz;
        }
    }
}

// round(W / d) with the correctly rounded f32 quotient, without a division per weight: with
// inv the correctly rounded 1/d, t = W * inv is within 2 ulp of W / d, hence within 2.5 ulp of
// its correctly rounded value; |t| <= 127 (|W| <= amax), so that is under 2.3e-5.  round() can tell
// the two apart only when t lies within that distance of a .5 boundary, and only there (about
// one weight in 10^4) is the quotient taken with the IEEE division.
// Off the tie window the nearest integer is unique, so rint (ties to even) gives the same code
// as round (ties away) there.
__device__ __forceinline__ int8_t repack_code(float w, float dd, float inv) {
    if (dd == 0.0f) return 0;
    const float t = __fmul_rn(w, inv);
    const float r = rintf(t);
    // (d below 2^-100 also takes the division: there 1/d and W * (1/d) could leave the
    // normal range, where the 2-ulp bound does not hold.)
    if (!(fabsf(t - r) < 0.5f - 3.0e-5f) || !(fabsf(t) < 256.0f) || dd < 7.9e-31f)
        return static_cast<int8_t>(roundf(__fdiv_rn(w, dd)));
    return static_cast<int8_t>(static_cast<int>(r));
}

constexpr int kRepackWarps = kNextThreads / 32;
constexpr int kQ80Block = 34;
constexpr int kWarpOut = 32 * kQ80Block;  // 1088 bytes per warp iteration

template <bool GRID>
__global__ void __launch_bounds__(kNextThreads)
    repack_kernel(const uint8_t *__restrict__ w, const float *__restrict__ aux,
                  uint8_t *__restrict__ out, int64_t nblocks, int64_t nb, int gcols) {
    __shared__ __align__(16) uint8_t stage[kRepackWarps][kWarpOut];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    uint8_t *st = stage[warp];
    const float s_tensor = GRID ? 0.0f : __ldg(aux);
    for (int64_t wb0 = (static_cast<int64_t>(blockIdx.x) * kRepackWarps + warp) * 32;
         wb0 < nblocks; wb0 += static_cast<int64_t>(gridDim.x) * kRepackWarps * 32) {
        const int64_t gb = wb0 + lane;
        const int nblk = static_cast<int>(nblocks - wb0 < 32 ? nblocks - wb0 : 32);
        if (lane < nblk) {
            const uint4 *src = reinterpret_cast<const uint4 *>(w + gb * 32);
            const uint4 v0 = __ldg(src), v1 = __ldg(src + 1);
            float s = s_tensor;
            if (GRID) {
                const int64_t r = gb / nb;
                const int64_t b = gb - r * nb;
                s = __ldg(aux + (r >> 7) * gcols + ((b * 32) >> 7));
            }
            const uint32_t words[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
            float W[32];
            float amax = 0.0f;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                uint32_t lo, hi;
                e4m3x4_to_f16x2x2(words[q], lo, hi);
                const __half2 l2 = *reinterpret_cast<const __half2 *>(&lo);
                const __half2 h2 = *reinterpret_cast<const __half2 *>(&hi);
                W[4 * q + 0] = __fmul_rn(__low2float(l2), s);
                W[4 * q + 1] = __fmul_rn(__high2float(l2), s);
                W[4 * q + 2] = __fmul_rn(__low2float(h2), s);
                W[4 * q + 3] = __fmul_rn(__high2float(h2), s);
#pragma unroll
                for (int k = 0; k < 4; ++k) amax = fmaxf(amax, fabsf(W[4 * q + k]));
            }
            const float dd = __fdiv_rn(amax, 127.0f);
            const float inv = dd != 0.0f ? __frcp_rn(dd) : 0.0f;
            uint16_t *o16 = reinterpret_cast<uint16_t *>(st + lane * kQ80Block);
            o16[0] = __half_as_ushort(__float2half_rn(dd));
#pragma unroll
            for (int k = 0; k < 32; k += 2) {
                const uint32_t c0 = static_cast<uint8_t>(repack_code(W[k], dd, inv));
                const uint32_t c1 = static_cast<uint8_t>(repack_code(W[k + 1], dd, inv));
                o16[1 + k / 2] = static_cast<uint16_t>(c0 | (c1 << 8));
            }
        }
        __syncwarp();
        // The warp's output is contiguous: 16-byte stores (the slab base and every warp's
        // offset, a multiple of 1088, are 16-byte aligned), bytes for a partial last group.
        const int bytes = nblk * kQ80Block;
        const int n16 = bytes / 16;
        uint8_t *dst = out + wb0 * kQ80Block;
        for (int i = lane; i < n16; i += 32)
            reinterpret_cast<uint4 *>(dst)[i] = reinterpret_cast<const uint4 *>(st)[i];
        for (int i = n16 * 16 + lane; i < bytes; i += 32) dst[i] = st[i];
        __syncwarp();
    }
}

bool aligned_to(const void *p, uintptr_t n) {
    return (reinterpret_cast<uintptr_t>(p) & (n - 1)) == 0;
}

int sm_count() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
    return sms;
}

template <bool GRID>
int repack_entry(const uint8_t *w, const float *aux, void *out, int64_t out_f, int64_t in_f,
                 void *stream) {
    if (in_f < 32 || (in_f % 32) != 0 || in_f > (1LL << 24)) return MEMQ_ERR_SHAPE;
    if (out_f < 0 || out_f > (1LL << 31) - 1) return MEMQ_ERR_SHAPE;
    if (out_f == 0) return MEMQ_OK;
    if (!w || !aux || !out) return MEMQ_ERR_NULL;
    if (!aligned_to(w, 16) || !aligned_to(out, 16) || !aligned_to(aux, 4)) return MEMQ_ERR_ALIGN;
    const int sms = sm_count();
    if (sms <= 0) return MEMQ_ERR_LAUNCH;
    const int64_t nb = in_f / 32;
    const int64_t nblocks = out_f * nb;
    const int64_t groups = (nblocks + 31) / 32;
    const int64_t want = (groups + kRepackWarps - 1) / kRepackWarps;
    const unsigned grid = static_cast<unsigned>(want < 8LL * sms ? want : 8LL * sms);
    repack_kernel<GRID><<<grid, kNextThreads, 0, static_cast<cudaStream_t>(stream)>>>(
        w, aux, static_cast<uint8_t *>(out), nblocks, nb, static_cast<int>((in_f + 127) / 128));
    return cudaGetLastError() == cudaSuccess ? MEMQ_OK : MEMQ_ERR_LAUNCH;
}

}  // namespace
}  // namespace memq

extern "C" int memq_silu_mul_q8_1(const float *gate, const float *up, float *z, int8_t *qs,
                                  float *d, int64_t ncols, int64_t rows, void *stream) {
    using namespace memq;
    if (ncols < 32 || (ncols % 32) != 0 || ncols > (1LL << 30) || rows < 0) return MEMQ_ERR_SHAPE;
    if (rows == 0) return MEMQ_OK;
    if (!gate || !up || !qs || !d) return MEMQ_ERR_NULL;
    if (!aligned_to(gate, 16) || !aligned_to(up, 16) || (z && !aligned_to(z, 16)) ||
        !aligned_to(qs, 4) || !aligned_to(d, 4))
        return MEMQ_ERR_ALIGN;
    const int sms = sm_count();
    if (sms <= 0) return MEMQ_ERR_LAUNCH;
    const int64_t n4 = rows * ncols / 4;
    const int64_t want = (n4 + kNextThreads - 1) / kNextThreads;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(want < 16LL * sms ? want : 16LL * sms));
    cfg.blockDim = dim3(kNextThreads);
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, silu_mul_q8_1_kernel, gate, up, z, qs, d, n4);
    return e == cudaSuccess ? MEMQ_OK : MEMQ_ERR_LAUNCH;
}

extern "C" int memq_repack_e4m3_q8_0(const uint8_t *w, const float *w_scale, void *out,
                                     int64_t out_f, int64_t in_f, void *stream) {
    return memq::repack_entry<false>(w, w_scale, out, out_f, in_f, stream);
}

extern "C" int memq_repack_e4m3_blk128_q8_0(const uint8_t *w, const float *grid, void *out,
                                            int64_t out_f, int64_t in_f, void *stream) {
    return memq::repack_entry<true>(w, grid, out, out_f, in_f, stream);
}
