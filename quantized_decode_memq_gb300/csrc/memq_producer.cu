// memq_producer.cu -- the fused RMSNorm -> q8_1 producer (memq_rmsnorm_q8_1).
//
// Operation: q8_fuse_gate.rs (memra-engine 0.125.0), module doc and `run_shape` -- the shipped
// two-launch chain `rms_norm` then `quantize_q8_1`, fused into one launch (`rms_norm_zq8_f32`)
// that emits f32 z, int8 qs and one f32 scale per 32-element block.
//
// Design (one CTA per row, the row held in registers):
//   * each thread owns V float4 slices of x (and, up to V = 8, of w), loaded once: x with an
//     L2-coherent load (it is typically the previous launch's output, see memq_dev.cuh), w
//     through the read-only path since every row shares it;
//   * sum of x^2: f32 per thread, f64 across threads (warp shuffles + a shared-memory step),
//     then r = 1/sqrt(ss/ncols + eps) with IEEE f32 divide and square root;
//   * z = (x*r)*w in f32; a 32-element block is 8 consecutive float4 slices, i.e. 8 adjacent
//     lanes, so the block amax is a 3-step xor shuffle inside each 8-lane group;
//   * d = amax/127 and qs = round(z/d) (IEEE division, ties away from zero) in f32.
// Launched with programmatic stream serialization: it releases the next launch at entry (so a
// following GEMV can start streaming its weights) and waits for its own predecessors before
// reading x.
#include <cmath>
#include <cstdint>

#include "memq.h"
#include "memq_dev.cuh"

namespace memq {
namespace {

__device__ __forceinline__ int8_t quant1(float z, float dd) {
    return dd != 0.0f ? static_cast<int8_t>(roundf(__fdiv_rn(z, dd))) : static_cast<int8_t>(0);
}

// V float4 slices per thread.  Up to V = 8 the CTA has at most 256 threads and keeps w in
// registers from the first load; at V = 16 (rows wider than 8192) it has up to 512 threads and
// reads w only in the second pass, to stay within 128 registers.
template <int V>
__global__ void __launch_bounds__(V <= 8 ? 256 : 512)
    rmsnorm_q8_1_kernel(const float *__restrict__ x, const float *__restrict__ w,
                        float *__restrict__ z, int8_t *__restrict__ qs, float *__restrict__ d,
                        int ncols, float eps) {
    griddep_launch_dependents();
    griddep_wait();

    __shared__ double red[32];
    __shared__ float r_shared;

    const int tid = threadIdx.x;
    const int nthr = blockDim.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int nf4 = ncols >> 2;
    const int64_t row = blockIdx.x;

    const float4 *xr = reinterpret_cast<const float4 *>(x + row * ncols);
    const float4 *w4 = reinterpret_cast<const float4 *>(w);

    constexpr bool kKeepW = V <= 8;
    float4 xv[V], wv[kKeepW ? V : 1];
#pragma unroll
    for (int v = 0; v < V; ++v) {
        const int f = tid + v * nthr;
        if (f < nf4) {
            xv[v] = __ldcg(xr + f);
            if (kKeepW) wv[kKeepW ? v : 0] = __ldg(w4 + f);
        } else {
            xv[v] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (kKeepW) wv[kKeepW ? v : 0] = xv[v];
        }
    }

    float ss = 0.0f;
#pragma unroll
    for (int v = 0; v < V; ++v) {
        ss = fmaf(xv[v].x, xv[v].x, ss);
        ss = fmaf(xv[v].y, xv[v].y, ss);
        ss = fmaf(xv[v].z, xv[v].z, ss);
        ss = fmaf(xv[v].w, xv[v].w, ss);
    }
    double s = warp_sum(static_cast<double>(ss));
    if (lane == 0) red[warp] = s;
    __syncthreads();
    if (warp == 0) {
        double t = lane < (nthr >> 5) ? red[lane] : 0.0;
        t = warp_sum(t);
        // mean and r in IEEE f32 (correctly rounded divide and square root): a few ulp in all.
        if (lane == 0)
            r_shared = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(
                __fdiv_rn(static_cast<float>(t), static_cast<float>(ncols)), eps)));
    }
    __syncthreads();
    const float r = r_shared;

    const int nb = ncols >> 5;
    float4 *z4 = z ? reinterpret_cast<float4 *>(z + row * ncols) : nullptr;
    uint32_t *q4 = reinterpret_cast<uint32_t *>(qs + row * ncols);
#pragma unroll
    for (int v = 0; v < V; ++v) {
        const int f = tid + v * nthr;
        float4 wk;
        if (kKeepW)
            wk = wv[kKeepW ? v : 0];
        else
            wk = f < nf4 ? __ldg(w4 + f) : make_float4(0.f, 0.f, 0.f, 0.f);
        float4 zz;
        zz.x = __fmul_rn(__fmul_rn(xv[v].x, r), wk.x);
        zz.y = __fmul_rn(__fmul_rn(xv[v].y, r), wk.y);
        zz.z = __fmul_rn(__fmul_rn(xv[v].z, r), wk.z);
        zz.w = __fmul_rn(__fmul_rn(xv[v].w, r), wk.w);
        float am = fmaxf(fmaxf(fabsf(zz.x), fabsf(zz.y)), fmaxf(fabsf(zz.z), fabsf(zz.w)));
        am = fmaxf(am, __shfl_xor_sync(kFullMask, am, 1));
        am = fmaxf(am, __shfl_xor_sync(kFullMask, am, 2));
        am = fmaxf(am, __shfl_xor_sync(kFullMask, am, 4));
        const float dd = __fdiv_rn(am, 127.0f);
        if (f < nf4) {
            const uint32_t packed = static_cast<uint32_t>(static_cast<uint8_t>(quant1(zz.x, dd))) |
                                    static_cast<uint32_t>(static_cast<uint8_t>(quant1(zz.y, dd))) << 8 |
                                    static_cast<uint32_t>(static_cast<uint8_t>(quant1(zz.z, dd))) << 16 |
                                    static_cast<uint32_t>(static_cast<uint8_t>(quant1(zz.w, dd))) << 24;
            q4[f] = packed;
            if (z4) z4[f] = zz;
            if ((tid & 7) == 0) d[row * nb + (f >> 3)] = dd;
        }
    }
}

template <int V>
cudaError_t launch_v(const float *x, const float *w, float *z, int8_t *qs, float *d, int ncols,
                     int rows, float eps, int threads, cudaStream_t st) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(rows));
    cfg.blockDim = dim3(static_cast<unsigned>(threads));
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, rmsnorm_q8_1_kernel<V>, x, w, z, qs, d, ncols, eps);
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

}  // namespace
}  // namespace memq

extern "C" int memq_rmsnorm_q8_1(const float *x, const float *w, float *z, int8_t *qs, float *d,
                                 int64_t ncols, int64_t rows, float eps, void *stream) {
    using namespace memq;
    if (ncols < 32 || ncols > MEMQ_MAX_NCOLS || (ncols % 32) != 0) return MEMQ_ERR_SHAPE;
    if (rows < 0 || rows > 0x7fffffffLL) return MEMQ_ERR_SHAPE;
    if (!(eps >= 0.0f) || std::isinf(eps)) return MEMQ_ERR_SHAPE;
    if (rows == 0) return MEMQ_OK;  // empty input: nothing to read or write, pointers unused
    if (!x || !w || !qs || !d) return MEMQ_ERR_NULL;
    if (!aligned(x, 16) || !aligned(w, 16) || (z && !aligned(z, 16)) || !aligned(qs, 4) ||
        !aligned(d, 4))
        return MEMQ_ERR_ALIGN;

    // V float4 slices per thread: the smallest power of two that keeps the CTA at <= 256
    // threads (up to 512 threads once V reaches 16).
    const int nf4 = static_cast<int>(ncols / 4);
    int v = 1;
    while (v < 16 && (nf4 + v - 1) / v > 256) v *= 2;
    const int threads = (((nf4 + v - 1) / v) + 31) / 32 * 32;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int nc = static_cast<int>(ncols), nr = static_cast<int>(rows);
    cudaError_t e;
    switch (v) {
        case 1: e = launch_v<1>(x, w, z, qs, d, nc, nr, eps, threads, st); break;
        case 2: e = launch_v<2>(x, w, z, qs, d, nc, nr, eps, threads, st); break;
        case 4: e = launch_v<4>(x, w, z, qs, d, nc, nr, eps, threads, st); break;
        case 8: e = launch_v<8>(x, w, z, qs, d, nc, nr, eps, threads, st); break;
        default: e = launch_v<16>(x, w, z, qs, d, nc, nr, eps, threads, st); break;
    }
    return e == cudaSuccess ? MEMQ_OK : MEMQ_ERR_LAUNCH;
}
