// memq_mla.cu -- the t <= 8 MLA decode attention kernels: absorb_q, decompress_v, attn_gathered.
//
// Operations: mla_decode_arm_gate.rs (memra-engine 0.125.0), module doc and `main` -- geometry
// nh = 64 heads, kv_rank = 512, d_nope = d_v = 256, d_rope = 0, a top-k gather of n_slots = 2048
// rows from a cache of kv rows, t_q in {1, 2, 4, 8}; each kernel has "split twins" whose outputs
// must equal the unsplit kernel's bit for bit (the split changes launch geometry only).
//
//   absorb_q      out[t][h][r] = sum_d q_nope[t][h][d] * wk_b[h][r][d]
//   decompress_v  out[t][h][v] = sum_r o_lat[t][h][r] * wv_b[h][v][r]
//   attn_gathered out[t][h][:] = softmax_j(scale * (q_lat[t][h] . c_j + q_pe[t][h] . c_j,rope)) . c_j
//                 over the gathered rows c_j = cache[idx[t][j]]
//
// head_gemv_kernel (absorb_q, decompress_v): a per-head batched GEMV over f32 weights (33.5 MB
// at the page geometry, read once: HBM-bound).  CTA (h, part) takes rows [part*rows/split,
// (part+1)*rows/split) of head h; a warp streams whole weight rows as float4s (two rows at a
// time), the t activation rows of head h sit in shared memory.  A row's sum is the lane's
// float4s in increasing order, then a fixed xor-shuffle tree: the same operations for every
// split, so the split twins are bit-identical by construction.
//
// attn_gathered_kernel: every head of query row t gathers the same n_slots rows, so a CTA
// serves a group of H heads from one staged copy of them, and a cluster of 8 CTAs splits the
// slots into 8 fixed ranges.  Each CTA runs an online softmax over its range (running max m,
// sum l, outputs rescaled by exp(m_old - m_new) per staged chunk of 16 rows); the 8 partials
// are merged through distributed shared memory in part order.  The slot ranges, chunks and
// merge order do not depend on H, which is the entry point's `split` (H = 8 / split), so the
// split twins are bit-identical.  No global scratch: the partials live in shared memory.
//
// Plain stream-ordered launches (no programmatic dependent launch): every input is complete
// when a kernel starts.
#include <cmath>
#include <cstdint>

#include "memq.h"
#include "memq_dev.cuh"

namespace memq {
namespace {

constexpr int kMlaThreads = 256;
constexpr int kMlaWarps = kMlaThreads / 32;
constexpr int kMaxT = 8;
constexpr int kMaxHeads = 1 << 16;
constexpr int64_t kMaxGrid = (int64_t{1} << 31) - 1;
constexpr int kMaxRope = 128;  // with kv_rank <= 1024: at most 152 KB of shared memory

// ------------------------------------------------------------------------------------------
// Per-head batched GEMV.  CV = cols / 128 float4s per lane per row (2 or 4 at the page
// geometry; any cols that is a multiple of 128 up to 1024).
// ------------------------------------------------------------------------------------------
template <int CV>
__global__ void __launch_bounds__(kMlaThreads)
    head_gemv_kernel(const float *__restrict__ x, const float *__restrict__ w,
                     float *__restrict__ out, int t, int nh, int rows, int split) {
    extern __shared__ __align__(16) float sx[];  // [t][cols]
    constexpr int cols = CV * 128;
    const int h = blockIdx.x / split;
    const int part = blockIdx.x - h * split;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int i = threadIdx.x; i < t * cols / 4; i += kMlaThreads) {
        const int tt = i / (cols / 4), k = i - tt * (cols / 4);
        reinterpret_cast<float4 *>(sx)[i] =
            __ldg(reinterpret_cast<const float4 *>(x + (static_cast<int64_t>(tt) * nh + h) * cols) + k);
    }
    __syncthreads();
    const int r0 = static_cast<int>(static_cast<int64_t>(part) * rows / split);
    const int r1 = static_cast<int>(static_cast<int64_t>(part + 1) * rows / split);
    const float4 *wh = reinterpret_cast<const float4 *>(w + static_cast<int64_t>(h) * rows * cols);
    const float4 *sx4 = reinterpret_cast<const float4 *>(sx);
    for (int i = r0 + 2 * warp; i < r1; i += 2 * kMlaWarps) {
        const bool two = i + 1 < r1;
        float4 wa[CV], wb[CV];
#pragma unroll
        for (int c = 0; c < CV; ++c) {
            wa[c] = __ldcs(wh + static_cast<int64_t>(i) * (cols / 4) + lane + 32 * c);
            wb[c] = two ? __ldcs(wh + static_cast<int64_t>(i + 1) * (cols / 4) + lane + 32 * c)
                        : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        for (int tt = 0; tt < t; ++tt) {
            float pa = 0.f, pb = 0.f;
#pragma unroll
            for (int c = 0; c < CV; ++c) {
                const float4 xv = sx4[tt * (cols / 4) + lane + 32 * c];
                pa = fmaf(xv.x, wa[c].x, pa);
                pa = fmaf(xv.y, wa[c].y, pa);
                pa = fmaf(xv.z, wa[c].z, pa);
                pa = fmaf(xv.w, wa[c].w, pa);
                pb = fmaf(xv.x, wb[c].x, pb);
                pb = fmaf(xv.y, wb[c].y, pb);
                pb = fmaf(xv.z, wb[c].z, pb);
                pb = fmaf(xv.w, wb[c].w, pb);
            }
            pa = warp_sum(pa);
            pb = warp_sum(pb);
            if (lane == 0) {
                out[(static_cast<int64_t>(tt) * nh + h) * rows + i] = pa;
                if (two) out[(static_cast<int64_t>(tt) * nh + h) * rows + i + 1] = pb;
            }
        }
    }
}

// ------------------------------------------------------------------------------------------
// Gathered attention.  One cluster of kParts CTAs per (t, group of H heads); CTA `part` of the
// cluster takes the fixed slot range [part * per, (part + 1) * per) and keeps, per head, the
// running max m, sum l and unnormalised output acc[kv_rank] of an online softmax over that
// range, kRowsC staged rows at a time.  The partials are then combined through distributed
// shared memory, part 0 first.  Nothing in a (t, h, r) output's arithmetic depends on H, so
// every head grouping (the `split` of the entry point) gives the same bits.
// ------------------------------------------------------------------------------------------
constexpr int kParts = 8;   // slot parts per (t, head group) = CTAs per cluster
constexpr int kRowsC = 16;  // gathered rows staged per step (>= 8 so the rows buffer can hold
                            // the H x kv_rank partial outputs for the combine)

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// All threads of every CTA in the cluster arrive; shared-memory writes before it are visible to
// the cluster's reads after it.
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                     : "memory");
}
// f32 at the same shared-memory offset as `p`, in the shared memory of cluster CTA `rank`.
__device__ __forceinline__ float ld_dsmem(const float *p, uint32_t rank) {
    uint32_t a;
    float v;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(smem_u32(p)), "r"(rank));
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(a) : "memory");
    return v;
}

template <int KV, int H>
__global__ void __cluster_dims__(kParts, 1, 1) __launch_bounds__(kMlaThreads)
    attn_gathered_kernel(const float *__restrict__ q_lat, const float *__restrict__ q_pe,
                         const float *__restrict__ cache, const int32_t *__restrict__ idx,
                         float *__restrict__ out, int nh, int d_rope, int n_slots, float scale) {
    constexpr int kv_rank = KV * 128;
    constexpr int KD = (kv_rank + kMlaThreads - 1) / kMlaThreads;  // output dims per thread
    extern __shared__ __align__(16) float sm[];
    const int row_len = kv_rank + d_rope;
    const int row_pad = (row_len + 3) & ~3;  // float4-aligned rows in shared memory
    float *sq = sm;                           // [H][row_pad]   the group's queries
    float *rows = sq + H * row_pad;           // [kRowsC][row_pad], then [H][kv_rank] partials
    float *ss = rows + kRowsC * row_pad;      // [kRowsC][H]    scaled scores of the chunk
    float *pw = ss + kRowsC * H;              // [kRowsC][H]    softmax weights of the chunk
    float *smm = pw + kRowsC * H;             // [H] running max
    float *smn = smm + H;                     // [H] the chunk's new max
    float *sal = smn + H;                     // [H] rescale factor exp(m_old - m_new)
    float *sl = sal + H;                      // [H] running sum

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int part = static_cast<int>(cluster_ctarank());
    const int ngrp = (nh + H - 1) / H;
    const int grp = blockIdx.x / kParts;
    const int tt = grp / ngrp, h0 = (grp - tt * ngrp) * H;

    for (int i = tid; i < H * row_len; i += kMlaThreads) {
        const int hh = i / row_len, k = i - hh * row_len;
        const int64_t th = static_cast<int64_t>(tt) * nh + min(h0 + hh, nh - 1);
        sq[hh * row_pad + k] = k < kv_rank ? __ldg(q_lat + th * kv_rank + k)
                                           : __ldg(q_pe + th * d_rope + (k - kv_rank));
    }
    if (tid < H) {
        smm[tid] = -INFINITY;
        sl[tid] = 0.f;
    }
    const int per = ((n_slots + kParts - 1) / kParts + kRowsC - 1) / kRowsC * kRowsC;
    const int j_begin = min(part * per, n_slots), j_end = min(j_begin + per, n_slots);
    const int32_t *ix = idx + static_cast<int64_t>(tt) * n_slots;

    float acc[KD][H];
#pragma unroll
    for (int k = 0; k < KD; ++k)
#pragma unroll
        for (int hh = 0; hh < H; ++hh) acc[k][hh] = 0.f;

    for (int j0 = j_begin; j0 < j_end; j0 += kRowsC) {
        const int nj = min(kRowsC, j_end - j0);
        __syncthreads();  // the previous chunk's rows and weights are no longer read
        for (int i = tid; i < nj * (kv_rank / 4); i += kMlaThreads) {
            const int j = i / (kv_rank / 4), k = i - j * (kv_rank / 4);
            const float *src = cache + static_cast<int64_t>(__ldg(ix + j0 + j)) * row_len + 4 * k;
            float4 v;
            if (row_len % 4 == 0) {
                v = __ldg(reinterpret_cast<const float4 *>(src));
            } else {
                v = make_float4(__ldg(src), __ldg(src + 1), __ldg(src + 2), __ldg(src + 3));
            }
            reinterpret_cast<float4 *>(rows + j * row_pad)[k] = v;
        }
        for (int i = tid; i < nj * d_rope; i += kMlaThreads) {
            const int j = i / d_rope, k = i - j * d_rope;
            rows[j * row_pad + kv_rank + k] =
                __ldg(cache + static_cast<int64_t>(__ldg(ix + j0 + j)) * row_len + kv_rank + k);
        }
        __syncthreads();
        // Scores: warp w takes rows w, w + 8; a lane's partial covers its float4s of the latent
        // part in order, then its rope floats; a fixed xor tree sums the lanes.
        for (int j = warp; j < nj; j += kMlaWarps) {
            const float4 *r4 = reinterpret_cast<const float4 *>(rows + j * row_pad);
            float4 rv[KV];
#pragma unroll
            for (int c = 0; c < KV; ++c) rv[c] = r4[lane + 32 * c];
#pragma unroll
            for (int hh = 0; hh < H; ++hh) {
                const float4 *q4 = reinterpret_cast<const float4 *>(sq + hh * row_pad);
                float s = 0.f;
#pragma unroll
                for (int c = 0; c < KV; ++c) {
                    const float4 a = q4[lane + 32 * c];
                    s = fmaf(a.x, rv[c].x, s);
                    s = fmaf(a.y, rv[c].y, s);
                    s = fmaf(a.z, rv[c].z, s);
                    s = fmaf(a.w, rv[c].w, s);
                }
                for (int k = lane; k < d_rope; k += 32)
                    s = fmaf(sq[hh * row_pad + kv_rank + k], rows[j * row_pad + kv_rank + k], s);
                s = warp_sum(s);
                if (lane == 0) ss[j * H + hh] = __fmul_rn(scale, s);
            }
        }
        __syncthreads();
        // Online softmax step, per head: new max over the chunk, weights, rescale factor.
        if (tid < nj * H) {
            const int hh = tid % H, j = tid / H;
            const float mo = smm[hh];
            float mc = mo;
            for (int q = 0; q < nj; ++q) mc = fmaxf(mc, ss[q * H + hh]);
            pw[tid] = expf(ss[tid] - mc);
            if (j == 0) {
                sal[hh] = mo == -INFINITY ? 0.f : expf(mo - mc);
                smn[hh] = mc;
            }
        }
        __syncthreads();
#pragma unroll
        for (int k = 0; k < KD; ++k) {
            const int d = tid + k * kMlaThreads;
            if (d < kv_rank) {
#pragma unroll
                for (int hh = 0; hh < H; ++hh) acc[k][hh] *= sal[hh];
                for (int j = 0; j < nj; ++j) {
                    const float rv = rows[j * row_pad + d];
#pragma unroll
                    for (int hh = 0; hh < H; ++hh) acc[k][hh] = fmaf(pw[j * H + hh], rv, acc[k][hh]);
                }
            }
        }
        if (tid < H) {
            float lc = 0.f;
            for (int j = 0; j < nj; ++j) lc += pw[j * H + tid];
            sl[tid] = fmaf(sl[tid], sal[tid], lc);
            smm[tid] = smn[tid];
        }
    }
    __syncthreads();  // the rows buffer is free: it takes this part's partial outputs
    float *sacc = rows;
#pragma unroll
    for (int k = 0; k < KD; ++k) {
        const int d = tid + k * kMlaThreads;
        if (d < kv_rank) {
#pragma unroll
            for (int hh = 0; hh < H; ++hh) sacc[hh * kv_rank + d] = acc[k][hh];
        }
    }
    cluster_sync_all();
    // Combine: this CTA finalises outputs [c0, c1) of the group's H x kv_rank, parts in order.
    const int c0 = part * (H * kv_rank) / kParts, c1 = (part + 1) * (H * kv_rank) / kParts;
    for (int i = c0 + tid; i < c1; i += kMlaThreads) {
        const int hh = i / kv_rank, d = i - hh * kv_rank;
        float mx = -INFINITY;
#pragma unroll
        for (int q = 0; q < kParts; ++q) mx = fmaxf(mx, ld_dsmem(smm + hh, q));
        float lsum = 0.f, o = 0.f;
#pragma unroll
        for (int q = 0; q < kParts; ++q) {
            const float mq = ld_dsmem(smm + hh, q);
            const float wq = mq == -INFINITY ? 0.f : expf(mq - mx);
            lsum = fmaf(ld_dsmem(sl + hh, q), wq, lsum);
            o = fmaf(ld_dsmem(sacc + i, q), wq, o);
        }
        if (h0 + hh < nh)
            out[(static_cast<int64_t>(tt) * nh + h0 + hh) * kv_rank + d] = __fdiv_rn(o, lsum);
    }
    cluster_sync_all();  // no CTA leaves while another still reads its shared memory
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int sm_count() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
    return sms;
}

int head_gemv_entry(const float *x, const float *w, float *out, int t, int nh, int rows, int cols,
                    int split, void *stream) {
    if (t < 1 || t > kMaxT) return MEMQ_ERR_M_RANGE;
    if (nh < 1 || nh > kMaxHeads || rows < 1 || cols < 128 || cols % 128 != 0 || cols > 1024 ||
        split < 0)
        return MEMQ_ERR_SHAPE;
    if (!x || !w || !out) return MEMQ_ERR_NULL;
    if (!aligned16(x) || !aligned16(w) || (reinterpret_cast<uintptr_t>(out) & 3u)) return MEMQ_ERR_ALIGN;
    const int sms = sm_count();
    if (sms <= 0) return MEMQ_ERR_LAUNCH;
    if (split == 0) split = (4 * sms + nh - 1) / nh;
    if (split > rows) split = rows;
    if (static_cast<int64_t>(nh) * split > kMaxGrid) split = static_cast<int>(kMaxGrid / nh);
    const size_t smem = static_cast<size_t>(t) * cols * sizeof(float);
    const dim3 grid(static_cast<unsigned>(nh * split));
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    switch (cols / 128) {
        case 1: head_gemv_kernel<1><<<grid, kMlaThreads, smem, st>>>(x, w, out, t, nh, rows, split); break;
        case 2: head_gemv_kernel<2><<<grid, kMlaThreads, smem, st>>>(x, w, out, t, nh, rows, split); break;
        case 4: head_gemv_kernel<4><<<grid, kMlaThreads, smem, st>>>(x, w, out, t, nh, rows, split); break;
        case 8: head_gemv_kernel<8><<<grid, kMlaThreads, smem, st>>>(x, w, out, t, nh, rows, split); break;
        default: return MEMQ_ERR_SHAPE;
    }
    return cudaGetLastError() == cudaSuccess ? MEMQ_OK : MEMQ_ERR_LAUNCH;
}

}  // namespace
}  // namespace memq

extern "C" int memq_mla_absorb_q(const float *q_nope, const float *wk_b, float *out, int t,
                                 int nh, int d_nope, int kv_rank, int split, void *stream) {
    return memq::head_gemv_entry(q_nope, wk_b, out, t, nh, kv_rank, d_nope, split, stream);
}

extern "C" int memq_mla_decompress_v(const float *o_lat, const float *wv_b, float *out, int t,
                                     int nh, int d_v, int kv_rank, int split, void *stream) {
    return memq::head_gemv_entry(o_lat, wv_b, out, t, nh, d_v, kv_rank, split, stream);
}

namespace memq {
namespace {

template <int KV, int H>
int launch_attn(const float *q_lat, const float *q_pe, const float *cache, const int32_t *idx,
                float *out, int nh, int d_rope, int t, int n_slots, float scale, cudaStream_t st) {
    const int row_pad = (KV * 128 + d_rope + 3) & ~3;
    const size_t smem = sizeof(float) * (static_cast<size_t>(row_pad) * (H + kRowsC) +
                                         2 * kRowsC * H + 4 * H);
    if (cudaFuncSetAttribute(attn_gathered_kernel<KV, H>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
        return MEMQ_ERR_LAUNCH;
    const unsigned groups = static_cast<unsigned>(t) * static_cast<unsigned>((nh + H - 1) / H);
    attn_gathered_kernel<KV, H><<<groups * kParts, kMlaThreads, smem, st>>>(
        q_lat, q_pe, cache, idx, out, nh, d_rope, n_slots, scale);
    return cudaGetLastError() == cudaSuccess ? MEMQ_OK : MEMQ_ERR_LAUNCH;
}

template <int KV>
int launch_attn_h(int H, const float *q_lat, const float *q_pe, const float *cache,
                  const int32_t *idx, float *out, int nh, int d_rope, int t, int n_slots,
                  float scale, cudaStream_t st) {
    switch (H) {
        case 8: return launch_attn<KV, 8>(q_lat, q_pe, cache, idx, out, nh, d_rope, t, n_slots, scale, st);
        case 4: return launch_attn<KV, 4>(q_lat, q_pe, cache, idx, out, nh, d_rope, t, n_slots, scale, st);
        case 2: return launch_attn<KV, 2>(q_lat, q_pe, cache, idx, out, nh, d_rope, t, n_slots, scale, st);
        default: return launch_attn<KV, 1>(q_lat, q_pe, cache, idx, out, nh, d_rope, t, n_slots, scale, st);
    }
}

}  // namespace
}  // namespace memq

extern "C" int memq_mla_attn_gathered(const float *q_lat, const float *q_pe, const float *cache,
                                      const int32_t *idx, float *out, int nh, int kv_rank,
                                      int d_rope, int t, int n_slots, float scale, int split,
                                      void *stream) {
    using namespace memq;
    if (t < 1 || t > kMaxT) return MEMQ_ERR_M_RANGE;
    if (nh < 1 || nh > kMaxHeads || kv_rank < 128 || kv_rank % 128 != 0 || kv_rank > 1024 || d_rope < 0 ||
        d_rope > kMaxRope || n_slots < 1 || !(split == 0 || split == 1 || split == 2 ||
                                               split == 4 || split == 8) ||
        !std::isfinite(scale))
        return MEMQ_ERR_SHAPE;
    if (!q_lat || !cache || !idx || !out || (d_rope > 0 && !q_pe)) return MEMQ_ERR_NULL;
    if (!aligned16(cache) || (reinterpret_cast<uintptr_t>(q_lat) & 3u) ||
        (reinterpret_cast<uintptr_t>(q_pe) & 3u) || (reinterpret_cast<uintptr_t>(out) & 3u) ||
        (reinterpret_cast<uintptr_t>(idx) & 3u))
        return MEMQ_ERR_ALIGN;
    if (split == 0) {
        // the widest head group that still gives every SM a cluster member
        const int sms = sm_count();
        if (sms <= 0) return MEMQ_ERR_LAUNCH;
        split = 8;
        for (int s = 1; s <= 8; s *= 2) {
            const int h = 8 / s;
            if (static_cast<int64_t>(t) * ((nh + h - 1) / h) * kParts >= sms) {
                split = s;
                break;
            }
        }
    }
    const int H = 8 / split;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    switch (kv_rank / 128) {
        case 1: return launch_attn_h<1>(H, q_lat, q_pe, cache, idx, out, nh, d_rope, t, n_slots, scale, st);
        case 2: return launch_attn_h<2>(H, q_lat, q_pe, cache, idx, out, nh, d_rope, t, n_slots, scale, st);
        case 4: return launch_attn_h<4>(H, q_lat, q_pe, cache, idx, out, nh, d_rope, t, n_slots, scale, st);
        case 8: return launch_attn_h<8>(H, q_lat, q_pe, cache, idx, out, nh, d_rope, t, n_slots, scale, st);
        default: return MEMQ_ERR_SHAPE;
    }
}
