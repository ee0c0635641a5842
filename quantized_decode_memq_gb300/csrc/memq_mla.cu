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
// Every dot product here has the same shape: lane l of a warp sums, in order, the products of
// its float4s (float4 index l + 32 c, c ascending; components x, y, z, w), then the 32 lane
// partials are added along the xor tree of offsets 16, 8, 4, 2, 1.  xor_reduce_scatter() runs
// that tree for many dots at once with fewer shuffles and the same bits, so how dots are
// batched (which the split and the head grouping change) never changes a result.
//
// head_gemv_kernel (absorb_q, decompress_v): a per-head batched GEMV over f32 weights (33.5 MB
// at the page geometry, read once: HBM-bound).  CTA (h, part) takes rows [part*rows/split,
// (part+1)*rows/split) of head h, contiguous in memory; a producer warp streams them into a
// shared-memory ring by bulk copies while 8 consumer warps take 2 rows of each stage (4 for
// t >= 4 on rows of <= 256 floats) against the t activation rows of head h (in shared memory);
// a warp releases a stage only after using what it loaded from it.  The default split fills one
// wave of resident CTAs.
//
// attn_gathered_kernel: every head of query row t gathers the same n_slots rows, so a CTA
// serves a group of H heads from one staged copy of them, and a cluster of 8 CTAs splits the
// slots into 8 fixed ranges.  The gathered rows stream into a ring of shared-memory stages by
// bulk copies (one per row, completing on an mbarrier per stage; each warp issues 2 rows of a
// chunk), issued S - 1 chunks ahead of the compute.  Each CTA runs an online softmax over its
// range (running max m, sum l, outputs rescaled by exp(m_old - m_new) per chunk of 16 rows);
// one warp per head runs the softmax step, every thread accumulates two output dims of every
// head of the group.  The 8 partials are merged through
// distributed shared memory in part order.  The slot ranges, chunks and merge order do not
// depend on H, which is the entry point's `split` (H = 8 / split), so the split twins are
// bit-identical.  No global scratch: the partials live in shared memory.
//
// All three use programmatic dependent launch.  absorb_q / decompress_v stream their constant
// weights while the preceding grid finishes and read x after griddepcontrol.wait, through L2;
// attn_gathered only sets up its barriers before the wait (every one of its inputs may come from
// the preceding grid) and then reads through L2 and the async proxy.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>

#include "memq.h"
#include "memq_dev.cuh"

namespace memq {
namespace {

// Device fault word of this translation unit: bit 2 = an attention kernel's bounded wait for
// its gathered rows expired (the kernel then stops streaming, finishes its barriers and
// returns); bit 3 = the same in absorb_q / decompress_v.
__device__ unsigned int g_mla_fault = 0;
constexpr unsigned int kFaultAttnWait = 4u;

constexpr int kMlaThreads = 256;
constexpr int kMlaWarps = kMlaThreads / 32;
constexpr int kMaxT = 8;
constexpr int kMaxHeads = 1 << 16;
constexpr int64_t kMaxGrid = (int64_t{1} << 31) - 1;
constexpr int kMaxRope = 128;  // with kv_rank <= 1024 the attention kernel fits shared memory

__host__ __device__ constexpr int ilog2(int v) { return v <= 1 ? 0 : 1 + ilog2(v / 2); }

// Sums v[e] over the 32 lanes for every e < NV (a power of two <= 32) along the xor tree of
// offsets 16, 8, 4, 2, 1, each step adding the partner's partial to one's own -- the tree of
// warp_sum, so each sum is bit-identical to warp_sum of that element.  At the step of offset o a
// lane sends the half of its remaining elements that its partner keeps (lanes with bit o set
// keep the upper half), so NV sums take NV - 1 + 5 - log2(NV) shuffles instead of 5 NV.
// On return lane l holds, in v[0], the sum of element l >> (5 - log2 NV).
template <int NV>
__device__ __forceinline__ float xor_reduce_scatter(float (&v)[NV], int lane) {
#pragma unroll
    for (int s = 0; s < 5; ++s) {
        const int off = 16 >> s;
        const int n = NV >> s;  // elements this lane still holds
        if (n > 1) {
            const bool upper = (lane & off) != 0;
#pragma unroll
            for (int i = 0; i < n / 2; ++i) {
                const float send = upper ? v[i] : v[i + n / 2];
                const float keep = upper ? v[i + n / 2] : v[i];
                v[i] = keep + __shfl_xor_sync(kFullMask, send, off);
            }
        } else {
            v[0] += __shfl_xor_sync(kFullMask, v[0], off);
        }
    }
    return v[0];
}

// ------------------------------------------------------------------------------------------
// Per-head batched GEMV.  CTA (h, part) owns rows [r0, r1) of head h, which are contiguous in
// memory: a producer warp streams them into a ring of S stages of 8 * kHeadRB rows with one bulk
// copy per stage (full barrier: transaction bytes; empty barrier: one arrival per consumer
// warp), while the 8 consumer warps take kHeadRB rows of each stage.  CV = cols / 128 float4s
// per lane per row; T = t rounded up to a power of two (rows of x beyond t are zero in shared
// memory and their sums are not stored).
// ------------------------------------------------------------------------------------------
// Rows per consumer warp per stage: 4 for several tokens on rows of <= 256 floats (the x rows
// read from shared memory then serve 4 weight rows), else 2.
__host__ __device__ constexpr int head_rb(int CV, int T) { return T >= 4 && CV <= 2 ? 4 : 2; }
constexpr int kHeadThreads = kMlaThreads + 32;  // + the producer warp
constexpr int kHeadMaxStages = 4;
constexpr unsigned int kFaultHeadWait = 8u;

struct HeadArgs {
    const float *x, *w;
    float *out;
    int t, nh, rows, split, stages;
};

template <int CV, int T>
__global__ void __launch_bounds__(kHeadThreads)
    head_gemv_kernel(const __grid_constant__ HeadArgs a) {
    constexpr int cols = CV * 128;
    constexpr int kHeadRB = head_rb(CV, T);
    constexpr int kHeadRows = kMlaWarps * kHeadRB;  // rows per stage
    constexpr int NV = kHeadRB * T;
    constexpr int kLaneShift = 5 - ilog2(NV);  // lane l holds element l >> kLaneShift
    constexpr uint32_t row_bytes = cols * 4u;
    extern __shared__ __align__(128) float hsm[];
    uint64_t *full = reinterpret_cast<uint64_t *>(hsm);  // [kHeadMaxStages]
    uint64_t *empty = full + kHeadMaxStages;             // [kHeadMaxStages]
    float *sx = hsm + 4 * kHeadMaxStages + 16;           // [T][cols] (128-byte aligned)
    float *ring = sx + T * cols;                         // [S][kHeadRows][cols]
    griddep_launch_dependents();
    const int S = a.stages, split = a.split, rows = a.rows, nh = a.nh, t = a.t;
    const int h = blockIdx.x / split;
    const int part = blockIdx.x - h * split;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r0 = static_cast<int>(static_cast<int64_t>(part) * rows / split);
    const int r1 = static_cast<int>(static_cast<int64_t>(part + 1) * rows / split);
    const int nst = (r1 - r0 + kHeadRows - 1) / kHeadRows;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kHeadMaxStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kMlaWarps);
        }
        mbar_init_fence();
    }
    __syncthreads();
    if (warp == kMlaWarps) {
        // Producer: stage st holds rows r0 + st * kHeadRows ...; slot st % S is reused once the
        // consumers released stage st - S.
        const uint64_t pol = l2_evict_first_policy();
        const float *src = a.w + (static_cast<int64_t>(h) * rows + r0) * cols;
        bool ok = true;
        int st = 0;
        for (; st < nst && ok; ++st) {
            const int slot = st % S;
            // The first S copies go out before the preceding grid has finished; the bounded
            // waits for released stages start only once it has, so that a long predecessor
            // never counts against this launch's own progress.
            if (st == S) griddep_wait();
            if (st >= S) ok = warp_wait_bounded(&empty[slot], static_cast<uint32_t>((st / S - 1) & 1));
            if (!ok) break;
            const int nrs = min(kHeadRows, r1 - r0 - st * kHeadRows);
            if (lane == 0) {
                mbar_arrive_expect_tx(&full[slot], static_cast<uint32_t>(nrs) * row_bytes);
                bulk_g2s(ring + static_cast<int64_t>(slot) * kHeadRows * cols,
                         src + static_cast<int64_t>(st) * kHeadRows * cols,
                         static_cast<uint32_t>(nrs) * row_bytes, &full[slot], pol);
            }
            __syncwarp();
        }
        if (!ok && lane == 0) atomicOr(&g_mla_fault, kFaultHeadWait);
        // Every copy issued must land before the CTA's shared memory goes away.
        for (int q = max(0, st - S); q < st; ++q)
            (void)warp_wait_bounded(&full[q % S], static_cast<uint32_t>((q / S) & 1));
        return;
    }
    // Consumers: x rows of head h into shared memory (overlapping the first weight copies).  x
    // may be the preceding launch's output: wait for that grid, then read through L2.
    griddep_wait();
    for (int i = threadIdx.x; i < T * cols / 4; i += kMlaThreads) {
        const int tt = i / (cols / 4), k = i - tt * (cols / 4);
        reinterpret_cast<float4 *>(sx)[i] =
            tt < t ? __ldcg(reinterpret_cast<const float4 *>(a.x + (static_cast<int64_t>(tt) * nh + h) * cols) + k)
                   : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    asm volatile("bar.sync 1, %0;" ::"n"(kMlaThreads) : "memory");
    const float4 *sx4 = reinterpret_cast<const float4 *>(sx);
    const int my_e = lane >> kLaneShift;
    const int my_b = my_e / T, my_t = my_e - my_b * T;
    const bool writer = (lane & ((1 << kLaneShift) - 1)) == 0;
    for (int st = 0; st < nst; ++st) {
        const int slot = st % S;
        if (!warp_wait_bounded(&full[slot], static_cast<uint32_t>((st / S) & 1))) {
            if (lane == 0) atomicOr(&g_mla_fault, kFaultHeadWait);
            break;
        }
        const int i = r0 + st * kHeadRows + warp * kHeadRB;  // this warp's first row
        const float4 *wr = reinterpret_cast<const float4 *>(ring + static_cast<int64_t>(slot) * kHeadRows * cols) +
                           warp * kHeadRB * (cols / 4);
        float4 wv[kHeadRB][CV];
#pragma unroll
        for (int b = 0; b < kHeadRB; ++b)
#pragma unroll
            for (int c = 0; c < CV; ++c) wv[b][c] = wr[b * (cols / 4) + lane + 32 * c];
        float p[NV];
#pragma unroll
        for (int tt = 0; tt < T; ++tt) {
            float4 xv[CV];
#pragma unroll
            for (int c = 0; c < CV; ++c) xv[c] = sx4[tt * (cols / 4) + lane + 32 * c];
#pragma unroll
            for (int b = 0; b < kHeadRB; ++b) {
                float s = 0.f;
#pragma unroll
                for (int c = 0; c < CV; ++c) {
                    s = fmaf(xv[c].x, wv[b][c].x, s);
                    s = fmaf(xv[c].y, wv[b][c].y, s);
                    s = fmaf(xv[c].z, wv[b][c].z, s);
                    s = fmaf(xv[c].w, wv[b][c].w, s);
                }
                p[b * T + tt] = s;
            }
        }
        // Release the stage only now: every lane has used (so received) the weights it loaded
        // from it.  An arrival right after issuing the loads would let the next bulk copy
        // overwrite the stage while loads are still in flight.
        __syncwarp();
        if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(&empty[slot])) : "memory");
        const float sum = xor_reduce_scatter<NV>(p, lane);
        if (writer && my_t < t && i + my_b < r1)
            a.out[(static_cast<int64_t>(my_t) * nh + h) * rows + i + my_b] = sum;
    }
}

// ------------------------------------------------------------------------------------------
// Gathered attention.  One cluster of kParts CTAs per (t, group of H heads); CTA `part` of the
// cluster takes the fixed slot range [part * per, (part + 1) * per) and keeps, per head, the
// running max m, sum l and unnormalised output acc[kv_rank] of an online softmax over that
// range, kRowsC gathered rows at a time.  KV = kv_rank / 128.
// ------------------------------------------------------------------------------------------
constexpr int kParts = 8;   // slot parts per (t, head group) = CTAs per cluster
constexpr int kRowsC = 16;  // gathered rows per chunk (>= 8 so one stage can hold the H x
                            // kv_rank partial outputs for the merge)
constexpr int kMaxStages = 4;
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

struct AttnArgs {
    const float *q_lat, *q_pe, *cache;
    const int32_t *idx;
    float *out;
    int nh, d_rope, n_slots, stages;
    float scale;
};

template <int KV, int H>
__global__ void __cluster_dims__(kParts, 1, 1) __launch_bounds__(kMlaThreads, H <= 2 ? 3 : 2)
    attn_gathered_kernel(const __grid_constant__ AttnArgs a) {
    constexpr int kv_rank = KV * 128;
    constexpr int KP = (kv_rank / 2 + kMlaThreads - 1) / kMlaThreads;  // output dim pairs per thread
    constexpr int NV = 2 * H;                                     // dots per warp per chunk
    constexpr int kLaneShift = 5 - ilog2(NV);
    extern __shared__ __align__(16) float sm[];
    griddep_launch_dependents();
    const int d_rope = a.d_rope, n_slots = a.n_slots, S = a.stages, nh = a.nh;
    const int row_len = kv_rank + d_rope;
    const int row_pad = (row_len + 3) & ~3;  // float4-aligned rows in shared memory
    const int stage_f = kRowsC * row_pad;
    // Bulk copies need 16-byte aligned rows in global memory: row_len % 4 == 0.  Otherwise the
    // rows are staged with plain loads into one stage, synchronously.
    const bool bulk = (row_len & 3) == 0;
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm);  // [kMaxStages] rows landed
    float *sq = sm + 2 * kMaxStages;                     // [H][row_pad]   the group's queries
    float *ring = sq + H * row_pad;                      // [S][kRowsC][row_pad]
    float *ss = ring + S * stage_f;                      // [kRowsC][H] scaled scores
    float *pw = ss + kRowsC * H;                         // [kRowsC][H] softmax weights
    float *smm = pw + kRowsC * H;                        // [H] running max
    float *sal = smm + H;                                // [H] rescale factor exp(m_old - m_new)
    float *sl = sal + H;                                 // [H] running sum

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int part = static_cast<int>(cluster_ctarank());
    const int ngrp = (nh + H - 1) / H;
    const int grp = blockIdx.x / kParts;
    const int tt = grp / ngrp, h0 = (grp - tt * ngrp) * H;

    const int per = ((n_slots + kParts - 1) / kParts + kRowsC - 1) / kRowsC * kRowsC;
    const int j_begin = min(part * per, n_slots), j_end = min(j_begin + per, n_slots);
    const int nchunks = (j_end - j_begin + kRowsC - 1) / kRowsC;
    const int32_t *ix = a.idx + static_cast<int64_t>(tt) * n_slots;
    const uint32_t row_bytes = static_cast<uint32_t>(row_len) * 4u;

    if (tid == 0) {
        for (int s = 0; s < kMaxStages; ++s) mbar_init(&bars[s], 1);
        mbar_init_fence();
    }
    // Every input may be the preceding grid's output (the absorbed query, the top-k indices,
    // the newest cache row): wait for it, then read through L2 (or the async proxy) only.
    griddep_wait();
    for (int i = tid; i < H * row_len; i += kMlaThreads) {
        const int hh = i / row_len, k = i - hh * row_len;
        const int64_t th = static_cast<int64_t>(tt) * nh + min(h0 + hh, nh - 1);
        sq[hh * row_pad + k] = k < kv_rank ? __ldcg(a.q_lat + th * kv_rank + k)
                                           : __ldcg(a.q_pe + th * d_rope + (k - kv_rank));
    }
    if (tid < H) {
        smm[tid] = -INFINITY;
        sl[tid] = 0.f;
    }
    __syncthreads();
    // The lane's latent query slices of all H heads in registers when they take <= 64 of them.
    constexpr bool kQReg = H * KV <= 16;
    float4 qreg[kQReg ? H : 1][kQReg ? KV : 1];
    if constexpr (kQReg) {
#pragma unroll
        for (int hh = 0; hh < H; ++hh)
#pragma unroll
            for (int k = 0; k < KV; ++k)
                qreg[hh][k] = reinterpret_cast<const float4 *>(sq + hh * row_pad)[lane + 32 * k];
    }

    // Every warp issues the bulk copies of 2 rows of each chunk, S - 1 chunks ahead (lane r < 2
    // copies row 2 * warp + r), so no warp carries all 16 copy issues; warp 0 lane 0 announces
    // the chunk's bytes with the stage barrier's single arrival (the phase cannot complete
    // before that arrival, whatever order the copies land in).  `nidx` holds the gather index of
    // the lane's row in the next chunk to issue, loaded one chunk ahead.
    constexpr int kRowsPerWarp = kRowsC / kMlaWarps;
    static_assert(kRowsPerWarp * kMlaWarps == kRowsC && kRowsPerWarp <= 32, "rows of a chunk per warp");
    const int my_row = warp * kRowsPerWarp + lane;  // meaningful for lane < kRowsPerWarp
    int issued = 0;
    int nidx = 0;
    if (bulk && lane < kRowsPerWarp && j_begin + my_row < j_end) nidx = __ldcg(ix + j_begin + my_row);
    auto issue_next = [&]() {  // every warp, in step; chunk `issued` into stage issued % S
        if (issued >= nchunks) return;
        const int j0 = j_begin + issued * kRowsC;
        const int nj = min(kRowsC, j_end - j0);
        uint64_t *bar = &bars[issued % S];
        if (warp == 0 && lane == 0) mbar_arrive_expect_tx(bar, static_cast<uint32_t>(nj) * row_bytes);
        if (lane < kRowsPerWarp && my_row < nj)
            bulk_g2s_plain(ring + (issued % S) * stage_f + my_row * row_pad,
                           a.cache + static_cast<int64_t>(nidx) * row_len, row_bytes, bar);
        ++issued;
        const int jn = j0 + kRowsC + my_row;
        if (lane < kRowsPerWarp && issued < nchunks && jn < j_end) nidx = __ldcg(ix + jn);
    };
    if (bulk)
        for (int c = 0; c < S - 1; ++c) issue_next();

    // Output accumulators.  Blocked (H % 4 == 0 and at least 16 outputs per thread): thread tid
    // owns heads 4 hg .. 4 hg + 3 (hg = tid / kTpg) and the dim quads dq + q kTpg (dq = tid %
    // kTpg, q < kDq), so per gathered row one 16-byte load of the row and one of the 4 weights
    // feed 16 FMAs per quad.  Otherwise thread tid owns the dim pairs 2(tid + 256 k) of every
    // head.  The f32 operations per (head, dim) are the same either way.
    constexpr bool kBlocked = H % 4 == 0 && H * KV >= 32;
    constexpr int kNg = kBlocked ? H / 4 : 1;               // head groups of 4
    constexpr int kTpg = kMlaThreads / kNg;                 // threads per head group
    constexpr int kDq = kBlocked ? kv_rank / (4 * kTpg) : 1;  // dim quads per thread
    const int hg = tid / kTpg, dq = tid - hg * kTpg;
    float4 acc4[kDq][kBlocked ? 4 : 1];
    float2 acc[kBlocked ? 1 : KP][kBlocked ? 1 : H];
    if constexpr (kBlocked) {
#pragma unroll
        for (int q = 0; q < kDq; ++q)
#pragma unroll
            for (int hh = 0; hh < 4; ++hh) acc4[q][hh] = make_float4(0.f, 0.f, 0.f, 0.f);
    } else {
#pragma unroll
        for (int k = 0; k < KP; ++k)
#pragma unroll
            for (int hh = 0; hh < H; ++hh) acc[k][hh] = make_float2(0.f, 0.f);
    }

    bool failed = false;  // this thread's wait for a stage gave up
    for (int c = 0; c < nchunks; ++c) {
        const int j0 = j_begin + c * kRowsC;
        const int nj = min(kRowsC, j_end - j0);
        const float *rows = ring + (bulk ? (c % S) * stage_f : 0);
        if (bulk) {
            if (!warp_wait_bounded(&bars[c % S], static_cast<uint32_t>((c / S) & 1))) {
                failed = true;
                if (lane == 0) atomicOr(&g_mla_fault, kFaultAttnWait);
            }
        } else {
            __syncthreads();  // every thread is done with the previous chunk's rows
            float *dst = ring;
            for (int i = tid; i < nj * row_len; i += kMlaThreads) {
                const int j = i / row_len, k = i - j * row_len;
                dst[j * row_pad + k] = __ldcg(a.cache + static_cast<int64_t>(__ldcg(ix + j0 + j)) * row_len + k);
            }
            __syncthreads();
        }
        // Scores: warp w takes rows w and w + 8 for all H heads (2H dots, one reduce-scatter);
        // both rows stay in registers while the heads' queries stream past them.
        {
            float p[NV];
            const int ja = warp < nj ? warp : 0;  // rows past the chunk end: computed, not stored
            const int jb = warp + kMlaWarps < nj ? warp + kMlaWarps : 0;
            const float4 *ra = reinterpret_cast<const float4 *>(rows + ja * row_pad);
            const float4 *rb = reinterpret_cast<const float4 *>(rows + jb * row_pad);
            float4 rva[KV], rvb[KV];
#pragma unroll
            for (int k = 0; k < KV; ++k) {
                rva[k] = ra[lane + 32 * k];
                rvb[k] = rb[lane + 32 * k];
            }
#pragma unroll
            for (int hh = 0; hh < H; ++hh) {
                const float4 *q4 = reinterpret_cast<const float4 *>(sq + hh * row_pad);
                float sa = 0.f, sb = 0.f;
#pragma unroll
                for (int k = 0; k < KV; ++k) {
                    const float4 qv = kQReg ? qreg[kQReg ? hh : 0][kQReg ? k : 0] : q4[lane + 32 * k];
                    sa = fmaf(qv.x, rva[k].x, sa);
                    sa = fmaf(qv.y, rva[k].y, sa);
                    sa = fmaf(qv.z, rva[k].z, sa);
                    sa = fmaf(qv.w, rva[k].w, sa);
                    sb = fmaf(qv.x, rvb[k].x, sb);
                    sb = fmaf(qv.y, rvb[k].y, sb);
                    sb = fmaf(qv.z, rvb[k].z, sb);
                    sb = fmaf(qv.w, rvb[k].w, sb);
                }
                for (int k = lane; k < d_rope; k += 32) {
                    const float qk = sq[hh * row_pad + kv_rank + k];
                    sa = fmaf(qk, rows[ja * row_pad + kv_rank + k], sa);
                    sb = fmaf(qk, rows[jb * row_pad + kv_rank + k], sb);
                }
                p[hh] = sa;
                p[H + hh] = sb;
            }
            const float sum = xor_reduce_scatter<NV>(p, lane);
            const int e = lane >> kLaneShift;
            const int j = warp + (e / H) * kMlaWarps, hh = e % H;
            if ((lane & ((1 << kLaneShift) - 1)) == 0 && j < nj) ss[j * H + hh] = __fmul_rn(a.scale, sum);
        }
        // The chunk's scores are complete; a wait that gave up anywhere stops every warp here,
        // together (the barrier's OR is the same in every thread).
        if (__syncthreads_or(failed)) break;
        // Every thread has also finished chunk c - 1 (its accumulate precedes these scores), so
        // stage (c - 1) % S is free: chunk c + S - 1 goes there.
        if (bulk) issue_next();
        // Online softmax step: warp hh < H updates head hh, lane j < nj holding score j.  The
        // chunk's max is a shuffle max (exact), its weight sum a fixed xor tree over lanes 0-15.
        if (warp < H) {
            const int hh = warp;
            const float mo = smm[hh];
            const float s = lane < nj ? ss[lane * H + hh] : -INFINITY;
            float mc = fmaxf(mo, s);
#pragma unroll
            for (int off = 8; off >= 1; off >>= 1) mc = fmaxf(mc, __shfl_xor_sync(kFullMask, mc, off));
            const float pj = lane < nj ? expf(s - mc) : 0.f;
            if (lane < nj) pw[lane * H + hh] = pj;
            float lc = pj;
#pragma unroll
            for (int off = 8; off >= 1; off >>= 1) lc += __shfl_xor_sync(kFullMask, lc, off);
            if (lane == 0) {
                const float al = mo == -INFINITY ? 0.f : expf(mo - mc);
                sal[hh] = al;
                sl[hh] = fmaf(sl[hh], al, lc);
                smm[hh] = mc;
            }
        }
        __syncthreads();
        // Accumulate (the rescale by exp(m_old - m_new), then the chunk's rows in order).
        if constexpr (kBlocked) {
            const float4 al = reinterpret_cast<const float4 *>(sal)[hg];
#pragma unroll
            for (int q = 0; q < kDq; ++q) {
                acc4[q][0].x *= al.x; acc4[q][0].y *= al.x; acc4[q][0].z *= al.x; acc4[q][0].w *= al.x;
                acc4[q][1].x *= al.y; acc4[q][1].y *= al.y; acc4[q][1].z *= al.y; acc4[q][1].w *= al.y;
                acc4[q][2].x *= al.z; acc4[q][2].y *= al.z; acc4[q][2].z *= al.z; acc4[q][2].w *= al.z;
                acc4[q][3].x *= al.w; acc4[q][3].y *= al.w; acc4[q][3].z *= al.w; acc4[q][3].w *= al.w;
            }
            auto row_step = [&](int j) {
                const float4 pv = reinterpret_cast<const float4 *>(pw + j * H)[hg];
                const float pj[4] = {pv.x, pv.y, pv.z, pv.w};
#pragma unroll
                for (int q = 0; q < kDq; ++q) {
                    const float4 rv = reinterpret_cast<const float4 *>(rows + j * row_pad)[dq + q * kTpg];
#pragma unroll
                    for (int hh = 0; hh < 4; ++hh) {
                        acc4[q][hh].x = fmaf(pj[hh], rv.x, acc4[q][hh].x);
                        acc4[q][hh].y = fmaf(pj[hh], rv.y, acc4[q][hh].y);
                        acc4[q][hh].z = fmaf(pj[hh], rv.z, acc4[q][hh].z);
                        acc4[q][hh].w = fmaf(pj[hh], rv.w, acc4[q][hh].w);
                    }
                }
            };
            if (nj == kRowsC) {
#pragma unroll
                for (int j = 0; j < kRowsC; ++j) row_step(j);
            } else {
                for (int j = 0; j < nj; ++j) row_step(j);
            }
        } else {
        // Thread tid owns the dim pairs (2p, 2p + 1), p = tid + 256 k; one 8-byte
        // load per row serves both dims.
#pragma unroll
        for (int k = 0; k < KP; ++k) {
            const int d = 2 * (tid + k * kMlaThreads);
            if (d < kv_rank) {
                float al[H];
#pragma unroll
                for (int hh = 0; hh < H; ++hh) al[hh] = sal[hh];
#pragma unroll
                for (int hh = 0; hh < H; ++hh) {
                    acc[k][hh].x *= al[hh];
                    acc[k][hh].y *= al[hh];
                }
                for (int j = 0; j < nj; ++j) {
                    const float2 rv = *reinterpret_cast<const float2 *>(rows + j * row_pad + d);
                    float pj[H];
                    if constexpr (H % 4 == 0) {
#pragma unroll
                        for (int q = 0; q < H / 4; ++q) {
                            const float4 v4 = reinterpret_cast<const float4 *>(pw + j * H)[q];
                            pj[4 * q] = v4.x;
                            pj[4 * q + 1] = v4.y;
                            pj[4 * q + 2] = v4.z;
                            pj[4 * q + 3] = v4.w;
                        }
                    } else if constexpr (H == 2) {
                        const float2 v2 = *reinterpret_cast<const float2 *>(pw + j * 2);
                        pj[0] = v2.x;
                        pj[1] = v2.y;
                    } else {
#pragma unroll
                        for (int hh = 0; hh < H; ++hh) pj[hh] = pw[j * H + hh];
                    }
#pragma unroll
                    for (int hh = 0; hh < H; ++hh) {
                        acc[k][hh].x = fmaf(pj[hh], rv.x, acc[k][hh].x);
                        acc[k][hh].y = fmaf(pj[hh], rv.y, acc[k][hh].y);
                    }
                }
            }
        }
        }
        // No barrier here: the next chunk's score barrier orders this accumulate before the
        // stage's reuse and before the next softmax step rewrites the weights.
    }
    if (bulk && warp == 0) {
        // Every copy issued (by any warp: all issue in step) must land before the stages take
        // the partials or the CTA exits (all of them already have unless a wait gave up).
        for (int c = max(0, issued - S); c < issued; ++c)
            (void)warp_wait_bounded(&bars[c % S], static_cast<uint32_t>((c / S) & 1));
    }
    __syncthreads();
    float *sacc = ring;  // this part's partial outputs [H][kv_rank] (fits one stage)
    if constexpr (kBlocked) {
#pragma unroll
        for (int q = 0; q < kDq; ++q)
#pragma unroll
            for (int hh = 0; hh < 4; ++hh)
                reinterpret_cast<float4 *>(sacc + (4 * hg + hh) * kv_rank)[dq + q * kTpg] = acc4[q][hh];
    } else {
#pragma unroll
        for (int k = 0; k < KP; ++k) {
            const int d = 2 * (tid + k * kMlaThreads);
            if (d < kv_rank) {
#pragma unroll
                for (int hh = 0; hh < H; ++hh) *reinterpret_cast<float2 *>(sacc + hh * kv_rank + d) = acc[k][hh];
            }
        }
    }
    cluster_sync_all();
    // Merge: this CTA finalises outputs [c0, c1) of the group's H x kv_rank, parts in order.
    const int c0 = part * (H * kv_rank) / kParts, c1 = (part + 1) * (H * kv_rank) / kParts;
    for (int i = c0 + tid; i < c1; i += kMlaThreads) {
        const int hh = i / kv_rank, d = i - hh * kv_rank;
        float mq[kParts];
        float mx = -INFINITY;
#pragma unroll
        for (int q = 0; q < kParts; ++q) {
            mq[q] = ld_dsmem(smm + hh, q);
            mx = fmaxf(mx, mq[q]);
        }
        float lsum = 0.f, o = 0.f;
#pragma unroll
        for (int q = 0; q < kParts; ++q) {
            const float wq = mq[q] == -INFINITY ? 0.f : expf(mq[q] - mx);
            lsum = fmaf(ld_dsmem(sl + hh, q), wq, lsum);
            o = fmaf(ld_dsmem(sacc + i, q), wq, o);
        }
        if (h0 + hh < nh)
            a.out[(static_cast<int64_t>(tt) * nh + h0 + hh) * kv_rank + d] = __fdiv_rn(o, lsum);
    }
    cluster_sync_all();  // no CTA leaves while another still reads its shared memory
}

// ------------------------------------------------------------------------------------------
// Gathered attention on the tensor cores (d_rope == 0, kv_rank <= 512): the same cluster
// schedule, slot ranges, online softmax and merge as attn_gathered_kernel, with both
// contractions of a 16-row chunk as mma.sync.m16n8k8 TF32 products in three terms
// (3xTF32): x = hi + lo with hi = x truncated to TF32 (exact) and lo = x - hi (exact in f32; the
// MMA reads its TF32 part), and x y ~ lo_x hi_y + hi_x lo_y + hi_x hi_y, the dropped lo lo
// term and the truncation of lo each below 2^-20 |x y|.
//   scores: S[j][h] = sum_k c_j[k] q_h[k] with M = the chunk's 16 rows, N = 8 heads (the group's
//     H, the rest zero), K = kv_rank split into 8 contiguous slices, one per warp; the 8 warp
//     partials of each (j, h) are added in warp order by the softmax step.
//   outputs: O[d][h] = O[d][h] al_h + sum_j c_j[d] p_j[h] with M = 16 dims (MMA rows g and g + 8
//     = dims 2g and 2g + 1 of the tile), N = 8 heads, K = the chunk's rows in two k8 steps; warp w
//     owns dims [w kv_rank / 8, (w + 1) kv_rank / 8).
// Each output element of an MMA depends only on its own row of A and column of B, and the
// K slicing, the k8 steps and the partial order do not depend on H, so the split twins stay
// bit-identical.  Rows are kv_rank + 8 floats apart in shared memory (8 banks), which makes
// every fragment load conflict-free.
// ------------------------------------------------------------------------------------------
__device__ __forceinline__ void tf32_split(float x, uint32_t &hi, uint32_t &lo) {
    const uint32_t b = __float_as_uint(x) & 0xFFFFE000u;
    hi = b;
    lo = __float_as_uint(x - __uint_as_float(b));
}

__device__ __forceinline__ void mma_tf32_16808(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1) {
    asm("mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// c += A B in three TF32 terms, the small cross terms first.
__device__ __forceinline__ void mma_3xtf32(float (&c)[4], const uint32_t (&ah)[4],
                                           const uint32_t (&al)[4], uint32_t bh0, uint32_t bh1,
                                           uint32_t bl0, uint32_t bl1) {
    mma_tf32_16808(c, al, bh0, bh1);
    mma_tf32_16808(c, ah, bl0, bl1);
    mma_tf32_16808(c, ah, bh0, bh1);
}

constexpr int kTcHeads = 8;  // MMA N: the head columns of a group (H of them in use)
// Row stride of the warp partials of the scores (floats): 10, so the softmax warp's 16 lanes
// reading one head of 16 rows hit 16 distinct banks (a stride of 8 put 4 rows on each bank).
constexpr int kRedRow = 10;

template <int KV, int H>
__global__ void __cluster_dims__(kParts, 1, 1) __launch_bounds__(kMlaThreads, 2)
    attn_gathered_tc_kernel(const __grid_constant__ AttnArgs a) {
    constexpr int kv_rank = KV * 128;
    constexpr int KS = kv_rank / 64;  // k8 steps of a warp's K slice (kv_rank / 8 wide)
    constexpr int MT = KV;            // 16-dim tiles of a warp's output dims (kv_rank / 8)
    constexpr int row_pad = kv_rank + 8;
    constexpr int stage_f = kRowsC * row_pad;
    extern __shared__ __align__(16) float sm[];
    griddep_launch_dependents();
    const int n_slots = a.n_slots, S = a.stages, nh = a.nh;
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm);       // [kMaxStages] rows landed
    float *ring = sm + 2 * kMaxStages;                        // [S][kRowsC][row_pad]
    float *red = ring + S * stage_f;                          // [kMlaWarps][kRowsC][kRedRow] partials
    float *pw = red + kMlaWarps * kRowsC * kRedRow;           // [kRowsC][8] softmax weights
    float *smm = pw + kRowsC * kTcHeads;                      // [8] running max
    float *sal = smm + kTcHeads;                              // [8] rescale factor
    float *sl = sal + kTcHeads;                               // [8] running sum

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, t = lane & 3;
    const int part = static_cast<int>(cluster_ctarank());
    const int ngrp = (nh + H - 1) / H;
    const int grp = blockIdx.x / kParts;
    const int tt = grp / ngrp, h0 = (grp - tt * ngrp) * H;

    const int per = ((n_slots + kParts - 1) / kParts + kRowsC - 1) / kRowsC * kRowsC;
    const int j_begin = min(part * per, n_slots), j_end = min(j_begin + per, n_slots);
    const int nchunks = (j_end - j_begin + kRowsC - 1) / kRowsC;
    const int32_t *ix = a.idx + static_cast<int64_t>(tt) * n_slots;
    constexpr uint32_t row_bytes = static_cast<uint32_t>(kv_rank) * 4u;

    if (tid == 0) {
        for (int s = 0; s < kMaxStages; ++s) mbar_init(&bars[s], 1);
        mbar_init_fence();
    }
    if (tid < kRowsC * kTcHeads) pw[tid] = 0.f;  // columns >= H stay zero
    if (tid < kTcHeads) {
        smm[tid] = -INFINITY;
        sal[tid] = 0.f;
        sl[tid] = 0.f;
    }
    // Every input may be the preceding grid's output: wait for it, then read through L2 (or the
    // async proxy) only.
    griddep_wait();
    // Bulk copies of the chunks' rows as in attn_gathered_kernel: every warp issues 2 rows of a
    // chunk, S - 1 chunks ahead; warp 0 lane 0 announces the chunk's bytes.
    constexpr int kRowsPerWarp = kRowsC / kMlaWarps;
    const int my_row = warp * kRowsPerWarp + lane;  // meaningful for lane < kRowsPerWarp
    int issued = 0;
    int nidx = 0;
    if (lane < kRowsPerWarp && j_begin + my_row < j_end) nidx = __ldcg(ix + j_begin + my_row);
    auto issue_next = [&]() {
        if (issued >= nchunks) return;
        const int j0 = j_begin + issued * kRowsC;
        const int nj = min(kRowsC, j_end - j0);
        uint64_t *bar = &bars[issued % S];
        if (warp == 0 && lane == 0) mbar_arrive_expect_tx(bar, static_cast<uint32_t>(nj) * row_bytes);
        if (lane < kRowsPerWarp && my_row < nj)
            bulk_g2s_plain(ring + (issued % S) * stage_f + my_row * row_pad,
                           a.cache + static_cast<int64_t>(nidx) * kv_rank, row_bytes, bar);
        ++issued;
        const int jn = j0 + kRowsC + my_row;
        if (lane < kRowsPerWarp && issued < nchunks && jn < j_end) nidx = __ldcg(ix + jn);
    };
    for (int c = 0; c < S - 1; ++c) issue_next();
    // The group's queries, staged in the ring's last stage (no copy writes it before the first
    // chunk's score barrier), zero for the columns >= H.
    float *sq = ring + (S - 1) * stage_f;  // [8][row_pad]
    for (int i = tid; i < kTcHeads * kv_rank; i += kMlaThreads) {
        const int hh = i / kv_rank, k = i - hh * kv_rank;
        const int64_t th = static_cast<int64_t>(tt) * nh + min(h0 + hh, nh - 1);
        sq[hh * row_pad + k] = hh < H ? __ldcg(a.q_lat + th * kv_rank + k) : 0.f;
    }
    __syncthreads();
    // The warp's B fragments of q: lane (g, t) holds q_g[kb + 8s + 2t] and q_g[kb + 8s + 2t + 1]
    // (MMA k slots t and t + 4; the rows' A fragments use the same pairing).
    const int kb = warp * (kv_rank / kMlaWarps);
    uint32_t qh[KS][2], ql[KS][2];
#pragma unroll
    for (int s = 0; s < KS; ++s) {
        const float2 qv = *reinterpret_cast<const float2 *>(sq + g * row_pad + kb + 8 * s + 2 * t);
        tf32_split(qv.x, qh[s][0], ql[s][0]);
        tf32_split(qv.y, qh[s][1], ql[s][1]);
    }
    // (the score barrier of chunk 0 orders these reads before chunk S - 1's copy into the stage)

    float acc[MT][4];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.f;
    const int d_base = warp * (kv_rank / kMlaWarps);
    bool failed = false;
    for (int c = 0; c < nchunks; ++c) {
        const int j0 = j_begin + c * kRowsC;
        const int nj = min(kRowsC, j_end - j0);
        const float *rows = ring + (c % S) * stage_f;
        if (!warp_wait_bounded(&bars[c % S], static_cast<uint32_t>((c / S) & 1))) {
            failed = true;
            if (lane == 0) atomicOr(&g_mla_fault, kFaultAttnWait);
        }
        // Scores of the warp's K slice (rows >= nj hold stale data: computed, never used), in
        // kChains independent MMA chains over the k8 steps s = kChains i + r, added in a fixed
        // tree at the end (short dependency chains; the same order for every H).
        {
            constexpr int kChains = KS >= 4 ? 4 : KS;
            float sp[kChains][4];
#pragma unroll
            for (int r = 0; r < kChains; ++r) sp[r][0] = sp[r][1] = sp[r][2] = sp[r][3] = 0.f;
            const float *ra = rows + g * row_pad + kb + 2 * t;
            const float *rb = ra + 8 * row_pad;
#pragma unroll
            for (int s = 0; s < KS; ++s) {
                const float2 va = *reinterpret_cast<const float2 *>(ra + 8 * s);
                const float2 vb = *reinterpret_cast<const float2 *>(rb + 8 * s);
                uint32_t ah[4], al[4];
                tf32_split(va.x, ah[0], al[0]);
                tf32_split(vb.x, ah[1], al[1]);
                tf32_split(va.y, ah[2], al[2]);
                tf32_split(vb.y, ah[3], al[3]);
                mma_3xtf32(sp[s % kChains], ah, al, qh[s][0], qh[s][1], ql[s][0], ql[s][1]);
            }
            float sc[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                if constexpr (kChains == 4) sc[e] = (sp[0][e] + sp[1][e]) + (sp[2][e] + sp[3][e]);
                else if constexpr (kChains == 2) sc[e] = sp[0][e] + sp[1][e];
                else sc[e] = sp[0][e];
            }
            float *rw = red + warp * (kRowsC * kRedRow);
            *reinterpret_cast<float2 *>(rw + g * kRedRow + 2 * t) = make_float2(sc[0], sc[1]);
            *reinterpret_cast<float2 *>(rw + (g + 8) * kRedRow + 2 * t) = make_float2(sc[2], sc[3]);
        }
        // The partials are complete, and every thread is done with chunk c - 1, whose stage
        // takes chunk c + S - 1.  A wait that gave up anywhere stops every warp here, together.
        if (__syncthreads_or(failed)) break;
        issue_next();
        // Online softmax step: warp hh < H updates head hh, lane j < 16 holding row j's score
        // (the 8 warp partials added in warp order, then scaled).
        if (warp < H) {
            const int hh = warp;
            const float mo = smm[hh];
            float s = -INFINITY;
            if (lane < nj) {
                float v = 0.f;
#pragma unroll
                for (int w = 0; w < kMlaWarps; ++w) v += red[(w * kRowsC + lane) * kRedRow + hh];
                s = __fmul_rn(a.scale, v);
            }
            float mc = fmaxf(mo, s);
#pragma unroll
            for (int off = 8; off >= 1; off >>= 1) mc = fmaxf(mc, __shfl_xor_sync(kFullMask, mc, off));
            const float pj = lane < nj ? expf(s - mc) : 0.f;
            if (lane < kRowsC) pw[lane * kTcHeads + hh] = pj;
            float lc = pj;
#pragma unroll
            for (int off = 8; off >= 1; off >>= 1) lc += __shfl_xor_sync(kFullMask, lc, off);
            if (lane == 0) {
                const float alv = mo == -INFINITY ? 0.f : expf(mo - mc);
                sal[hh] = alv;
                sl[hh] = fmaf(sl[hh], alv, lc);
                smm[hh] = mc;
            }
        }
        __syncthreads();
        // Outputs: rescale, then the chunk's rows in two k8 steps (rows >= nj read as zero).
        {
            const float al0 = sal[2 * t], al1 = sal[2 * t + 1];
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
                acc[mt][0] *= al0;
                acc[mt][1] *= al1;
                acc[mt][2] *= al0;
                acc[mt][3] *= al1;
            }
#pragma unroll
            for (int ks = 0; ks < 2; ++ks) {
                const int r0 = 8 * ks + t, r1 = r0 + 4;
                uint32_t bh0, bl0, bh1, bl1;
                tf32_split(pw[r0 * kTcHeads + g], bh0, bl0);
                tf32_split(pw[r1 * kTcHeads + g], bh1, bl1);
                // rows past the chunk's end read as zero (their weights are zero, their stage
                // rows stale); a full chunk needs no test
                const bool ok0 = nj == kRowsC || r0 < nj, ok1 = nj == kRowsC || r1 < nj;
                // MMA rows g and g + 8 of a 16-dim tile are the adjacent dims 2g and 2g + 1: one
                // 8-byte load per row
                const float *p0 = rows + r0 * row_pad + d_base + 2 * g;
                const float *p1 = rows + r1 * row_pad + d_base + 2 * g;
#pragma unroll
                for (int mt = 0; mt < MT; ++mt) {
                    const float2 v0 = ok0 ? *reinterpret_cast<const float2 *>(p0 + 16 * mt) : make_float2(0.f, 0.f);
                    const float2 v1 = ok1 ? *reinterpret_cast<const float2 *>(p1 + 16 * mt) : make_float2(0.f, 0.f);
                    uint32_t ah[4], al[4];
                    tf32_split(v0.x, ah[0], al[0]);
                    tf32_split(v0.y, ah[1], al[1]);
                    tf32_split(v1.x, ah[2], al[2]);
                    tf32_split(v1.y, ah[3], al[3]);
                    mma_3xtf32(acc[mt], ah, al, bh0, bh1, bl0, bl1);
                }
            }
        }
        // No barrier here: the next chunk's score barrier orders this chunk's reads before the
        // stage's reuse and before the next softmax step rewrites the weights.
    }
    if (warp == 0) {
        // Every copy issued must land before the stages take the partials or the CTA exits.
        for (int c = max(0, issued - S); c < issued; ++c)
            (void)warp_wait_bounded(&bars[c % S], static_cast<uint32_t>((c / S) & 1));
    }
    __syncthreads();
    float *sacc = ring;  // this part's partial outputs [H][kv_rank] (fits one stage)
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
        const int d = d_base + 16 * mt + 2 * g;  // acc[mt]: dims d, d + 1 x heads 2t, 2t + 1
        if (2 * t < H)
            *reinterpret_cast<float2 *>(sacc + (2 * t) * kv_rank + d) = make_float2(acc[mt][0], acc[mt][2]);
        if (2 * t + 1 < H)
            *reinterpret_cast<float2 *>(sacc + (2 * t + 1) * kv_rank + d) = make_float2(acc[mt][1], acc[mt][3]);
    }
    cluster_sync_all();
    // Merge: this CTA finalises outputs [c0, c1) of the group's H x kv_rank, parts in order.
    const int c0 = part * (H * kv_rank) / kParts, c1 = (part + 1) * (H * kv_rank) / kParts;
    for (int i = c0 + tid; i < c1; i += kMlaThreads) {
        const int hh = i / kv_rank, d = i - hh * kv_rank;
        float mq[kParts];
        float mx = -INFINITY;
#pragma unroll
        for (int q = 0; q < kParts; ++q) {
            mq[q] = ld_dsmem(smm + hh, q);
            mx = fmaxf(mx, mq[q]);
        }
        float lsum = 0.f, o = 0.f;
#pragma unroll
        for (int q = 0; q < kParts; ++q) {
            const float wq = mq[q] == -INFINITY ? 0.f : expf(mq[q] - mx);
            lsum = fmaf(ld_dsmem(sl + hh, q), wq, lsum);
            o = fmaf(ld_dsmem(sacc + i, q), wq, o);
        }
        if (h0 + hh < nh)
            a.out[(static_cast<int64_t>(tt) * nh + h0 + hh) * kv_rank + d] = __fdiv_rn(o, lsum);
    }
    cluster_sync_all();  // no CTA leaves while another still reads its shared memory
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

constexpr int kMaxDevices = 64;

// SM count of the current device (queried once per device).
int sm_count() {
    static std::atomic<int> cache[kMaxDevices];
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    if (dev < kMaxDevices && (sms = cache[dev].load(std::memory_order_relaxed)) > 0) return sms;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
    if (dev < kMaxDevices) cache[dev].store(sms, std::memory_order_relaxed);
    return sms;
}

// Lets `kern` use the device's whole opt-in shared memory, once per (kernel, device); `done`
// is the caller's per-kernel record (one bit per device).
bool allow_max_smem(const void *kern, std::atomic<uint64_t> &done) {
    int dev = 0, optin = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    const uint64_t bit = dev < kMaxDevices ? (uint64_t{1} << dev) : 0;
    if (bit && (done.load(std::memory_order_acquire) & bit)) return true;
    if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, optin) != cudaSuccess)
        return false;
    if (bit) done.fetch_or(bit, std::memory_order_acq_rel);
    return true;
}

template <int CV, int T>
int launch_head(const float *x, const float *w, float *out, int t, int nh, int rows, int split,
                cudaStream_t st) {
    const auto kern = head_gemv_kernel<CV, T>;
    const size_t fixed = sizeof(float) * (4 * kHeadMaxStages + 16 + static_cast<size_t>(T) * CV * 128);
    const size_t stage = sizeof(float) * static_cast<size_t>(kMlaWarps * head_rb(CV, T)) * CV * 128;
    // As many stages as fit in about half an SM's shared memory (two CTAs per SM), 2 to 4.
    const int stages = std::max(2, std::min(kHeadMaxStages,
                                            static_cast<int>((100 * 1024 - static_cast<int64_t>(fixed)) /
                                                             static_cast<int64_t>(stage))));
    const size_t smem = fixed + stages * stage;
    static std::atomic<uint64_t> attr_done{0};
    if (!allow_max_smem(reinterpret_cast<const void *>(kern), attr_done)) return MEMQ_ERR_LAUNCH;
    if (split == 0) {
        // one wave of resident CTAs over all heads (CTAs per SM queried once per device)
        static std::atomic<int> occ_cache[kMaxDevices];
        const int sms = sm_count();
        int dev = 0, occ = 0;
        if (sms <= 0 || cudaGetDevice(&dev) != cudaSuccess) return MEMQ_ERR_LAUNCH;
        if (dev < kMaxDevices) occ = occ_cache[dev].load(std::memory_order_relaxed);
        if (occ <= 0) {
            if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kHeadThreads, smem) != cudaSuccess)
                return MEMQ_ERR_LAUNCH;
            occ = std::max(occ, 1);
            if (dev < kMaxDevices) occ_cache[dev].store(occ, std::memory_order_relaxed);
        }
        split = static_cast<int>(std::max<int64_t>(1, static_cast<int64_t>(occ) * sms / nh));
    }
    if (split > rows) split = rows;
    if (static_cast<int64_t>(nh) * split > kMaxGrid) split = static_cast<int>(kMaxGrid / nh);
    const HeadArgs args{x, w, out, t, nh, rows, split, stages};
    // Programmatic dependent launch: the weight stream may start while the preceding grid
    // finishes; the consumers wait for it before reading x.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(nh * split));
    cfg.blockDim = dim3(kHeadThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args) == cudaSuccess ? MEMQ_OK : MEMQ_ERR_LAUNCH;
}

template <int CV>
int launch_head_t(const float *x, const float *w, float *out, int t, int nh, int rows, int split,
                  cudaStream_t st) {
    if (t <= 1) return launch_head<CV, 1>(x, w, out, t, nh, rows, split, st);
    if (t <= 2) return launch_head<CV, 2>(x, w, out, t, nh, rows, split, st);
    if (t <= 4) return launch_head<CV, 4>(x, w, out, t, nh, rows, split, st);
    return launch_head<CV, 8>(x, w, out, t, nh, rows, split, st);
}

int head_gemv_entry(const float *x, const float *w, float *out, int t, int nh, int rows, int cols,
                    int split, void *stream) {
    if (t < 1 || t > kMaxT) return MEMQ_ERR_M_RANGE;
    if (nh < 1 || nh > kMaxHeads || rows < 1 || cols < 128 || cols % 128 != 0 || cols > 1024 ||
        split < 0)
        return MEMQ_ERR_SHAPE;
    if (!x || !w || !out) return MEMQ_ERR_NULL;
    if (!aligned16(x) || !aligned16(w) || (reinterpret_cast<uintptr_t>(out) & 3u)) return MEMQ_ERR_ALIGN;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    switch (cols / 128) {
        case 1: return launch_head_t<1>(x, w, out, t, nh, rows, split, st);
        case 2: return launch_head_t<2>(x, w, out, t, nh, rows, split, st);
        case 4: return launch_head_t<4>(x, w, out, t, nh, rows, split, st);
        case 8: return launch_head_t<8>(x, w, out, t, nh, rows, split, st);
        default: return MEMQ_ERR_SHAPE;
    }
}

template <int KV, int H>
int launch_attn(const AttnArgs &args0, int t, cudaStream_t st) {
    AttnArgs args = args0;
    const int row_len = KV * 128 + args.d_rope;
    const int row_pad = (row_len + 3) & ~3;
    const size_t fixed = sizeof(uint64_t) * kMaxStages +
                         sizeof(float) * (static_cast<size_t>(H) * row_pad + 2 * kRowsC * H + 3 * H + 4);
    const size_t stage = sizeof(float) * static_cast<size_t>(kRowsC) * row_pad;
    // As many stages as fit in the share of an SM's shared memory of one of the CTAs the
    // register budget allows per SM (three for H <= 2, else two), 2 to 4.
    const int64_t budget = H <= 2 ? 72 * 1024 : 112 * 1024;
    int stages = static_cast<int>((budget - static_cast<int64_t>(fixed)) / static_cast<int64_t>(stage));
    stages = std::max(2, std::min(kMaxStages, stages));
    if ((row_len & 3) != 0) stages = 1;  // plain loads: one stage
    args.stages = stages;
    const size_t smem = fixed + stages * stage;
    static std::atomic<uint64_t> attr_done{0};
    if (!allow_max_smem(reinterpret_cast<const void *>(attn_gathered_kernel<KV, H>), attr_done))
        return MEMQ_ERR_LAUNCH;
    const unsigned groups = static_cast<unsigned>(t) * static_cast<unsigned>((args.nh + H - 1) / H);
    // Programmatic dependent launch (the cluster shape comes from the kernel's attribute).
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(groups * kParts);
    cfg.blockDim = dim3(kMlaThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, attn_gathered_kernel<KV, H>, args) == cudaSuccess ? MEMQ_OK
                                                                                      : MEMQ_ERR_LAUNCH;
}

// The tensor-core kernel (d_rope == 0): as many 16-row stages as fit beside the fixed part in
// the share of one of two CTAs per SM, 2 to kMaxStages.
template <int KV, int H>
int launch_attn_tc(const AttnArgs &args0, int t, cudaStream_t st) {
    AttnArgs args = args0;
    constexpr int row_pad = KV * 128 + 8;
    const size_t fixed = sizeof(float) * (2 * kMaxStages + kMlaWarps * kRowsC * kRedRow + kRowsC * kTcHeads +
                                          3 * kTcHeads);
    const size_t stage = sizeof(float) * static_cast<size_t>(kRowsC) * row_pad;
    const int64_t budget = 112 * 1024;
    int stages = static_cast<int>((budget - static_cast<int64_t>(fixed)) / static_cast<int64_t>(stage));
    stages = std::max(2, std::min(kMaxStages, stages));
    args.stages = stages;
    const size_t smem = fixed + stages * stage;
    static std::atomic<uint64_t> attr_done{0};
    if (!allow_max_smem(reinterpret_cast<const void *>(attn_gathered_tc_kernel<KV, H>), attr_done))
        return MEMQ_ERR_LAUNCH;
    const unsigned groups = static_cast<unsigned>(t) * static_cast<unsigned>((args.nh + H - 1) / H);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(groups * kParts);
    cfg.blockDim = dim3(kMlaThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, attn_gathered_tc_kernel<KV, H>, args) == cudaSuccess ? MEMQ_OK
                                                                                         : MEMQ_ERR_LAUNCH;
}

// Which attention kernel serves a call is fixed by (t, kv_rank, d_rope), never by the split, so
// the split twins run the same arithmetic: the tensor-core kernel for t >= 2, d_rope == 0 and
// kv_rank <= 512, the f32 kernel otherwise (measured on GB300 at the page geometry, us, tensor
// cores against f32: t = 1 44.6 / 39.6, t = 2 45.7 / 47.3, t = 4 51.9 / 64.5, t = 8 97 / 121;
// at t = 1 the 8-head MMA tiles are mostly idle for lack of query rows per SM).
template <int KV>
int launch_attn_h(int H, const AttnArgs &args, int t, cudaStream_t st) {
    if constexpr (KV <= 4) {
        if (args.d_rope == 0 && t >= 2) {
            switch (H) {
                case 8: return launch_attn_tc<KV, 8>(args, t, st);
                case 4: return launch_attn_tc<KV, 4>(args, t, st);
                case 2: return launch_attn_tc<KV, 2>(args, t, st);
                default: return launch_attn_tc<KV, 1>(args, t, st);
            }
        }
    }
    switch (H) {
        case 8: return launch_attn<KV, 8>(args, t, st);
        case 4: return launch_attn<KV, 4>(args, t, st);
        case 2: return launch_attn<KV, 2>(args, t, st);
        default: return launch_attn<KV, 1>(args, t, st);
    }
}

}  // namespace
}  // namespace memq

// Internal: this translation unit's device fault word (not part of the public header).
int memq_internal_fault_mla(unsigned int *out, bool clear) {
    if (cudaMemcpyFromSymbol(out, memq::g_mla_fault, sizeof(unsigned int)) != cudaSuccess) return 1;
    if (!clear) return 0;
    const unsigned int zero = 0;
    return cudaMemcpyToSymbol(memq::g_mla_fault, &zero, sizeof(zero)) == cudaSuccess ? 0 : 1;
}

extern "C" int memq_mla_absorb_q(const float *q_nope, const float *wk_b, float *out, int t,
                                 int nh, int d_nope, int kv_rank, int split, void *stream) {
    return memq::head_gemv_entry(q_nope, wk_b, out, t, nh, kv_rank, d_nope, split, stream);
}

extern "C" int memq_mla_decompress_v(const float *o_lat, const float *wv_b, float *out, int t,
                                     int nh, int d_v, int kv_rank, int split, void *stream) {
    return memq::head_gemv_entry(o_lat, wv_b, out, t, nh, d_v, kv_rank, split, stream);
}

extern "C" int memq_mla_attn_gathered(const float *q_lat, const float *q_pe, const float *cache,
                                      const int32_t *idx, float *out, int nh, int kv_rank,
                                      int d_rope, int t, int n_slots, float scale, int split,
                                      void *stream) {
    using namespace memq;
    if (t < 1 || t > kMaxT) return MEMQ_ERR_M_RANGE;
    if (nh < 1 || nh > kMaxHeads || kv_rank < 128 || kv_rank % 128 != 0 || kv_rank > 1024 ||
        d_rope < 0 || d_rope > kMaxRope || n_slots < 1 ||
        !(split == 0 || split == 1 || split == 2 || split == 4 || split == 8) || !std::isfinite(scale))
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
    const AttnArgs args{q_lat, q_pe, cache, idx, out, nh, d_rope, n_slots, 0, scale};
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    switch (kv_rank / 128) {
        case 1: return launch_attn_h<1>(H, args, t, st);
        case 2: return launch_attn_h<2>(H, args, t, st);
        case 4: return launch_attn_h<4>(H, args, t, st);
        case 8: return launch_attn_h<8>(H, args, t, st);
        default: return MEMQ_ERR_SHAPE;
    }
}
