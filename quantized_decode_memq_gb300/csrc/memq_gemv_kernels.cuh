// memq_gemv_kernels.cuh -- weight-stream GEMVs against a q8_1 activation, m <= 8 activation
// rows, and the fused RMSNorm -> q8_1 -> GEMV decode step.  Included once per container by
// memq_gemv_e4m3.cu, memq_gemv_blk128.cu and memq_gemv_q8_0.cu (one translation unit each, so
// they compile in parallel).
//
// Operations: gemv_e4m3_bench.rs (memra-engine 0.125.0), module doc -- "THE COMPARISON" (arm
// E4M3: raw E4M3 bytes, one per-tensor scale; arm Q8_0: ggml block_q8_0, 34 B per 32 weights)
// and "THE BLOCK-128 ARM" (E4M3 plus an f32 [ceil(out_f/128), ceil(in_f/128)] scale grid).
//
// Fast path (the "stream" or tile kernel), one skeleton for all three containers:
//   * CTA c owns output rows [R0, R1), an equal share (+-1 row) of out_f.  It walks its rows in
//     16-row tiles and each tile's K dimension in chunks of 32 blocks (1 KB of E4M3, 1088 B of
//     Q8_0 per row).
//   * One producer warp fills a shared ring of S stages: a full tile (or the first 8 rows of a
//     ragged one) arrives as one 2-D tensor copy (cp.async.bulk.tensor, L2 evict-first) into row
//     slots padded against bank conflicts, leftover rows as 1-D bulk copies, all completing on
//     the stage's "full" mbarrier.  Eight consumer warps wait on it (bounded), compute, and
//     release the stage on its "empty" mbarrier.
//   * E4M3 / block-128, and Q8_0 from a few activation rows on: consumer warp w takes blocks
//     4w..4w+3 of every stage and computes them on the tensor cores (mma.sync m16n8k16, f16
//     operands, f32 accumulation); E4M3 -> f16 (hardware cvt) and int8 -> f16 are exact and f16 x
//     f16 products are exact in f32.  At the end of a tile each warp leaves its partial sums in
//     shared memory; after one barrier among the consumers the 8 partials of each (row, token)
//     are added in warp order (deterministic) and stored.
//   * Q8_0 with dp4a: warp w takes rows 2w and 2w + 1 (one per half-warp), lane l blocks l % 16
//     and l % 16 + 16 of every stage; dp4a gives the exact int32 dot product of each block.
//   * The activation is read once per CTA, after the wait for the preceding launch: as f16 MMA
//     fragments, as staged qs / d, or in the dp4a record-aligned layout.  The producer starts
//     streaming before that wait (programmatic dependent launch): it never reads what the
//     preceding launch writes.
// The K-outer kernel (memq_gemv_kouter.cuh) serves CTAs of 8 to 16 rows with wide activations.
// Generic path: a plain warp-per-row kernel with byte loads for anything the fast path does not
// take (unaligned pointers, Q8_0 rows that are not 16-byte aligned).
#pragma once

#include <algorithm>
#include <cmath>
#include <atomic>
#include <cstdint>
#include <cuda.h>
#include <cuda_fp16.h>
#include <mutex>

#include "memq.h"
#include "memq_dev.cuh"

namespace memq {

namespace {

// Device-side fault word of this translation unit (bit 0: a consumer's bounded mbarrier wait
// expired; bit 1: the producer's).  memq_device_fault reads and clears all of them.
__device__ unsigned int g_memq_fault = 0;

constexpr int kWarps = 8;                    // consumer warps
constexpr int kThreads = (kWarps + 1) * 32;  // + one producer warp
constexpr int kConsumerThreads = kWarps * 32;
constexpr int kBarConsumers = 1;             // named barrier id used by the consumer warps

// kQ80T is Q8_0 computed on the tensor cores (taken from kQ80MmaMinM activation rows up); the
// public Q8_0 entry points choose between kQ80 and kQ80T.
enum Kind : int { kE4M3 = 0, kBlk = 1, kQ80 = 2, kQ80T = 3 };
constexpr int kQ80MmaMinM = 3;

constexpr bool is_q80(int kind) { return kind == kQ80 || kind == kQ80T; }

// Which Q8_0 path a call takes.  dp4a reads the activation once per weight row, so from a few
// activation rows on it is bound by shared-memory bandwidth; the tensor-core path reads it once
// per 16-row block step but needs 16-row tiles and a larger staged activation.  Measured on
// GB300 (back-to-back, DRAM-cold): tensor cores win from m = 6 on every shape (17408 x 5120,
// m = 8: 23 us against 49 us; 5120 x 17408, m = 6: 38 against 47 us), from m = 5 when the
// activation is small enough to keep several CTAs per SM (17408 x 5120, m = 5: 20.7 against
// 34.6 us), and from m = 4 with many rows (17408 x 5120: 19.6 against 20.8 us; 12288 x 5120:
// 15.3 against 16.0 us).  At m = 3 dp4a on two CTAs per SM is ahead there (17408 x 5120: 17.9
// against 22.1 us; 12288 x 5120: 14.2 against 15.7 us).  With 5120 rows the tile kernel's
// tensor-core launch has a floor of ~12.4 us (16-row tiles leave CTAs with one full and one
// ragged tile), so dp4a stays ahead up to m = 4 there (10.9 against 12.5 us at m = 4) unless
// the K-outer kernel applies (it is tried first); with a 17408-wide activation at m = 3-5, or
// 1024 rows, dp4a is as fast or faster.
inline bool q80_on_tensor_cores(int64_t out_f, int64_t in_f, int m) {
    if (m >= 6) return true;
    if (m < kQ80MmaMinM || m * in_f > 40960 || out_f < 2048) return false;
    return m >= 5 || (m >= 4 && out_f >= 8192);
}

// Q8_0 with dp4a: rows per consumer warp in a tile (q80_pair_row: the two half-warps take two
// adjacent rows).
constexpr int kQ8RowsPerWarp = 2;

// Stream-kernel geometry per container.  A stage holds 32 blocks of every tile row.
//   E4M3 / block-128: 16-row tiles (one m16 MMA row tile); row slots padded to 1056 bytes (a row
//   stride of 32 bytes modulo the 128-byte bank period): a warp's 8-byte fragment loads cover
//   rows g = 0..7 at byte 8t of a block, and each group of 16 lanes (rows 4i..4i+3) then hits
//   32 distinct banks, so the loads are conflict-free.
//   Q8_0 (dp4a): 8 * kQ8RowsPerWarp-row tiles, 1088-byte row slots (34-byte blocks).
//   Q8_0 (tensor cores): 16-row tiles, row slots padded to 1104 bytes.
template <int KIND>
struct Geo {
    static constexpr bool kMma = KIND != kQ80;
    static constexpr int kBlockBytes = is_q80(KIND) ? 34 : 32;
    static constexpr int kTileRows = kMma ? 16 : kWarps * kQ8RowsPerWarp;
    static constexpr int kChunkBlocks = 32;
    static constexpr int kSlot = kChunkBlocks * kBlockBytes + (!kMma ? 0 : is_q80(KIND) ? 16 : 32);
    static constexpr int kStage = kTileRows * kSlot;
    static constexpr int kMinStages = 3;
    // Register budget: three (tensor-core kernels) or four (Q8_0 with dp4a) CTAs per SM; the
    // plan (plan_stream) may use fewer.
    static constexpr int kMinCtasPerSm = kMma ? 3 : 4;
    // CTAs per SM one launch uses (at most kMinCtasPerSm).
    static constexpr int kCtasPerLaunch = kMinCtasPerSm;
    static constexpr int kMaxStages = 12;
    static constexpr int kWarpBlocks = kChunkBlocks / kWarps;  // E4M3: blocks per warp per stage
};

// Weight matrices one launch may cover (sharing the activation: gate / up, q / k / v).
constexpr int kMaxGroup = 4;

struct StreamArgs {
    const uint8_t *w;
    const float *aux;  // per-tensor scale (E4M3) or grid (block-128); unused for Q8_0
    const int8_t *qs;
    const float *d;
    float *y;
    int64_t out_f;
    int64_t row_bytes;
    int in_f;
    int nb;     // in_f / 32
    int gcols;  // ceil(in_f / 128)
    int stages;
    int grid_rows;  // block-128: grid rows staged per CTA (bound)
    // Fused decode step only: the f32 activation rows and RMSNorm weight the prologue
    // quantizes, and where CTA 0 publishes the q8_1 activation (z optional).
    const float *x;
    const float *wn;
    float eps;
    float *z_out;
    // Shared-memory layout (bytes); barriers at 0.
    uint32_t off_part, off_bfrag, off_qs, off_d, off_grid, off_red, off_ring;
    // Row strides of the staged activation: qstr bytes per token row of qs (in_f, or padded to
    // 32 mod 128 where the tensor-core consumers convert B fragments from it), dstr floats per
    // token row of d (padded to 4 mod 16, so the scales of tokens 0, 2, 4, 6 one warp loads fall
    // on different banks).
    int qstr, dstr;
    int use_tma;  // 1: full tiles (and 8-row halves) come as one tensor copy each
    int ctas_per_sm;  // host: CTAs per SM the plan sized shared memory for
    // The launch's matrices: matrix i owns CTAs [mat_cta[i], mat_cta[i+1]); each CTA takes w,
    // aux, y and out_f above from its matrix.  A plain GEMV is a group of one.
    int nmat;
    int mat_cta[kMaxGroup + 1];
    const uint8_t *mat_w[kMaxGroup];
    const float *mat_aux[kMaxGroup];
    float *mat_y[kMaxGroup];
    int64_t mat_out_f[kMaxGroup];
};

// Tensor maps over the weight plane viewed as [out_f rows][row_bytes / 8] 64-bit elements, box
// = one chunk slot (kSlot bytes, i.e. the 1 KB / 1088 B chunk plus the row padding of the shared
// layout) x `rows`: `tile` covers a whole tile, `oct` 8 rows.  A box lands in shared memory as
// rows of kSlot bytes, exactly the ring's stage layout; columns past the end of a row read as
// zero and rows past out_f too.  The padding columns of a chunk overlap the next chunk of the
// same row (they are never used).
struct TmaMaps {
    CUtensorMap tile;
    CUtensorMap oct;
};

struct TmaGroup {
    TmaMaps m[kMaxGroup];
};

// Where the consumers read the activation from.
enum ActMode : int {
    kActGlobal = 0,  // qs and d straight from global memory (L1/L2)
    kActSmem = 1,    // qs (int8) and d staged in shared memory once per CTA
    kActFrag = 2,    // E4M3 / block-128 / Q8_0 on the tensor cores: f16 MMA B fragments and d
                     // staged in shared memory; Q8_0 with dp4a: the activation staged in the
                     // record-aligned layout of q80_stage_lane (and d)
};

__device__ __forceinline__ void fault(unsigned bit) { atomicOr(&g_memq_fault, bit); }

__device__ __forceinline__ void named_barrier_consumers() {
    asm volatile("bar.sync %0, %1;" ::"n"(kBarConsumers), "n"(kConsumerThreads) : "memory");
}

// The consumer barrier that also ORs a predicate over the consumer threads.
__device__ __forceinline__ bool named_barrier_consumers_or(bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(v)), "n"(kBarConsumers), "n"(kConsumerThreads)
        : "memory");
    return r != 0;
}


// ---------------------------------------------------------------------------------------------
// E4M3 / block-128 stage: tensor-core inner products.
//
// Per 32-weight block, two m16n8k16 MMAs with A = the tile's 16 weight rows (E4M3 decoded to
// f16 by the hardware cvt) and B = the q8_1 activation of up to 8 tokens (int8 -> f16), both
// exact, accumulating in f32; the 16x8 block result is then scaled by d[token][block] (and the
// grid entry) into f32 accumulators.  The dot product is order-free, so the K index inside a
// block is permuted: thread (g, t) = (lane/4, lane%4) supplies physical columns 8t..8t+7 of its
// rows for MMA slots {2t, 2t+1, 2t+8, 2t+9} (first MMA: 8t..8t+3, second: 8t+4..8t+7), and the
// B fragment of token g uses exactly the same map.  The B fragments come precomputed from
// shared memory (kActFrag) or are converted from the int8 activation (kActSmem, kActGlobal).
// acc[0..3] = rows (g, g+8) x tokens (2t, 2t+1) of the tile.
// ---------------------------------------------------------------------------------------------
template <int KIND, int M, int MODE, bool FULL>
__device__ __forceinline__ void mma_stage(const StreamArgs &a, const uint8_t *stage,
                                          const uint8_t *sm, int64_t row0, int64_t row_last,
                                          int64_t grow_base, int kb0, int nblk, int lane,
                                          float (&acc)[4]) {
    using G = Geo<KIND>;
    const int g = lane >> 2;
    const int t = lane & 3;
    const uint4 *bfrag = reinterpret_cast<const uint4 *>(sm + a.off_bfrag);
    const int8_t *s_qs = reinterpret_cast<const int8_t *>(sm + a.off_qs);
    const float *s_d = reinterpret_cast<const float *>(sm + a.off_d);
    float grp[4] = {0.f, 0.f, 0.f, 0.f};  // block-128: the sum over this 128-column group
#pragma unroll
    for (int b = 0; b < G::kWarpBlocks; ++b) {
        if (FULL || b < nblk) {
            const int kb = kb0 + b;
            uint32_t bq[4] = {0u, 0u, 0u, 0u};
            {
                // B column g is token g; columns g >= M load token M - 1 (no divergent branch):
                // an MMA column depends only on its own B column, and those are never stored
                const int gq = g < M ? g : M - 1;
                if (MODE == kActFrag) {
                    const uint4 v = bfrag[(gq * (a.nb | 1) + kb) * 4 + t];
                    bq[0] = v.x;
                    bq[1] = v.y;
                    bq[2] = v.z;
                    bq[3] = v.w;
                } else {
                    const uint2 qv = MODE == kActSmem
                                         ? lds64(s_qs + gq * a.qstr + 32 * kb + 8 * t)
                                         : __ldcg(reinterpret_cast<const uint2 *>(
                                               a.qs + static_cast<int64_t>(gq) * a.in_f + 32 * kb + 8 * t));
                    s8x4_to_f16x2x2(qv.x, bq[0], bq[1]);
                    s8x4_to_f16x2x2(qv.y, bq[2], bq[3]);
                }
            }
            float k0 = 0.f, k1 = 0.f;
            if (MODE == kActGlobal) {
                if (2 * t < M) k0 = __ldcg(a.d + (2 * t) * a.nb + kb);
                if (2 * t + 1 < M) k1 = __ldcg(a.d + (2 * t + 1) * a.nb + kb);
            } else {
                if (2 * t < M) k0 = s_d[(2 * t) * a.dstr + kb];
                if (2 * t + 1 < M) k1 = s_d[(2 * t + 1) * a.dstr + kb];
            }
            const uint8_t *pa = stage + g * G::kSlot + 32 * b + 8 * t;
            const uint2 wa = lds64(pa);
            const uint2 wb = lds64(pa + 8 * G::kSlot);
            uint32_t a0, a1, a2, a3;
            float c[4] = {0.f, 0.f, 0.f, 0.f};
            e4m3x4_to_f16x2x2(wa.x, a0, a2);
            e4m3x4_to_f16x2x2(wb.x, a1, a3);
            mma_f16_16816(c, a0, a1, a2, a3, bq[0], bq[1]);
            e4m3x4_to_f16x2x2(wa.y, a0, a2);
            e4m3x4_to_f16x2x2(wb.y, a1, a3);
            mma_f16_16816(c, a0, a1, a2, a3, bq[2], bq[3]);
            float(&dst)[4] = KIND == kBlk ? grp : acc;
            dst[0] = fmaf(c[0], k0, dst[0]);
            dst[1] = fmaf(c[1], k1, dst[1]);
            dst[2] = fmaf(c[2], k0, dst[2]);
            dst[3] = fmaf(c[3], k1, dst[3]);
        }
    }
    if (KIND == kBlk) {
        // The grid entries of this thread's two tile rows for the warp's 128-column group (kb0 is
        // a multiple of 4, so a warp's blocks never straddle two groups), from the CTA's staged
        // grid rows.
        const int64_t r0 = row0 + g > row_last ? row_last : row0 + g;
        const int64_t r8 = row0 + g + 8 > row_last ? row_last : row0 + g + 8;
        const float *s_grid = reinterpret_cast<const float *>(sm + a.off_grid);
        const float g0 = s_grid[((r0 >> 7) - grow_base) * a.gcols + (kb0 >> 2)];
        const float g8 = s_grid[((r8 >> 7) - grow_base) * a.gcols + (kb0 >> 2)];
        acc[0] = fmaf(grp[0], g0, acc[0]);
        acc[1] = fmaf(grp[1], g0, acc[1]);
        acc[2] = fmaf(grp[2], g8, acc[2]);
        acc[3] = fmaf(grp[3], g8, acc[3]);
    }
}

// ---------------------------------------------------------------------------------------------
// Q8_0 stage on the tensor cores (kQ80T): as mma_stage, with A = the int8 weights of the tile's
// 16 rows (int8 -> f16 exact).  Every product is an integer of magnitude <= 127^2 and a block's
// 32 of them sum to < 2^24, so the MMA's f32 block sum is the exact integer dot product -- the
// same value dp4a gives.  A record is 34 bytes (f16 d_w, then 32 int8); the thread's 8 weight
// bytes start 2 bytes into it, i.e. 4-byte aligned for odd blocks of the warp and 2 mod 4 for
// even ones (the stage, its row slots and the warp's 4-block slice are 8-byte aligned), read
// with two or three 4-byte loads.  The block result of (row, token) is scaled by
// d_w[row] * d_x[token], in that order, as in the dp4a stage.
// ---------------------------------------------------------------------------------------------
__device__ __forceinline__ uint2 q80_weights8(const uint8_t *rec, bool odd) {
    // rec: the record start + 8t; returns its bytes [2, 10).  `odd` is a constant after the
    // caller's unrolling.
    if (odd) {
        return make_uint2(lds32(rec + 2), lds32(rec + 6));
    } else {
        const uint32_t a = lds32(rec), b = lds32(rec + 4), c = lds32(rec + 8);
        return make_uint2(__funnelshift_r(a, b, 16), __funnelshift_r(b, c, 16));
    }
}

template <int M, int MODE, bool FULL>
__device__ __forceinline__ void mma_stage_q80(const StreamArgs &a, const uint8_t *stage,
                                              const uint8_t *sm, int kb0, int nblk, int lane,
                                              float (&acc)[4]) {
    using G = Geo<kQ80T>;
    const int g = lane >> 2;
    const int t = lane & 3;
    const uint4 *bfrag = reinterpret_cast<const uint4 *>(sm + a.off_bfrag);
    const int8_t *s_qs = reinterpret_cast<const int8_t *>(sm + a.off_qs);
    const float *s_d = reinterpret_cast<const float *>(sm + a.off_d);
    const uint8_t *row0 = stage + g * G::kSlot;
    const uint8_t *row8 = row0 + 8 * G::kSlot;
#pragma unroll
    for (int b = 0; b < G::kWarpBlocks; ++b) {
        if (FULL || b < nblk) {
            const int kb = kb0 + b;
            uint32_t bq[4] = {0u, 0u, 0u, 0u};
            {
                // B column g is token g; columns g >= M load token M - 1 (no divergent branch):
                // an MMA column depends only on its own B column, and those are never stored
                const int gq = g < M ? g : M - 1;
                if (MODE == kActFrag) {
                    const uint4 v = bfrag[(gq * (a.nb | 1) + kb) * 4 + t];
                    bq[0] = v.x;
                    bq[1] = v.y;
                    bq[2] = v.z;
                    bq[3] = v.w;
                } else {
                    const uint2 qv = MODE == kActSmem
                                         ? lds64(s_qs + gq * a.qstr + 32 * kb + 8 * t)
                                         : __ldcg(reinterpret_cast<const uint2 *>(
                                               a.qs + static_cast<int64_t>(gq) * a.in_f + 32 * kb + 8 * t));
                    s8x4_to_f16x2x2(qv.x, bq[0], bq[1]);
                    s8x4_to_f16x2x2(qv.y, bq[2], bq[3]);
                }
            }
            float k0 = 0.f, k1 = 0.f;
            if (MODE == kActGlobal) {
                if (2 * t < M) k0 = __ldcg(a.d + (2 * t) * a.nb + kb);
                if (2 * t + 1 < M) k1 = __ldcg(a.d + (2 * t + 1) * a.nb + kb);
            } else {
                if (2 * t < M) k0 = s_d[(2 * t) * a.dstr + kb];
                if (2 * t + 1 < M) k1 = s_d[(2 * t + 1) * a.dstr + kb];
            }
            const uint8_t *r0 = row0 + 34 * b;
            const uint8_t *r8 = row8 + 34 * b;
            const float dw0 = __half2float(__ushort_as_half(static_cast<unsigned short>(lds16(r0))));
            const float dw8 = __half2float(__ushort_as_half(static_cast<unsigned short>(lds16(r8))));
            const uint2 wa = q80_weights8(r0 + 8 * t, b & 1);
            const uint2 wb = q80_weights8(r8 + 8 * t, b & 1);
            uint32_t a0, a1, a2, a3;
            float c[4] = {0.f, 0.f, 0.f, 0.f};
            s8x4_to_f16x2x2(wa.x, a0, a2);
            s8x4_to_f16x2x2(wb.x, a1, a3);
            mma_f16_16816(c, a0, a1, a2, a3, bq[0], bq[1]);
            s8x4_to_f16x2x2(wa.y, a0, a2);
            s8x4_to_f16x2x2(wb.y, a1, a3);
            mma_f16_16816(c, a0, a1, a2, a3, bq[2], bq[3]);
            acc[0] = fmaf(c[0], dw0 * k0, acc[0]);
            acc[1] = fmaf(c[1], dw0 * k1, acc[1]);
            acc[2] = fmaf(c[2], dw8 * k0, acc[2]);
            acc[3] = fmaf(c[3], dw8 * k1, acc[3]);
        }
    }
}

// ---------------------------------------------------------------------------------------------
// Q8_0 stage: the warp's row, lane l owns block l.  The block's 32 weights start 2 bytes into a
// 34-byte record, so they are re-aligned from 4-byte shared loads with funnel shifts; dp4a then
// gives the exact int32 dot product with the activation block.
// ---------------------------------------------------------------------------------------------
// kActFrag (the default for dp4a): the activation is staged once per CTA in a layout that
// matches the 34-byte records as they sit in the stage, so no weight word needs realigning.
// Lane l reads the nine 4-byte words of its row slot that cover its record, from byte
// (34*l) & ~3: for an even block the record starts on a word (word 0 = f16 scale, then
// q0 q1; word 8 = q30 q31 and the next record's scale), for an odd block two bytes into one
// (word 0 = the previous record's last two codes, then the scale; words 1..8 = q0..q31).  The
// staged activation of block kb (12 words per (token, block), 9 used) has the activation bytes
// under the weight bytes of that layout and zeros under everything else, so nine dp4a give the
// block's exact int32 dot product, and the scale comes out of word 0.
constexpr int kQ8ActWords = 12;  // words per (token, block) of the staged dp4a activation

__device__ __forceinline__ void q80_act_layout(const uint32_t *q, bool odd, uint32_t *dst) {
    // q: the block's 8 activation words; dst: 9 words (see above)
    if (odd) {
        dst[0] = 0u;
#pragma unroll
        for (int i = 0; i < 8; ++i) dst[i + 1] = q[i];
    } else {
        dst[0] = q[0] << 16;
#pragma unroll
        for (int i = 1; i < 8; ++i) dst[i] = __funnelshift_r(q[i - 1], q[i], 16);
        dst[8] = q[7] >> 16;
    }
}

// Q8_0 with dp4a and the record-aligned activation (kActFrag): the rows of a 16-row tile a lane
// works on.  Warp w takes rows 2w and 2w + 1: lanes 0-15 read row 2w and lanes 16-31 row 2w + 1,
// lane l blocks l % 16 and l % 16 + 16.  Lane k of a half-warp reads the words of record k from
// word floor(8.5 k) of its row: for k < 16 these fall on 16 distinct banks, and the next row
// lies one 1088-byte slot (272 words, 16 banks) away -- on the complementary 16 banks -- so every
// 4-byte load of the warp is conflict-free (the same holds for blocks 16-31).
__device__ __forceinline__ int q80_pair_row(int warp, int lane) { return 2 * warp + (lane >> 4); }

template <int M, int MODE>
__device__ __forceinline__ void q80_block_plain(const StreamArgs &a, const uint8_t *slot,
                                                const uint8_t *sm, int kb0, int b,
                                                float (&acc)[M]) {
    const int kb = kb0 + b;
    const int qstart = 34 * b + 2;
    const int abase = qstart & ~3;
    const uint32_t sh = static_cast<uint32_t>(qstart & 3) * 8u;  // 0 or 16
    uint32_t wv[9];
#pragma unroll
    for (int i = 0; i < 8; ++i) wv[i] = lds32(slot + abase + 4 * i);
    wv[8] = sh ? lds32(slot + abase + 32) : 0u;
    uint32_t qw[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) qw[i] = __funnelshift_r(wv[i], wv[i + 1], sh);
    const float dw = __half2float(__ushort_as_half(static_cast<unsigned short>(lds16(slot + 34 * b))));
    const int8_t *s_qs = reinterpret_cast<const int8_t *>(sm + a.off_qs);
    const float *s_d = reinterpret_cast<const float *>(sm + a.off_d);
#pragma unroll
    for (int j = 0; j < M; ++j) {
        uint4 x0, x1;
        float dj;
        if (MODE == kActSmem) {
            x0 = lds128(s_qs + j * a.qstr + 32 * kb);
            x1 = lds128(s_qs + j * a.qstr + 32 * kb + 16);
            dj = s_d[j * a.dstr + kb];
        } else {
            const uint4 *qx = reinterpret_cast<const uint4 *>(a.qs + static_cast<int64_t>(j) * a.in_f + 32 * kb);
            x0 = __ldcg(qx);
            x1 = __ldcg(qx + 1);
            dj = __ldcg(a.d + j * a.nb + kb);
        }
        int s = 0;
        s = __dp4a(static_cast<int>(qw[0]), static_cast<int>(x0.x), s);
        s = __dp4a(static_cast<int>(qw[1]), static_cast<int>(x0.y), s);
        s = __dp4a(static_cast<int>(qw[2]), static_cast<int>(x0.z), s);
        s = __dp4a(static_cast<int>(qw[3]), static_cast<int>(x0.w), s);
        s = __dp4a(static_cast<int>(qw[4]), static_cast<int>(x1.x), s);
        s = __dp4a(static_cast<int>(qw[5]), static_cast<int>(x1.y), s);
        s = __dp4a(static_cast<int>(qw[6]), static_cast<int>(x1.z), s);
        s = __dp4a(static_cast<int>(qw[7]), static_cast<int>(x1.w), s);
        acc[j] = fmaf(static_cast<float>(s), dw * dj, acc[j]);
    }
}

// The lane's share of a Q8_0 stage (q80_pair_row): blocks k and k + 16 (k = lane % 16) of its
// row, whose slot is `slot`, accumulated into acc in block order.  The block products are exact
// integers and the f32 operations per (row, token) are the same in every activation mode, so the
// modes give bit-identical outputs.
template <int M, int MODE>
__device__ __forceinline__ void q80_stage_lane(const StreamArgs &a, const uint8_t *slot,
                                               const uint8_t *sm, int kb0, int nblk, int lane,
                                               float (&acc)[M]) {
    const int k = lane & 15;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int b = k + 16 * h;
        if (b >= nblk) break;
        if constexpr (MODE == kActFrag) {
            // record-aligned activation: nine dp4a over the record's word window
            const bool odd = k & 1;  // kb0 is even; blocks k and k + 16 share k's parity
            const int kb = kb0 + b;
            const uint32_t *act = reinterpret_cast<const uint32_t *>(sm + a.off_bfrag);
            const float *s_d = reinterpret_cast<const float *>(sm + a.off_d);
            const uint8_t *rec = slot + ((34 * b) & ~3);
            uint32_t w[9];
#pragma unroll
            for (int i = 0; i < 9; ++i) w[i] = lds32(rec + 4 * i);
            const uint32_t dbits = odd ? (w[0] >> 16) : (w[0] & 0xffffu);
            const float dw = __half2float(__ushort_as_half(static_cast<unsigned short>(dbits)));
#pragma unroll
            for (int j = 0; j < M; ++j) {
                const uint32_t *aj = act + (j * a.nb + kb) * kQ8ActWords;
                const uint4 x0 = lds128(aj);
                const uint4 x1 = lds128(aj + 4);
                const uint32_t x2 = lds32(aj + 8);
                int s0 = 0, s1 = 0;
                s0 = __dp4a(static_cast<int>(w[0]), static_cast<int>(x0.x), s0);
                s1 = __dp4a(static_cast<int>(w[1]), static_cast<int>(x0.y), s1);
                s0 = __dp4a(static_cast<int>(w[2]), static_cast<int>(x0.z), s0);
                s1 = __dp4a(static_cast<int>(w[3]), static_cast<int>(x0.w), s1);
                s0 = __dp4a(static_cast<int>(w[4]), static_cast<int>(x1.x), s0);
                s1 = __dp4a(static_cast<int>(w[5]), static_cast<int>(x1.y), s1);
                s0 = __dp4a(static_cast<int>(w[6]), static_cast<int>(x1.z), s0);
                s1 = __dp4a(static_cast<int>(w[7]), static_cast<int>(x1.w), s1);
                s0 = __dp4a(static_cast<int>(w[8]), static_cast<int>(x2), s0);
                acc[j] = fmaf(static_cast<float>(s0 + s1), dw * s_d[j * a.dstr + kb], acc[j]);
            }
        } else {
            q80_block_plain<M, MODE>(a, slot, sm, kb0, b, acc);
        }
    }
}

// ---------------------------------------------------------------------------------------------
// Fused decode step: every CTA quantizes the m activation rows itself (the RMSNorm -> q8_1
// producer of memq_rmsnorm_q8_1 with the same per-element arithmetic: f32 per-thread sum of
// squares, f64 across threads, IEEE f32 divide / square root, z = (x*r)*w, 8-lane block amax,
// d = amax/127, qs = round(z/d)) into shared memory, while its producer warp already streams
// weights.  The values are identical in every CTA; CTA 0 also writes them to qs/d (and z).
// ---------------------------------------------------------------------------------------------
__device__ __forceinline__ int8_t quant_q8(float z, float dd) {
    return dd != 0.0f ? static_cast<int8_t>(roundf(__fdiv_rn(z, dd))) : static_cast<int8_t>(0);
}

template <int M>
__device__ __forceinline__ void fused_quantize(const StreamArgs &a, int8_t *s_qs, float *s_d,
                                               double *s_red, float *s_r) {
    const int tid = threadIdx.x;  // consumer threads 0..255
    const int lane = tid & 31, warp = tid >> 5;
    const int nf4 = a.in_f >> 2;
    const bool publish = blockIdx.x == 0;
    const float4 *w4 = reinterpret_cast<const float4 *>(a.wn);
    // Rows up to kKeep * 1024 wide keep x in registers between the two passes (one read per
    // CTA); wider rows read it twice (the second read hits L1).
    constexpr int kKeep = 8;
    const bool keep = nf4 <= kKeep * kConsumerThreads;
    for (int j = 0; j < M; ++j) {
        const float4 *xr = reinterpret_cast<const float4 *>(a.x + static_cast<int64_t>(j) * a.in_f);
        float4 xk[kKeep];
        float ss = 0.f;
        if (keep) {
#pragma unroll
            for (int v = 0; v < kKeep; ++v) {
                const int f = tid + v * kConsumerThreads;
                xk[v] = f < nf4 ? __ldcg(xr + f) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int v = 0; v < kKeep; ++v) {
                ss = fmaf(xk[v].x, xk[v].x, ss);
                ss = fmaf(xk[v].y, xk[v].y, ss);
                ss = fmaf(xk[v].z, xk[v].z, ss);
                ss = fmaf(xk[v].w, xk[v].w, ss);
            }
        } else {
            for (int f = tid; f < nf4; f += kConsumerThreads) {
                const float4 v = __ldcg(xr + f);
                ss = fmaf(v.x, v.x, ss);
                ss = fmaf(v.y, v.y, ss);
                ss = fmaf(v.z, v.z, ss);
                ss = fmaf(v.w, v.w, ss);
            }
        }
        const double s = warp_sum(static_cast<double>(ss));
        if (lane == 0) s_red[warp] = s;
        named_barrier_consumers();
        if (warp == 0) {
            double t = lane < kWarps ? s_red[lane] : 0.0;
            t = warp_sum(t);
            if (lane == 0)
                *s_r = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(
                    __fdiv_rn(static_cast<float>(t), static_cast<float>(a.in_f)), a.eps)));
        }
        named_barrier_consumers();
        const float r = *s_r;
        for (int f0 = 0, v = 0; f0 < nf4; f0 += kConsumerThreads, ++v) {
            const int f = f0 + tid;
            const bool act = f < nf4;
            float4 xv = make_float4(0.f, 0.f, 0.f, 0.f), wv = xv;
            if (keep) {
#pragma unroll
                for (int u = 0; u < kKeep; ++u)
                    if (u == v) xv = xk[u];
            }
            if (act) {
                if (!keep) xv = __ldcg(xr + f);
                wv = __ldg(w4 + f);
            }
            float4 zz;
            zz.x = __fmul_rn(__fmul_rn(xv.x, r), wv.x);
            zz.y = __fmul_rn(__fmul_rn(xv.y, r), wv.y);
            zz.z = __fmul_rn(__fmul_rn(xv.z, r), wv.z);
            zz.w = __fmul_rn(__fmul_rn(xv.w, r), wv.w);
            float am = fmaxf(fmaxf(fabsf(zz.x), fabsf(zz.y)), fmaxf(fabsf(zz.z), fabsf(zz.w)));
            am = fmaxf(am, __shfl_xor_sync(kFullMask, am, 1));
            am = fmaxf(am, __shfl_xor_sync(kFullMask, am, 2));
            am = fmaxf(am, __shfl_xor_sync(kFullMask, am, 4));
            const float dd = __fdiv_rn(am, 127.0f);
            if (act) {
                const uint32_t packed =
                    static_cast<uint32_t>(static_cast<uint8_t>(quant_q8(zz.x, dd))) |
                    static_cast<uint32_t>(static_cast<uint8_t>(quant_q8(zz.y, dd))) << 8 |
                    static_cast<uint32_t>(static_cast<uint8_t>(quant_q8(zz.z, dd))) << 16 |
                    static_cast<uint32_t>(static_cast<uint8_t>(quant_q8(zz.w, dd))) << 24;
                reinterpret_cast<uint32_t *>(s_qs + j * a.qstr)[f] = packed;
                if ((tid & 7) == 0) s_d[j * a.dstr + (f >> 3)] = dd;
                if (publish) {
                    reinterpret_cast<uint32_t *>(const_cast<int8_t *>(a.qs) + static_cast<int64_t>(j) * a.in_f)[f] = packed;
                    if ((tid & 7) == 0) const_cast<float *>(a.d)[j * a.nb + (f >> 3)] = dd;
                    if (a.z_out) reinterpret_cast<float4 *>(a.z_out + static_cast<int64_t>(j) * a.in_f)[f] = zz;
                }
            }
        }
        named_barrier_consumers();  // s_red / s_r are reused by the next row
    }
}

// ---------------------------------------------------------------------------------------------
// The stream kernel (see the file header for the schedule).
// ---------------------------------------------------------------------------------------------
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Single-thread bounded wait (the producer's lane 0).
__device__ __forceinline__ bool thread_wait_bounded(uint64_t *bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity))
        if (clock64() - t0 > kWaitCycles) return false;
    return true;
}

template <int KIND, int M, int MODE, bool FUSE>
__global__ void __launch_bounds__(kThreads, Geo<KIND>::kMinCtasPerSm)
    gemv_stream_kernel(const __grid_constant__ StreamArgs args, const __grid_constant__ TmaGroup tg) {
    using G = Geo<KIND>;
    constexpr int TR = G::kTileRows;
    extern __shared__ __align__(128) uint8_t smem[];
    griddep_launch_dependents();

    // This CTA's matrix, and its share of that matrix's rows.
    int mi = 0;
    while (mi + 1 < args.nmat && static_cast<int>(blockIdx.x) >= args.mat_cta[mi + 1]) ++mi;
    StreamArgs a = args;
    a.w = args.mat_w[mi];
    a.aux = args.mat_aux[mi];
    a.y = args.mat_y[mi];
    a.out_f = args.mat_out_f[mi];
    const TmaMaps &tm = tg.m[mi];
    const int64_t cta = static_cast<int64_t>(blockIdx.x) - args.mat_cta[mi];
    const int64_t ncta = args.mat_cta[mi + 1] - args.mat_cta[mi];

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int S = a.stages;

    const int64_t R0 = cta * a.out_f / ncta;
    const int64_t R1 = (cta + 1) * a.out_f / ncta;
    const int ntiles = static_cast<int>((R1 - R0 + TR - 1) / TR);
    const int nch = (a.nb + G::kChunkBlocks - 1) / G::kChunkBlocks;
    const int items = ntiles * nch;

    uint64_t *full = reinterpret_cast<uint64_t *>(smem);
    uint64_t *empty = full + S;
    uint64_t *act_bar = full + 2 * S;  // the activation's bulk copies
    uint8_t *ring = smem + a.off_ring;
    float *part = reinterpret_cast<float *>(smem + a.off_part);  // [2][kWarps][TR][M]

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kWarps);
        }
        mbar_init(act_bar, 1);
        mbar_init_fence();
    }
    __syncthreads();

    if (warp == kWarps) {
        // ------------------------------- producer warp ---------------------------------------
        if (lane == 0) {
            const uint64_t pol = l2_evict_first_policy();
            // Tensor copies need 128-byte aligned destinations: every stage base is, given a
            // 128-byte aligned ring (checked here, else rows are copied one by one).
            const bool use_tma = a.use_tma && (smem_u32(ring) & 127u) == 0;
            if (use_tma) {
                tma_prefetch_map(&tm.tile);
                if (TR > 8) tma_prefetch_map(&tm.oct);
            }
            int tile = 0, ch = 0, s = 0;
            uint32_t eph = 0;  // parity of the empty-barrier phase awaited before a reuse
            for (int it = 0; it < items; ++it) {
                // The first S stages go out before the preceding grid has finished; the bounded
                // waits for released stages start only once it has, so that a long predecessor
                // never counts against this launch's own progress.
                if (it == S) griddep_wait();
                if (it >= S && !thread_wait_bounded(&empty[s], eph)) {
                    fault(2u);
                    break;
                }
                const int64_t r0 = R0 + static_cast<int64_t>(tile) * TR;
                const int rc = static_cast<int>(R1 - r0 < TR ? R1 - r0 : TR);
                const int kb = ch * G::kChunkBlocks;
                const int nblk = min(G::kChunkBlocks, a.nb - kb);
                const uint32_t bytes = static_cast<uint32_t>(nblk * G::kBlockBytes);
                const uint8_t *src = a.w + r0 * a.row_bytes + static_cast<int64_t>(kb) * G::kBlockBytes;
                uint8_t *dst = ring + s * G::kStage;
                // Rows [0, boxed) come as tensor copies (whole tile, or its first 8 rows: both
                // land 128-byte aligned), the rest row by row.
                const int boxed = !use_tma ? 0 : rc == TR ? TR : rc >= 8 ? 8 : 0;
                mbar_arrive_expect_tx(&full[s], static_cast<uint32_t>(boxed * G::kSlot) +
                                                    bytes * static_cast<uint32_t>(rc - boxed));
                const int tx = kb * G::kBlockBytes / 8;
                if (boxed == TR)
                    tma_load_2d(dst, &tm.tile, tx, static_cast<int>(r0), &full[s], pol);
                else if (boxed == 8)
                    tma_load_2d(dst, &tm.oct, tx, static_cast<int>(r0), &full[s], pol);
                for (int rr = boxed; rr < rc; ++rr)
                    bulk_g2s(dst + rr * G::kSlot, src + rr * a.row_bytes, bytes, &full[s], pol);
                if (++ch == nch) {
                    ch = 0;
                    ++tile;
                }
                // Use k of a stage (items kS..kS+S-1) waits for phase k-1 of its empty barrier:
                // parity 0 for k = 1, then alternating, so flip on every wrap after the second.
                if (++s == S) {
                    s = 0;
                    if (it >= 2 * S - 1) eph ^= 1u;
                }
            }
        }
        return;
    }

    // --------------------------------- consumer warps ------------------------------------------
    // Constants first (the per-tensor scale, the block-128 grid rows this CTA touches): they do
    // not depend on the preceding launch, so they are staged while it finishes.
    float scale = 1.0f;
    if (KIND == kE4M3) scale = __ldg(a.aux);
    const int64_t grow_base = R0 >> 7;
    if (KIND == kBlk) {
        float *dst = reinterpret_cast<float *>(smem + a.off_grid);
        const int nrows = static_cast<int>(((R1 - 1) >> 7) - grow_base + 1);
        const int n = nrows * a.gcols;
        for (int i = threadIdx.x; i < n; i += kConsumerThreads)
            dst[i] = __ldg(a.aux + grow_base * a.gcols + i);
    }
    griddep_wait();
    bool ok = true;
    // The activation (written by the preceding launch): qs and d into shared memory with one
    // bulk copy each (one L2 round trip), or computed here in the fused decode step.  For the
    // f16 MMA fragments (E4M3 / block-128 / Q8_0 on the tensor cores) of an activation of at most
    // kDirectItems items the consumers read qs straight from global memory (at most three rounds
    // of loads per thread) and write the fragments while d is copied; a larger one is staged and
    // converted in place (measured on GB300: 4096 x 4096 m = 1 5.17 -> 4.98 us with the direct
    // read, 1024 x 5120 m = 8 4.68 -> 4.86 us).
    //
    // Fragment layout: entry (g, kb, t) = uint4 (g * (nb | 1) + kb) * 4 + t holds
    // q[g][32kb + 8t .. 8t+7] as four f16x2 registers (token rows of an odd number of 64-byte
    // blocks, so the two tokens of a quarter-warp's 16-byte loads fall on different bank halves).
    // Item j = (g * nb + kb) * 4 + t is 8 bytes of qs at byte 8j of [M][in_f].
    constexpr bool kFragMma = G::kMma && MODE == kActFrag;
    constexpr int kR = 4;  // items per thread in flight
    constexpr int kDirectItems = 3 * kR * kConsumerThreads;
    const int n_items = a.nb * M * 4;
    const bool direct = kFragMma && !FUSE && n_items <= kDirectItems;
    // dp4a: the record-aligned layout of up to 512 blocks is built from global memory likewise
    const bool direct_q80 = KIND == kQ80 && MODE == kActFrag && !FUSE && a.nb * M <= 2 * kConsumerThreads;
    const int pad = 4 * ((a.nb | 1) - a.nb);
    // token of item j: j / (4 nb) as a multiply-high by ceil(2^32 / (4 nb)), exact here since
    // j * 4nb < 2^32 (n <= 14.5K items fit the shared memory)
    const uint32_t magic = 0xFFFFFFFFu / static_cast<uint32_t>(4 * a.nb) + 1u;
    uint4 *bfrag = reinterpret_cast<uint4 *>(smem + a.off_bfrag);
    auto frag_store = [&](int j, uint2 qv) {
        uint4 v;
        s8x4_to_f16x2x2(qv.x, v.x, v.y);
        s8x4_to_f16x2x2(qv.y, v.z, v.w);
        bfrag[j + pad * static_cast<int>(__umulhi(static_cast<uint32_t>(j), magic))] = v;
    };
    if (FUSE) {
        double *s_red = reinterpret_cast<double *>(smem + a.off_red);  // [kWarps] + r
        fused_quantize<M>(a, reinterpret_cast<int8_t *>(smem + a.off_qs),
                          reinterpret_cast<float *>(smem + a.off_d), s_red,
                          reinterpret_cast<float *>(s_red + kWarps));
    } else if (MODE != kActGlobal) {
        // one bulk copy per activation array, or one per token row where the staged rows are
        // padded (row sizes and strides are multiples of 16 bytes there)
        const uint32_t qbytes = direct || direct_q80 ? 0u : static_cast<uint32_t>(M * a.in_f);
        const uint32_t dbytes = static_cast<uint32_t>(M * a.nb * 4);
        const bool d_bulk = (a.nb & 3) == 0 && (reinterpret_cast<uintptr_t>(a.d) & 15u) == 0;
        if (threadIdx.x == 0) {
            mbar_arrive_expect_tx(act_bar, qbytes + (d_bulk ? dbytes : 0u));
            if (qbytes) {
                if (a.qstr == a.in_f) {
                    bulk_g2s_plain(smem + a.off_qs, a.qs, qbytes, act_bar);
                } else {
                    for (int j = 0; j < M; ++j)
                        bulk_g2s_plain(smem + a.off_qs + j * a.qstr, a.qs + static_cast<int64_t>(j) * a.in_f,
                                       static_cast<uint32_t>(a.in_f), act_bar);
                }
            }
            if (d_bulk) {
                if (a.dstr == a.nb) {
                    bulk_g2s_plain(smem + a.off_d, a.d, dbytes, act_bar);
                } else {
                    for (int j = 0; j < M; ++j)
                        bulk_g2s_plain(smem + a.off_d + j * a.dstr * 4, a.d + j * a.nb,
                                       static_cast<uint32_t>(a.nb * 4), act_bar);
                }
            }
        }
        if (!d_bulk) {
            float *dst = reinterpret_cast<float *>(smem + a.off_d);
            for (int i = threadIdx.x; i < M * a.nb; i += kConsumerThreads) {
                const int j = i / a.nb;
                dst[i + j * (a.dstr - a.nb)] = __ldcg(a.d + i);
            }
        }
        if (direct) {
            const uint2 *src = reinterpret_cast<const uint2 *>(a.qs);
            for (int j0 = threadIdx.x; j0 < n_items; j0 += kR * kConsumerThreads) {
                uint2 qv[kR];
#pragma unroll
                for (int r = 0; r < kR; ++r) {
                    const int j = j0 + r * kConsumerThreads;
                    qv[r] = j < n_items ? __ldcg(src + j) : make_uint2(0u, 0u);
                }
#pragma unroll
                for (int r = 0; r < kR; ++r)
                    if (j0 + r * kConsumerThreads < n_items) frag_store(j0 + r * kConsumerThreads, qv[r]);
            }
        }
        if (!warp_wait_bounded(act_bar, 0)) {
            // Record the fault; give the activation copy and the ring's first stages a bounded
            // chance to land before the CTA stops consuming (and eventually exits).
            if (lane == 0) fault(1u);
            (void)warp_wait_bounded(act_bar, 0);
            for (int j = 0; j < min(items, S); ++j) (void)warp_wait_bounded(&full[j], 0);
            ok = false;
        }
    }
    if (MODE == kActFrag && KIND == kQ80) {
        // The dp4a layout of the whole activation (q80_stage_lane): per (token, block) nine words
        // in a 12-word record, read and written as 16-byte vectors (records 48 bytes apart: the
        // eight 16-byte accesses of a quarter-warp fall on distinct bank groups), from global
        // memory for small activations, else from the staged qs.
        uint8_t *dst = smem + a.off_bfrag;
        const int n = a.nb * M;
        for (int i = threadIdx.x; i < n; i += kConsumerThreads) {
            const int j = i / a.nb, kb = i - j * a.nb;
            uint4 v0, v1;
            if (direct_q80) {
                const uint4 *src = reinterpret_cast<const uint4 *>(a.qs + static_cast<int64_t>(j) * a.in_f + 32 * kb);
                v0 = __ldcg(src);
                v1 = __ldcg(src + 1);
            } else {
                const uint8_t *src = smem + a.off_qs + j * a.qstr + 32 * kb;
                v0 = lds128(src);
                v1 = lds128(src + 16);
            }
            const uint32_t q[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
            uint32_t o[9];
            q80_act_layout(q, kb & 1, o);
            uint8_t *rec = dst + static_cast<size_t>(i) * (kQ8ActWords * 4);
            *reinterpret_cast<uint4 *>(rec) = make_uint4(o[0], o[1], o[2], o[3]);
            *reinterpret_cast<uint4 *>(rec + 16) = make_uint4(o[4], o[5], o[6], o[7]);
            *reinterpret_cast<uint32_t *>(rec + 32) = o[8];
        }
    } else if (kFragMma && !direct) {
        // qs (staged, or computed by the fused step) is at the top of the fragment region: item j
        // reads 8 bytes at
        // off_qs + 8j = off_bfrag + 8n + 64PM + 8j (n = 4 nb M items, P = (nb | 1) - nb) and
        // writes 16 bytes at off_bfrag + 16j + 64Pg, which can only overlap the sources of items
        // j' <= j.  So items are converted in increasing order, in chunks whose sources are all
        // read into registers before the chunk's first write.
        const uint8_t *src = smem + a.off_qs;
        for (int j0 = 0; j0 < n_items; j0 += kR * kConsumerThreads) {
            uint2 qv[kR];
#pragma unroll
            for (int r = 0; r < kR; ++r) {
                const int j = j0 + r * kConsumerThreads + threadIdx.x;
                qv[r] = j < n_items ? lds64(src + 8 * j) : make_uint2(0u, 0u);
            }
            named_barrier_consumers();
#pragma unroll
            for (int r = 0; r < kR; ++r) {
                const int j = j0 + r * kConsumerThreads + threadIdx.x;
                if (j < n_items) frag_store(j, qv[r]);
            }
        }
    }
    named_barrier_consumers();

    int c_stage = 0;
    uint32_t c_phase = 0;
    int consumed = 0;
    for (int tile = 0; tile < ntiles; ++tile) {
        const int64_t r0 = R0 + static_cast<int64_t>(tile) * TR;
        const int rc = static_cast<int>(R1 - r0 < TR ? R1 - r0 : TR);
        float acc_m[4] = {0.f, 0.f, 0.f, 0.f};
        float acc_q[M];
#pragma unroll
        for (int j = 0; j < M; ++j) acc_q[j] = 0.f;

        for (int ch = 0; ch < nch; ++ch) {
            if (ok && !warp_wait_bounded(&full[c_stage], c_phase)) {
                // Record the fault, give the copies that may be in flight a bounded chance to
                // land, and stop consuming; the tile barriers below still run.
                if (lane == 0) fault(1u);
                int st = c_stage;
                uint32_t ph = c_phase;
                for (int j = consumed + 1; j < min(items, consumed + S); ++j) {
                    if (++st == S) {
                        st = 0;
                        ph ^= 1u;
                    }
                    (void)warp_wait_bounded(&full[st], ph);
                }
                ok = false;
            }
            if (ok) {
                const int kbc = ch * G::kChunkBlocks;
                const int nblk = min(G::kChunkBlocks, a.nb - kbc);
                const uint8_t *stage = ring + c_stage * G::kStage;
                if constexpr (KIND == kQ80T) {
                    const int kb0 = kbc + warp * G::kWarpBlocks;
                    const int n = min(G::kWarpBlocks, nblk - warp * G::kWarpBlocks);
                    const uint8_t *st = stage + warp * G::kWarpBlocks * G::kBlockBytes;
                    if (n == G::kWarpBlocks)
                        mma_stage_q80<M, MODE, true>(a, st, smem, kb0, n, lane, acc_m);
                    else if (n > 0)
                        mma_stage_q80<M, MODE, false>(a, st, smem, kb0, n, lane, acc_m);
                } else if (G::kMma) {
                    const int kb0 = kbc + warp * G::kWarpBlocks;
                    const int n = min(G::kWarpBlocks, nblk - warp * G::kWarpBlocks);
                    const uint8_t *st = stage + warp * G::kWarpBlocks * G::kBlockBytes;
                    if (n == G::kWarpBlocks)
                        mma_stage<KIND, M, MODE, true>(a, st, smem, r0, R1 - 1, grow_base, kb0, n, lane, acc_m);
                    else if (n > 0)
                        mma_stage<KIND, M, MODE, false>(a, st, smem, r0, R1 - 1, grow_base, kb0, n, lane, acc_m);
                } else {
                    const int row = q80_pair_row(warp, lane);
                    if (row < rc)
                        q80_stage_lane<M, MODE>(a, stage + row * G::kSlot, smem, kbc, nblk, lane, acc_q);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[c_stage]);
                ++consumed;
            }
            if (++c_stage == S) {
                c_stage = 0;
                c_phase ^= 1u;
            }
        }

        if (G::kMma) {
            // Per-warp partials of this tile -> shared memory; then sum the 8 warp partials of
            // each (row, token) in warp order and store y.
            float *pw = part + ((tile & 1) * kWarps + warp) * TR * M;
            const int g = lane >> 2, t = lane & 3;
            if (2 * t < M) {
                pw[g * M + 2 * t] = acc_m[0];
                pw[(g + 8) * M + 2 * t] = acc_m[2];
            }
            if (2 * t + 1 < M) {
                pw[g * M + 2 * t + 1] = acc_m[1];
                pw[(g + 8) * M + 2 * t + 1] = acc_m[3];
            }
            // A tile that any consumer warp gave up on is not stored (its sums are incomplete).
            const bool bad = named_barrier_consumers_or(!ok);
            for (int idx = threadIdx.x; !bad && idx < rc * M; idx += kConsumerThreads) {
                const int row = idx / M, tok = idx - row * M;
                const float *pt = part + (tile & 1) * kWarps * TR * M + row * M + tok;
                float v = 0.f;
#pragma unroll
                for (int w = 0; w < kWarps; ++w) v += pt[w * TR * M];
                a.y[static_cast<int64_t>(tok) * a.out_f + r0 + row] = v * scale;
            }
        } else {
            // sum over the 16 lanes of each half-warp: the warp's two rows
            const int row = q80_pair_row(warp, lane);
#pragma unroll
            for (int j = 0; j < M; ++j) {
                float v = acc_q[j];
#pragma unroll
                for (int o = 8; o > 0; o >>= 1) v += __shfl_xor_sync(kFullMask, v, o);
                if ((lane & 15) == 0 && row < rc && ok) a.y[static_cast<int64_t>(j) * a.out_f + r0 + row] = v;
            }
        }
    }
}

// ---------------------------------------------------------------------------------------------
// Generic kernel: one warp per output row, byte-granular global loads, any alignment.
// ---------------------------------------------------------------------------------------------
constexpr int kGenericWarps = 8;

template <int KIND>
__global__ void __launch_bounds__(kGenericWarps * 32)
    gemv_generic_kernel(const uint8_t *__restrict__ w, const float *__restrict__ aux,
                        const int8_t *__restrict__ qs, const float *__restrict__ d,
                        float *__restrict__ y, int64_t out_f, int in_f, int m) {
    const int lane = threadIdx.x & 31;
    const int64_t r = static_cast<int64_t>(blockIdx.x) * kGenericWarps + (threadIdx.x >> 5);
    if (r >= out_f) return;
    const int nb = in_f / 32;
    const int gcols = (in_f + 127) / 128;
    const int64_t row_bytes = (KIND == kQ80) ? static_cast<int64_t>(nb) * 34 : in_f;
    const uint8_t *wr = w + r * row_bytes;
    float acc[MEMQ_MAX_M];
    for (int j = 0; j < MEMQ_MAX_M; ++j) acc[j] = 0.f;
    for (int kb = lane; kb < nb; kb += 32) {
        float wf[32];
        float bscale = 1.0f;
        if (KIND == kQ80) {
            const uint8_t *blk = wr + static_cast<int64_t>(kb) * 34;
            bscale = __half2float(__ushort_as_half(static_cast<unsigned short>(blk[0] | (blk[1] << 8))));
            for (int t = 0; t < 32; ++t) wf[t] = static_cast<float>(static_cast<int8_t>(blk[2 + t]));
        } else {
            for (int t = 0; t < 32; t += 2) {
                const uint32_t two = wr[32 * kb + t] | (static_cast<uint32_t>(wr[32 * kb + t + 1]) << 8);
                const uint32_t h2 = e4m3x2_to_f16x2(two);
                wf[t] = __half2float(__ushort_as_half(static_cast<unsigned short>(h2 & 0xffffu)));
                wf[t + 1] = __half2float(__ushort_as_half(static_cast<unsigned short>(h2 >> 16)));
            }
            if (KIND == kBlk) bscale = aux[(r >> 7) * gcols + (kb >> 2)];
        }
        for (int j = 0; j < m; ++j) {
            const int8_t *qx = qs + static_cast<int64_t>(j) * in_f + 32 * kb;
            float p = 0.f;
            for (int t = 0; t < 32; ++t) p = fmaf(wf[t], static_cast<float>(qx[t]), p);
            acc[j] = fmaf(p, bscale * d[static_cast<int64_t>(j) * nb + kb], acc[j]);
        }
    }
    const float scale = (KIND == kE4M3) ? aux[0] : 1.0f;
    for (int j = 0; j < m; ++j) {
        const float v = warp_sum(acc[j]);
        if (lane == 0) y[static_cast<int64_t>(j) * out_f + r] = v * scale;
    }
}

// ---------------------------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------------------------
struct DeviceInfo {
    int sms = 0;
    int smem_optin = 0;  // per CTA
    int smem_sm = 0;     // per SM
};

constexpr int kMaxDevices = 64;
DeviceInfo g_dev[kMaxDevices];
std::once_flag g_dev_once[kMaxDevices];
std::atomic<uint64_t> g_attr_set[4][kMaxDevices];  // [kind]: bit per (M, mode, fused) set

bool aligned(const void *p, uintptr_t n) { return (reinterpret_cast<uintptr_t>(p) & (n - 1)) == 0; }

// A small direct-mapped cache of per-call host results (occupancy answers, tensor maps), guarded
// by a mutex.  An entry is only reused for an identical key: everything the value depends on is
// part of the key, so nothing goes stale.
template <class Key, class Val, int N>
class HostCache {
  public:
    bool get(const Key &k, uint64_t h, Val &v) {
        std::lock_guard<std::mutex> lock(mu_);
        const Slot &e = slot_[h % N];
        if (!e.used || !(e.key == k)) return false;
        v = e.val;
        return true;
    }
    void put(const Key &k, uint64_t h, const Val &v) {
        std::lock_guard<std::mutex> lock(mu_);
        Slot &e = slot_[h % N];
        e.used = true;
        e.key = k;
        e.val = v;
    }

  private:
    struct Slot {
        bool used = false;
        Key key{};
        Val val{};
    };
    std::mutex mu_;
    Slot slot_[N];
};

inline uint64_t mix_hash(uint64_t h, uint64_t v) {
    h ^= v + 0x9E3779B97F4A7C15ull + (h << 6) + (h >> 2);
    return h;
}

struct OccKey {
    const void *fn;
    uint32_t smem;
    int dev;
    bool operator==(const OccKey &o) const { return fn == o.fn && smem == o.smem && dev == o.dev; }
};
HostCache<OccKey, int, 256> g_occ_cache;

// cudaOccupancyMaxActiveBlocksPerMultiprocessor for kThreads-thread CTAs, cached per (kernel,
// dynamic shared memory, device).
template <class Kern>
cudaError_t occupancy(int &per_sm, Kern kern, uint32_t smem, int dev) {
    const OccKey k{reinterpret_cast<const void *>(kern), smem, dev};
    const uint64_t h = mix_hash(mix_hash(reinterpret_cast<uintptr_t>(k.fn), smem), static_cast<uint64_t>(dev));
    if (g_occ_cache.get(k, h, per_sm)) return cudaSuccess;
    const cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, smem);
    if (e == cudaSuccess) g_occ_cache.put(k, h, per_sm);
    return e;
}
uint32_t align_up(uint32_t v, uint32_t a) { return (v + a - 1) / a * a; }

cudaError_t device_info(int &dev, DeviceInfo &info) {
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    cudaError_t err = cudaSuccess;
    std::call_once(g_dev_once[dev], [&] {
        DeviceInfo di;
        err = cudaDeviceGetAttribute(&di.sms, cudaDevAttrMultiProcessorCount, dev);
        if (err == cudaSuccess)
            err = cudaDeviceGetAttribute(&di.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        if (err == cudaSuccess)
            err = cudaDeviceGetAttribute(&di.smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
        if (err == cudaSuccess) g_dev[dev] = di;
    });
    if (err != cudaSuccess) return err;
    info = g_dev[dev];
    return info.sms > 0 ? cudaSuccess : cudaErrorInvalidDevice;
}

// cuTensorMapEncodeTiled, fetched from the driver through the runtime once per process (the
// library does not link the driver API directly).  Null when the driver does not provide it.
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled() {
    static const EncodeTiledFn fn = [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return static_cast<EncodeTiledFn>(nullptr);
        return reinterpret_cast<EncodeTiledFn>(p);
    }();
    return fn;
}

struct MapKey {
    int kind;
    const void *w;
    int64_t out_f;
    int64_t row_bytes;
    int dev;
    bool operator==(const MapKey &o) const {
        return kind == o.kind && w == o.w && out_f == o.out_f && row_bytes == o.row_bytes &&
               dev == o.dev;
    }
};
// Tensor maps of recently used weight planes (a decode loop reuses the same few hundred).
HostCache<MapKey, TmaMaps, 1024> g_map_cache;

// Builds the two tensor maps of the weight plane (see TmaMaps) and sets a.use_tma; on any
// failure the producer copies every row with its own bulk copy instead.  Encoded maps are
// cached per (container, weight pointer, rows, row bytes, device).
template <int KIND>
void make_maps(StreamArgs &a, TmaMaps &tm, int dev) {
    using G = Geo<KIND>;
    a.use_tma = 0;
    const MapKey key{KIND, a.w, a.out_f, a.row_bytes, dev};
    const uint64_t h = mix_hash(mix_hash(mix_hash(reinterpret_cast<uintptr_t>(a.w),
                                                  static_cast<uint64_t>(a.out_f)),
                                         static_cast<uint64_t>(a.row_bytes)),
                                static_cast<uint64_t>(KIND * 64 + dev));
    if (g_map_cache.get(key, h, tm)) {
        a.use_tma = 1;
        return;
    }
    const EncodeTiledFn enc = encode_tiled();
    if (!enc || a.row_bytes % 16 != 0 || a.out_f > (1ll << 31) - 1) return;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(a.row_bytes / 8),
                                static_cast<cuuint64_t>(a.out_f)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(a.row_bytes)};
    const cuuint32_t estr[2] = {1, 1};
    const int heights[2] = {G::kTileRows, 8};
    CUtensorMap *maps[2] = {&tm.tile, &tm.oct};
    for (int i = 0; i < 2; ++i) {
        const cuuint32_t box[2] = {static_cast<cuuint32_t>(G::kSlot / 8),
                                   static_cast<cuuint32_t>(heights[i])};
        if (enc(maps[i], CU_TENSOR_MAP_DATA_TYPE_UINT64, 2, const_cast<uint8_t *>(a.w), dims,
                strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return;
    }
    a.use_tma = 1;
    g_map_cache.put(key, h, tm);
}

template <int KIND, int M, int MODE, bool FUSE>
cudaError_t launch_stream(StreamArgs a, uint32_t smem_bytes, int dev, const DeviceInfo &info,
                          cudaStream_t st) {
    auto kern = gemv_stream_kernel<KIND, M, MODE, FUSE>;
    const uint64_t bit = 1ull << ((M - 1) + 8 * MODE + (FUSE ? 32 : 0));
    if (!(g_attr_set[KIND][dev].load(std::memory_order_acquire) & bit)) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             info.smem_optin);
        if (e != cudaSuccess) return e;
        g_attr_set[KIND][dev].fetch_or(bit, std::memory_order_acq_rel);
    }
    // Ring depth: as many stages as fit when the CTAs that registers allow per SM share its
    // shared memory (more stages = more weight bytes in flight), at least kMinStages.
    using G = Geo<KIND>;
    const uint32_t fixed = smem_bytes;  // everything except the ring and its barriers
    int per_sm = 0;
    cudaError_t e = occupancy(per_sm, kern, fixed + G::kMinStages * (G::kStage + 16) + 128, dev);
    if (e != cudaSuccess) return e;
    per_sm = std::max(std::min({per_sm, G::kMinCtasPerSm, a.ctas_per_sm}), 1);
    // A CTA with a short sweep (at most 8 stage loads: ragged 1024-row shapes) takes at most 4
    // stages: its ring then leaves shared memory for the next launch's CTAs to become resident
    // and start streaming while this launch drains (measured on GB300, 1024 x 5120 m = 1: E4M3
    // 4.25 -> 3.38 us, Q8_0 3.86 -> 3.27 us; 17408 x 5120, 20 loads per CTA, keeps its 6).
    int64_t rows_sum = 0;
    for (int i = 0; i < a.nmat; ++i) rows_sum += a.mat_out_f[i];
    const int64_t rows_cta = (rows_sum + static_cast<int64_t>(info.sms) * per_sm - 1) /
                             (static_cast<int64_t>(info.sms) * per_sm);
    const int64_t loads_cta = (rows_cta + G::kTileRows - 1) / G::kTileRows *
                              ((a.nb + G::kChunkBlocks - 1) / G::kChunkBlocks);
    const int s_max = loads_cta <= 8 ? std::min(4, G::kMaxStages) : G::kMaxStages;
    int S = G::kMinStages;
    for (int s = s_max; s >= G::kMinStages; --s) {
        const uint32_t need = fixed + align_up(static_cast<uint32_t>((2 * s + 1) * 8), 128) +
                              static_cast<uint32_t>(s * G::kStage);
        if (need <= static_cast<uint32_t>(info.smem_optin) &&
            static_cast<int64_t>(need + 1024) * per_sm <= info.smem_sm) {
            S = s;
            break;
        }
    }
    const uint32_t bars = align_up(static_cast<uint32_t>((2 * S + 1) * 8), 128);
    // Shift every region past the barriers.
    a.stages = S;
    a.off_part += bars;
    a.off_grid += bars;
    a.off_bfrag += bars;
    a.off_qs += bars;
    a.off_d += bars;
    a.off_red += bars;
    a.off_ring += bars;
    smem_bytes = fixed + bars + static_cast<uint32_t>(S * G::kStage);
    e = occupancy(per_sm, kern, smem_bytes, dev);
    if (e != cudaSuccess) return e;
    per_sm = std::max(per_sm, 1);
    // One wave of CTAs, split over the launch's matrices in proportion to their rows (rounded
    // up, so no matrix gets more rows per CTA than the plan assumed), never more CTAs than rows.
    const int64_t total = static_cast<int64_t>(info.sms) * std::min({per_sm, G::kCtasPerLaunch, a.ctas_per_sm});
    int64_t rows_all = 0;
    for (int i = 0; i < a.nmat; ++i) rows_all += a.mat_out_f[i];
    int64_t grid = 0;
    for (int i = 0; i < a.nmat; ++i) {
        int64_t n = (total * a.mat_out_f[i] + rows_all - 1) / rows_all;
        n = std::max<int64_t>(1, std::min<int64_t>(n, a.mat_out_f[i]));
        a.mat_cta[i] = static_cast<int>(grid);
        grid += n;
    }
    a.mat_cta[a.nmat] = static_cast<int>(grid);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem_bytes;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    TmaGroup tg = {};
    int tma_ok = 1;
    for (int i = 0; i < a.nmat; ++i) {
        StreamArgs ai = a;
        ai.w = a.mat_w[i];
        ai.out_f = a.mat_out_f[i];
        make_maps<KIND>(ai, tg.m[i], dev);
        tma_ok &= ai.use_tma;
    }
    a.use_tma = tma_ok;
    return cudaLaunchKernelEx(&cfg, kern, a, tg);
}

template <int KIND, int MODE, bool FUSE>
cudaError_t launch_stream_m(int m, StreamArgs a, uint32_t smem, int dev, const DeviceInfo &info,
                            cudaStream_t st) {
    if constexpr (KIND == kQ80T) {  // only taken from kQ80MmaMinM = 3 rows up
        switch (m) {
            case 3: return launch_stream<KIND, 3, MODE, FUSE>(a, smem, dev, info, st);
            case 4: return launch_stream<KIND, 4, MODE, FUSE>(a, smem, dev, info, st);
            case 5: return launch_stream<KIND, 5, MODE, FUSE>(a, smem, dev, info, st);
            case 6: return launch_stream<KIND, 6, MODE, FUSE>(a, smem, dev, info, st);
            case 7: return launch_stream<KIND, 7, MODE, FUSE>(a, smem, dev, info, st);
            case 8: return launch_stream<KIND, 8, MODE, FUSE>(a, smem, dev, info, st);
            default: return cudaErrorInvalidValue;
        }
    } else {
        switch (m) {
            case 1: return launch_stream<KIND, 1, MODE, FUSE>(a, smem, dev, info, st);
            case 2: return launch_stream<KIND, 2, MODE, FUSE>(a, smem, dev, info, st);
            case 3: return launch_stream<KIND, 3, MODE, FUSE>(a, smem, dev, info, st);
            case 4: return launch_stream<KIND, 4, MODE, FUSE>(a, smem, dev, info, st);
            case 5: return launch_stream<KIND, 5, MODE, FUSE>(a, smem, dev, info, st);
            case 6: return launch_stream<KIND, 6, MODE, FUSE>(a, smem, dev, info, st);
            case 7: return launch_stream<KIND, 7, MODE, FUSE>(a, smem, dev, info, st);
            default: return launch_stream<KIND, 8, MODE, FUSE>(a, smem, dev, info, st);
        }
    }
}

// Shared-memory plan of the stream kernel.  Fixed part: tile partials (E4M3 / block-128), the
// CTA's grid rows (block-128), the staged activation, and a ring of at least kMinStages stages
// (the barrier block and the final ring depth are added at launch).  The activation lives in
// shared memory -- int8 qs + scales, plus its f16 MMA fragments for E4M3 / block-128 when they
// also fit -- and the plan takes the largest CTA count per SM (at most kMinCtasPerSm) for which
// that fits; only an activation too large for one CTA per SM is read from global memory.  The
// fused decode step always needs the int8 + scales there (it computes them) and fails the plan
// if they do not fit.
template <int KIND>
bool plan_stream(int64_t out_f, int64_t in_f, int m, bool fuse, const DeviceInfo &info,
                 StreamArgs &a, uint32_t &smem, int &mode) {
    using G = Geo<KIND>;
    const int nb = static_cast<int>(in_f / 32);
    const uint32_t optin = static_cast<uint32_t>(info.smem_optin);
    const uint32_t part = G::kMma ? align_up(static_cast<uint32_t>(2 * kWarps * G::kTileRows * m * 4), 128) : 0u;
    // Grid rows one CTA can touch: rows per CTA at one CTA per SM, over 128, plus two.
    const int64_t rows_cta = (out_f + info.sms - 1) / info.sms;
    const int grid_rows = static_cast<int>(rows_cta / 128 + 2);
    const int gcols = static_cast<int>((in_f + 127) / 128);
    const uint32_t gridb = KIND == kBlk ? align_up(static_cast<uint32_t>(grid_rows * gcols * 4), 128) : 0u;
    // Activation staging: the dp4a layout (Q8_0) sits beside the staged int8 qs; the f16 MMA
    // fragments (E4M3 / block-128 / Q8_0 on the tensor cores) are built in place over it, so
    // their region holds the qs at its top and no separate qs region is needed.
    const uint32_t frag = G::kMma ? align_up(static_cast<uint32_t>(m * (nb | 1) * 64), 128)
                                  : align_up(static_cast<uint32_t>(nb * m * 4 * kQ8ActWords), 128);
    // Staged rows: from m = 5 (where 3 or 4 tokens' scales meet in one warp load) d padded to 4
    // mod 16 floats and qs to 32 mod 128 bytes where the tensor-core consumers read it per block
    // (kActSmem); the in-place fragment build and the dp4a layouts read qs contiguous.  Measured
    // on GB300, 17408 x 5120: m = 8 E4M3 18.0 -> 16.1 us, Q8_0 23.6 -> 19.1 us; at m <= 4 the
    // per-row copies cost more than the 2-way conflicts they remove (5120 x 5120 m = 3 +2%).
    const int dstr = m >= 5 ? nb + ((4 - nb) & 15) : nb;
    const int qstr_smem = G::kMma && m >= 5 ? static_cast<int>(in_f + ((32 - in_f) & 127)) : static_cast<int>(in_f);
    const uint32_t qsb = align_up(static_cast<uint32_t>(m * in_f), 128);
    const uint32_t qsb_smem = align_up(static_cast<uint32_t>(m * qstr_smem), 128);
    const uint32_t frag_act = G::kMma ? frag : frag + qsb;
    const uint32_t db = align_up(static_cast<uint32_t>(m * dstr * 4), 128);
    // block-128 with a staged activation: the CTA's d * grid table
    const uint32_t red = fuse ? align_up((kWarps + 1) * 8, 128) : 0u;
    const uint32_t ring_min = static_cast<uint32_t>(G::kMinStages * G::kStage) + 128;
    const uint32_t base = part + gridb + red + ring_min;
    if (base > optin) return false;
    // Small problems: fewer CTAs per SM when a CTA would get fewer than kMinRowsPerCta rows
    // (measured: 1024 x 5120 runs 20-30% faster at one CTA per SM than with 2-3 rows per CTA;
    // from about 7 rows per CTA up, more CTAs per SM are faster).
    constexpr int64_t kMinRowsPerCta = 4;
    // Preferred CTAs per SM, measured on GB300 (back-to-back launches, DRAM-cold):
    //  * E4M3 / block-128: two when every CTA then gets at least two full 16-row tiles (17408 x
    //    5120: 15.0 us against 16.1 us with three), else three (5120 x 5120: 6.3 against 7.9 us;
    //    5120 x 17408: 17.2 against 21.8 us).  CTAs of one launch sharing an SM do not stream at
    //    equal rates, so fewer and larger CTAs shorten the tail -- unless a CTA's rows make only
    //    one full tile and a ragged one, or its staged activation leaves a shallow ring.
    //  * Q8_0 with dp4a: two by the same rule (17408 x 5120: 15.5 against 15.9 us with three,
    //    12288 x 5120: 11.1 against 11.6 us -- each CTA's deeper ring keeps more weight bytes in
    //    flight per SM), else four, three when the staged activation is large (5120 x 17408:
    //    17.5 against 19.1 us).
    int pref = G::kMinCtasPerSm;
    const bool two_tiles = out_f >= static_cast<int64_t>(info.sms) * 2 * 2 * G::kTileRows;
    if (KIND == kE4M3 || KIND == kBlk)
        pref = two_tiles ? 2 : 3;
    else if (KIND == kQ80)
        pref = two_tiles ? 2 : static_cast<int64_t>(m) * in_f > 8192 ? 3 : 4;
    const int k_rows = static_cast<int>(std::min<int64_t>(
        pref, std::max<int64_t>(1, out_f / (static_cast<int64_t>(info.sms) * kMinRowsPerCta))));
    int ctas = k_rows;
    mode = kActGlobal;
    for (int k = k_rows; k >= 1; --k) {
        // Shared memory one CTA may use and still leave room for k CTAs per SM.
        const uint32_t budget = std::min(optin, static_cast<uint32_t>(info.smem_sm / k - 1024));
        if (base + frag_act + db <= budget) {
            mode = kActFrag;
        } else if (base + qsb_smem + db <= budget) {
            mode = kActSmem;
        } else {
            continue;
        }
        ctas = k;
        break;
    }
    if (fuse && mode == kActGlobal) return false;
    a.grid_rows = grid_rows;
    a.ctas_per_sm = ctas;
    a.qstr = mode == kActSmem ? qstr_smem : static_cast<int>(in_f);
    a.dstr = mode == kActGlobal ? nb : dstr;
    a.off_part = 0;
    a.off_grid = a.off_part + part;
    uint32_t off = a.off_grid + gridb;
    a.off_bfrag = off;
    if (mode == kActFrag) off += frag;
    if (G::kMma && mode == kActFrag) {
        // the int8 qs at the top of the fragment region (16-byte aligned: 32 nb m + 64 P m)
        a.off_qs = a.off_bfrag + static_cast<uint32_t>(m * (nb | 1) * 64 - m * in_f);
    } else {
        a.off_qs = off;
        if (mode != kActGlobal) off += mode == kActSmem ? qsb_smem : qsb;
    }
    a.off_d = off;
    if (mode != kActGlobal) off += db;
    a.off_red = off;
    off += red;  // cross-warp scratch of the fused prologue
    a.off_ring = off;
    smem = off;  // fixed part; the ring is added in launch_stream
    return true;
}

template <int KIND, bool FUSE>
cudaError_t launch_planned(int m, int mode, StreamArgs a, uint32_t smem, int dev,
                           const DeviceInfo &info, cudaStream_t st) {
    if (mode == kActFrag) return launch_stream_m<KIND, kActFrag, FUSE>(m, a, smem, dev, info, st);
    if (mode == kActSmem) return launch_stream_m<KIND, kActSmem, FUSE>(m, a, smem, dev, info, st);
    if constexpr (!FUSE) return launch_stream_m<KIND, kActGlobal, false>(m, a, smem, dev, info, st);
    return cudaErrorInvalidValue;
}

}  // namespace
}  // namespace memq

#include "memq_gemv_kouter.cuh"

namespace memq {
namespace {

template <int KIND>
int check_gemv_args(const uint8_t *w, const float *aux, const int8_t *qs, const float *d,
                    float *y, int64_t out_f, int64_t in_f, int m) {
    if (m < 1 || m > MEMQ_MAX_M) return MEMQ_ERR_M_RANGE;
    if (in_f < 32 || (in_f % 32) != 0 || in_f > (1LL << 24)) return MEMQ_ERR_SHAPE;
    if (out_f < 0 || out_f > (1LL << 31) - 1) return MEMQ_ERR_SHAPE;
    if (out_f == 0) return MEMQ_OK;
    if (!w || !qs || !d || !y || (!is_q80(KIND) && !aux)) return MEMQ_ERR_NULL;
    if (!aligned(d, 4) || !aligned(y, 4) || (aux && !aligned(aux, 4))) return MEMQ_ERR_ALIGN;
    return -1;  // valid, work to do
}

template <int KIND>
StreamArgs base_args(const uint8_t *w, const float *aux, const int8_t *qs, const float *d,
                     float *y, int64_t out_f, int64_t in_f) {
    StreamArgs a = {};
    a.w = w;
    a.aux = aux;
    a.qs = qs;
    a.qstr = static_cast<int>(in_f);
    a.dstr = static_cast<int>(in_f / 32);
    a.d = d;
    a.y = y;
    a.out_f = out_f;
    a.row_bytes = is_q80(KIND) ? in_f / 32 * 34 : in_f;
    a.in_f = static_cast<int>(in_f);
    a.nb = static_cast<int>(in_f / 32);
    a.gcols = static_cast<int>((in_f + 127) / 128);
    a.nmat = 1;
    a.mat_w[0] = w;
    a.mat_aux[0] = aux;
    a.mat_y[0] = y;
    a.mat_out_f[0] = out_f;
    return a;
}

template <int KIND>
bool fast_path_ok(const uint8_t *w, const int8_t *qs, int64_t in_f) {
    const int64_t row_bytes = is_q80(KIND) ? in_f / 32 * 34 : in_f;
    return aligned(w, 16) && aligned(qs, 16) && (row_bytes % 16) == 0 &&
           (!is_q80(KIND) || ((in_f / 32) % 8) == 0);
}

template <int KIND>
int gemv_entry(const uint8_t *w, const float *aux, const int8_t *qs, const float *d, float *y,
               int64_t out_f, int64_t in_f, int m, void *stream) {
    const int rc = check_gemv_args<KIND>(w, aux, qs, d, y, out_f, in_f, m);
    if (rc >= 0) return rc;
    int dev = 0;
    DeviceInfo info;
    if (device_info(dev, info) != cudaSuccess) return MEMQ_ERR_LAUNCH;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if constexpr (KIND == kE4M3 || KIND == kBlk) {
        if (fast_path_ok<KIND>(w, qs, in_f)) {
            const cudaError_t ek = launch_kouter_m<KIND>(m, 1, &w, &aux, &y, &out_f, qs, d, in_f, dev, info, st);
            if (ek != cudaErrorNotSupported) return ek == cudaSuccess ? MEMQ_OK : MEMQ_ERR_LAUNCH;
        }
    }
    StreamArgs a = base_args<KIND>(w, aux, qs, d, y, out_f, in_f);
    uint32_t smem = 0;
    int mode = kActGlobal;
    cudaError_t e;
    if (fast_path_ok<KIND>(w, qs, in_f) && plan_stream<KIND>(out_f, in_f, m, false, info, a, smem, mode)) {
        e = launch_planned<KIND, false>(m, mode, a, smem, dev, info, st);
    } else {
        const int64_t blocks = (out_f + kGenericWarps - 1) / kGenericWarps;
        constexpr int GK = KIND == kQ80T ? kQ80 : KIND;
        gemv_generic_kernel<GK><<<static_cast<unsigned>(blocks), kGenericWarps * 32, 0, st>>>(
            w, aux, qs, d, y, out_f, static_cast<int>(in_f), m);
        e = cudaGetLastError();
    }
    return e == cudaSuccess ? MEMQ_OK : MEMQ_ERR_LAUNCH;
}

// A group of GEMVs sharing one activation (qs, d, in_f, m) in one launch: the matrices' rows
// are split over the CTAs in proportion, each CTA streams one matrix, and every CTA stages the
// same activation.  Taken when every matrix is on the fast path; otherwise one GEMV per matrix.
template <int KIND>
int group_entry(int count, const uint8_t *const *w, const float *const *aux, float *const *y,
                const int64_t *out_f, const int8_t *qs, const float *d, int64_t in_f, int m,
                void *stream) {
    if (count < 1 || count > kMaxGroup) return MEMQ_ERR_SHAPE;
    if (!w || !y || !out_f || (!is_q80(KIND) && !aux)) return MEMQ_ERR_NULL;
    int64_t rows_all = 0;
    bool fast = true;
    for (int i = 0; i < count; ++i) {
        const int rc = check_gemv_args<KIND>(w[i], is_q80(KIND) ? nullptr : aux[i], qs, d, y[i],
                                             out_f[i], in_f, m);
        if (rc > 0) return rc;
        if (rc == MEMQ_OK) return MEMQ_ERR_SHAPE;  // an empty matrix in a group
        rows_all += out_f[i];
        fast = fast && fast_path_ok<KIND>(w[i], qs, in_f);
    }
    if (!fast) {
        for (int i = 0; i < count; ++i) {
            const int rc = gemv_entry<KIND>(w[i], is_q80(KIND) ? nullptr : aux[i], qs, d, y[i],
                                            out_f[i], in_f, m, stream);
            if (rc != MEMQ_OK) return rc;
        }
        return MEMQ_OK;
    }
    int dev = 0;
    DeviceInfo info;
    if (device_info(dev, info) != cudaSuccess) return MEMQ_ERR_LAUNCH;
    if constexpr (KIND == kE4M3 || KIND == kBlk) {
        const cudaError_t ek = launch_kouter_m<KIND>(m, count, w, aux, y, out_f, qs, d, in_f, dev,
                                                     info, static_cast<cudaStream_t>(stream));
        if (ek != cudaErrorNotSupported) return ek == cudaSuccess ? MEMQ_OK : MEMQ_ERR_LAUNCH;
    }
    StreamArgs a = base_args<KIND>(w[0], is_q80(KIND) ? nullptr : aux[0], qs, d, y[0], out_f[0], in_f);
    a.nmat = count;
    for (int i = 0; i < count; ++i) {
        a.mat_w[i] = w[i];
        a.mat_aux[i] = is_q80(KIND) ? nullptr : aux[i];
        a.mat_y[i] = y[i];
        a.mat_out_f[i] = out_f[i];
    }
    uint32_t smem = 0;
    int mode = kActGlobal;
    if (!plan_stream<KIND>(rows_all, in_f, m, false, info, a, smem, mode)) {
        for (int i = 0; i < count; ++i) {
            const int rc = gemv_entry<KIND>(w[i], is_q80(KIND) ? nullptr : aux[i], qs, d, y[i],
                                            out_f[i], in_f, m, stream);
            if (rc != MEMQ_OK) return rc;
        }
        return MEMQ_OK;
    }
    const cudaError_t e = launch_planned<KIND, false>(m, mode, a, smem, dev, info,
                                                      static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MEMQ_OK : MEMQ_ERR_LAUNCH;
}

// The fused decode step: RMSNorm -> q8_1 of x (m rows) and the GEMV in one launch when the plan
// allows it, else memq_rmsnorm_q8_1 followed by the GEMV.  Either way qs / d (and z when given)
// receive the activation.
template <int KIND>
int fused_check(const float *x, const float *wn, float eps, const uint8_t *w, const float *aux,
                int8_t *qs, float *d, float *z, float *y, int64_t out_f, int64_t in_f, int m) {
    // check_gemv_args: > 0 an error; MEMQ_OK when out_f == 0 (nothing to multiply, the
    // activation is still produced); < 0 work to do
    const int rc = check_gemv_args<KIND>(w, aux, qs, d, y, out_f, in_f, m);
    if (rc > 0) return rc;
    if (in_f > MEMQ_MAX_NCOLS) return MEMQ_ERR_SHAPE;
    if (!(eps >= 0.0f) || eps == INFINITY) return MEMQ_ERR_SHAPE;
    if (!x || !wn || !qs || !d) return MEMQ_ERR_NULL;
    if (!aligned(x, 16) || !aligned(wn, 16) || (z && !aligned(z, 16)) || !aligned(qs, 4) ||
        !aligned(d, 4))
        return MEMQ_ERR_ALIGN;
    return MEMQ_OK;
}

template <int KIND>
int fused_entry(const float *x, const float *wn, float eps, const uint8_t *w, const float *aux,
                int8_t *qs, float *d, float *z, float *y, int64_t out_f, int64_t in_f, int m,
                void *stream) {
    const int rc = fused_check<KIND>(x, wn, eps, w, aux, qs, d, z, y, out_f, in_f, m);
    if (rc != MEMQ_OK) return rc;
    int dev = 0;
    DeviceInfo info;
    if (device_info(dev, info) != cudaSuccess) return MEMQ_ERR_LAUNCH;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (out_f > 0 && fast_path_ok<KIND>(w, qs, in_f)) {
        StreamArgs a = base_args<KIND>(w, aux, qs, d, y, out_f, in_f);
        a.x = x;
        a.wn = wn;
        a.eps = eps;
        a.z_out = z;
        uint32_t smem = 0;
        int mode = kActSmem;
        if (plan_stream<KIND>(out_f, in_f, m, true, info, a, smem, mode)) {
            const cudaError_t e = launch_planned<KIND, true>(m, mode, a, smem, dev, info, st);
            return e == cudaSuccess ? MEMQ_OK : MEMQ_ERR_LAUNCH;
        }
    }
    const int r = memq_rmsnorm_q8_1(x, wn, z, qs, d, in_f, m, eps, stream);
    if (r != MEMQ_OK || out_f == 0) return r;
    return gemv_entry<KIND>(w, aux, qs, d, y, out_f, in_f, m, stream);
}

// One decode step for a caller whose activation rows and outputs live in host memory: the
// arguments are checked as the fused step checks them (nothing is enqueued on an error), then
// x_host -> x_dev, `step()` (the fused step on the device buffers), y_dev -> y_host,
// and a wait for the stream.  Past the checks, a failure still waits for the stream, so that
// no copy is left reading or writing the host buffers when the call returns.
template <int KIND, typename Step>
int host_step_entry(const float *x_host, float *x_dev, const float *wn, float eps,
                    const uint8_t *w, const float *aux, int8_t *qs, float *d, float *z,
                    float *y_dev, float *y_host, int64_t out_f, int64_t in_f, int m, void *stream,
                    Step step) {
    const int rc = fused_check<KIND>(x_dev, wn, eps, w, aux, qs, d, z, y_dev, out_f, in_f, m);
    if (rc != MEMQ_OK) return rc;
    if (!x_host || (out_f > 0 && !y_host)) return MEMQ_ERR_NULL;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const size_t x_bytes = sizeof(float) * static_cast<size_t>(m) * static_cast<size_t>(in_f);
    const size_t y_bytes = sizeof(float) * static_cast<size_t>(m) * static_cast<size_t>(out_f);
    int r = cudaMemcpyAsync(x_dev, x_host, x_bytes, cudaMemcpyHostToDevice, st) == cudaSuccess
                ? MEMQ_OK
                : MEMQ_ERR_LAUNCH;
    if (r == MEMQ_OK) r = step();
    if (r == MEMQ_OK && y_bytes > 0 &&
        cudaMemcpyAsync(y_host, y_dev, y_bytes, cudaMemcpyDeviceToHost, st) != cudaSuccess)
        r = MEMQ_ERR_LAUNCH;
    const bool waited = cudaStreamSynchronize(st) == cudaSuccess;
    return r != MEMQ_OK ? r : waited ? MEMQ_OK : MEMQ_ERR_LAUNCH;
}

// Reads (and optionally clears) this translation unit's device fault word.
inline cudaError_t read_fault(unsigned int *out, bool clear) {
    cudaError_t e = cudaMemcpyFromSymbol(out, g_memq_fault, sizeof(unsigned int));
    if (e != cudaSuccess || !clear) return e;
    const unsigned int zero = 0;
    return cudaMemcpyToSymbol(g_memq_fault, &zero, sizeof(zero));
}

}  // namespace
}  // namespace memq

