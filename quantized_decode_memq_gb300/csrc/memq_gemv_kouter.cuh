// memq_gemv_kouter.cuh -- the K-outer weight-stream GEMV for E4M3 and block-128 weights.
// Included by memq_gemv_kernels.cuh (after the tile kernel and its helpers), inside the same
// namespace.
//
// Operations: gemv_e4m3_bench.rs (memra-engine 0.125.0), module doc -- "THE COMPARISON" (arm
// E4M3) and "THE BLOCK-128 ARM"; m <= 8 activation rows read against one weight stream (module
// doc, "grid.y=m and _b2/_b4/_b8 bit-parity arms").
//
// Schedule.  CTA c owns output rows [R0, R1), an equal share (+-1 row) of out_f, and sweeps K in
// the outer loop: a stage of the shared ring holds ALL of the CTA's rows (up to 16 * TILES per
// pass; more rows take more passes) for a K-chunk of kw 32-blocks, plus that chunk of the q8_1
// activation (qs and d of every token).  So
//   * a CTA never walks a ragged tile: 17 rows cost one sweep, not a 16-row and a 1-row sweep;
//   * nothing is staged per CTA before the stream starts: the activation chunk arrives with its
//     stage (the weights of the first stages are requested before the preceding grid has
//     finished, their activation chunks right after it has);
//   * the B fragments of a block (the activation of up to 8 tokens, int8 -> f16 exact) are built
//     once per stage and serve every 16-row tile of the CTA.
// The producer warp issues per stage one 2-D tensor copy of the pass's rows (rows of `slot`
// bytes: the kw*32 weight bytes plus 32 bytes that keep the consumers' fragment loads
// bank-conflict free; a pass one row longer than the box gets a 1-D bulk copy for it), and one
// tensor copy each for the activation's qs and d.  Consumer warp w takes blocks 4w..4w+3 of the
// stage's 32-block chunk for all row tiles; each block's 16 x 32 x 8 product is two
// mma.sync.m16n8k16 (E4M3 -> f16 by the hardware cvt and int8 -> f16 are exact, products exact
// in f32, f32 accumulation), scaled by d[token][block] (block-128: the warp's 128-column group
// sum scaled by the grid entry of the row).  At the end of a pass the eight warps' partial sums
// of each (row, token) are added in warp order (deterministic) and stored.  Per (row, token)
// these are the tile kernel's f32 operations in the tile kernel's order: the two kernels agree
// bit for bit.
#pragma once

namespace memq {
namespace {

// Row tiles of 16 per pass: the kernel is compiled for passes of up to 16 rows (three CTAs per
// SM) and of up to 64 rows (two CTAs per SM).
constexpr int kKoMaxTiles = 4;
constexpr int kKoMinStages = 3;
constexpr int kKoMaxStages = 12;
constexpr int kKoKw = 32;                // 32-blocks per stage: the tile kernel's chunk
// Per container: bytes of a 32-weight block, of a row's K-chunk, and of a row slot in a stage
// (the chunk plus padding that keeps the consumers' fragment loads bank-conflict free: E4M3 /
// block-128 rows 32 bytes apart modulo the 128-byte bank period, Q8_0 rows 80, as in the tile
// kernel).
// The stage's activation chunk: token rows of kw 32-blocks of qs padded to 1056 bytes and of kw
// scales padded to 36 floats (the tensor copies' boxes are that wide and read the next chunk's
// first bytes, or zeros past the end), so the B-fragment loads of 8 tokens (rows 32 bytes apart
// modulo the 128-byte bank period) and the scale loads of tokens 2t (rows 8 banks apart) are
// bank-conflict free.
constexpr int kKoActRow = kKoKw * 32 + 32;  // bytes per token row of qs in a stage
constexpr int kKoDRow = kKoKw + 4;          // floats per token row of d in a stage

template <int KIND>
struct KoGeo {
    static constexpr int kBlockBytes = KIND == kQ80T ? 34 : 32;
    static constexpr int kChunk = kKoKw * kBlockBytes;
    static constexpr int kSlot = kChunk + (KIND == kQ80T ? 16 : 32);
};

struct KoArgs {
    int nmat;
    int mat_cta[kMaxGroup + 1];
    const uint8_t *mat_w[kMaxGroup];
    const float *mat_aux[kMaxGroup];
    float *mat_y[kMaxGroup];
    int64_t mat_out_f[kMaxGroup];
    int64_t row_bytes;
    int in_f;
    int nb;         // in_f / 32
    int gcols;      // ceil(in_f / 128)
    int box_rows[kMaxGroup];  // per matrix: rows of the weight tensor box (the fewest a pass
                              // holds); a pass with more rows copies the rest row by row
    int stage;      // bytes per stage (weights of the largest pass + activation)
    int act_qs;     // offset of the stage's qs chunk [m][kKoActRow]
    int act_d;      // offset of the stage's d chunk [m][kKoDRow] (f32)
    int act_bytes;  // bytes the two activation copies complete per stage
    int stages;
    uint32_t off_part, off_grid, off_ring;
};

// Tensor maps: per matrix the weight plane as [out_f][row_bytes / 8] 64-bit elements with boxes
// of slot bytes x box_rows rows (one copy per stage brings a pass's rows); the activation qs as
// [m][in_f / 8] 64-bit elements, box kKoActRow bytes x m rows; d as [m][in_f / 32] f32, box
// kKoDRow x m.
struct KoMaps {
    CUtensorMap w8[kMaxGroup];
    CUtensorMap qs;
    CUtensorMap d;
};

__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

// Rows [P0, P1) of pass p of a CTA with rows [R0, R1): passes of near-equal size.
__device__ __forceinline__ void ko_pass_rows(int64_t R0, int64_t R1, int npass, int p,
                                             int64_t &P0, int64_t &P1) {
    const int64_t R = R1 - R0;
    P0 = R0 + R * p / npass;
    P1 = R0 + R * (p + 1) / npass;
}

// One consumer warp's share of a stage: blocks 4w .. 4w+3 of the 32-block chunk that starts at
// block kbc (the same blocks, in the same order, as the tile kernel's warp w), for the pass's T
// row tiles.  acc[rt][0..3] = rows (16rt + g, 16rt + g + 8) x tokens (2t, 2t+1).  The f32
// operations per (row, token) are exactly the tile kernel's (block results scaled by d in block
// order; block-128: the warp's four blocks -- one 128-column group -- summed, then scaled by the
// grid entry), so both kernels give bit-identical outputs and either may serve a call.
// ro[rt][0 / 1]: byte offsets of this thread's rows 16rt + g and 16rt + g + 8 in the stage, both
// clamped to the pass's last row (rows past it are computed from a valid row and never stored,
// and no load leaves the stage's weight region).
// Q8_0 on the tensor cores: the same share of a stage with A = the int8 weights of the pass's
// rows (int8 -> f16 exact) and each block's (row, token) result scaled by d_w[row] * d_x[token]
// -- per (row, token) exactly the tile kernel's Q8_0 tensor-core operations in its order
// (mma_stage_q80), so either kernel may serve a call.  The warp's four records start 136w bytes
// into each 1104-byte row slot, so a record's weight bytes are 4-byte aligned for odd blocks and
// 2 mod 4 for even ones (q80_weights8).
template <int M, int TILES, bool FULL>
__device__ __forceinline__ void ko_stage_q80(const KoArgs &a, const uint8_t *stage, int T,
                                             const int (&ro)[TILES][2], int kbc, int warp,
                                             int lane, float (&acc)[TILES][4]) {
    const int g = lane >> 2;
    const int t = lane & 3;
    const int j0 = 4 * warp;
    const int nblk = FULL ? 4 : min(4, a.nb - kbc - j0);
    if (!FULL && nblk <= 0) return;
    // B column g is token g; columns g >= M read token M - 1 (no divergent branch): an MMA
    // column depends only on its own B column, and those columns are never stored
    const uint8_t *aq = stage + a.act_qs + (g < M ? g : M - 1) * kKoActRow + 32 * j0 + 8 * t;
    const float *ad = reinterpret_cast<const float *>(stage + a.act_d) + 2 * t * kKoDRow + j0;
    const uint8_t *pa = stage + 34 * j0;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
        if (FULL || b < nblk) {
            uint32_t bq[4] = {0u, 0u, 0u, 0u};
            {
                const uint2 qv = lds64(aq + 32 * b);
                s8x4_to_f16x2x2(qv.x, bq[0], bq[1]);
                s8x4_to_f16x2x2(qv.y, bq[2], bq[3]);
            }
            const float k0 = 2 * t < M ? ad[b] : 0.f;
            const float k1 = 2 * t + 1 < M ? ad[kKoDRow + b] : 0.f;
#pragma unroll
            for (int rt = 0; rt < TILES; ++rt) {
                if (TILES == 1 || rt < T) {
                    const uint8_t *r0 = pa + ro[rt][0] + 34 * b;
                    const uint8_t *r8 = pa + ro[rt][1] + 34 * b;
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
                    acc[rt][0] = fmaf(c[0], dw0 * k0, acc[rt][0]);
                    acc[rt][1] = fmaf(c[1], dw0 * k1, acc[rt][1]);
                    acc[rt][2] = fmaf(c[2], dw8 * k0, acc[rt][2]);
                    acc[rt][3] = fmaf(c[3], dw8 * k1, acc[rt][3]);
                }
            }
        }
    }
}

template <int KIND, int M, int TILES, bool FULL>
__device__ __forceinline__ void ko_stage(const KoArgs &a, const uint8_t *stage, const float *s_grid,
                                         int64_t P0, int64_t P1, int64_t grow_base, int T,
                                         const int (&ro)[TILES][2], int kbc, int warp, int lane,
                                         float (&acc)[TILES][4]) {
    if constexpr (KIND == kQ80T) {
        ko_stage_q80<M, TILES, FULL>(a, stage, T, ro, kbc, warp, lane, acc);
    } else {
    const int g = lane >> 2;
    const int t = lane & 3;
    const int j0 = 4 * warp;
    const int nblk = FULL ? 4 : min(4, a.nb - kbc - j0);
    if (!FULL && nblk <= 0) return;
    // this thread's activation bytes (token g) and scales (tokens 2t, 2t+1) of block j0
    // B column g is token g; columns g >= M read token M - 1 (no divergent branch): an MMA
    // column depends only on its own B column, and those columns are never stored
    const uint8_t *aq = stage + a.act_qs + (g < M ? g : M - 1) * kKoActRow + 32 * j0 + 8 * t;
    const float *ad = reinterpret_cast<const float *>(stage + a.act_d) + 2 * t * kKoDRow + j0;
    const uint8_t *pa = stage + 32 * j0 + 8 * t;
    float grp[TILES][4];
#pragma unroll
    for (int rt = 0; rt < TILES; ++rt) grp[rt][0] = grp[rt][1] = grp[rt][2] = grp[rt][3] = 0.f;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
        if (FULL || b < nblk) {
            uint32_t bq[4] = {0u, 0u, 0u, 0u};
            {
                const uint2 qv = lds64(aq + 32 * b);
                s8x4_to_f16x2x2(qv.x, bq[0], bq[1]);
                s8x4_to_f16x2x2(qv.y, bq[2], bq[3]);
            }
            const float k0 = 2 * t < M ? ad[b] : 0.f;
            const float k1 = 2 * t + 1 < M ? ad[kKoDRow + b] : 0.f;
#pragma unroll
            for (int rt = 0; rt < TILES; ++rt) {
                if (TILES == 1 || rt < T) {
                    const uint2 wa = lds64(pa + ro[rt][0] + 32 * b);
                    const uint2 wb = lds64(pa + ro[rt][1] + 32 * b);
                    uint32_t a0, a1, a2, a3;
                    float c[4] = {0.f, 0.f, 0.f, 0.f};
                    e4m3x4_to_f16x2x2(wa.x, a0, a2);
                    e4m3x4_to_f16x2x2(wb.x, a1, a3);
                    mma_f16_16816(c, a0, a1, a2, a3, bq[0], bq[1]);
                    e4m3x4_to_f16x2x2(wa.y, a0, a2);
                    e4m3x4_to_f16x2x2(wb.y, a1, a3);
                    mma_f16_16816(c, a0, a1, a2, a3, bq[2], bq[3]);
                    float(&dst)[4] = KIND == kBlk ? grp[rt] : acc[rt];
                    dst[0] = fmaf(c[0], k0, dst[0]);
                    dst[1] = fmaf(c[1], k1, dst[1]);
                    dst[2] = fmaf(c[2], k0, dst[2]);
                    dst[3] = fmaf(c[3], k1, dst[3]);
                }
            }
        }
    }
    if (KIND == kBlk) {
        // the grid entries of this thread's two rows for the warp's 128-column group
        const int col = (kbc + j0) >> 2;
#pragma unroll
        for (int rt = 0; rt < TILES; ++rt) {
            if (TILES == 1 || rt < T) {
                const int64_t ra = min(P0 + 16 * rt + g, P1 - 1);
                const int64_t rb = min(P0 + 16 * rt + g + 8, P1 - 1);
                const float ga = s_grid[((ra >> 7) - grow_base) * a.gcols + col];
                const float gb = s_grid[((rb >> 7) - grow_base) * a.gcols + col];
                acc[rt][0] = fmaf(grp[rt][0], ga, acc[rt][0]);
                acc[rt][1] = fmaf(grp[rt][1], ga, acc[rt][1]);
                acc[rt][2] = fmaf(grp[rt][2], gb, acc[rt][2]);
                acc[rt][3] = fmaf(grp[rt][3], gb, acc[rt][3]);
            }
        }
    }
    }  // E4M3 / block-128
}

template <int KIND, int M, int TILES>
__global__ void __launch_bounds__(kThreads, TILES == 1 ? 3 : 2)
    gemv_kouter_kernel(const __grid_constant__ KoArgs args, const __grid_constant__ KoMaps maps) {
    constexpr int kPassRows = 16 * TILES;
    extern __shared__ __align__(128) uint8_t smem[];
    griddep_launch_dependents();

    int mi = 0;
    while (mi + 1 < args.nmat && static_cast<int>(blockIdx.x) >= args.mat_cta[mi + 1]) ++mi;
    const KoArgs &a = args;
    const uint8_t *w = a.mat_w[mi];
    const float *aux = a.mat_aux[mi];
    float *y = a.mat_y[mi];
    const int64_t out_f = a.mat_out_f[mi];
    const int64_t cta = static_cast<int64_t>(blockIdx.x) - a.mat_cta[mi];
    const int64_t ncta = a.mat_cta[mi + 1] - a.mat_cta[mi];
    const int64_t R0 = cta * out_f / ncta;
    const int64_t R1 = (cta + 1) * out_f / ncta;
    const int npass = static_cast<int>((R1 - R0 + kPassRows - 1) / kPassRows);
    const int nch = (a.nb + kKoKw - 1) / kKoKw;
    const int items = npass * nch;
    const int S = a.stages;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    uint64_t *full = reinterpret_cast<uint64_t *>(smem);
    uint64_t *empty = full + S;
    uint8_t *ring = smem + a.off_ring;
    float *part = reinterpret_cast<float *>(smem + a.off_part);  // [kWarps][TILES][16][M]
    // Tensor copies need 128-byte aligned destinations (stage offsets are multiples of 128): a
    // ring that is not would be a fault, so record it and do nothing.
    if ((smem_u32(ring) & 127u) != 0) {
        if (threadIdx.x == 0) fault(2u);
        return;
    }

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kWarps);
        }
        mbar_init_fence();
    }
    __syncthreads();

    if (warp == kWarps) {
        // ------------------------------- producer warp ---------------------------------------
        if (lane == 0 && items > 0) {
            const uint64_t pol = l2_evict_first_policy();
            tma_prefetch_map(&maps.w8[mi]);
            tma_prefetch_map(&maps.qs);
            tma_prefetch_map(&maps.d);
            // The item cursor walks (pass, K-chunk) in order without divisions: the single
            // producer thread shares its SM sub-partition with busy consumer warps, so a long
            // dependent chain per stage (64-bit divisions) would delay every copy it issues.
            using KG = KoGeo<KIND>;
            const int last_nbytes = (a.nb - (nch - 1) * kKoKw) * KG::kBlockBytes;
            const int box_rows = a.box_rows[mi];
            struct Cursor {
                int p, ch, rows, boxed;
                int64_t P0;
            };
            auto start_pass = [&](Cursor &c, int p) {
                int64_t P0, P1;
                ko_pass_rows(R0, R1, npass, p, P0, P1);
                c.p = p;
                c.ch = 0;
                c.P0 = P0;
                c.rows = static_cast<int>(P1 - P0);
                c.boxed = min(c.rows, box_rows);
            };
            auto advance = [&](Cursor &c) {
                if (++c.ch == nch) start_pass(c, c.p + 1);
            };
            // Bytes the item's weight copies complete: boxed rows whole slots (box = slot bytes),
            // the rows left over only the chunk's weight bytes.
            auto weight_bytes = [&](const Cursor &c) -> uint32_t {
                const int nbytes = c.ch == nch - 1 ? last_nbytes : KG::kChunk;
                return static_cast<uint32_t>(c.boxed * KG::kSlot + nbytes * (c.rows - c.boxed));
            };
            auto issue_weights = [&](const Cursor &c, int s) {
                const int kb = c.ch * kKoKw;
                uint8_t *dst = ring + s * a.stage;
                tma_load_2d(dst, &maps.w8[mi], kb * KG::kBlockBytes / 8, static_cast<int>(c.P0), &full[s], pol);
                const uint32_t nbytes = static_cast<uint32_t>(c.ch == nch - 1 ? last_nbytes : KG::kChunk);
                const uint8_t *src = w + c.P0 * a.row_bytes + static_cast<int64_t>(kb) * KG::kBlockBytes;
                for (int r = c.boxed; r < c.rows; ++r)
                    bulk_g2s(dst + r * KG::kSlot, src + r * a.row_bytes, nbytes, &full[s], pol);
            };
            auto issue_act = [&](int ch, int s) {
                uint8_t *dst = ring + s * a.stage;
                tma_load_2d_plain(dst + a.act_qs, &maps.qs, ch * kKoKw * 4, 0, &full[s]);
                tma_load_2d_plain(dst + a.act_d, &maps.d, ch * kKoKw, 0, &full[s]);
            };
            // The first stages' weights go out before the preceding grid has finished (their
            // barriers announce the weight bytes without arriving); once it has, their
            // activation chunks follow with the arrival.  The bounded waits for released stages
            // start only after that, so a long predecessor never counts against this launch.
            const int pre = min(S, items);
            Cursor c;
            start_pass(c, 0);
            for (int it = 0; it < pre; ++it) {
                mbar_expect_tx(&full[it], weight_bytes(c));
                issue_weights(c, it);
                advance(c);
            }
            griddep_wait();
            for (int it = 0, ch = 0; it < pre; ++it) {
                mbar_arrive_expect_tx(&full[it], static_cast<uint32_t>(a.act_bytes));
                issue_act(ch, it);
                if (++ch == nch) ch = 0;
            }
            // Item it >= S goes to stage it % S once its use it / S - 1 has been released
            // (empty-barrier phase it / S - 1, parity ep).
            int s = 0;
            uint32_t ep = 0;
            for (int it = pre; it < items; ++it) {
                if (!thread_wait_bounded(&empty[s], ep)) {
                    fault(2u);
                    break;
                }
                mbar_arrive_expect_tx(&full[s], weight_bytes(c) + static_cast<uint32_t>(a.act_bytes));
                issue_weights(c, s);
                issue_act(c.ch, s);
                advance(c);
                if (++s == S) {
                    s = 0;
                    ep ^= 1u;
                }
            }
        }
        return;
    }

    // --------------------------------- consumer warps ------------------------------------------
    float scale = 1.0f;
    if (KIND == kE4M3) scale = __ldg(aux);
    const int64_t grow_base = R0 >> 7;
    float *s_grid = reinterpret_cast<float *>(smem + a.off_grid);
    if (KIND == kBlk) {
        const int nrows = static_cast<int>(((R1 - 1) >> 7) - grow_base + 1);
        for (int i = threadIdx.x; i < nrows * a.gcols; i += kConsumerThreads)
            s_grid[i] = __ldg(aux + grow_base * a.gcols + i);
        named_barrier_consumers();
    }
    bool ok = true;
    int it = 0;
    int s = 0;         // stage of item it (it % S)
    uint32_t ph = 0;   // parity of the full-barrier phase awaited for item it ((it / S) & 1)
    for (int p = 0; p < npass; ++p) {
        int64_t P0, P1;
        ko_pass_rows(R0, R1, npass, p, P0, P1);
        const int rows = static_cast<int>(P1 - P0);
        const int T = (rows + 15) >> 4;
        int ro[TILES][2];
#pragma unroll
        for (int rt = 0; rt < TILES; ++rt) {
            ro[rt][0] = min(16 * rt + (lane >> 2), rows - 1) * KoGeo<KIND>::kSlot;
            ro[rt][1] = min(16 * rt + (lane >> 2) + 8, rows - 1) * KoGeo<KIND>::kSlot;
        }
        float acc[TILES][4];
#pragma unroll
        for (int rt = 0; rt < TILES; ++rt)
            acc[rt][0] = acc[rt][1] = acc[rt][2] = acc[rt][3] = 0.f;
        for (int ch = 0; ch < nch; ++ch, ++it) {
            if (ok && !warp_wait_bounded(&full[s], ph)) {
                // Record the fault, give the copies that may be in flight a bounded chance to
                // land, and stop consuming; the pass barriers below still run.
                if (lane == 0) fault(1u);
                for (int j = it + 1; j < min(items, it + S); ++j)
                    (void)warp_wait_bounded(&full[j % S], static_cast<uint32_t>((j / S) & 1));
                ok = false;
            }
            if (ok) {
                const uint8_t *stg = ring + static_cast<int64_t>(s) * a.stage;
                if ((ch + 1) * kKoKw <= a.nb)
                    ko_stage<KIND, M, TILES, true>(a, stg, s_grid, P0, P1, grow_base, T, ro, ch * kKoKw, warp, lane, acc);
                else
                    ko_stage<KIND, M, TILES, false>(a, stg, s_grid, P0, P1, grow_base, T, ro, ch * kKoKw, warp, lane, acc);
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[s]);
            }
            if (++s == S) {
                s = 0;
                ph ^= 1u;
            }
        }
        // Per-warp partials of the pass -> shared memory; then the 8 warp partials of each
        // (row, token) are added in warp order and stored.
        const int g = lane >> 2, t = lane & 3;
        float *pw = part + warp * TILES * 16 * M;
#pragma unroll
        for (int rt = 0; rt < TILES; ++rt) {
            if (rt < T) {
                if (2 * t < M) {
                    pw[(rt * 16 + g) * M + 2 * t] = acc[rt][0];
                    pw[(rt * 16 + g + 8) * M + 2 * t] = acc[rt][2];
                }
                if (2 * t + 1 < M) {
                    pw[(rt * 16 + g) * M + 2 * t + 1] = acc[rt][1];
                    pw[(rt * 16 + g + 8) * M + 2 * t + 1] = acc[rt][3];
                }
            }
        }
        const bool bad = named_barrier_consumers_or(!ok);
        // y may be read or written by the preceding grid: store only once it has completed
        // (already so, since every stage's activation was requested after it had; the wait
        // states it and costs nothing then).
        griddep_wait();
        for (int idx = threadIdx.x; !bad && idx < rows * M; idx += kConsumerThreads) {
            const int row = idx / M, tok = idx - row * M;
            const float *pt = part + row * M + tok;
            float v = 0.f;
#pragma unroll
            for (int ww = 0; ww < kWarps; ++ww) v += pt[ww * TILES * 16 * M];
            y[static_cast<int64_t>(tok) * out_f + P0 + row] = v * scale;
        }
        named_barrier_consumers();  // the partial buffer is rewritten by the next pass
    }
}


// ---------------------------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------------------------
// When the K-outer kernel is used: CTAs of 8 to 16 rows at three CTAs per SM (one 16-row tile
// per pass, K-chunks of 32 blocks, one tensor copy per stage), and an activation of at least
// kKoMinAct = m * in_f bytes -- the size from which the tile kernel's per-CTA staging (1.125 to
// 3.125 bytes per activation byte) costs ring stages or CTAs per SM.  Measured on GB300
// (back-to-back launches, E4M3, us, K-outer against the tile kernel): 5120 x 17408 m = 1 16.7 /
// 17.2, m = 2 17.5 / 25.8, m = 4 17.4 / 26.2; 5120 x 5120 m = 1 7.6 / 6.5, m = 2 7.8 / 7.3,
// m = 4 7.4 / 9.6.  Below the threshold the tile kernel's once-per-CTA activation fragments
// beat K-outer's per-stage fragment conversion.  Larger CTAs stay on the tile kernel: 17408 x
// 5120 in 16-row passes at three CTAs per SM gives m = 4 16.9 / 17.0 but m = 8 19.6 / 18.0, at
// two CTAs per SM 17.9 / 17.0 and 18.4 / 18.0.
constexpr int kKoCtasPerSm = 3;
constexpr int kKoTiles = 1;
constexpr int64_t kKoMinAct = 16384;
// From m = 3: K-outer from 15360 activation bytes, i.e. also 3 x 5120 (5120 x 5120 m = 3,
// K-outer against the tile kernel: E4M3 7.1 / 7.4 us, block-128 7.15 / 7.2 us, Q8_0 8.5 us
// against 9.2 us for dp4a); at m = 2 the general threshold stays (Q8_0 5120 x 5120: 7.9 against
// 7.8 us, 4096 x 4096: 6.6 against 5.2).
constexpr int64_t kKoMinActM3 = 15360;
inline int64_t ko_min_act(int kind, int m) {
    (void)kind;
    return m >= 3 ? kKoMinActM3 : kKoMinAct;
}
std::atomic<uint64_t> g_ko_attr[3][kMaxDevices];  // [E4M3, block-128, Q8_0]: bit per m set

// Encodes (or finds in the cache) a 2-D tensor map over `base` viewed as [rows][cols] elements
// of `esize` bytes (row stride `stride` bytes), box (bx, by).  `tag` separates the map kinds in
// the cache key.
inline bool ko_map(CUtensorMap &map, int tag, const void *base, int64_t rows, int64_t cols,
                   int64_t stride, int esize, int bx, int by, int dev) {
    const MapKey key{tag * 1000000 + bx * 1000 + by, base, rows, (cols << 32) | stride, dev};
    const uint64_t h = mix_hash(mix_hash(reinterpret_cast<uintptr_t>(base), static_cast<uint64_t>(rows)),
                                static_cast<uint64_t>(key.kind) * 131 + static_cast<uint64_t>(dev));
    TmaMaps cached;
    if (g_map_cache.get(key, h, cached)) {
        map = cached.tile;
        return true;
    }
    const EncodeTiledFn enc = encode_tiled();
    if (!enc) return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(stride)};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(bx), static_cast<cuuint32_t>(by)};
    const cuuint32_t estr[2] = {1, 1};
    const CUtensorMapDataType dt = esize == 8 ? CU_TENSOR_MAP_DATA_TYPE_UINT64 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    if (enc(&map, dt, 2, const_cast<void *>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return false;
    cached.tile = map;
    g_map_cache.put(key, h, cached);
    return true;
}

// The most rows a CTA of the K-outer split holds: kKoCtasPerSm CTAs per SM, shared by the
// matrices in proportion to their rows (the split launch_kouter makes).
inline int64_t ko_rmax(int nmat, const int64_t *out_f, const DeviceInfo &info) {
    const int64_t total = static_cast<int64_t>(info.sms) * kKoCtasPerSm;
    int64_t rows_all = 0, rmax = 0;
    for (int i = 0; i < nmat; ++i) rows_all += out_f[i];
    for (int i = 0; i < nmat; ++i) {
        int64_t n = (total * out_f[i] + rows_all - 1) / rows_all;
        n = std::max<int64_t>(1, std::min<int64_t>(n, out_f[i]));
        rmax = std::max(rmax, (out_f[i] + n - 1) / n);
    }
    return rmax;
}

// Whether a Q8_0 call (or group) runs K-outer on the tensor cores: m >= 2 and the activation
// and CTA-size conditions of launch_kouter.  The Q8_0 entry points decide their path (tensor
// cores or dp4a) with it before launching.  Measured on GB300 (back-to-back, us, K-outer against
// dp4a): 5120 x 17408 m = 2 22.1 / 23.4, m = 4 22.2 / 35.9, m = 8 22.1 / 62.2; 5120 x 5120
// m = 3 8.5 / 9.2, m = 4 8.9 / 10.9, m = 8 8.0 / 19.9; at m = 1 dp4a (15.8 us at 5120 x 17408).
inline bool q80_kouter_applies(int nmat, const int64_t *out_f, int64_t in_f, int m,
                               const int8_t *qs, const float *d, const DeviceInfo &info) {
    if (m < 2 || in_f % 128 != 0 || !aligned(qs, 16) || !aligned(d, 16) ||
        m * in_f < ko_min_act(kQ80T, m))
        return false;
    const int64_t r = ko_rmax(nmat, out_f, info);
    return r >= 8 && r <= 16 * kKoTiles;
}

// Plans and launches the K-outer kernel for a group of nmat E4M3 / block-128 / Q8_0 matrices
// sharing one activation.  Returns cudaErrorNotSupported (nothing launched) when the K-outer path does
// not apply -- a CTA would get more than 16 rows, the activation scales cannot be copied as
// tensor boxes (in_f % 128 != 0, or qs / d not 16-byte aligned), or the ring would be too
// shallow -- and the caller falls back to the tile kernel.
template <int KIND, int M>
cudaError_t launch_kouter(int nmat, const uint8_t *const *w, const float *const *aux,
                          float *const *y, const int64_t *out_f, const int8_t *qs, const float *d,
                          int64_t in_f, int dev, const DeviceInfo &info, cudaStream_t st) {
    static_assert(KIND == kE4M3 || KIND == kBlk || KIND == kQ80T,
                  "K-outer path: E4M3, block-128 and Q8_0 on the tensor cores");
    using KG = KoGeo<KIND>;
    constexpr int TILES = kKoTiles;
    constexpr int kPassRows = 16 * TILES;
    if (in_f % 128 != 0 || !aligned(d, 16) || !aligned(qs, 16) || M * in_f < ko_min_act(KIND, M))
        return cudaErrorNotSupported;
    KoArgs a = {};
    a.nmat = nmat;
    a.row_bytes = in_f / 32 * KG::kBlockBytes;
    a.in_f = static_cast<int>(in_f);
    a.nb = static_cast<int>(in_f / 32);
    a.gcols = static_cast<int>((in_f + 127) / 128);
    // CTAs: kKoCtasPerSm per SM, split over the matrices in proportion to their rows.
    const int64_t total = static_cast<int64_t>(info.sms) * kKoCtasPerSm;
    int64_t rows_all = 0;
    for (int i = 0; i < nmat; ++i) rows_all += out_f[i];
    int64_t grid = 0, rmax = 0;
    int pass_rows = 0;  // the most rows any pass of any CTA holds
    for (int i = 0; i < nmat; ++i) {
        int64_t n = (total * out_f[i] + rows_all - 1) / rows_all;
        n = std::max<int64_t>(1, std::min<int64_t>(n, out_f[i]));
        a.mat_cta[i] = static_cast<int>(grid);
        a.mat_w[i] = w[i];
        a.mat_aux[i] = aux[i];
        a.mat_y[i] = y[i];
        a.mat_out_f[i] = out_f[i];
        grid += n;
        rmax = std::max(rmax, (out_f[i] + n - 1) / n);
        // this matrix's CTAs hold floor(out_f / n) or that + 1 rows; a pass then holds between
        // box_rows and pass_rows rows
        int lo = 1 << 30;
        for (int64_t r = out_f[i] / n; r <= (out_f[i] + n - 1) / n; ++r) {
            if (r < 1) continue;
            const int64_t np = (r + kPassRows - 1) / kPassRows;
            lo = std::min(lo, static_cast<int>(r / np));
            pass_rows = std::max(pass_rows, static_cast<int>((r + np - 1) / np));
        }
        a.box_rows[i] = lo;
    }
    a.mat_cta[nmat] = static_cast<int>(grid);
    // CTAs of 8 to 16 rows: fewer rows leave stages mostly activation and tiles mostly padding
    // (1024 x 5120, m = 4: 8.2 us against 4.4 us on the tile kernel, which uses fewer CTAs there)
    if (rmax > kPassRows || rmax < 8) return cudaErrorNotSupported;
    a.act_qs = static_cast<int>(align_up(static_cast<uint32_t>(pass_rows * KG::kSlot), 128));
    a.act_d = a.act_qs + static_cast<int>(align_up(static_cast<uint32_t>(M * kKoActRow), 128));
    a.stage = a.act_d + static_cast<int>(align_up(static_cast<uint32_t>(M * kKoDRow * 4), 128));
    a.act_bytes = M * kKoActRow + M * kKoDRow * 4;
    // Shared memory: barriers, the pass partials, the block-128 grid rows, the ring.
    const uint32_t part = align_up(static_cast<uint32_t>(kWarps * kPassRows * M * 4), 128);
    const int grid_rows = static_cast<int>(rmax / 128 + 2);
    const uint32_t gridb = KIND == kBlk ? align_up(static_cast<uint32_t>(grid_rows * a.gcols * 4), 128) : 0u;
    const uint32_t budget = std::min(static_cast<uint32_t>(info.smem_optin),
                                     static_cast<uint32_t>(info.smem_sm / kKoCtasPerSm - 1024));
    const uint32_t bars = align_up(static_cast<uint32_t>(2 * kKoMaxStages * 8), 128);
    if (bars + part + gridb + static_cast<uint32_t>(kKoMinStages * a.stage) > budget)
        return cudaErrorNotSupported;
    // At most 3 stages when the K sweep is short (<= 8 chunks): a ring holding most of a CTA's
    // rows is mostly requested before the preceding launch ends and competes with its tail
    // (measured on GB300, 5120 x 5120 m = 4: 7.07 us with 4 stages, 6.35 with 3; 5120 x 17408,
    // 17 chunks: no change).
    const int nch = (a.nb + kKoKw - 1) / kKoKw;
    const uint32_t cap = nch <= 8 ? 3u : static_cast<uint32_t>(kKoMaxStages);
    a.stages = static_cast<int>(std::min<uint32_t>(cap, (budget - bars - part - gridb) / a.stage));
    a.off_part = bars;
    a.off_grid = a.off_part + part;
    a.off_ring = a.off_grid + gridb;
    const uint32_t smem = a.off_ring + static_cast<uint32_t>(a.stages * a.stage);

    KoMaps maps = {};
    for (int i = 0; i < nmat; ++i)
        if (!ko_map(maps.w8[i], 1, w[i], out_f[i], a.row_bytes / 8, a.row_bytes, 8, KG::kSlot / 8,
                    a.box_rows[i], dev))
            return cudaErrorNotSupported;
    if (!ko_map(maps.qs, 2, qs, M, in_f / 8, in_f, 8, kKoActRow / 8, M, dev) ||
        !ko_map(maps.d, 3, d, M, in_f / 32, in_f / 8, 4, kKoDRow, M, dev))
        return cudaErrorNotSupported;

    auto kern = gemv_kouter_kernel<KIND, M, TILES>;
    const int ki = KIND == kBlk ? 1 : KIND == kQ80T ? 2 : 0;
    const uint64_t bit = 1ull << (M - 1);
    if (!(g_ko_attr[ki][dev].load(std::memory_order_acquire) & bit)) {
        const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   info.smem_optin);
        if (e != cudaSuccess) return e;
        g_ko_attr[ki][dev].fetch_or(bit, std::memory_order_acq_rel);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, a, maps);
}

template <int KIND>
cudaError_t launch_kouter_m(int m, int nmat, const uint8_t *const *w, const float *const *aux,
                            float *const *y, const int64_t *out_f, const int8_t *qs,
                            const float *d, int64_t in_f, int dev, const DeviceInfo &info,
                            cudaStream_t st) {
    switch (m) {
        // Q8_0 at m = 1 stays on dp4a (q80_kouter_applies)
        case 1:
            if constexpr (KIND == kQ80T) return cudaErrorNotSupported;
            else return launch_kouter<KIND, 1>(nmat, w, aux, y, out_f, qs, d, in_f, dev, info, st);
        case 2: return launch_kouter<KIND, 2>(nmat, w, aux, y, out_f, qs, d, in_f, dev, info, st);
        case 3: return launch_kouter<KIND, 3>(nmat, w, aux, y, out_f, qs, d, in_f, dev, info, st);
        case 4: return launch_kouter<KIND, 4>(nmat, w, aux, y, out_f, qs, d, in_f, dev, info, st);
        case 5: return launch_kouter<KIND, 5>(nmat, w, aux, y, out_f, qs, d, in_f, dev, info, st);
        case 6: return launch_kouter<KIND, 6>(nmat, w, aux, y, out_f, qs, d, in_f, dev, info, st);
        case 7: return launch_kouter<KIND, 7>(nmat, w, aux, y, out_f, qs, d, in_f, dev, info, st);
        default: return launch_kouter<KIND, 8>(nmat, w, aux, y, out_f, qs, d, in_f, dev, info, st);
    }
}

}  // namespace
}  // namespace memq
