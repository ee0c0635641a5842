/*
 * memq.h -- C ABI of libmemq: the m <= 8 quantized decode chain on GB300 (sm_103a).
 *
 * Two stages, each one asynchronous kernel launch on the caller's CUDA stream:
 *
 *   1. memq_rmsnorm_q8_1      f32 rows -> RMSNorm -> q8_1 activation (int8 qs + f32 d per 32)
 *   2. memq_gemv_e4m3         raw FP8 E4M3 weights, one per-tensor f32 scale   (1.0 B/weight)
 *      memq_gemv_e4m3_blk128  E4M3 weights + f32 block-128 scale grid          (1.0 B/weight)
 *      memq_gemv_q8_0         ggml block_q8_0 weights (f16 scale + 32 int8)     (1.0625 B/weight)
 *
 * Around them: the fused decode steps memq_rmsnorm_q8_1_gemv_* (stage 1 inside the GEMV
 * launch), the decode step for host-resident rows memq_decode_step_host, the grouped GEMVs memq_gemv_*_group, the silu(gate) * up -> q8_1 producer
 * memq_silu_mul_q8_1, the load-time repack of E4M3 weights into a Q8_0 slab,
 * memq_repack_e4m3[_blk128]_q8_0, and the t <= 8 MLA decode attention kernels memq_mla_absorb_q,
 * memq_mla_attn_gathered and memq_mla_decompress_v.
 *
 * The operations are the ones defined on the memra-engine 0.125.0 source pages:
 * q8_fuse_gate.rs (module doc: the `rms_norm` -> `quantize_q8_1` chain and the fused
 * `rms_norm_zq8_f32` producer), gemv_e4m3_bench.rs (module doc, "THE COMPARISON" and "THE
 * BLOCK-128 ARM", and the container generators `synth_e4m3`, `synth_blk_grid`, `synth_q8_0`)
 * and mla_decode_arm_gate.rs (module doc and `main`: the MLA kernels and their split twins).
 *
 * Conventions for every entry point:
 *   - Pointers named "device" must be device-accessible memory of the current CUDA device
 *     (cudaMalloc / torch CUDA tensors).  The caller owns every buffer; the library never
 *     allocates, frees or keeps a pointer after the call returns.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Calls only enqueue work;
 *     they never synchronize (except memq_decode_step_host and memq_device_fault, which wait
 *     for the stream).  Results are ready when the stream reaches the launch.  Launches
 *     may begin before the preceding work on the stream has finished (programmatic dependent
 *     launch), but read nothing the stream wrote before that work is complete; callers see
 *     plain stream order.
 *   - Arguments are validated on the host before anything is launched; on any error the call
 *     returns a nonzero memq_status and writes nothing.  A launch failure returns
 *     MEMQ_ERR_LAUNCH.  Device-side waits are bounded: if one ever expires, the kernel records
 *     a fault bit that memq_device_fault() reports, and returns without hanging.
 *   - Outputs must not alias inputs.
 *   - Row-major layouts throughout; "m" is the number of activation rows (decode tokens),
 *     1 <= m <= 8.
 */
#ifndef MEMQ_H
#define MEMQ_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum memq_status {
    MEMQ_OK = 0,
    MEMQ_ERR_NULL = 1,    /* a required pointer is NULL */
    MEMQ_ERR_SHAPE = 2,   /* a size is out of range or not a multiple of 32 */
    MEMQ_ERR_ALIGN = 3,   /* a pointer breaks its documented alignment */
    MEMQ_ERR_M_RANGE = 4, /* m outside [1, 8] */
    MEMQ_ERR_LAUNCH = 5,  /* the CUDA launch (or a device query before it) failed */
    MEMQ_ERR_DEVICE = 6   /* memq_device_fault() could not read the device fault word */
} memq_status;

/* Maximum activation rows per GEMV call. */
#define MEMQ_MAX_M 8
/* Largest row width accepted by memq_rmsnorm_q8_1. */
#define MEMQ_MAX_NCOLS 32768

/*
 * memq_rmsnorm_q8_1 -- fused RMSNorm -> q8_1 producer.
 * Defined by q8_fuse_gate.rs (module doc; `run_shape` compares the two-launch `rms_norm` +
 * `quantize_q8_1` chain with the fused `rms_norm_zq8_f32`).  For each row r < rows:
 *     z[r][i] = (x[r][i] * rr) * w[i],   rr = 1 / sqrt(sum_i x[r][i]^2 / ncols + eps)
 * then for each 32-element block b of the row:
 *     d[r][b]  = max_{i in b} |z[r][i]| / 127              (f32)
 *     qs[r][i] = round(z[r][i] / d[r][b]) (ties away from zero), or 0 when d[r][b] == 0
 * so |qs| <= 127 and the block's largest |z| maps to +-127.
 *   x   device, f32 [rows][ncols], 16-byte aligned
 *   w   device, f32 [ncols], 16-byte aligned (one weight vector shared by all rows)
 *   z   device, f32 [rows][ncols], 16-byte aligned, or NULL to skip writing z
 *   qs  device, int8 [rows][ncols], 4-byte aligned
 *   d   device, f32 [rows][ncols/32]
 *   ncols: 32 <= ncols <= MEMQ_MAX_NCOLS, ncols % 32 == 0;  eps >= 0;  rows >= 0, where
 *   rows == 0 is a no-op that accepts NULL pointers.
 * Numerics: the row statistic is accumulated in f32 per thread and f64 across threads, r uses
 * IEEE f32 divide and square root; z uses f32 products; qs uses an IEEE f32 division z/d.
 */
int memq_rmsnorm_q8_1(const float *x, const float *w, float *z, int8_t *qs, float *d,
                      int64_t ncols, int64_t rows, float eps, void *stream);

/*
 * memq_gemv_e4m3 -- y = s * W_e4m3 . X_q8_1 (per-tensor scale).
 * Defined by gemv_e4m3_bench.rs (module doc, "THE COMPARISON", arm E4M3: raw checkpoint E4M3
 * bytes as the weight stream, row_bytes == in_f; `synth_e4m3`).  For j < m, r < out_f:
 *     y[j][r] = s * sum_i e4m3(w[r][i]) * d[j][i/32] * qs[j][i]
 *   w        device, uint8 E4M3 codes [out_f][in_f] (0x7F/0xFF are NaN and propagate)
 *   w_scale  device, one f32 (the per-tensor scale s); read by the kernel, so it may change
 *            between graph replays
 *   qs, d    device, the q8_1 activation: int8 [m][in_f] and f32 [m][in_f/32]
 *   y        device, f32 [m][out_f]
 *   in_f % 32 == 0, 32 <= in_f <= 2^24; 1 <= m <= MEMQ_MAX_M; out_f >= 0, where out_f == 0
 *   is a no-op that accepts NULL pointers.
 * The fast path wants w and qs 16-byte aligned; other alignments take a slower generic kernel
 * with the same results contract.
 * Numerics (all three containers): a 32-block's product of weights and activation codes is
 * formed on the tensor cores from exactly converted operands (E4M3 -> f16 and int8 -> f16 are
 * exact, products exact in f32, f32 accumulation), or for Q8_0 at small m as an exact int32
 * dp4a dot product; it is scaled by d (and the grid entry / f16 block scale) and summed in f32
 * in a fixed order per (row, token).  E4M3 and block-128: on the fast path that order does not
 * depend on m, on how the launch splits the rows, or on which of the library's kernels serves
 * the call, so a row's outputs are bit-identical whether it is computed alone, in an m-batch,
 * or in a group.
 * Q8_0: the same holds within each of its two paths (dp4a at m = 1; tensor cores from m = 2
 * when each CTA gets 8 to 16 rows of a wide activation, from m = 4 to 6 on other shapes); across
 * them the block sums are the same exact integers added in another order, and results agree
 * within the GEMV tolerance.
 */
int memq_gemv_e4m3(const uint8_t *w, const float *w_scale, const int8_t *qs, const float *d,
                   float *y, int64_t out_f, int64_t in_f, int m, void *stream);

/*
 * memq_gemv_e4m3_blk128 -- y = (G (x) W_e4m3) . X_q8_1 with a block-128 scale grid.
 * Defined by gemv_e4m3_bench.rs (module doc, "THE BLOCK-128 ARM": the raw E4M3 plane plus a
 * resident f32 [ceil(out_f/128), ceil(in_f/128)] grid in F8BlockGrid order; `synth_blk_grid`):
 *     y[j][r] = sum_i grid[r/128][i/128] * e4m3(w[r][i]) * d[j][i/32] * qs[j][i]
 *   grid  device, f32 [ceil(out_f/128)][ceil(in_f/128)] row-major; a partial edge tile uses
 *         its own entry.  Other arguments as memq_gemv_e4m3.
 */
int memq_gemv_e4m3_blk128(const uint8_t *w, const float *grid, const int8_t *qs, const float *d,
                          float *y, int64_t out_f, int64_t in_f, int m, void *stream);

/*
 * memq_gemv_q8_0 -- y = W_q8_0 . X_q8_1.
 * Defined by gemv_e4m3_bench.rs (module doc, arm Q8_0, row_bytes = in_f/32*34; `synth_q8_0`:
 * ggml block_q8_0 = a little-endian f16 scale then 32 int8 weights, 34 bytes per 32 weights):
 *     y[j][r] = sum_i f16(blk(r, i/32).d) * blk(r, i/32).qs[i%32] * d[j][i/32] * qs[j][i]
 *   w   device, out_f rows of in_f/32 blocks of 34 bytes, rows packed back to back
 *   Other arguments as memq_gemv_e4m3.  The fast path wants w and qs 16-byte aligned and
 *   in_f % 256 == 0 (so every row starts 16-byte aligned); anything else takes the generic
 *   kernel.  The full int8 range (including -128) is accepted in both operands.
 */
int memq_gemv_q8_0(const void *w, const int8_t *qs, const float *d, float *y, int64_t out_f,
                   int64_t in_f, int m, void *stream);

/*
 * Fused decode step: memq_rmsnorm_q8_1 on the m rows of x followed by the GEMV on the resulting
 * q8_1 activation, as one launch.  Every CTA of the GEMV quantizes x itself (same arithmetic
 * as memq_rmsnorm_q8_1) while its weight stream is already in flight, so the producer's latency
 * leaves the critical path (the "two launches -> one" of q8_fuse_gate.rs, module doc, carried
 * one stage further into the GEMV of gemv_e4m3_bench.rs).
 *   x    device, f32 [m][in_f], 16-byte aligned;  wn  device, f32 [in_f], 16-byte aligned
 *   eps  >= 0
 *   qs, d  device outputs: the q8_1 activation (int8 [m][in_f], f32 [m][in_f/32]); required
 *   z      device output f32 [m][in_f] (16-byte aligned) or NULL
 *   y      device output f32 [m][out_f]
 *   Weight arguments as the matching GEMV.  in_f <= MEMQ_MAX_NCOLS.  When the single-launch
 *   plan does not apply (alignment, shared memory) the call makes the same two launches as
 *   memq_rmsnorm_q8_1 + memq_gemv_*, with the same outputs.  out_f == 0 only produces qs / d / z.
 */
int memq_rmsnorm_q8_1_gemv_e4m3(const float *x, const float *wn, float eps, const uint8_t *w,
                                const float *w_scale, int8_t *qs, float *d, float *z, float *y,
                                int64_t out_f, int64_t in_f, int m, void *stream);
int memq_rmsnorm_q8_1_gemv_e4m3_blk128(const float *x, const float *wn, float eps,
                                       const uint8_t *w, const float *grid, int8_t *qs, float *d,
                                       float *z, float *y, int64_t out_f, int64_t in_f, int m,
                                       void *stream);
int memq_rmsnorm_q8_1_gemv_q8_0(const float *x, const float *wn, float eps, const void *w,
                                int8_t *qs, float *d, float *z, float *y, int64_t out_f,
                                int64_t in_f, int m, void *stream);

/* The weight containers of the GEMVs, for the entry points that take one as an argument. */
typedef enum memq_container {
    MEMQ_CONTAINER_E4M3 = 0,        /* memq_gemv_e4m3: aux = the per-tensor w_scale */
    MEMQ_CONTAINER_E4M3_BLK128 = 1, /* memq_gemv_e4m3_blk128: aux = the block-128 grid */
    MEMQ_CONTAINER_Q8_0 = 2         /* memq_gemv_q8_0: aux is not read (may be NULL) */
} memq_container;

/*
 * memq_decode_step_host -- one decode step for a caller whose activation rows and outputs are
 * in HOST memory (a host-side sampler or scheduler that hands over one token's hidden rows and
 * reads the projection back): copies x_host to x_dev, runs memq_rmsnorm_q8_1_gemv_<container>
 * on the device buffers, copies y_dev to y_host, and waits for the stream.  The operation is the
 * fused step's (q8_fuse_gate.rs, module doc; the GEMV of gemv_e4m3_bench.rs, "THE
 * COMPARISON"); the copies and the wait are the host path around it, in one native call.
 *   container  a memq_container; any other value returns MEMQ_ERR_SHAPE
 *   x_host     host, f32 [m][in_f] (page-locked memory gives the asynchronous, fastest copy;
 *              pageable memory works)
 *   x_dev      device, f32 [m][in_f], 16-byte aligned: the caller's device buffer for the copy
 *   y_dev      device, f32 [m][out_f]: the caller's device buffer for the result
 *   y_host     host, f32 [m][out_f]; may be NULL when out_f == 0
 *   wn, eps, w, aux, qs, d, z, out_f, in_f, m: as memq_rmsnorm_q8_1_gemv_<container> (x = x_dev,
 *              y = y_dev; aux = w_scale or grid, not read for Q8_0), with the same checks
 * Unlike the other entry points this call WAITS: it returns once the stream has finished
 * everything enqueued on it up to and including the copy to y_host, so y_host holds the
 * result, bit-identical to memq_rmsnorm_q8_1_gemv_<container> on x_dev.  Arguments are
 * checked before anything is enqueued (an error writes nothing); a failing copy, launch or
 * wait returns MEMQ_ERR_LAUNCH after the stream has been waited for, so no copy still touches
 * the host buffers.  Not for stream capture (it waits).
 */
int memq_decode_step_host(int container, const float *x_host, float *x_dev, const float *wn,
                          float eps, const void *w, const float *aux, int8_t *qs, float *d,
                          float *z, float *y_dev, float *y_host, int64_t out_f, int64_t in_f,
                          int m, void *stream);

/*
 * memq_gemv_*_group -- up to 4 GEMVs of the same container that share one activation (qs, d,
 * in_f, m), e.g. the gate and up projections, or q and k/v, in ONE launch: the matrices' rows
 * are split over the CTAs in proportion; every output equals the corresponding single
 * memq_gemv_* call bit for bit.  w, w_scale / grid, y and out_f are HOST arrays of `count`
 * entries (device pointers / row counts), read during the call only.  Per matrix the
 * single-call rules apply; every out_f must be >= 1.  If any matrix is off the fast path (an
 * unaligned pointer, Q8_0 rows not 16-byte aligned) the call falls back to one launch per
 * matrix.  It serves the gate and up projections, which read the same activation (q8_fuse_gate.rs,
 * `main`, lists that site among those not yet fused).
 * Errors: MEMQ_ERR_SHAPE (count outside [1, 4], an empty matrix, a bad size), MEMQ_ERR_NULL,
 * MEMQ_ERR_ALIGN, MEMQ_ERR_M_RANGE, MEMQ_ERR_LAUNCH.
 */
int memq_gemv_e4m3_group(int count, const uint8_t *const *w, const float *const *w_scale,
                         float *const *y, const int64_t *out_f, const int8_t *qs, const float *d,
                         int64_t in_f, int m, void *stream);
int memq_gemv_e4m3_blk128_group(int count, const uint8_t *const *w, const float *const *grid,
                                float *const *y, const int64_t *out_f, const int8_t *qs,
                                const float *d, int64_t in_f, int m, void *stream);
int memq_gemv_q8_0_group(int count, const void *const *w, float *const *y, const int64_t *out_f,
                         const int8_t *qs, const float *d, int64_t in_f, int m, void *stream);

/*
 * memq_silu_mul_q8_1 -- the silu(gate) * up -> q8_1 activation producer.
 * Named on q8_fuse_gate.rs (`main`: the expert-ff width 1536, the "silu/gate*up -> q8_1"
 * fusion site).  For each row r < rows and column i < ncols:
 *     z[r][i] = silu(gate[r][i]) * up[r][i],   silu(g) = g / (1 + exp(-g))   (f32)
 * then per 32-element block exactly as memq_rmsnorm_q8_1: d = amax/127, qs = round(z/d).
 *   gate, up  device f32 [rows][ncols], 16-byte aligned (typically the two GEMV outputs)
 *   z         device f32 [rows][ncols], 16-byte aligned, or NULL to skip writing z
 *   qs        device int8 [rows][ncols], 4-byte aligned;  d  device f32 [rows][ncols/32]
 *   ncols     multiple of 32, 32 <= ncols <= 2^30;  rows >= 0 (0 = no-op)
 * Errors: MEMQ_ERR_SHAPE, MEMQ_ERR_NULL, MEMQ_ERR_ALIGN, MEMQ_ERR_LAUNCH.
 */
int memq_silu_mul_q8_1(const float *gate, const float *up, float *z, int8_t *qs, float *d,
                       int64_t ncols, int64_t rows, void *stream);

/*
 * memq_repack_e4m3_q8_0 / memq_repack_e4m3_blk128_q8_0 -- load-time conversion of E4M3
 * weights into ggml block_q8_0 records (gemv_e4m3_bench.rs, module doc "QUESTION": the
 * shipping path converts FP8 weights into Q8_0 once, at load time, ARM B').  For each row r and 32-block
 * b of the row, with W[i] = e4m3(w[r][i]) * s in f32 (s = *w_scale, or grid[r/128][i/128]):
 *     d = max_{i in b} |W[i]| / 127  (f32),  stored as f16 (round to nearest even)
 *     qs[i] = round(W[i] / d)  (f32 quotient, ties away from zero; 0 when d == 0)
 * so that out can be passed to memq_gemv_q8_0 in place of (w, scale).  The f32 operations are
 * IEEE (one rounding each), so the slab is bit-reproducible.
 *   w        device E4M3 bytes [out_f][in_f], 16-byte aligned
 *   w_scale  device f32, one value;  grid  device f32 [ceil(out_f/128)][ceil(in_f/128)]
 *   out      device bytes [out_f][in_f/32 * 34], 16-byte aligned (the slab is contiguous)
 *   in_f     multiple of 32;  out_f >= 0 (0 = no-op)
 * NaN weight codes (0x7F / 0xFF) are outside the contract.  Not for the decode loop: it reads
 * 1 byte and writes 1.0625 bytes per weight, once at load.
 * Errors: MEMQ_ERR_SHAPE, MEMQ_ERR_NULL, MEMQ_ERR_ALIGN, MEMQ_ERR_LAUNCH.
 */
int memq_repack_e4m3_q8_0(const uint8_t *w, const float *w_scale, void *out, int64_t out_f,
                          int64_t in_f, void *stream);
int memq_repack_e4m3_blk128_q8_0(const uint8_t *w, const float *grid, void *out, int64_t out_f,
                                 int64_t in_f, void *stream);

/*
 * The t <= 8 MLA decode attention kernels of mla_decode_arm_gate.rs (module doc and `main`: 64
 * heads, kv_rank 512, d_nope = d_v = 256, d_rope 0, a top-k gather of 2048 rows from a pool of
 * cached latent rows, t_q in {1, 2, 4, 8}).  All f32, row-major, with t in [1, 8] query rows
 * (MEMQ_ERR_M_RANGE otherwise).  `split` is launch geometry only (0 = the library's choice):
 * for absorb_q / decompress_v, s >= 1 CTAs share the rows of one head; for attn_gathered,
 * s in {1, 2, 4, 8} puts 8 / s heads in each CTA.  For every split the outputs are
 * bit-identical (each output element is produced by the same floating-point operations in the
 * same order), which is the "split twin" property the page gates on.
 *
 * memq_mla_absorb_q:     out[t][h][r] = sum_{d < d_nope} q_nope[t][h][d] * wk_b[h][r][d]
 *   q_nope device [t][nh][d_nope], 16-byte aligned;  wk_b device [nh][kv_rank][d_nope],
 *   16-byte aligned;  out device [t][nh][kv_rank], 4-byte aligned.
 * memq_mla_decompress_v: out[t][h][v] = sum_{r < kv_rank} o_lat[t][h][r] * wv_b[h][v][r]
 *   o_lat device [t][nh][kv_rank], 16-byte aligned;  wv_b device [nh][d_v][kv_rank], 16-byte
 *   aligned;  out device [t][nh][d_v], 4-byte aligned.
 * The reduced dimension (d_nope, resp. kv_rank) must be 128, 256, 512 or 1024; the other >= 1;
 * 1 <= nh <= 65536.
 *
 * memq_mla_attn_gathered: for each query row t and head h, over the gathered slots j < n_slots
 * with c_j = cache[idx[t][j]] (kv_rank latent floats, then d_rope rope floats):
 *     s_j = scale * (q_lat[t][h] . c_j[:kv_rank] + q_pe[t][h] . c_j[kv_rank:])
 *     out[t][h][:] = sum_j softmax(s)_j * c_j[:kv_rank]
 *   q_lat device [t][nh][kv_rank];  q_pe device [t][nh][d_rope] (may be NULL when d_rope == 0)
 *   cache device [pool][kv_rank + d_rope], 16-byte aligned;  idx device int32 [t][n_slots],
 *   each in [0, pool) (not checked: an index outside the pool is outside the contract)
 *   out device [t][nh][kv_rank];  q_lat, q_pe, idx, out 4-byte aligned
 *   kv_rank in {128, 256, 512, 1024};  0 <= d_rope <= 128;  n_slots >= 1;  scale finite.
 * Numerics of attn_gathered: an online softmax over 8 fixed slot ranges of 16-slot chunks,
 * merged in range order.  With t >= 2, d_rope == 0 and kv_rank <= 512 (the page geometry) the
 * scores and outputs are tensor-core products in three TF32 terms (hi = the value truncated to
 * TF32, lo = the exact remainder at TF32 precision; per-product error below 3 * 2^-20 of
 * |x y|), otherwise f32 FMAs.  The choice depends on (t, kv_rank, d_rope) only, so the split
 * twins run the same arithmetic.
 * Errors: MEMQ_ERR_SHAPE, MEMQ_ERR_NULL, MEMQ_ERR_ALIGN, MEMQ_ERR_M_RANGE, MEMQ_ERR_LAUNCH.
 */
int memq_mla_absorb_q(const float *q_nope, const float *wk_b, float *out, int t, int nh,
                      int d_nope, int kv_rank, int split, void *stream);
int memq_mla_decompress_v(const float *o_lat, const float *wv_b, float *out, int t, int nh,
                          int d_v, int kv_rank, int split, void *stream);
int memq_mla_attn_gathered(const float *q_lat, const float *q_pe, const float *cache,
                           const int32_t *idx, float *out, int nh, int kv_rank, int d_rope, int t,
                           int n_slots, float scale, int split, void *stream);

/* Human-readable name of a memq_status value (static storage; never NULL). */
const char *memq_status_string(int status);

/*
 * memq_device_fault -- read and clear the current device's fault word.
 * Synchronizes `stream`, then stores the word in *fault_out (0 = no fault) and resets it.
 * Bit 0: a GEMV consumer's bounded wait on a shared-memory barrier expired; bit 1: the GEMV
 * producer's.  A CTA that gave up stores no output for the tile it was on or any later one
 * (rows it finished before may already be stored), waits (bounded) for its copies in flight
 * and returns; the call's outputs are invalid.  Bit 2: an
 * memq_mla_attn_gathered CTA's bounded wait for its gathered rows expired; bit 3: the same in
 * memq_mla_absorb_q / memq_mla_decompress_v.  That CTA stopped streaming, waited (bounded) for
 * its copies in flight and returned; the call's outputs are invalid.
 * Returns MEMQ_ERR_NULL for a NULL fault_out, MEMQ_ERR_DEVICE if the copy fails.
 */
int memq_device_fault(void *stream, uint32_t *fault_out);

/* ABI version of this header: (major << 16) | minor. */
int memq_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MEMQ_H */
