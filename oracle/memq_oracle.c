/*
 * memq_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, obviously correct CPU oracle of the m <= 8 quantized decode chain, written in
 * f64 from the definitions on the source pages of memra-engine 0.125.0:
 *   - q8_fuse_gate.rs, module doc and `run_shape`: the fused RMSNorm -> q8_1 producer
 *     (z = x * rsqrt(mean(x^2) + eps) * w, then per 32-element block d = amax/127 and
 *     qs = round(z/d), emitted as f32 z, int8 qs and an f32 per-block scale d);
 *   - gemv_e4m3_bench.rs, module doc ("THE COMPARISON", "THE BLOCK-128 ARM") and the
 *     generators `synth_e4m3`, `synth_blk_grid`, `synth_q8_0`: the m=1..8 GEMV of a q8_1
 *     activation against three weight containers (raw E4M3 + one per-tensor scale, E4M3 + an
 *     f32 [ceil(out_f/128), ceil(in_f/128)] block-128 scale grid, ggml block_q8_0).
 *
 * Only the tests, the package's smoke check and the bench's CPU-baseline leg may load this
 * library.  It shares no code, header or table with the CUDA path and includes nothing from it.
 * Every sum here is a straight loop in the definition's order; there is no blocking, fusion or
 * reordering.  No fast-math: build with plain -O2.
 *
 * Parity pins (what each function is checked against, by the CPU tests):
 *   memq_oracle_e4m3     closed-form spot values of the OCP E4M3 format + all 256 codes vs the
 *                        float8_e4m3fn decode of a tensor library (NaN exactly at 0x7F/0xFF)
 *   memq_oracle_f16      all 65536 codes vs numpy.float16
 *   memq_oracle_rmsnorm  closed forms (constant rows) + a library rms_norm in f64
 *   memq_oracle_quantize closed forms, rounding-tie cases, invariants |qs|<=127, amax -> +-127,
 *                        |z - d*qs| <= d/2
 *   memq_oracle_gemv_*   library matmul of independently dequantized operands on small
 *                        shapes, one-hot activations, sign-flip / zero / constant-grid
 *                        identities, and the exact cross-container identity
 *   memq_oracle_silu_mul the identity silu(x) - silu(-x) = x, silu(0) = 0, a library logistic
 *                        function, and the q8_1 quantizer's own pins on its output
 *   memq_oracle_f16_bits all representable binade boundaries and random f32 values vs the
 *                        float16 conversion of numpy (round to nearest even, subnormals)
 *   memq_oracle_repack_q8_0  brute-force nearest code over all 255 values, amax -> +-127,
 *                        constant / zero blocks, dequantization error <= d/2, and the GEMV of
 *                        the repacked slab against the GEMV of the E4M3 source within the
 *                        quantization bound
 *
 *   memq_oracle_mla_*    library einsum / softmax of the same operands; closed forms
 *                        (attention over identical rows returns the row, a one-slot gather
 *                        returns that slot, scale 0 gives the mean of the rows); the rope term
 *                        equals the same problem on concatenated queries and rows; a zeroed
 *                        head's weights give that head a zero output
 *
 * Also from the pages: q8_fuse_gate.rs, `main` -- the silu(gate)*up -> q8_1 activation producer
 * named for the 1536-wide expert site; gemv_e4m3_bench.rs, module doc "QUESTION" -- the ship
 * path converts FP8 weights into a Q8_0 copy once, at load time ("ARM B'"); mla_decode_arm_gate.rs,
 * module doc and `main` -- the t <= 8 MLA decode attention kernels absorb_q, decompress_v and
 * attn_gathered.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>

/* ---------------------------------------------------------------------------------------------
 * Format decoders.
 * ------------------------------------------------------------------------------------------- */

/* FP8 E4M3 (OCP "E4M3FN"): 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits, no infinities;
 * exponent 15 with mantissa 7 is NaN -- gemv_e4m3_bench.rs, `synth_e4m3` doc: "Magnitude 0x7F is
 * the e4m3 NaN code". */
double memq_oracle_e4m3(uint8_t b)
{
    int sign = (b >> 7) & 1;
    int expo = (b >> 3) & 15;
    int mant = b & 7;
    double mag;
    if (expo == 15 && mant == 7)
        return NAN;
    if (expo == 0)
        mag = ldexp((double)mant, -9);                 /* subnormal: mant/8 * 2^(1-7) */
    else
        mag = ldexp(1.0 + (double)mant / 8.0, expo - 7);
    return sign ? -mag : mag;
}

/* IEEE-754 binary16, the block_q8_0 scale (gemv_e4m3_bench.rs, `synth_q8_0`: "d = f16 0x1400 =
 * 2^-10"; two little-endian bytes at the start of each 34-byte block). */
double memq_oracle_f16(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int expo = (h >> 10) & 31;
    int frac = h & 1023;
    double mag;
    if (expo == 31)
        mag = frac ? NAN : INFINITY;
    else if (expo == 0)
        mag = ldexp((double)frac, -24);
    else
        mag = ldexp(1.0 + (double)frac / 1024.0, expo - 15);
    return sign ? -mag : mag;
}

void memq_oracle_e4m3_table(double *out256)
{
    for (int b = 0; b < 256; ++b)
        out256[b] = memq_oracle_e4m3((uint8_t)b);
}

void memq_oracle_f16_decode(const uint16_t *h, int64_t n, double *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = memq_oracle_f16(h[i]);
}

/* ---------------------------------------------------------------------------------------------
 * Stage 1: RMSNorm, then q8_1 quantization (q8_fuse_gate.rs, module doc: `rms_norm` then
 * `quantize_q8_1`, fused as `rms_norm_zq8_f32`).
 * ------------------------------------------------------------------------------------------- */

/* z[r][i] = x[r][i] * r_row * w[i],  r_row = 1 / sqrt(sum_i x[r][i]^2 / ncols + eps).
 * x: [rows][ncols] f32, w: [ncols] f32, z: [rows][ncols] f64.  eps arrives as the f32 the
 * callers use (1e-6f in `run_shape`) and is promoted to f64. */
void memq_oracle_rmsnorm(const float *x, const float *w, int64_t rows, int64_t ncols, float eps,
                         double *z)
{
    for (int64_t r = 0; r < rows; ++r) {
        const float *xr = x + r * ncols;
        double ss = 0.0;
        for (int64_t i = 0; i < ncols; ++i)
            ss += (double)xr[i] * (double)xr[i];
        double rr = 1.0 / sqrt(ss / (double)ncols + (double)eps);
        for (int64_t i = 0; i < ncols; ++i)
            z[r * ncols + i] = (double)xr[i] * rr * (double)w[i];
    }
}

/* Per 32-element block of each row: amax = max |z|, d = amax / 127 stored as an f32 (the q8_1
 * scale is an f32 per block), qs = round(z / d) with ties away from zero, and qs = 0 when d = 0
 * (the `id = 1/d` branch named in q8_fuse_gate.rs, `Xorshift64::next_f32` doc).
 * z: [rows][ncols] f64 -> d: [rows][ncols/32] f32, qs: [rows][ncols] int8,
 * ratio: [rows][ncols] f64 = z / d (the exact quotient whose rounding gives qs), may be NULL. */
void memq_oracle_quantize_q8_1(const double *z, int64_t rows, int64_t ncols, float *d,
                               int8_t *qs, double *ratio)
{
    int64_t nb = ncols / 32;
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t b = 0; b < nb; ++b) {
            const double *zb = z + r * ncols + b * 32;
            double amax = 0.0;
            for (int k = 0; k < 32; ++k)
                if (fabs(zb[k]) > amax)
                    amax = fabs(zb[k]);
            float dd = (float)(amax / 127.0);
            d[r * nb + b] = dd;
            for (int k = 0; k < 32; ++k) {
                int64_t i = r * ncols + b * 32 + k;
                double t = (dd != 0.0f) ? zb[k] / (double)dd : 0.0;
                qs[i] = (int8_t)round(t);
                if (ratio)
                    ratio[i] = t;
            }
        }
    }
}

/* ---------------------------------------------------------------------------------------------
 * Stage 2: y[j][r] = sum_i W(r, i) * X(j, i), with X(j, i) = d[j][i/32] * qs[j][i] the
 * dequantized q8_1 activation row j (j < m) and W the dequantized weight
 * (gemv_e4m3_bench.rs, "THE COMPARISON" and "THE BLOCK-128 ARM").
 *
 * Every GEMV takes an optional list of output rows (row_idx, nrows; NULL = all out_f rows in
 * order) so that full-size problems can be checked on sampled rows.  Outputs are
 * y[j][t] and sabs[j][t] = sum_i |W(r,i) X(j,i)| for t < nrows, r = row_idx[t].
 * ------------------------------------------------------------------------------------------- */

static double act(const int8_t *qs, const float *d, int64_t in_f, int64_t j, int64_t i)
{
    return (double)d[j * (in_f / 32) + i / 32] * (double)qs[j * in_f + i];
}

/* Raw E4M3 plane [out_f][in_f] (row stride in_f, 1 byte per weight), one per-tensor scale:
 * W(r, i) = scale * e4m3(w[r][i]). */
void memq_oracle_gemv_e4m3(const uint8_t *w, float scale, const int8_t *qs, const float *d,
                           int64_t out_f, int64_t in_f, int m, const int64_t *row_idx,
                           int64_t nrows, double *y, double *sabs)
{
    double tab[256];
    memq_oracle_e4m3_table(tab);
    if (!row_idx)
        nrows = out_f;
    for (int64_t t = 0; t < nrows; ++t) {
        int64_t r = row_idx ? row_idx[t] : t;
        for (int j = 0; j < m; ++j) {
            double acc = 0.0, s = 0.0;
            for (int64_t i = 0; i < in_f; ++i) {
                double p = (double)scale * tab[w[r * in_f + i]] * act(qs, d, in_f, j, i);
                acc += p;
                s += fabs(p);
            }
            y[j * nrows + t] = acc;
            sabs[j * nrows + t] = s;
        }
    }
}

/* E4M3 plane plus the block-128 scale grid, f32 [ceil(out_f/128)][ceil(in_f/128)] row-major
 * (the `F8BlockGrid` order): W(r, i) = grid[r/128][i/128] * e4m3(w[r][i]); a partial edge tile
 * keeps its own grid entry. */
void memq_oracle_gemv_e4m3_blk128(const uint8_t *w, const float *grid, const int8_t *qs,
                                  const float *d, int64_t out_f, int64_t in_f, int m,
                                  const int64_t *row_idx, int64_t nrows, double *y, double *sabs)
{
    double tab[256];
    int64_t gcols = (in_f + 127) / 128;
    memq_oracle_e4m3_table(tab);
    if (!row_idx)
        nrows = out_f;
    for (int64_t t = 0; t < nrows; ++t) {
        int64_t r = row_idx ? row_idx[t] : t;
        for (int j = 0; j < m; ++j) {
            double acc = 0.0, s = 0.0;
            for (int64_t i = 0; i < in_f; ++i) {
                double g = (double)grid[(r / 128) * gcols + i / 128];
                double p = g * tab[w[r * in_f + i]] * act(qs, d, in_f, j, i);
                acc += p;
                s += fabs(p);
            }
            y[j * nrows + t] = acc;
            sabs[j * nrows + t] = s;
        }
    }
}

/* ggml block_q8_0 rows: in_f/32 blocks of 34 bytes per row, each an f16 scale (little-endian,
 * bytes 0-1) followed by 32 int8 weights: W(r, i) = f16(block.d) * block.qs[i % 32]. */
void memq_oracle_gemv_q8_0(const uint8_t *w, const int8_t *qs, const float *d, int64_t out_f,
                           int64_t in_f, int m, const int64_t *row_idx, int64_t nrows, double *y,
                           double *sabs)
{
    int64_t nb = in_f / 32;
    if (!row_idx)
        nrows = out_f;
    for (int64_t t = 0; t < nrows; ++t) {
        int64_t r = row_idx ? row_idx[t] : t;
        for (int j = 0; j < m; ++j) {
            double acc = 0.0, s = 0.0;
            for (int64_t i = 0; i < in_f; ++i) {
                const uint8_t *blk = w + (r * nb + i / 32) * 34;
                double dw = memq_oracle_f16((uint16_t)(blk[0] | (blk[1] << 8)));
                double p = dw * (double)(int8_t)blk[2 + i % 32] * act(qs, d, in_f, j, i);
                acc += p;
                s += fabs(p);
            }
            y[j * nrows + t] = acc;
            sabs[j * nrows + t] = s;
        }
    }
}

/* ---------------------------------------------------------------------------------------------
 * The silu(gate) * up -> q8_1 activation producer (q8_fuse_gate.rs, `main`: the expert-ff site,
 * "silu/gate*up -> q8_1").  z = silu(g) * u with silu(g) = g / (1 + exp(-g)), in f64; the q8_1
 * step is memq_oracle_quantize_q8_1 on z.  g, u: [n] f32 -> z: [n] f64.
 * ------------------------------------------------------------------------------------------- */
void memq_oracle_silu_mul(const float *g, const float *u, int64_t n, double *z)
{
    for (int64_t i = 0; i < n; ++i) {
        double gi = (double)g[i];
        z[i] = gi / (1.0 + exp(-gi)) * (double)u[i];
    }
}

/* ---------------------------------------------------------------------------------------------
 * Load-time repack of E4M3 weights into a Q8_0 slab (gemv_e4m3_bench.rs, module doc
 * "QUESTION": the shipping path converts FP8 weights into Q8_0 once, at load time).
 *
 * The pages fix the two formats but not the arithmetic of the conversion; the reading taken is
 * the q8_1 rule applied to the dequantized weights, per 32-block of a row:
 *   W[k] = e4m3(w[k]) * s  (s = the per-tensor scale, or grid[r/128][i/128]),
 *   amax = max |W|,  d = amax / 127,  stored as f16 (round to nearest, ties to even),
 *   qs[k] = round(W[k] / d) (ties away from zero), qs = 0 when d = 0.
 * Floating point decides the integer codes here, so this function takes those decisions in the
 * precision of the GPU kernel, IEEE f32 (one rounded product, one rounded quotient each); with
 * -ffp-contract=off the result is the exact f32 evaluation of these formulas.
 * ------------------------------------------------------------------------------------------- */

/* f64 -> IEEE binary16 bits, round to nearest, ties to even; subnormals; overflow -> inf. */
uint16_t memq_oracle_f16_bits(double v)
{
    uint16_t sign = 0;
    if (v != v)
        return 0x7E00;
    if (v < 0 || (v == 0 && 1.0 / v < 0)) {
        sign = 0x8000;
        v = -v;
    }
    if (v == 0)
        return sign;
    /* exponent of the f16 quantum: 2^(e - 10) for a normal value in [2^e, 2^(e+1)), e >= -14;
     * subnormals share the quantum 2^-24 */
    int e = 0;
    double m = frexp(v, &e); /* v = m * 2^e, m in [0.5, 1) */
    e -= 1;                  /* v in [2^e, 2^(e+1)) */
    if (e < -14)
        e = -14;
    double q = ldexp(1.0, e - 10);
    double k = rint(v / q); /* the division by a power of two is exact; rint = ties to even */
    double r = k * q;
    (void)m;
    if (r >= 65536.0)
        return sign | 0x7C00;
    /* encode r */
    if (r < ldexp(1.0, -14))
        return sign | (uint16_t)k; /* subnormal: r = k * 2^-24 */
    int er = 0;
    double mr = frexp(r, &er); /* r = mr * 2^er, mr in [0.5, 1) */
    er -= 1;
    uint16_t mant = (uint16_t)((mr * 2.0 - 1.0) * 1024.0);
    return sign | (uint16_t)((er + 15) << 10) | mant;
}

/* w: [out_f][in_f] E4M3 bytes; aux: the per-tensor scale (grid = 0, aux[0]) or the f32 grid
 * [ceil(out_f/128)][ceil(in_f/128)] (grid = 1).  out: [out_f][in_f/32 * 34] bytes (f16 d
 * little-endian, then 32 int8).  dout (may be NULL): the f32 d of every block. */
void memq_oracle_repack_q8_0(const uint8_t *w, const float *aux, int grid, int64_t out_f,
                             int64_t in_f, uint8_t *out, float *dout)
{
    int64_t nb = in_f / 32, gcols = (in_f + 127) / 128;
    for (int64_t r = 0; r < out_f; ++r) {
        for (int64_t b = 0; b < nb; ++b) {
            float W[32];
            float amax = 0.0f;
            for (int k = 0; k < 32; ++k) {
                int64_t i = b * 32 + k;
                float s = grid ? aux[(r / 128) * gcols + i / 128] : aux[0];
                volatile float p = (float)memq_oracle_e4m3(w[r * in_f + i]) * s;
                W[k] = p;
                if (fabsf(W[k]) > amax)
                    amax = fabsf(W[k]);
            }
            volatile float d = amax / 127.0f;
            uint8_t *blk = out + (r * nb + b) * 34;
            uint16_t h = memq_oracle_f16_bits((double)d);
            blk[0] = (uint8_t)(h & 0xFF);
            blk[1] = (uint8_t)(h >> 8);
            if (dout)
                dout[r * nb + b] = d;
            for (int k = 0; k < 32; ++k) {
                volatile float t = (d != 0.0f) ? W[k] / d : 0.0f;
                blk[2 + k] = (uint8_t)(int8_t)roundf(t);
            }
        }
    }
}

/* ---------------------------------------------------------------------------------------------
 * t <= 8 MLA decode attention (mla_decode_arm_gate.rs: the three kernels `absorb_q`,
 * `decompress_v` and `attn_gathered`, geometry nh = 64 heads, kv_rank = 512, d_nope = d_v = 256,
 * d_rope = 0, a top-k gather of n_slots rows from a cache of kv rows).  The pages give shapes and
 * call sequences only; the readings:
 *   absorb_q      out[t][h][r] = sum_d q_nope[t][h][d] * wk_b[h][r][d]       (wk_b [nh][kv_rank][d_nope])
 *   decompress_v  out[t][h][v] = sum_r o_lat[t][h][r] * wv_b[h][v][r]        (wv_b [nh][d_v][kv_rank])
 *   attn_gathered per (t, h), over the gathered rows c_j = cache[idx[t][j]] (kv_rank + d_rope
 *                 floats): s_j = scale * (q_lat[t][h] . c_j[0:kv_rank] + q_pe[t][h] . c_j[kv_rank:]),
 *                 p = softmax(s), out[t][h][r] = sum_j p_j * c_j[r]          (out [t][nh][kv_rank])
 * Each also returns sabs, the sum of |terms| of every output (the scale of its rounding error).
 * ------------------------------------------------------------------------------------------- */

/* The per-head product shared by absorb_q and decompress_v: out[t][h][i] = sum_k x[t][h][k] *
 * w[h][i][k], x [t][nh][cols], w [nh][rows][cols], out / sabs [t][nh][rows]. */
void memq_oracle_mla_head_gemv(const float *x, const float *w, int t, int nh, int rows, int cols,
                               double *out, double *sabs)
{
    for (int tt = 0; tt < t; ++tt)
        for (int h = 0; h < nh; ++h)
            for (int i = 0; i < rows; ++i) {
                double acc = 0.0, s = 0.0;
                const float *xr = x + ((int64_t)tt * nh + h) * cols;
                const float *wr = w + ((int64_t)h * rows + i) * cols;
                for (int k = 0; k < cols; ++k) {
                    double p = (double)xr[k] * (double)wr[k];
                    acc += p;
                    s += fabs(p);
                }
                out[((int64_t)tt * nh + h) * rows + i] = acc;
                sabs[((int64_t)tt * nh + h) * rows + i] = s;
            }
}

/* out, cabs: [t][nh][kv_rank]; cabs[t][h][r] = max_j |c_j[r]| (the scale of the output's
 * error).  scores (may be NULL): [t][nh][n_slots], the s_j. */
void memq_oracle_mla_attn_gathered(const float *q_lat, const float *q_pe, const float *cache,
                                   const int32_t *idx, int nh, int kv_rank, int d_rope, int t,
                                   int n_slots, float scale, double *out, double *cabs,
                                   double *scores)
{
    const int row = kv_rank + d_rope;
    double *s = (double *)malloc(sizeof(double) * (size_t)n_slots);
    for (int tt = 0; tt < t; ++tt)
        for (int h = 0; h < nh; ++h) {
            const float *q = q_lat + ((int64_t)tt * nh + h) * kv_rank;
            const float *qp = q_pe + ((int64_t)tt * nh + h) * d_rope;
            double m = -INFINITY;
            for (int j = 0; j < n_slots; ++j) {
                const float *c = cache + (int64_t)idx[(int64_t)tt * n_slots + j] * row;
                double dot = 0.0;
                for (int r = 0; r < kv_rank; ++r)
                    dot += (double)q[r] * (double)c[r];
                for (int r = 0; r < d_rope; ++r)
                    dot += (double)qp[r] * (double)c[kv_rank + r];
                s[j] = (double)scale * dot;
                if (scores)
                    scores[((int64_t)tt * nh + h) * n_slots + j] = s[j];
                if (s[j] > m)
                    m = s[j];
            }
            double l = 0.0;
            for (int j = 0; j < n_slots; ++j)
                l += exp(s[j] - m);
            double *o = out + ((int64_t)tt * nh + h) * kv_rank;
            double *ca = cabs + ((int64_t)tt * nh + h) * kv_rank;
            for (int r = 0; r < kv_rank; ++r) {
                o[r] = 0.0;
                ca[r] = 0.0;
            }
            for (int j = 0; j < n_slots; ++j) {
                const float *c = cache + (int64_t)idx[(int64_t)tt * n_slots + j] * row;
                double pj = exp(s[j] - m) / l;
                for (int r = 0; r < kv_rank; ++r) {
                    o[r] += pj * (double)c[r];
                    if (fabs((double)c[r]) > ca[r])
                        ca[r] = fabs((double)c[r]);
                }
            }
        }
    free(s);
}
