/*
 * MXFP8 block-scaled quantization: plain scalar CPU oracle.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the package smoke check and the
 * CPU-baseline leg of the benchmark may load this file's library.  The CUDA
 * path never calls it and shares no code with it.
 *
 * What it computes (the MXFP8 quantize operation of "[Common] Experimental
 * CuTeDSL MXFP8 backends in C++ via TVM-FFI", TransformerEngine PR #3137,
 * sections "Description" and the quantization-config review of `to_key()`,
 * whose fields name dtype, fp8_dtype, rowwise, colwise, with_dbias and
 * with_noop; 32-element blocks per the review "Why are the non-32-divisible
 * shapes omitted?"):
 *
 *   A BF16 matrix x[M,N] (row-major) is cut into blocks of 32 elements,
 *   1x32 along a row (rowwise) and 32x1 down a column (colwise).  For every
 *   block with amax = max |x| over its 32 elements the block gets an E8M0
 *   scale byte
 *         e = clamp(k + 127, 0, 254),   k = smallest integer with
 *                                          amax <= Fmax * 2^k,
 *   i.e. k = ceil(log2(amax / Fmax)); an all-zero block gets e = 127.
 *   Each element becomes q = RNE-saturate_F(x * 2^(127 - e)), F = E4M3
 *   (Fmax 448) or E5M2 (Fmax 57344).  The optional dbias is the fp32 column
 *   sum of the unquantized input.
 *
 * Everything is evaluated exactly in double precision: a BF16 value has 8
 * significant bits, the scale is a power of two, so x * 2^(127-e) is exact
 * and the only rounding is the single FP8 rounding.  FP8 layouts follow the
 * bit layouts quoted on the cudnn-frontend PR #593 page ("frost" block-scale
 * GEMMs, FP8 data-type discussion): E4M3 = 1 sign, 4 exponent (bias 7),
 * 3 mantissa bits, no infinity, S.1111.111 = NaN; E5M2 = 1 sign, 5 exponent
 * (bias 15), 2 mantissa bits, IEEE-style infinities and NaNs.
 *
 * NaN / Inf inputs are outside the contract: parity unpinned for them.
 */
#include <math.h>
#include <stdint.h>
#include <stddef.h>

#define MXO_E4M3 0
#define MXO_E5M2 1
#define MXO_BLOCK 32

/* Per-format constants, written from the bit layouts above. */
static int mxo_mbits(int fmt) { return fmt == MXO_E4M3 ? 3 : 2; }
static int mxo_ebits(int fmt) { return fmt == MXO_E4M3 ? 4 : 5; }
static int mxo_bias(int fmt) { return fmt == MXO_E4M3 ? 7 : 15; }
/* Largest finite magnitude: E4M3 0.1111.110 = 1.75 * 2^8; E5M2 0.11110.11 = 1.75 * 2^15. */
double mxo_fp8_max(int fmt) { return fmt == MXO_E4M3 ? 448.0 : 57344.0; }

/* BF16 bit pattern -> exact value: 1 sign, 8 exponent (bias 127), 7 mantissa. */
double mxo_bf16_to_double(uint16_t u)
{
    int sign = (u >> 15) & 1;
    int ef = (u >> 7) & 0xFF;
    int m = u & 0x7F;
    double mag;
    if (ef == 0xFF)
        mag = m ? NAN : INFINITY;
    else if (ef == 0)
        mag = ldexp((double)m, 1 - 127 - 7);            /* subnormal */
    else
        mag = ldexp((double)(128 + m), ef - 127 - 7);   /* (1 + m/128) * 2^(ef-127) */
    return sign ? -mag : mag;
}

/* FP8 byte -> exact value. */
double mxo_fp8_decode(uint8_t b, int fmt)
{
    const int mbits = mxo_mbits(fmt), ebits = mxo_ebits(fmt), bias = mxo_bias(fmt);
    const int sign = b >> 7;
    const int ef = (b >> mbits) & ((1 << ebits) - 1);
    const int m = b & ((1 << mbits) - 1);
    double mag;
    if (fmt == MXO_E4M3 && ef == 15 && m == 7)
        return NAN;
    if (fmt == MXO_E5M2 && ef == 31) {
        if (m)
            return NAN;
        mag = INFINITY;
    } else if (ef == 0) {
        mag = ldexp((double)m, 1 - bias - mbits);
    } else {
        mag = ldexp((double)((1 << mbits) + m), ef - bias - mbits);
    }
    return sign ? -mag : mag;
}

/*
 * Exact value -> FP8 byte, round to nearest with ties to even mantissa,
 * saturating every finite overflow (and +-Inf) to +-Fmax.  The sign of a
 * result that rounds to zero is kept (-tiny -> 0x80).
 */
uint8_t mxo_fp8_encode(double v, int fmt)
{
    const int mbits = mxo_mbits(fmt), bias = mxo_bias(fmt);
    const int emin = 1 - bias;                /* exponent of the smallest normal */
    const double fmax = mxo_fp8_max(fmt);
    const int sign = signbit(v) ? 1 : 0;
    double a = fabs(v), r;
    int ex, e2, ef, m;

    if (isnan(a))
        return (uint8_t)((sign << 7) | 0x7F);  /* S.1111.111 / S.11111.11 */
    if (a == 0.0)
        return (uint8_t)(sign << 7);
    if (isinf(a)) {
        r = fmax;
    } else {
        /* Spacing of representable values around a: 2^(max(floor(log2 a), emin) - mbits). */
        frexp(a, &e2);                         /* a = f * 2^e2, f in [0.5, 1) */
        ex = e2 - 1;                           /* floor(log2 a) */
        if (ex < emin)
            ex = emin;
        const double quantum = ldexp(1.0, ex - mbits);
        r = nearbyint(a / quantum) * quantum;  /* default mode: ties to even */
        if (r > fmax)
            r = fmax;
    }
    if (r == 0.0)
        return (uint8_t)(sign << 7);
    frexp(r, &e2);
    ex = e2 - 1;
    if (ex < emin) {
        ef = 0;
        m = (int)(r / ldexp(1.0, emin - mbits));
    } else {
        ef = ex + bias;
        m = (int)(r / ldexp(1.0, ex - mbits)) - (1 << mbits);
    }
    return (uint8_t)((sign << 7) | (ef << mbits) | m);
}

/* E8M0 block exponent e for a block whose largest magnitude is amax. */
int mxo_block_exponent(double amax, int fmt)
{
    const double fmax = mxo_fp8_max(fmt);
    int k, e;
    if (amax == 0.0)
        return 127;
    /* smallest integer k with amax <= fmax * 2^k, found by search from a guess */
    k = ilogb(amax) - ilogb(fmax);
    while (amax > ldexp(fmax, k))
        k++;
    while (amax <= ldexp(fmax, k - 1))
        k--;
    e = k + 127;
    if (e < 0)
        e = 0;
    if (e > 254)
        e = 254;
    return e;
}

/* E8M0 byte -> scale value 2^(e-127) (255 is NaN). */
double mxo_e8m0_decode(uint8_t e)
{
    return e == 255 ? NAN : ldexp(1.0, (int)e - 127);
}

/*
 * Flat quantize of x[M,N] (BF16 bits, row-major).  Any of the four output
 * pairs may be NULL to skip that direction; dbias may be NULL.  With
 * Cr = ceil(N/32) and Rc = ceil(M/32):
 *   out_row[i*N + j], scale_row[i*Cr + j/32]   (1x32 blocks along a row)
 *   out_col[i*N + j], scale_col[(i/32)*N + j]  (32x1 blocks down a column)
 * When N (or M) is not a multiple of 32 the last block of each row (column)
 * holds the remaining N % 32 (M % 32) elements, and its amax is taken over
 * those elements only (the reading adopted for shapes the source page's
 * kernels leave out: "Why are the non-32-divisible shapes omitted?").
 * Returns 0, or -1 if M or N is negative.
 */
int mxo_quantize(const uint16_t *x, int64_t M, int64_t N, int fmt,
                 uint8_t *out_row, uint8_t *scale_row,
                 uint8_t *out_col, uint8_t *scale_col, float *dbias)
{
    int64_t i, j, c, r, k;
    if (M < 0 || N < 0)
        return -1;
    const int64_t Cr = (N + MXO_BLOCK - 1) / MXO_BLOCK, Rc = (M + MXO_BLOCK - 1) / MXO_BLOCK;

    if (out_row && scale_row) {
        for (i = 0; i < M; i++) {
            for (c = 0; c < Cr; c++) {
                const int64_t j0 = c * MXO_BLOCK;
                const int64_t len = N - j0 < MXO_BLOCK ? N - j0 : MXO_BLOCK;
                const uint16_t *blk = x + i * N + j0;
                double amax = 0.0;
                for (k = 0; k < len; k++) {
                    double a = fabs(mxo_bf16_to_double(blk[k]));
                    if (a > amax)
                        amax = a;
                }
                const int e = mxo_block_exponent(amax, fmt);
                const double s = ldexp(1.0, 127 - e);
                scale_row[i * Cr + c] = (uint8_t)e;
                for (k = 0; k < len; k++)
                    out_row[i * N + j0 + k] = mxo_fp8_encode(mxo_bf16_to_double(blk[k]) * s, fmt);
            }
        }
    }

    if (out_col && scale_col) {
        for (r = 0; r < Rc; r++) {
            const int64_t i0 = r * MXO_BLOCK;
            const int64_t len = M - i0 < MXO_BLOCK ? M - i0 : MXO_BLOCK;
            for (j = 0; j < N; j++) {
                double amax = 0.0;
                for (k = 0; k < len; k++) {
                    double a = fabs(mxo_bf16_to_double(x[(i0 + k) * N + j]));
                    if (a > amax)
                        amax = a;
                }
                const int e = mxo_block_exponent(amax, fmt);
                const double s = ldexp(1.0, 127 - e);
                scale_col[r * N + j] = (uint8_t)e;
                for (k = 0; k < len; k++) {
                    const int64_t idx = (i0 + k) * N + j;
                    out_col[idx] = mxo_fp8_encode(mxo_bf16_to_double(x[idx]) * s, fmt);
                }
            }
        }
    }

    if (dbias) {
        for (j = 0; j < N; j++) {
            double acc = 0.0;
            for (i = 0; i < M; i++)
                acc += mxo_bf16_to_double(x[i * N + j]);
            dbias[j] = (float)acc;
        }
    }
    return 0;
}

/*
 * Grouped quantize: rows [offsets[g], offsets[g+1]) form group g; each
 * group is quantized as its own flat problem (its columnwise blocks start at
 * the group's first row, and its last block holds the rows the group has
 * left).  Row-indexed outputs (out_row, scale_row, out_col) sit at the
 * group's row offset; the group's ceil(rows_g/32) columnwise scale rows
 * follow those of the groups before it, i.e. start at scale row
 * sum_{h<g} ceil(rows_h/32) (= offsets[g]/32 when every offset is a
 * multiple of 32, the flat call's layout).  offsets has num_groups+1
 * entries.  Returns 0, or -1 when the offsets are not a prefix-sum vector
 * starting at 0, ending at total_rows and non-decreasing.
 */
int mxo_quantize_grouped(const uint16_t *x, int64_t total_rows, int64_t N, int num_groups,
                         const int64_t *offsets, int fmt,
                         uint8_t *out_row, uint8_t *scale_row,
                         uint8_t *out_col, uint8_t *scale_col)
{
    int g;
    if (num_groups < 0 || total_rows < 0 || N < 0)
        return -1;
    if (offsets[0] != 0 || offsets[num_groups] != total_rows)
        return -1;
    int64_t s0 = 0; /* first columnwise scale row of group g */
    for (g = 0; g < num_groups; g++)
        if (offsets[g + 1] < offsets[g])
            return -1;
    for (g = 0; g < num_groups; g++) {
        const int64_t r0 = offsets[g], rows = offsets[g + 1] - offsets[g];
        if (rows == 0)
            continue;
        mxo_quantize(x + r0 * N, rows, N, fmt,
                     out_row ? out_row + r0 * N : 0,
                     scale_row ? scale_row + r0 * ((N + MXO_BLOCK - 1) / MXO_BLOCK) : 0,
                     out_col ? out_col + r0 * N : 0, scale_col ? scale_col + s0 * N : 0,
                     0);
        s0 += (rows + MXO_BLOCK - 1) / MXO_BLOCK;
    }
    return 0;
}

/*
 * GEMM-ready ("swizzled") E8M0 scale layout.  The pages name a `swizzled`
 * config bit (TransformerEngine PR #3137, `to_key()` review) without giving
 * the layout; the reading used here is the layout block-scaled tensor-core
 * GEMMs take on Blackwell: a scale matrix of R rows x C scale columns is
 * padded to multiples of 128 rows and 4 columns and cut into 128x4 tiles of
 * 512 bytes, tiles stored row-tile major (all column tiles of row tile 0,
 * then row tile 1, ...); inside a tile, entry (r, c) sits at
 * (r % 32) * 16 + (r / 32) * 4 + c.  Padding entries are 0.
 */
int64_t mxo_swizzled_bytes(int64_t R, int64_t C)
{
    return ((R + 127) / 128 * 128) * ((C + 3) / 4 * 4);
}

int64_t mxo_swizzle_offset(int64_t r, int64_t c, int64_t C)
{
    const int64_t col_tiles = (C + 3) / 4;
    const int64_t tile = (r / 128) * col_tiles + c / 4;
    const int64_t rr = r % 128, cc = c % 4;
    return tile * 512 + (rr % 32) * 16 + (rr / 32) * 4 + cc;
}

/* plain[R][C] (row-major) -> out[mxo_swizzled_bytes(R, C)], padding zeroed. */
void mxo_swizzle_scales(const uint8_t *plain, int64_t R, int64_t C, uint8_t *out)
{
    int64_t r, c;
    const int64_t n = mxo_swizzled_bytes(R, C);
    for (r = 0; r < n; r++)
        out[r] = 0;
    for (r = 0; r < R; r++)
        for (c = 0; c < C; c++)
            out[mxo_swizzle_offset(r, c, C)] = plain[r * C + c];
}

/* Per-tensor amax: max |x| over the whole BF16 matrix, as fp32 (exact). */
float mxo_amax(const uint16_t *x, int64_t M, int64_t N)
{
    double amax = 0.0;
    int64_t i;
    for (i = 0; i < M * N; i++) {
        const double a = fabs(mxo_bf16_to_double(x[i]));
        if (a > amax)
            amax = a;
    }
    return (float)amax;
}

/*
 * Fused activation before the cast (the `with_act` / `activation` fields of the
 * config key on the PR #3137 page).  The pages do not give the formulas; the
 * reading used: the activation is evaluated in fp32 (the value the cast then
 * quantizes, and whose block amax sets the scale) from the BF16 input:
 *   1 ReLU      x > 0 ? x : +0
 *   2 SReLU     x > 0 ? x*x : +0            (squared ReLU, the FC1 epilogue of
 *                                            the Lightning W4A16 page)
 *   3 GeLU      x * sigmoid(2 sqrt(2/pi) (x + 0.044715 x^3))
 *               (= 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))), the tanh
 *               form, written without the cancellation of 1 + tanh for x << 0)
 *   4 SiLU      x * sigmoid(x)
 *   5 QGeLU     x * sigmoid(1.702 x)
 * with sigmoid(t) = 1 / (1 + e^-t) for t >= 0 and e^t / (1 + e^t) for t < 0
 * (no overflow, no cancellation).  mxo_activation_f64 is the exact-as-double
 * value; mxo_activation rounds it once to fp32: exact for ReLU and SReLU (a
 * BF16 square has 16 significant bits), within an ulp or so of the GPU's fp32
 * evaluation for the others.
 */
static double mxo_sigmoid(double t)
{
    if (t >= 0)
        return 1.0 / (1.0 + exp(-t));
    const double e = exp(t);
    return e / (1.0 + e);
}

double mxo_activation_f64(double x, int act)
{
    switch (act) {
    case 1: return x > 0 ? x : 0.0;
    case 2: return x > 0 ? x * x : 0.0;
    case 3: return x * mxo_sigmoid(2.0 * 0.7978845608028654 * (x + 0.044715 * x * x * x));
    case 4: return x * mxo_sigmoid(x);
    case 5: return x * mxo_sigmoid(1.702 * x);
    default: return x;
    }
}

float mxo_activation(double x, int act)
{
    return (float)mxo_activation_f64(x, act);
}

/*
 * Quantize fp32 values y[M,N] (already activated): same blocks (partial last
 * blocks included), scale rule and rounding as mxo_quantize, evaluated
 * exactly on the fp32 values; dbias (if requested) is the column sum of y.
 */
int mxo_quantize_f32(const float *y, int64_t M, int64_t N, int fmt,
                     uint8_t *out_row, uint8_t *scale_row,
                     uint8_t *out_col, uint8_t *scale_col, float *dbias)
{
    int64_t i, j, c, r, k;
    if (M < 0 || N < 0)
        return -1;
    const int64_t Cr = (N + MXO_BLOCK - 1) / MXO_BLOCK, Rc = (M + MXO_BLOCK - 1) / MXO_BLOCK;
    if (out_row && scale_row) {
        for (i = 0; i < M; i++) {
            for (c = 0; c < Cr; c++) {
                const int64_t j0 = c * MXO_BLOCK, len = N - j0 < MXO_BLOCK ? N - j0 : MXO_BLOCK;
                const float *blk = y + i * N + j0;
                double amax = 0.0;
                for (k = 0; k < len; k++)
                    if (fabs((double)blk[k]) > amax)
                        amax = fabs((double)blk[k]);
                const int e = mxo_block_exponent(amax, fmt);
                const double s = ldexp(1.0, 127 - e);
                scale_row[i * Cr + c] = (uint8_t)e;
                for (k = 0; k < len; k++)
                    out_row[i * N + j0 + k] = mxo_fp8_encode((double)blk[k] * s, fmt);
            }
        }
    }
    if (out_col && scale_col) {
        for (r = 0; r < Rc; r++) {
            const int64_t i0 = r * MXO_BLOCK, len = M - i0 < MXO_BLOCK ? M - i0 : MXO_BLOCK;
            for (j = 0; j < N; j++) {
                double amax = 0.0;
                for (k = 0; k < len; k++) {
                    const double a = fabs((double)y[(i0 + k) * N + j]);
                    if (a > amax)
                        amax = a;
                }
                const int e = mxo_block_exponent(amax, fmt);
                const double s = ldexp(1.0, 127 - e);
                scale_col[r * N + j] = (uint8_t)e;
                for (k = 0; k < len; k++) {
                    const int64_t idx = (i0 + k) * N + j;
                    out_col[idx] = mxo_fp8_encode((double)y[idx] * s, fmt);
                }
            }
        }
    }
    if (dbias) {
        for (j = 0; j < N; j++) {
            double acc = 0.0;
            for (i = 0; i < M; i++)
                acc += (double)y[i * N + j];
            dbias[j] = (float)acc;
        }
    }
    return 0;
}

/* y[i] = activation(x[i]) for a BF16 matrix, as fp32. */
void mxo_activate(const uint16_t *x, int64_t n, int act, float *y)
{
    int64_t i;
    for (i = 0; i < n; i++)
        y[i] = mxo_activation(mxo_bf16_to_double(x[i]), act);
}

/*
 * Gated activation before the cast (the GLU family: ReGLU, squared-ReLU GLU,
 * GeGLU, SwiGLU, QGeGLU for act = 1..5).  The pages name the fused activation
 * field but give neither the gated forms nor their layout; the reading used:
 * x is BF16 [M, 2N], its first N columns are the activation's input a and its
 * last N the linear input b, and the value cast is
 *     y[i][j] = act(a[i][j]) * b[i][j],   a = x[i][j], b = x[i][N + j],
 * evaluated in double (act as in mxo_activation_f64) and rounded once to fp32.
 * y is [M, N] fp32.
 */
void mxo_gate(const uint16_t *x, int64_t M, int64_t N, int act, float *y)
{
    int64_t i, j;
    for (i = 0; i < M; i++)
        for (j = 0; j < N; j++) {
            const double a = mxo_bf16_to_double(x[i * 2 * N + j]);
            const double b = mxo_bf16_to_double(x[i * 2 * N + N + j]);
            y[i * N + j] = (float)(mxo_activation_f64(a, act) * b);
        }
}

/*
 * Per-expert dbias of a grouped call (each expert's bias gradient, the
 * column sums of its own rows): dbias[g][j] = sum of x[i][j] over the rows i
 * of group g, in double, rounded once to fp32; an empty group gets zeros.
 * Returns -1 for offsets the grouped call rejects.
 */
int mxo_grouped_dbias(const uint16_t *x, int64_t total_rows, int64_t N, int num_groups,
                      const int64_t *offsets, float *dbias)
{
    int g;
    int64_t i, j;
    if (num_groups < 0 || total_rows < 0 || N < 0 || offsets[0] != 0 || offsets[num_groups] != total_rows)
        return -1;
    for (g = 0; g < num_groups; g++)
        if (offsets[g + 1] < offsets[g])
            return -1;
    for (g = 0; g < num_groups; g++)
        for (j = 0; j < N; j++) {
            double acc = 0.0;
            for (i = offsets[g]; i < offsets[g + 1]; i++)
                acc += mxo_bf16_to_double(x[i * N + j]);
            dbias[(int64_t)g * N + j] = (float)acc;
        }
    return 0;
}

/*
 * Backward fusion (the `with_dact` field of the config key on the PR #3137
 * page): the cast quantizes dY * act'(X) for a gradient dY and the
 * activation's input X, both BF16.  The pages give no formulas; the reading
 * used is the derivative of each activation of mxo_activation, evaluated in
 * fp32 and multiplied by dY in fp32:
 *   1 dReLU    X > 0 ? 1 : 0
 *   2 dSReLU   X > 0 ? 2X : 0
 *   3 dGeLU    s (1 + X (1-s) t'), s = sigmoid(t), t = 2 sqrt(2/pi) (X + 0.044715 X^3),
 *                                 t' = 2 sqrt(2/pi) (1 + 3 * 0.044715 X^2)
 *   4 dSiLU    s (1 + X (1-s)),   s = sigmoid(X)
 *   5 dQGeLU   s (1 + 1.702 X (1-s)), s = sigmoid(1.702 X)
 * with s and 1-s both taken from e = exp(-|t|) (no cancellation).  Here the
 * derivative is evaluated in double and the product dY * act'(X) rounded once
 * to fp32: exact for dReLU and dSReLU (a product of BF16 values and 2), within
 * a few fp32 ulps of the GPU's evaluation for the others.
 */
static void mxo_sigmoid_pair(double t, double *s, double *one_minus_s)
{
    const double e = exp(-fabs(t));
    const double inv = 1.0 / (1.0 + e);
    *s = t >= 0 ? inv : e * inv;
    *one_minus_s = t >= 0 ? e * inv : inv;
}

double mxo_dactivation_f64(double x, int act)
{
    double s, oms;
    switch (act) {
    case 1: return x > 0 ? 1.0 : 0.0;
    case 2: return x > 0 ? 2.0 * x : 0.0;
    case 3: {
        const double c = 2.0 * 0.7978845608028654;
        const double t = c * (x + 0.044715 * x * x * x), dt = c * (1.0 + 3.0 * 0.044715 * x * x);
        mxo_sigmoid_pair(t, &s, &oms);
        return s * (1.0 + x * oms * dt);   /* factored: keeps the sign when s underflows */
    }
    case 4:
        mxo_sigmoid_pair(x, &s, &oms);
        return s * (1.0 + x * oms);
    case 5:
        mxo_sigmoid_pair(1.702 * x, &s, &oms);
        return s * (1.0 + 1.702 * x * oms);
    default: return 1.0;
    }
}

/* y[i] = dY[i] * act'(X[i]) for BF16 matrices, rounded once to fp32. */
void mxo_dactivate(const uint16_t *dy, const uint16_t *x, int64_t n, int act, float *y)
{
    int64_t i;
    for (i = 0; i < n; i++)
        y[i] = (float)(mxo_bf16_to_double(dy[i]) * mxo_dactivation_f64(mxo_bf16_to_double(x[i]), act));
}

/*
 * Backward of the gated activation (mxo_gate): for y = act(a) * b and the
 * gradient g = dL/dy (BF16 [M, N]), the gradient of x = [a | b] is
 *     da = g * b * act'(a),   db = g * act(a),
 * each evaluated in double (act and act' as in mxo_activation_f64 /
 * mxo_dactivation_f64) and rounded once to fp32.  da and db are [M, N] fp32.
 */
void mxo_dgate(const uint16_t *g, const uint16_t *x, int64_t M, int64_t N, int act, float *da, float *db)
{
    int64_t i, j;
    for (i = 0; i < M; i++)
        for (j = 0; j < N; j++) {
            const double gv = mxo_bf16_to_double(g[i * N + j]);
            const double a = mxo_bf16_to_double(x[i * 2 * N + j]);
            const double b = mxo_bf16_to_double(x[i * 2 * N + N + j]);
            da[i * N + j] = (float)(gv * b * mxo_dactivation_f64(a, act));
            db[i * N + j] = (float)(gv * mxo_activation_f64(a, act));
        }
}
