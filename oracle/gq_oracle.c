/*
 * gq_oracle.c -- plain, slow CPU oracle for the grouped FP8 quantizer and the
 * grouped expert GEMMs.  TEST INFRASTRUCTURE ONLY: the tests, the smoke check
 * and the benchmark's CPU-baseline leg call it; the product path never does.
 * It shares no code, header or table with the CUDA library.
 *
 * What it computes, and where the pages define it:
 *
 *  - Split scan (row offsets, 128-row tile counts, scale offsets) -- the
 *    split_sizes / grouped_layout / m_splits partition of a token buffer
 *    (DeepGEMM issue 365, the unit test's grouped_layout; TransformerEngine
 *    PR 3224, "first_dims" and the alignment contract for m_splits).
 *  - MXFP8 1x32 quantisation with E8M0 scales, rowwise and columnwise, scales
 *    in the swizzled [outer/128][inner/128][32][4][4] layout with every
 *    extent taken from the group's own row count (TransformerEngine issue
 *    3484, "Describe the bug"; PR 3224, the group_quantize_mxfp8 fix).
 *  - Per-channel 128-row fp32-scale quantisation, op by op in fp32, as in the
 *    DeepGEMM issue's _per_channel_cast_to_fp8 (sf = amax/448, zero -> sf_val,
 *    clamp_min(1e-30), codes = e4m3(x * (1/sf))).
 *  - Grouped fprop Y_e = X_e W_e^T, dgrad dX_e = dY_e W_e and k-grouped
 *    wgrad dW_e = dY_e^T X_e over each group's live rows only, on the
 *    dequantised operands, accumulated in fp64 (TransformerEngine issue 3484,
 *    "Additional context: Scope"; DeepGEMM issue 365, the fp32 reference
 *    ref[e] = gy_e.t() @ s_e with empty experts skipped).
 *  - Grouped bias add y += b_g over each group's live rows, and the bias
 *    gradient db_g = column sums of dY over the group's live rows
 *    (TransformerEngine PR 3224: launch_grouped_bias_add with its zero-row
 *    guard, and the dbiases of the backward).
 *
 * Readings taken where the pages are silent (each listed in the design notes):
 *  - FP8 is float8_e4m3fn: bias 7, max 448, no infinities, NaN = S.1111.111,
 *    subnormals down to 2^-9; conversion rounds to nearest, ties to even, and
 *    saturates finite values to +-448; a value that rounds to zero keeps its
 *    sign.
 *  - The E8M0 block scale is 2^e with e = floor(log2(amax)) - 8 (8 = the
 *    largest e4m3 exponent), clamped to [-127, 127]; an all-zero block gets
 *    e = -127.  Codes are e4m3(x * 2^-e).
 *  - In the [32][4][4] atom the byte of (row r of a 128-row tile, scale
 *    column j of a 4-column group) sits at (r % 32) * 16 + (r / 32) * 4 + j.
 *    Rowwise atoms of a group are ordered [row tile][column tile]; columnwise
 *    atoms [column tile][row tile] (the m-tile is the inner stride).  Bytes of
 *    a group's last tile that cover no live row are 0.
 *  - Columnwise codes keep the buffer's [rows, cols] orientation.
 *  - Per-channel scales are stored [live_rows/128][cols] (block-major): the
 *    storage of the page's sf, which the page hands on as the view sf.T.
 *  - MX needs every split % 32 == 0, the per-channel recipe % 128 == 0, and
 *    cols % 128 == 0; anything else is rejected, not padded.
 */
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_OK 0
#define OR_ERR_INVALID_ARG (-1)
#define OR_ERR_ALIGNMENT (-2)
#define OR_ERR_SPLITS (-3)
#define OR_ERR_UNSUPPORTED (-4)

#define OR_RECIPE_MX 0
#define OR_RECIPE_CHANNEL 1

/* ------------------------------------------------------------------------ */
/* bf16 and float8_e4m3fn                                                    */
/* ------------------------------------------------------------------------ */

static double bf16_value(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static float bf16_value_f32(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Value of an e4m3fn byte: (-1)^s * 2^(E-7) * 1.mmm for E > 0,
 * (-1)^s * 2^-6 * 0.mmm for E == 0; S.1111.111 is NaN. */
double or_e4m3_decode(uint8_t b)
{
    int s = b >> 7, E = (b >> 3) & 15, m = b & 7;
    double v;
    if (E == 15 && m == 7)
        return NAN;
    if (E == 0)
        v = ldexp((double)m, -9);              /* m/8 * 2^-6 */
    else
        v = ldexp((double)(8 + m), E - 10);    /* (1 + m/8) * 2^(E-7) */
    return s ? -v : v;
}

/* Nearest e4m3fn value to v (ties to even mantissa), saturating to +-448.
 * v must be exactly the value to be rounded (the callers pass exact products). */
uint8_t or_e4m3_encode(double v)
{
    uint8_t sign = (signbit(v) ? 0x80 : 0x00);
    double a = fabs(v);
    int e2;
    double q, n;
    if (isnan(v))
        return 0x7F;
    if (a >= 448.0)
        return sign | 0x7E;
    /* quantum of the binade that holds a: 2^(E-3) for normals, 2^-9 below 2^-6 */
    if (a < ldexp(1.0, -6)) {
        e2 = -9;
    } else {
        int E;
        frexp(a, &E);          /* a = f * 2^E, f in [0.5, 1) => floor(log2 a) = E - 1 */
        e2 = (E - 1) - 3;
    }
    q = ldexp(a, -e2);         /* exact: a / quantum */
    n = floor(q);
    if (q - n > 0.5 || (q - n == 0.5 && fmod(n, 2.0) != 0.0))
        n += 1.0;
    /* n * 2^e2 is the rounded magnitude; now find its bit pattern */
    if (e2 == -9)
        return sign | (uint8_t)n;          /* n in [0, 8]; 8 is the smallest normal 0x08 */
    {
        int E = e2 + 3;                    /* floor(log2 a) */
        int code = ((E + 7) << 3) + ((int)n - 8);   /* n in [8, 16]; 16 carries into E+1 */
        if (code > 0x7E)
            code = 0x7E;
        return sign | (uint8_t)code;
    }
}

void or_e4m3_encode_array(const double* v, int64_t n, uint8_t* out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = or_e4m3_encode(v[i]);
}

void or_e4m3_decode_array(const uint8_t* b, int64_t n, double* out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = or_e4m3_decode(b[i]);
}

/* E8M0 exponent of a 32-element block: floor(log2 amax) - 8, clamped. */
int or_mx_scale_exponent(double amax)
{
    int E, e;
    if (amax == 0.0)
        return -127;
    frexp(amax, &E);
    e = (E - 1) - 8;
    if (e < -127)
        e = -127;
    if (e > 127)
        e = 127;
    return e;
}

/* ------------------------------------------------------------------------ */
/* Split scan                                                                */
/* ------------------------------------------------------------------------ */

static int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

/* Row offsets o_g, prefix of 128-row tile counts, and scale-buffer byte
 * offsets of every group.  splits == NULL means the uniform split
 * rows_cap / G (which must divide).  Arrays hold G + 1 entries. */
int or_split_scan(const int32_t* splits, int G, int64_t rows_cap, int64_t cols, int recipe,
                  int64_t* row_offset, int64_t* tile_prefix, int64_t* scale_offset)
{
    int64_t o = 0, t = 0;
    int align = (recipe == OR_RECIPE_CHANNEL) ? 128 : 32;
    if (G < 1 || G > 1024 || rows_cap < 0 || cols <= 0)
        return OR_ERR_INVALID_ARG;
    if (cols % 128 != 0)
        return OR_ERR_ALIGNMENT;
    if (splits == NULL && rows_cap % G != 0)
        return OR_ERR_ALIGNMENT;
    for (int g = 0; g < G; ++g) {
        int64_t m = splits ? (int64_t)splits[g] : rows_cap / G;
        if (m < 0 || m % align != 0)
            return OR_ERR_SPLITS;
        row_offset[g] = o;
        tile_prefix[g] = t;
        scale_offset[g] = (recipe == OR_RECIPE_CHANNEL) ? 4 * cols * (o / 128)
                                                        : 512 * (cols / 128) * t;
        o += m;
        t += ceil_div(m, 128);
    }
    if (o > rows_cap)
        return OR_ERR_SPLITS;
    row_offset[G] = o;
    tile_prefix[G] = t;
    scale_offset[G] = (recipe == OR_RECIPE_CHANNEL) ? 4 * cols * (o / 128)
                                                    : 512 * (cols / 128) * t;
    return OR_OK;
}

/* Byte position inside one 512-byte atom: row r of the 128-row tile and
 * scale column j (0..3) of the 4-column group. */
static int64_t atom_byte(int64_t r, int64_t j) { return (r % 32) * 16 + (r / 32) * 4 + j; }

/* ------------------------------------------------------------------------ */
/* MXFP8 1x32 quantisation                                                   */
/* ------------------------------------------------------------------------ */

int or_quantize_mx(const uint16_t* x, int64_t rows_cap, int64_t cols, const int32_t* splits, int G,
                   int rowwise, int colwise,
                   uint8_t* row_data, uint8_t* row_scale, int64_t row_scale_bytes,
                   uint8_t* col_data, uint8_t* col_scale, int64_t col_scale_bytes)
{
    int64_t *off = malloc(sizeof(int64_t) * (G + 1) * 3);
    int64_t *tp, *sb;
    int st;
    if (!off)
        return OR_ERR_INVALID_ARG;
    tp = off + (G + 1);
    sb = off + 2 * (G + 1);
    st = or_split_scan(splits, G, rows_cap, cols, OR_RECIPE_MX, off, tp, sb);
    if (st != OR_OK || (!rowwise && !colwise)) {
        free(off);
        return st != OR_OK ? st : OR_ERR_INVALID_ARG;
    }
    if ((rowwise && sb[G] > row_scale_bytes) || (colwise && sb[G] > col_scale_bytes)) {
        free(off);
        return OR_ERR_INVALID_ARG;
    }
    if (rowwise)
        memset(row_scale, 0, (size_t)sb[G]);
    if (colwise)
        memset(col_scale, 0, (size_t)sb[G]);

    for (int g = 0; g < G; ++g) {
        int64_t o = off[g], m = off[g + 1] - off[g], T = tp[g + 1] - tp[g];
        if (rowwise) {
#pragma omp parallel for schedule(static)
            for (int64_t lr = 0; lr < m; ++lr) {
                int64_t r = o + lr;
                for (int64_t j = 0; j < cols / 32; ++j) {
                    double amax = 0.0;
                    int e;
                    for (int64_t c = 32 * j; c < 32 * j + 32; ++c) {
                        double a = fabs(bf16_value(x[r * cols + c]));
                        if (a > amax)
                            amax = a;
                    }
                    e = or_mx_scale_exponent(amax);
                    for (int64_t c = 32 * j; c < 32 * j + 32; ++c)
                        row_data[r * cols + c] = or_e4m3_encode(ldexp(bf16_value(x[r * cols + c]), -e));
                    row_scale[sb[g] + ((lr / 128) * (cols / 128) + j / 4) * 512 +
                              atom_byte(lr % 128, j % 4)] = (uint8_t)(e + 127);
                }
            }
        }
        if (colwise) {
#pragma omp parallel for schedule(static)
            for (int64_t c = 0; c < cols; ++c) {
                for (int64_t b = 0; b < m / 32; ++b) {
                    double amax = 0.0;
                    int e;
                    for (int64_t lr = 32 * b; lr < 32 * b + 32; ++lr) {
                        double a = fabs(bf16_value(x[(o + lr) * cols + c]));
                        if (a > amax)
                            amax = a;
                    }
                    e = or_mx_scale_exponent(amax);
                    for (int64_t lr = 32 * b; lr < 32 * b + 32; ++lr)
                        col_data[(o + lr) * cols + c] =
                            or_e4m3_encode(ldexp(bf16_value(x[(o + lr) * cols + c]), -e));
                    col_scale[sb[g] + ((c / 128) * T + b / 4) * 512 + atom_byte(c % 128, b % 4)] =
                        (uint8_t)(e + 127);
                }
            }
        }
    }
    free(off);
    return OR_OK;
}

/* ------------------------------------------------------------------------ */
/* Per-channel 128-row fp32-scale quantisation (columnwise only)             */
/* ------------------------------------------------------------------------ */

int or_quantize_channel(const uint16_t* x, int64_t rows_cap, int64_t cols, const int32_t* splits,
                        int G, float zero_scale, uint8_t* col_data, float* col_scale,
                        int64_t col_scale_count)
{
    int64_t *off = malloc(sizeof(int64_t) * (G + 1) * 3);
    int64_t L;
    int st;
    if (!off)
        return OR_ERR_INVALID_ARG;
    st = or_split_scan(splits, G, rows_cap, cols, OR_RECIPE_CHANNEL, off, off + G + 1,
                       off + 2 * (G + 1));
    L = off[G];
    free(off);
    if (st != OR_OK)
        return st;
    if ((L / 128) * cols > col_scale_count)
        return OR_ERR_INVALID_ARG;
    /* Every group starts on a multiple of 128, so live row block b = rows
     * [128b, 128b + 128) lies inside one group. */
#pragma omp parallel for schedule(static)
    for (int64_t c = 0; c < cols; ++c) {
        for (int64_t b = 0; b < L / 128; ++b) {
            float amax = 0.0f, sf, rcp;
            for (int64_t r = 128 * b; r < 128 * b + 128; ++r) {
                float a = fabsf(bf16_value_f32(x[r * cols + c]));
                if (a > amax)
                    amax = a;
            }
            sf = amax / 448.0f;
            if (sf == 0.0f)
                sf = zero_scale;
            if (sf < 1e-30f)
                sf = 1e-30f;
            rcp = 1.0f / sf;
            for (int64_t r = 128 * b; r < 128 * b + 128; ++r) {
                volatile float q = bf16_value_f32(x[r * cols + c]) * rcp;   /* one fp32 rounding */
                col_data[r * cols + c] = or_e4m3_encode((double)q);
            }
            col_scale[b * cols + c] = sf;
        }
    }
    return OR_OK;
}

/* ------------------------------------------------------------------------ */
/* Dequantisation of single elements                                         */
/* ------------------------------------------------------------------------ */

typedef struct {
    int G;
    int64_t cols;
    const int64_t* off;   /* row offsets, G + 1 */
    const int64_t* tp;    /* tile prefix, G + 1 */
    const int64_t* sb;    /* scale byte offsets, G + 1 */
} layout_t;

static int group_of_row(const layout_t* l, int64_t r)
{
    int lo = 0, hi = l->G - 1;
    while (lo < hi) {            /* last g with off[g] <= r and a non-empty range */
        int mid = (lo + hi + 1) / 2;
        if (l->off[mid] <= r)
            lo = mid;
        else
            hi = mid - 1;
    }
    return lo;
}

/* Rowwise MX element (r, c): code * 2^(scale - 127). */
static double mx_row_elem(const layout_t* l, const uint8_t* data, const uint8_t* scale, int g,
                          int64_t r, int64_t c)
{
    int64_t lr = r - l->off[g];
    int64_t j = c / 32;
    uint8_t s = scale[l->sb[g] + ((lr / 128) * (l->cols / 128) + j / 4) * 512 +
                      atom_byte(lr % 128, j % 4)];
    return ldexp(or_e4m3_decode(data[r * l->cols + c]), (int)s - 127);
}

/* Columnwise MX element (r, c). */
static double mx_col_elem(const layout_t* l, const uint8_t* data, const uint8_t* scale, int g,
                          int64_t r, int64_t c)
{
    int64_t lr = r - l->off[g];
    int64_t b = lr / 32;
    int64_t T = l->tp[g + 1] - l->tp[g];
    uint8_t s = scale[l->sb[g] + ((c / 128) * T + b / 4) * 512 + atom_byte(c % 128, b % 4)];
    return ldexp(or_e4m3_decode(data[r * l->cols + c]), (int)s - 127);
}

/* Per-channel element (r, c): code * sf[r / 128][c]. */
static double ch_col_elem(const layout_t* l, const uint8_t* data, const float* scale, int64_t r,
                          int64_t c)
{
    return or_e4m3_decode(data[r * l->cols + c]) * (double)scale[(r / 128) * l->cols + c];
}

typedef struct {
    int64_t* buf;
    layout_t l;
} scan_t;

static int make_layout(scan_t* s, const int32_t* splits, int G, int64_t rows_cap, int64_t cols,
                       int recipe)
{
    int st;
    s->buf = malloc(sizeof(int64_t) * (G + 1) * 3);
    if (!s->buf)
        return OR_ERR_INVALID_ARG;
    st = or_split_scan(splits, G, rows_cap, cols, recipe, s->buf, s->buf + G + 1,
                       s->buf + 2 * (G + 1));
    s->l.G = G;
    s->l.cols = cols;
    s->l.off = s->buf;
    s->l.tp = s->buf + G + 1;
    s->l.sb = s->buf + 2 * (G + 1);
    if (st != OR_OK) {
        free(s->buf);
        s->buf = NULL;
    }
    return st;
}

/* Dequantise rows [0, L) of an MX operand into a dense fp64 [L, cols] array. */
static double* deq_mx(const layout_t* l, const uint8_t* data, const uint8_t* scale, int colwise)
{
    int64_t L = l->off[l->G];
    double* out = malloc(sizeof(double) * (size_t)(L > 0 ? L : 1) * (size_t)l->cols);
    if (!out)
        return NULL;
    for (int g = 0; g < l->G; ++g) {
#pragma omp parallel for schedule(static)
        for (int64_t r = l->off[g]; r < l->off[g + 1]; ++r)
            for (int64_t c = 0; c < l->cols; ++c)
                out[r * l->cols + c] = colwise ? mx_col_elem(l, data, scale, g, r, c)
                                               : mx_row_elem(l, data, scale, g, r, c);
    }
    return out;
}

static double* deq_ch(const layout_t* l, const uint8_t* data, const float* scale)
{
    int64_t L = l->off[l->G];
    double* out = malloc(sizeof(double) * (size_t)(L > 0 ? L : 1) * (size_t)l->cols);
    if (!out)
        return NULL;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < L; ++r)
        for (int64_t c = 0; c < l->cols; ++c)
            out[r * l->cols + c] = ch_col_elem(l, data, scale, r, c);
    return out;
}

/* ------------------------------------------------------------------------ */
/* Grouped GEMMs (fp64 on dequantised operands)                              */
/* ------------------------------------------------------------------------ */

/* fprop: Y[o_g + r, n] = sum_k X[o_g + r, k] * W_g[n, k].
 * x: rowwise MX [rows_cap, K] split by `splits`; w: rowwise MX [G*N, K] split
 * uniformly into G blocks of N rows.  Rows of y past the live total are not
 * written. */
int or_gemm_fprop(const uint8_t* x_data, const uint8_t* x_scale, const uint8_t* w_data,
                  const uint8_t* w_scale, const int32_t* splits, int G, int64_t rows_cap,
                  int64_t N, int64_t K, double* y)
{
    scan_t sx, sw;
    double *X, *W;
    int st = make_layout(&sx, splits, G, rows_cap, K, OR_RECIPE_MX);
    if (st != OR_OK)
        return st;
    st = make_layout(&sw, NULL, G, (int64_t)G * N, K, OR_RECIPE_MX);
    if (st != OR_OK) {
        free(sx.buf);
        return st;
    }
    X = deq_mx(&sx.l, x_data, x_scale, 0);
    W = deq_mx(&sw.l, w_data, w_scale, 0);
    for (int g = 0; g < G; ++g) {
#pragma omp parallel for schedule(static)
        for (int64_t r = sx.l.off[g]; r < sx.l.off[g + 1]; ++r)
            for (int64_t n = 0; n < N; ++n) {
                double acc = 0.0;
                const double* xr = X + r * K;
                const double* wr = W + ((int64_t)g * N + n) * K;
                for (int64_t k = 0; k < K; ++k)
                    acc += xr[k] * wr[k];
                y[r * N + n] = acc;
            }
    }
    free(X);
    free(W);
    free(sx.buf);
    free(sw.buf);
    return OR_OK;
}

/* dgrad: dX[o_g + r, k] = sum_n dY[o_g + r, n] * W_g[n, k].
 * dy: rowwise MX [rows_cap, N]; w: columnwise MX [G*N, K] (32-row blocks
 * along n, group-local layout with N rows per group). */
int or_gemm_dgrad(const uint8_t* dy_data, const uint8_t* dy_scale, const uint8_t* w_data,
                  const uint8_t* w_scale, const int32_t* splits, int G, int64_t rows_cap,
                  int64_t N, int64_t K, double* dx)
{
    scan_t sd, sw;
    double *D, *W;
    int st = make_layout(&sd, splits, G, rows_cap, N, OR_RECIPE_MX);
    if (st != OR_OK)
        return st;
    st = make_layout(&sw, NULL, G, (int64_t)G * N, K, OR_RECIPE_MX);
    if (st != OR_OK) {
        free(sd.buf);
        return st;
    }
    D = deq_mx(&sd.l, dy_data, dy_scale, 0);
    W = deq_mx(&sw.l, w_data, w_scale, 1);
    for (int g = 0; g < G; ++g) {
#pragma omp parallel for schedule(static)
        for (int64_t r = sd.l.off[g]; r < sd.l.off[g + 1]; ++r) {
            double* acc = calloc((size_t)K, sizeof(double));
            for (int64_t n = 0; n < N; ++n) {       /* sum over n in ascending order */
                double a = D[r * N + n];
                const double* wr = W + ((int64_t)g * N + n) * K;
                for (int64_t k = 0; k < K; ++k)
                    acc[k] += a * wr[k];
            }
            memcpy(dx + r * K, acc, sizeof(double) * (size_t)K);
            free(acc);
        }
    }
    free(D);
    free(W);
    free(sd.buf);
    free(sw.buf);
    return OR_OK;
}

/* wgrad: dW[g, n, k] = (accumulate ? dW[g, n, k] : 0) + sum_{r < m_g} dY[o_g + r, n] * X[o_g + r, k]
 * over the group's live rows only.  recipe selects MX columnwise operands
 * (uint8 E8M0 scales) or per-channel operands (fp32 scales). */
static int wgrad_common(const uint8_t* dy_data, const void* dy_scale, const uint8_t* x_data,
                        const void* x_scale, const int32_t* splits, int G, int64_t rows_cap,
                        int64_t N, int64_t K, int accumulate, double* dw, int recipe)
{
    scan_t sd, sx;
    double *D, *X;
    int st = make_layout(&sd, splits, G, rows_cap, N, recipe);
    if (st != OR_OK)
        return st;
    st = make_layout(&sx, splits, G, rows_cap, K, recipe);
    if (st != OR_OK) {
        free(sd.buf);
        return st;
    }
    if (recipe == OR_RECIPE_MX) {
        D = deq_mx(&sd.l, dy_data, (const uint8_t*)dy_scale, 1);
        X = deq_mx(&sx.l, x_data, (const uint8_t*)x_scale, 1);
    } else {
        D = deq_ch(&sd.l, dy_data, (const float*)dy_scale);
        X = deq_ch(&sx.l, x_data, (const float*)x_scale);
    }
    for (int g = 0; g < G; ++g) {
        int64_t o = sd.l.off[g], m = sd.l.off[g + 1] - o;
#pragma omp parallel for schedule(static)
        for (int64_t n = 0; n < N; ++n) {
            double* out = dw + ((int64_t)g * N + n) * K;
            double* acc = calloc((size_t)K, sizeof(double));
            for (int64_t r = 0; r < m; ++r) {       /* live rows only, ascending */
                double a = D[(o + r) * N + n];
                const double* xr = X + (o + r) * K;
                for (int64_t k = 0; k < K; ++k)
                    acc[k] += a * xr[k];
            }
            for (int64_t k = 0; k < K; ++k)
                out[k] = accumulate ? out[k] + acc[k] : acc[k];
            free(acc);
        }
    }
    free(D);
    free(X);
    free(sd.buf);
    free(sx.buf);
    return OR_OK;
}

int or_gemm_wgrad_mx(const uint8_t* dy_data, const uint8_t* dy_scale, const uint8_t* x_data,
                     const uint8_t* x_scale, const int32_t* splits, int G, int64_t rows_cap,
                     int64_t N, int64_t K, int accumulate, double* dw)
{
    return wgrad_common(dy_data, dy_scale, x_data, x_scale, splits, G, rows_cap, N, K,
                        accumulate, dw, OR_RECIPE_MX);
}

int or_gemm_wgrad_channel(const uint8_t* dy_data, const float* dy_scale, const uint8_t* x_data,
                          const float* x_scale, const int32_t* splits, int G, int64_t rows_cap,
                          int64_t N, int64_t K, int accumulate, double* dw)
{
    return wgrad_common(dy_data, dy_scale, x_data, x_scale, splits, G, rows_cap, N, K,
                        accumulate, dw, OR_RECIPE_CHANNEL);
}

/* ------------------------------------------------------------------------ */
/* Sampled outputs (for full-size workloads): one dot product per sample     */
/* ------------------------------------------------------------------------ */

/* kind: 0 fprop (i = row, j = n), 1 dgrad (i = row, j = k),
 *       2 wgrad MX (g, i = n, j = k), 3 wgrad per-channel (g, i = n, j = k).
 * For fprop/dgrad `g_idx` is ignored (the group follows from the row). */
int or_gemm_sample(int kind, const uint8_t* a_data, const void* a_scale, const uint8_t* b_data,
                   const void* b_scale, const int32_t* splits, int G, int64_t rows_cap,
                   int64_t N, int64_t K, int64_t n_samples, const int32_t* g_idx,
                   const int64_t* i_idx, const int64_t* j_idx, double* out)
{
    scan_t sa, sb;
    int recipe = (kind == 3) ? OR_RECIPE_CHANNEL : OR_RECIPE_MX;
    int64_t a_cols = (kind == 0) ? K : N;
    int st = make_layout(&sa, splits, G, rows_cap, a_cols, recipe);
    if (st != OR_OK)
        return st;
    if (kind <= 1)
        st = make_layout(&sb, NULL, G, (int64_t)G * N, K, OR_RECIPE_MX);
    else
        st = make_layout(&sb, splits, G, rows_cap, K, recipe);
    if (st != OR_OK) {
        free(sa.buf);
        return st;
    }
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t s = 0; s < n_samples; ++s) {
        double acc = 0.0;
        int64_t i = i_idx[s], j = j_idx[s];
        if (kind == 0) {
            int g = group_of_row(&sa.l, i);
            for (int64_t k = 0; k < K; ++k)
                acc += mx_row_elem(&sa.l, a_data, a_scale, g, i, k) *
                       mx_row_elem(&sb.l, b_data, b_scale, g, (int64_t)g * N + j, k);
        } else if (kind == 1) {
            int g = group_of_row(&sa.l, i);
            for (int64_t n = 0; n < N; ++n)
                acc += mx_row_elem(&sa.l, a_data, a_scale, g, i, n) *
                       mx_col_elem(&sb.l, b_data, b_scale, g, (int64_t)g * N + n, j);
        } else {
            int g = g_idx[s];
            for (int64_t r = sa.l.off[g]; r < sa.l.off[g + 1]; ++r) {
                if (kind == 2)
                    acc += mx_col_elem(&sa.l, a_data, a_scale, g, r, i) *
                           mx_col_elem(&sb.l, b_data, b_scale, g, r, j);
                else
                    acc += ch_col_elem(&sa.l, a_data, a_scale, r, i) *
                           ch_col_elem(&sb.l, b_data, b_scale, r, j);
            }
        }
        out[s] = acc;
    }
    free(sa.buf);
    free(sb.buf);
    return OR_OK;
}

/* ------------------------------------------------------------------------ */
/* Grouped bias add and bias gradient                                        */
/* ------------------------------------------------------------------------ */

/* Bias add: y[o_g + r, n] += bias[g, n] for every live row r of group g --
 * the grouped bias add that follows the grouped GEMM in TransformerEngine
 * PR 3224's forward sequence (launch_grouped_bias_add), which returns
 * before touching any data when the token total is 0.  Rows past the live
 * total are not touched.  MX split alignment (multiples of 32). */
int or_grouped_bias_add(double* y, const double* bias, const int32_t* splits, int G, int64_t rows_cap,
                        int64_t N)
{
    int64_t off[1025], tp[1025], sb[1025];
    if (G < 1 || G > 1024 || N <= 0)
        return OR_ERR_INVALID_ARG;
    int st = or_split_scan(splits, G, rows_cap, N, OR_RECIPE_MX, off, tp, sb);
    if (st != OR_OK)
        return st;
    if (off[G] == 0)
        return OR_OK;
    for (int g = 0; g < G; ++g)
        for (int64_t r = off[g]; r < off[g + 1]; ++r)
            for (int64_t n = 0; n < N; ++n)
                y[r * N + n] += bias[(int64_t)g * N + n];
    return OR_OK;
}

/* Bias gradient: db[g, c] = sum of dy[r, c] over the live rows r of group g,
 * in fp64 on the bf16 values -- the per-group dbiases that the grouped
 * linear's backward returns beside dinput and dweights (TransformerEngine
 * PR 3224, sequence diagram).  An empty group gets 0. */
int or_grouped_bias_grad(const uint16_t* dy, const int32_t* splits, int G, int64_t rows_cap, int64_t C,
                         double* db)
{
    int64_t off[1025], tp[1025], sb[1025];
    if (G < 1 || G > 1024 || C <= 0)
        return OR_ERR_INVALID_ARG;
    int st = or_split_scan(splits, G, rows_cap, C, OR_RECIPE_MX, off, tp, sb);
    if (st != OR_OK)
        return st;
    for (int g = 0; g < G; ++g)
        for (int64_t c = 0; c < C; ++c) {
            double acc = 0.0;
            for (int64_t r = off[g]; r < off[g + 1]; ++r)
                acc += bf16_value(dy[r * C + c]);
            db[(int64_t)g * C + c] = acc;
        }
    return OR_OK;
}

/* ------------------------------------------------------------------------ */
/* ScaledSReLU + MXFP8 quantisation of an fp32 activation                    */
/* ------------------------------------------------------------------------ */

/* MXFP8 1x32 quantisation of an fp32 [L, cols] array `a` (the live rows of
 * a grouped buffer), rowwise and columnwise, with the scale rule, codes and
 * swizzled layout of or_quantize_mx; the scale regions are zeroed first. */
static void mx_quantize_f32(const float* a, int64_t cols, const int64_t* off, const int64_t* tp,
                            const int64_t* sb, int G, uint8_t* row_data, uint8_t* row_scale,
                            uint8_t* col_data, uint8_t* col_scale)
{
    memset(row_scale, 0, (size_t)sb[G]);
    memset(col_scale, 0, (size_t)sb[G]);
    for (int g = 0; g < G; ++g) {
        int64_t o = off[g], m = off[g + 1] - off[g], T = tp[g + 1] - tp[g];
#pragma omp parallel for schedule(static)
        for (int64_t lr = 0; lr < m; ++lr) {
            int64_t r = o + lr;
            for (int64_t j = 0; j < cols / 32; ++j) {
                double amax = 0.0;
                int e;
                for (int64_t c = 32 * j; c < 32 * j + 32; ++c)
                    if (fabs((double)a[r * cols + c]) > amax)
                        amax = fabs((double)a[r * cols + c]);
                e = or_mx_scale_exponent(amax);
                for (int64_t c = 32 * j; c < 32 * j + 32; ++c)
                    row_data[r * cols + c] = or_e4m3_encode(ldexp((double)a[r * cols + c], -e));
                row_scale[sb[g] + ((lr / 128) * (cols / 128) + j / 4) * 512 + atom_byte(lr % 128, j % 4)] =
                    (uint8_t)(e + 127);
            }
        }
#pragma omp parallel for schedule(static)
        for (int64_t c = 0; c < cols; ++c) {
            for (int64_t b = 0; b < m / 32; ++b) {
                double amax = 0.0;
                int e;
                for (int64_t lr = 32 * b; lr < 32 * b + 32; ++lr)
                    if (fabs((double)a[(o + lr) * cols + c]) > amax)
                        amax = fabs((double)a[(o + lr) * cols + c]);
                e = or_mx_scale_exponent(amax);
                for (int64_t lr = 32 * b; lr < 32 * b + 32; ++lr)
                    col_data[(o + lr) * cols + c] = or_e4m3_encode(ldexp((double)a[(o + lr) * cols + c], -e));
                col_scale[sb[g] + ((c / 128) * T + b / 4) * 512 + atom_byte(c % 128, b % 4)] = (uint8_t)(e + 127);
            }
        }
    }
}


/* a = probs[r] * relu(y)^2 in fp32, op by op: t = max(y, 0); t = t * t;
 * a = t * probs[r] (the ScaledSReLU between fc1 and fc2 in TransformerEngine
 * issue 3484's reproducer, te.ops.ScaledSReLU, fed with per-token probs;
 * the pages name it without printing its arithmetic: squared ReLU scaled by
 * the row's prob is the plain reading).  Then MXFP8 1x32 quantisation of the
 * fp32 values, rowwise and columnwise, with the same scale rule, codes and
 * swizzled scale layout as or_quantize_mx.  Rows past the live total are
 * neither read nor written. */
int or_srelu_quantize_mx(const float* y, const float* probs, int64_t rows_cap, int64_t cols,
                         const int32_t* splits, int G, uint8_t* row_data, uint8_t* row_scale,
                         int64_t row_scale_bytes, uint8_t* col_data, uint8_t* col_scale,
                         int64_t col_scale_bytes)
{
    int64_t *off = malloc(sizeof(int64_t) * (G + 1) * 3);
    int64_t *tp, *sb, L;
    float* a;
    int st;
    if (!off)
        return OR_ERR_INVALID_ARG;
    tp = off + (G + 1);
    sb = off + 2 * (G + 1);
    st = or_split_scan(splits, G, rows_cap, cols, OR_RECIPE_MX, off, tp, sb);
    if (st != OR_OK) {
        free(off);
        return st;
    }
    if (sb[G] > row_scale_bytes || sb[G] > col_scale_bytes) {
        free(off);
        return OR_ERR_INVALID_ARG;
    }
    L = off[G];
    a = malloc(sizeof(float) * (size_t)(L > 0 ? L * cols : 1));
    if (!a) {
        free(off);
        return OR_ERR_INVALID_ARG;
    }
    for (int64_t r = 0; r < L; ++r)
        for (int64_t c = 0; c < cols; ++c) {
            float t = y[r * cols + c];
            t = t > 0.0f ? t : 0.0f;
            t = t * t;
            a[r * cols + c] = t * probs[r];
        }
    mx_quantize_f32(a, cols, off, tp, sb, G, row_data, row_scale, col_data, col_scale);
    free(a);
    free(off);
    return OR_OK;
}

/* ------------------------------------------------------------------------ */
/* NVFP4: E2M1 codes, 16-element blocks with E4M3 scales, and one fp32       */
/* second-level scale per group                                              */
/* ------------------------------------------------------------------------ */
/*
 * TransformerEngine PR 3224 names NVFP4 as a second quantiser on the same
 * grouped code paths (its NVFP4 note beside the MXFP8 changes) without
 * defining it.  Reading taken: the public NVFP4 format.
 *  - Codes are FP4 E2M1 (values +-{0, 0.5, 1, 1.5, 2, 3, 4, 6}); conversion
 *    rounds to nearest, ties to even, saturates to +-6, and a value that
 *    rounds to zero keeps its sign.  Two codes per byte, the element with the
 *    even index in the low nibble.
 *  - Group g's second-level scale, fp32: S_g = 2688 / amax_g (2688 = 448 * 6,
 *    the largest E4M3 scale times the largest E2M1 magnitude), S_g = 1 when
 *    amax_g == 0, clamped to FLT_MAX; amax_g is the largest |x| over the
 *    group's live rows.
 *  - Each block of 16 consecutive elements along the contraction axis, in
 *    fp32 op by op: s = (amax_b / 6) * S_g; its E4M3 byte sf = e4m3(s)
 *    (nearest-even, saturating); m = S_g / sf (0 when sf == 0, clamped to
 *    FLT_MAX); codes = e2m1(x * m).  The value a code stands for is
 *    e2m1(code) * sf / S_g.
 *  - Rowwise codes [rows_cap, cols/2] (blocks along a row); columnwise codes
 *    are stored transposed, [cols, rows_cap/2] (blocks of 16 rows, the
 *    column's codes contiguous), so that every GEMM operand is K-major.
 *  - Scale bytes use the 512-byte [32][4][4] atom of the MX layout with 16
 *    elements per scale, so an atom covers 128 rows (channels) x 64
 *    elements.  Group g's region starts at byte 512 * (cols/64) * (T_0 + ...
 *    + T_{g-1}), T_h = ceil(m_h / 128), for both orientations.  Rowwise
 *    atoms are ordered [128-row tile][64-column block]; columnwise atoms
 *    [128-column tile][64-row block], the group's 2 T_g row blocks the inner
 *    stride.  Entries that cover no live row are 0.
 */
static const double e2m1_magnitudes[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

/* Value of an E2M1 nibble: sign bit 3, then the magnitude index 0..7. */
double or_e2m1_decode(uint8_t code)
{
    double v = e2m1_magnitudes[code & 7];
    return (code & 8) ? -v : v;
}

/* Nearest E2M1 code to v (ties to the even magnitude index), saturating. */
uint8_t or_e2m1_encode(double v)
{
    uint8_t sign = signbit(v) ? 8 : 0;
    double a = fabs(v), quantum, q, n, r;
    if (isnan(v))
        return 7;
    if (a >= 6.0)
        return sign | 7;
    /* spacing of the codes around a: 0.5 below 2, 1 in [2, 4), 2 in [4, 6] */
    quantum = a < 2.0 ? 0.5 : (a < 4.0 ? 1.0 : 2.0);
    q = a / quantum;                 /* exact: quantum is a power of two */
    n = floor(q);
    if (q - n > 0.5 || (q - n == 0.5 && fmod(n, 2.0) != 0.0))
        n += 1.0;
    r = n * quantum;
    for (int c = 0; c < 8; ++c)
        if (e2m1_magnitudes[c] == r)
            return sign | (uint8_t)c;
    return sign | 7;
}

/* Second-level scale S_g of a group from its amax. */
float or_nv_global_scale(float amax)
{
    volatile float s;
    if (amax == 0.0f)
        return 1.0f;
    s = 2688.0f / amax;
    return s > FLT_MAX ? FLT_MAX : s;
}

/* One block of 16 elements x[0], x[stride], ...: its scale byte, and codes. */
static uint8_t nv_block(const uint16_t* x, int64_t stride, float S, uint8_t* codes)
{
    float amax = 0.0f, m = 0.0f;
    volatile float s;
    uint8_t sf;
    for (int i = 0; i < 16; ++i) {
        float a = fabsf(bf16_value_f32(x[i * stride]));
        if (a > amax)
            amax = a;
    }
    s = amax / 6.0f;
    s = s * S;
    sf = or_e4m3_encode((double)s);
    if (sf != 0) {
        volatile float mm = S / (float)or_e4m3_decode(sf);
        m = mm > FLT_MAX ? FLT_MAX : mm;
    }
    for (int i = 0; i < 16; ++i) {
        volatile float q = bf16_value_f32(x[i * stride]) * m;     /* one fp32 rounding */
        codes[i] = or_e2m1_encode((double)q);
    }
    return sf;
}

static void put_nibble(uint8_t* base, int64_t i, uint8_t code)
{
    if (i % 2 == 0)
        base[i / 2] = (uint8_t)((base[i / 2] & 0xF0) | (code & 0x0F));
    else
        base[i / 2] = (uint8_t)((base[i / 2] & 0x0F) | (uint8_t)(code << 4));
}

static uint8_t get_nibble(const uint8_t* base, int64_t i)
{
    return (uint8_t)((i % 2 == 0) ? (base[i / 2] & 0x0F) : (base[i / 2] >> 4));
}

/* Byte offset of group g's NVFP4 scale region for a buffer of `cols` columns. */
static int64_t nv_region(int64_t cols, int64_t tile_prefix) { return 512 * (cols / 64) * tile_prefix; }

int or_quantize_nvfp4(const uint16_t* x, int64_t rows_cap, int64_t cols, const int32_t* splits, int G,
                      int rowwise, int colwise, uint8_t* row_data, uint8_t* row_scale, int64_t row_scale_bytes,
                      uint8_t* col_data, uint8_t* col_scale, int64_t col_scale_bytes, float* amax_out)
{
    int64_t *off = malloc(sizeof(int64_t) * (G + 1) * 3);
    int64_t *tp, end;
    int st;
    if (!off)
        return OR_ERR_INVALID_ARG;
    tp = off + (G + 1);
    st = or_split_scan(splits, G, rows_cap, cols, OR_RECIPE_MX, off, tp, off + 2 * (G + 1));
    if (st != OR_OK || (!rowwise && !colwise)) {
        free(off);
        return st != OR_OK ? st : OR_ERR_INVALID_ARG;
    }
    end = nv_region(cols, tp[G]);
    if ((rowwise && end > row_scale_bytes) || (colwise && end > col_scale_bytes)) {
        free(off);
        return OR_ERR_INVALID_ARG;
    }
    if (colwise && rows_cap % 2 != 0) {
        free(off);
        return OR_ERR_ALIGNMENT;
    }
    if (rowwise)
        memset(row_scale, 0, (size_t)end);
    if (colwise)
        memset(col_scale, 0, (size_t)end);

    for (int g = 0; g < G; ++g) {
        int64_t o = off[g], m = off[g + 1] - off[g], T = tp[g + 1] - tp[g];
        int64_t sb = nv_region(cols, tp[g]);
        float amax = 0.0f, S;
        for (int64_t r = o; r < o + m; ++r)
            for (int64_t c = 0; c < cols; ++c) {
                float a = fabsf(bf16_value_f32(x[r * cols + c]));
                if (a > amax)
                    amax = a;
            }
        amax_out[g] = amax;
        S = or_nv_global_scale(amax);
        if (rowwise) {
#pragma omp parallel for schedule(static)
            for (int64_t lr = 0; lr < m; ++lr) {
                int64_t r = o + lr;
                uint8_t codes[16];
                for (int64_t j = 0; j < cols / 16; ++j) {
                    uint8_t sf = nv_block(x + r * cols + 16 * j, 1, S, codes);
                    for (int i = 0; i < 16; ++i)
                        put_nibble(row_data + r * (cols / 2), 16 * j + i, codes[i]);
                    row_scale[sb + ((lr / 128) * (cols / 64) + j / 4) * 512 + atom_byte(lr % 128, j % 4)] = sf;
                }
            }
        }
        if (colwise) {
#pragma omp parallel for schedule(static)
            for (int64_t c = 0; c < cols; ++c) {
                uint8_t codes[16];
                for (int64_t b = 0; b < m / 16; ++b) {
                    uint8_t sf = nv_block(x + (o + 16 * b) * cols + c, cols, S, codes);
                    for (int i = 0; i < 16; ++i)
                        put_nibble(col_data + c * (rows_cap / 2), o + 16 * b + i, codes[i]);
                    col_scale[sb + ((c / 128) * 2 * T + b / 4) * 512 + atom_byte(c % 128, b % 4)] = sf;
                }
            }
        }
    }
    free(off);
    return OR_OK;
}

/* NVFP4 element (r, c) of the [rows, cols] operand (group g), from rowwise
 * or transposed columnwise storage. */
static double nv_elem(const layout_t* l, int64_t rows_cap, const uint8_t* data, const uint8_t* scale,
                      const float* amax, int colwise, int g, int64_t r, int64_t c)
{
    int64_t lr = r - l->off[g], T = l->tp[g + 1] - l->tp[g];
    int64_t sb = nv_region(l->cols, l->tp[g]);
    uint8_t code, sf;
    if (!colwise) {
        int64_t j = c / 16;
        code = get_nibble(data + r * (l->cols / 2), c);
        sf = scale[sb + ((lr / 128) * (l->cols / 64) + j / 4) * 512 + atom_byte(lr % 128, j % 4)];
    } else {
        int64_t b = lr / 16;
        code = get_nibble(data + c * (rows_cap / 2), r);
        sf = scale[sb + ((c / 128) * 2 * T + b / 4) * 512 + atom_byte(c % 128, b % 4)];
    }
    return or_e2m1_decode(code) * or_e4m3_decode(sf) / (double)or_nv_global_scale(amax[g]);
}

/* Rows [0, L) of an NVFP4 operand as a dense fp64 [L, cols] array. */
static double* deq_nv(const layout_t* l, int64_t rows_cap, const uint8_t* data, const uint8_t* scale,
                      const float* amax, int colwise)
{
    int64_t L = l->off[l->G];
    double* out = malloc(sizeof(double) * (size_t)(L > 0 ? L : 1) * (size_t)l->cols);
    if (!out)
        return NULL;
    for (int g = 0; g < l->G; ++g) {
#pragma omp parallel for schedule(static)
        for (int64_t r = l->off[g]; r < l->off[g + 1]; ++r)
            for (int64_t c = 0; c < l->cols; ++c)
                out[r * l->cols + c] = nv_elem(l, rows_cap, data, scale, amax, colwise, g, r, c);
    }
    return out;
}

/* Grouped GEMMs on NVFP4 operands, fp64 on the dequantised values:
 *  kind 0 fprop: a = X rowwise [rows_cap, K], b = W rowwise [G*N, K];
 *                y[o_g + r, n] = sum_k X[o_g + r, k] W_g[n, k]
 *  kind 1 dgrad: a = dY rowwise [rows_cap, N], b = W columnwise (stored [K, G*N/2]);
 *                y[o_g + r, k] = sum_n dY[o_g + r, n] W_g[n, k]
 *  kind 2 wgrad: a = dY columnwise (stored [N, rows_cap/2]), b = X columnwise
 *                (stored [K, rows_cap/2]); y[g, n, k] = (accumulate ? y : 0)
 *                + sum over the live rows r of group g of dY[o_g + r, n] X[o_g + r, k]
 * a_amax / b_amax: the operands' per-group amax (weights: one per expert). */
int or_gemm_nvfp4(int kind, const uint8_t* a_data, const uint8_t* a_scale, const float* a_amax,
                  const uint8_t* b_data, const uint8_t* b_scale, const float* b_amax, const int32_t* splits,
                  int G, int64_t rows_cap, int64_t N, int64_t K, int accumulate, double* y)
{
    scan_t sa, sb;
    double *A, *B;
    int64_t wrows = (int64_t)G * N;
    int st;
    if (kind < 0 || kind > 2)
        return OR_ERR_INVALID_ARG;
    st = make_layout(&sa, splits, G, rows_cap, kind == 0 ? K : N, OR_RECIPE_MX);
    if (st != OR_OK)
        return st;
    if (kind == 2)
        st = make_layout(&sb, splits, G, rows_cap, K, OR_RECIPE_MX);
    else
        st = make_layout(&sb, NULL, G, wrows, K, OR_RECIPE_MX);
    if (st != OR_OK) {
        free(sa.buf);
        return st;
    }
    A = deq_nv(&sa.l, rows_cap, a_data, a_scale, a_amax, kind == 2);
    B = deq_nv(&sb.l, kind == 2 ? rows_cap : wrows, b_data, b_scale, b_amax, kind != 0);
    for (int g = 0; g < G; ++g) {
        int64_t o = sa.l.off[g], m = sa.l.off[g + 1] - o;
        if (kind == 0) {
#pragma omp parallel for schedule(static)
            for (int64_t r = o; r < o + m; ++r)
                for (int64_t n = 0; n < N; ++n) {
                    double acc = 0.0;
                    for (int64_t k = 0; k < K; ++k)
                        acc += A[r * K + k] * B[((int64_t)g * N + n) * K + k];
                    y[r * N + n] = acc;
                }
        } else if (kind == 1) {
#pragma omp parallel for schedule(static)
            for (int64_t r = o; r < o + m; ++r)
                for (int64_t k = 0; k < K; ++k) {
                    double acc = 0.0;
                    for (int64_t n = 0; n < N; ++n)
                        acc += A[r * N + n] * B[((int64_t)g * N + n) * K + k];
                    y[r * K + k] = acc;
                }
        } else {
#pragma omp parallel for schedule(static)
            for (int64_t n = 0; n < N; ++n)
                for (int64_t k = 0; k < K; ++k) {
                    double acc = 0.0;
                    for (int64_t r = o; r < o + m; ++r)
                        acc += A[r * N + n] * B[r * K + k];
                    y[((int64_t)g * N + n) * K + k] = accumulate ? y[((int64_t)g * N + n) * K + k] + acc : acc;
                }
        }
    }
    free(A);
    free(B);
    free(sa.buf);
    free(sb.buf);
    return OR_OK;
}

/* Sampled outputs of the NVFP4 GEMMs, one fp64 dot product each (kind and
 * operands as or_gemm_nvfp4; fprop (i = row, j = n), dgrad (i = row, j = k),
 * wgrad (g, i = n, j = k) without any accumulate term). */
int or_gemm_nvfp4_sample(int kind, const uint8_t* a_data, const uint8_t* a_scale, const float* a_amax,
                         const uint8_t* b_data, const uint8_t* b_scale, const float* b_amax, const int32_t* splits,
                         int G, int64_t rows_cap, int64_t N, int64_t K, int64_t n_samples, const int32_t* g_idx,
                         const int64_t* i_idx, const int64_t* j_idx, double* out)
{
    scan_t sa, sb;
    int64_t wrows = (int64_t)G * N;
    int st;
    if (kind < 0 || kind > 2)
        return OR_ERR_INVALID_ARG;
    st = make_layout(&sa, splits, G, rows_cap, kind == 0 ? K : N, OR_RECIPE_MX);
    if (st != OR_OK)
        return st;
    if (kind == 2)
        st = make_layout(&sb, splits, G, rows_cap, K, OR_RECIPE_MX);
    else
        st = make_layout(&sb, NULL, G, wrows, K, OR_RECIPE_MX);
    if (st != OR_OK) {
        free(sa.buf);
        return st;
    }
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t s = 0; s < n_samples; ++s) {
        double acc = 0.0;
        int64_t i = i_idx[s], j = j_idx[s];
        if (kind == 0) {
            int g = group_of_row(&sa.l, i);
            for (int64_t k = 0; k < K; ++k)
                acc += nv_elem(&sa.l, rows_cap, a_data, a_scale, a_amax, 0, g, i, k) *
                       nv_elem(&sb.l, wrows, b_data, b_scale, b_amax, 0, g, (int64_t)g * N + j, k);
        } else if (kind == 1) {
            int g = group_of_row(&sa.l, i);
            for (int64_t n = 0; n < N; ++n)
                acc += nv_elem(&sa.l, rows_cap, a_data, a_scale, a_amax, 0, g, i, n) *
                       nv_elem(&sb.l, wrows, b_data, b_scale, b_amax, 1, g, (int64_t)g * N + n, j);
        } else {
            int g = g_idx[s];
            for (int64_t r = sa.l.off[g]; r < sa.l.off[g + 1]; ++r)
                acc += nv_elem(&sa.l, rows_cap, a_data, a_scale, a_amax, 1, g, r, i) *
                       nv_elem(&sb.l, rows_cap, b_data, b_scale, b_amax, 1, g, r, j);
        }
        out[s] = acc;
    }
    free(sa.buf);
    free(sb.buf);
    return OR_OK;
}

/* ------------------------------------------------------------------------ */
/* ScaledSwiGLU + MXFP8 quantisation of an fp32 activation                   */
/* ------------------------------------------------------------------------ */
/*
 * TransformerEngine issue 3484 names ScaledSwiGLU (with ScaledClampedQGeGLU
 * and ScaledSiTUGLU) beside ScaledSReLU without defining it.  Reading taken:
 * the SwiGLU of Shazeer's "GLU Variants Improve Transformer", scaled by the
 * row's prob: the fc1 output of width 2n is split into a gate half
 * y[:, 0:n] and a linear half y[:, n:2n], and
 *     a[r, c] = (silu(y[r, c]) * y[r, n + c]) * probs[r],
 *     silu(x) = x / (1 + exp(-x)),
 * in fp32 op by op.  exp is this library's own: the argument is clamped to
 * [-87, 88] (outside it 1 + exp(-x) is 1, or the quotient is below 1e-36),
 * reduced by ln 2 in the Cody-Waite way (n = rint(x log2 e), r = x - n ln2_hi
 * - n ln2_lo with fused multiply-adds, ln2_hi holding 16 bits so n ln2_hi is
 * exact), the degree-7 Taylor polynomial of exp(r) is evaluated in Horner
 * form with fused multiply-adds, and the result is scaled by 2^n exactly.
 * Every step is one correctly rounded fp32 operation, so any two faithful
 * implementations give the same bits.
 */
float or_act_exp(float x)
{
    volatile float t, n, r, p;
    int32_t ni;
    uint32_t bits;
    float two_n;
    if (x < -87.0f)
        x = -87.0f;
    if (x > 88.0f)
        x = 88.0f;
    t = x * 0x1.715476p+0f;                    /* x * log2(e), rounded */
    n = rintf(t);
    r = fmaf(n, -0x1.62e4p-1f, x);             /* - n * ln2_hi */
    r = fmaf(n, -0x1.7f7d1cp-20f, r);          /* - n * ln2_lo */
    p = 0x1.a01a02p-13f;                       /* 1/7! */
    p = fmaf(p, r, 0x1.6c16c2p-10f);           /* 1/6! */
    p = fmaf(p, r, 0x1.111112p-7f);            /* 1/5! */
    p = fmaf(p, r, 0x1.555556p-5f);            /* 1/4! */
    p = fmaf(p, r, 0x1.555556p-3f);            /* 1/3! */
    p = fmaf(p, r, 0.5f);
    p = fmaf(p, r, 1.0f);
    p = fmaf(p, r, 1.0f);
    ni = (int32_t)n;
    bits = (uint32_t)(ni + 127) << 23;         /* 2^n, n in [-126, 127] */
    memcpy(&two_n, &bits, sizeof two_n);
    return p * two_n;
}

/* silu(x) = x / (1 + exp(-x)), fp32 op by op. */
float or_act_silu(float x)
{
    volatile float d = 1.0f + or_act_exp(-x);
    return x / d;
}

/* y: fp32 [rows_cap, 2 * cols] (gate half, then linear half); the activation
 * [rows_cap, cols] is MX-quantised rowwise and columnwise like
 * or_quantize_mx.  Rows past the live total are neither read nor written. */
int or_swiglu_quantize_mx(const float* y, const float* probs, int64_t rows_cap, int64_t cols,
                          const int32_t* splits, int G, uint8_t* row_data, uint8_t* row_scale,
                          int64_t row_scale_bytes, uint8_t* col_data, uint8_t* col_scale,
                          int64_t col_scale_bytes)
{
    int64_t *off = malloc(sizeof(int64_t) * (G + 1) * 3);
    int64_t *tp, *sb, L;
    float* a;
    int st;
    if (!off)
        return OR_ERR_INVALID_ARG;
    tp = off + (G + 1);
    sb = off + 2 * (G + 1);
    st = or_split_scan(splits, G, rows_cap, cols, OR_RECIPE_MX, off, tp, sb);
    if (st != OR_OK) {
        free(off);
        return st;
    }
    if (sb[G] > row_scale_bytes || sb[G] > col_scale_bytes) {
        free(off);
        return OR_ERR_INVALID_ARG;
    }
    L = off[G];
    a = malloc(sizeof(float) * (size_t)(L > 0 ? L * cols : 1));
    if (!a) {
        free(off);
        return OR_ERR_INVALID_ARG;
    }
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < L; ++r)
        for (int64_t c = 0; c < cols; ++c) {
            volatile float s = or_act_silu(y[r * 2 * cols + c]);
            volatile float t = s * y[r * 2 * cols + cols + c];
            a[r * cols + c] = t * probs[r];
        }
    mx_quantize_f32(a, cols, off, tp, sb, G, row_data, row_scale, col_data, col_scale);
    free(a);
    free(off);
    return OR_OK;
}
