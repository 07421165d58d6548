/*
 * Plain, slow, fp64 CPU oracle of the fused MLA query up-projection.
 *
 * TEST INFRASTRUCTURE. Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg load this library. It shares no code, header, table or
 * helper with the CUDA path, and the product path never calls it.
 *
 * What it computes (each function names the passage it follows):
 *   - TransformerEngine PR "Add support for fused Q Up-Proj GEMM/RoPE/Quant",
 *     description paragraph: the Q up-projection GEMM of DeepSeek-V3 training,
 *     followed by RoPE and MXFP8 quantization, with a 16-bit or an MXFP8
 *     projection (weights).
 *   - TransformerEngine PR "Add a backwards linear function to be used with the
 *     fused mla q up-proj", Greptile summary and sequence diagram: the query
 *     gradient goes through the RoPE backward (giving the pre-RoPE projection
 *     gradient), then the linear backward gives the input and weight
 *     gradients; review comment "BF16 bias gradient remains missing": the bias
 *     gradient belongs to that backward.
 *   - Megatron-LM PR "Fix fused MLA YaRN RoPE query kernel corrupting upstream
 *     tensor in-place", Problem section: the RoPE output must not overwrite its
 *     input, and a cos/sin table narrower than the rotary dim must never be
 *     read out of bounds.
 *
 * The pages print no formulas. Where they are silent the readings are:
 * rotate-half RoPE on the last Dr channels of each head (pair i, i+Dr/2);
 * column j of the cos/sin table serves rope channel j; bias added before the
 * rotation; MXFP8 = E4M3 (OCP "FN": max 448, no Inf) elements with one E8M0
 * power-of-two scale per 32 consecutive channels of a head, scale exponent
 * the smallest e with amax <= 448 * 2^e (= ceil(log2(amax/448))), elements
 * rounded to nearest-even with saturation.
 *
 * Every sum runs sequentially in index order in fp64. OpenMP splits only
 * independent outputs (rows) across threads, never one sum.
 *
 * Build: gcc -O2 -fopenmp -ffp-contract=off -fPIC -shared (no fast-math, no
 * FMA contraction, so the results are the same on x86-64 and aarch64).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_OK 0
#define ORACLE_ERR_ARG 1
#define ORACLE_ERR_ROPE_WIDTH 2
#define ORACLE_ERR_POS_RANGE 8

/* Threads the parallel loops below use (1 without OpenMP). */
int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ------------------------------------------------------------------ decode */

/* bf16 bit pattern -> exact double (bf16 is the top half of an fp32). */
double oracle_bf16_to_f64(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

void oracle_decode_bf16(int64_t n, const uint16_t *in, double *out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_bf16_to_f64(in[i]);
}

/* OCP E4M3 ("FN") code -> value: sign, 4-bit exponent with bias 7, 3-bit
 * mantissa; exponent field 0 holds subnormals m * 2^-9; S.1111.111 is NaN;
 * there is no infinity. */
double oracle_e4m3_decode(uint8_t code)
{
    int s = code >> 7, e = (code >> 3) & 15, m = code & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = ldexp((double)m, -9);
    else v = ldexp(1.0 + m / 8.0, e - 7);
    return s ? -v : v;
}

/* E8M0 scale byte -> 2^(byte - 127); 0xFF is NaN. */
double oracle_e8m0_decode(uint8_t byte)
{
    if (byte == 0xFF) return NAN;
    return ldexp(1.0, (int)byte - 127);
}

/* Dequantize rows of MXFP8: out[r, c] = decode(codes[r, c]) * 2^(scale[r, c/32] - 127). */
void oracle_mxfp8_dequantize(int64_t R, int64_t C, const uint8_t *codes, const uint8_t *scales,
                             double *out)
{
    int64_t nb = (C + 31) / 32;
    for (int64_t r = 0; r < R; ++r)
        for (int64_t c = 0; c < C; ++c)
            out[r * C + c] = oracle_e4m3_decode(codes[r * C + c]) *
                             oracle_e8m0_decode(scales[r * nb + c / 32]);
}

/* --------------------------------------------------------------- quantize */

/* Scale exponent of a block: the smallest integer e with amax <= 448 * 2^e,
 * clamped to [-127, 127]. Found by exact comparisons with 448 * 2^e (ldexp is
 * exact), not by a floating-point log. amax = 0 gives -127. */
int oracle_e8m0_exponent(double amax)
{
    int e;
    if (!(amax > 0.0)) return -127;
    (void)frexp(amax / 448.0, &e); /* estimate, fixed up below */
    while (e > -127 && amax <= ldexp(448.0, e - 1)) --e;
    while (e < 127 && amax > ldexp(448.0, e)) ++e;
    if (e < -127) e = -127;
    if (e > 127) e = 127;
    return e;
}

/* Round v to the nearest E4M3 value, ties to the even code, saturating to
 * +-448; NaN -> S.1111.111. The grid below 2^-6 is the subnormal step 2^-9;
 * in the binade [2^E, 2^(E+1)) the step is 2^(E-3). Dividing by a power of two
 * is exact, and rint() rounds half to even in the default rounding mode. */
uint8_t oracle_e4m3_encode(double v)
{
    uint8_t sign = signbit(v) ? 0x80 : 0x00;
    double a = fabs(v), step, r;
    int E;
    if (isnan(v)) return (uint8_t)(sign | 0x7F);
    if (a >= 448.0) return (uint8_t)(sign | 0x7E);
    if (a < ldexp(1.0, -6)) {
        step = ldexp(1.0, -9);
    } else {
        (void)frexp(a, &E); /* a = f * 2^E, f in [0.5, 1) -> binade exponent E-1 */
        step = ldexp(1.0, (E - 1) - 3);
    }
    r = rint(a / step) * step;
    if (r > 448.0) r = 448.0;
    if (r == 0.0) return sign;
    if (r < ldexp(1.0, -6)) return (uint8_t)(sign | (uint8_t)(r / ldexp(1.0, -9)));
    (void)frexp(r, &E);
    E -= 1;                                                /* r in [2^E, 2^(E+1)) */
    {
        int m = (int)(ldexp(r, -E) * 8.0 - 8.0);         /* exact, 0..7 */
        return (uint8_t)(sign | ((E + 7) << 3) | m);
    }
}

/* Rowwise MXFP8 quantization of in[R, C] (row stride ld_in), blocks of 32
 * consecutive elements along a row (the last block of a row may be partial;
 * its amax covers only its valid elements). A block holding a NaN or an
 * infinity gets scale 0xFF and NaN codes that keep each element's sign.
 * codes: [R, C] dense; scales: [R, ceil(C/32)] dense. */
void oracle_mxfp8_quantize(int64_t R, int64_t C, const double *in, int64_t ld_in, uint8_t *codes,
                           uint8_t *scales)
{
    int64_t nb = (C + 31) / 32;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < R; ++r) {
        for (int64_t b = 0; b < nb; ++b) {
            int64_t c0 = b * 32, c1 = c0 + 32 < C ? c0 + 32 : C;
            double amax = 0.0;
            int nonfinite = 0;
            for (int64_t c = c0; c < c1; ++c) {
                double v = in[r * ld_in + c];
                if (!isfinite(v)) nonfinite = 1;
                else if (fabs(v) > amax) amax = fabs(v);
            }
            if (nonfinite) {
                scales[r * nb + b] = 0xFF;
                for (int64_t c = c0; c < c1; ++c)
                    codes[r * C + c] = (uint8_t)((signbit(in[r * ld_in + c]) ? 0x80 : 0) | 0x7F);
                continue;
            }
            {
                int e = oracle_e8m0_exponent(amax);
                scales[r * nb + b] = (uint8_t)(e + 127);
                for (int64_t c = c0; c < c1; ++c)
                    codes[r * C + c] = oracle_e4m3_encode(ldexp(in[r * ld_in + c], -e));
            }
        }
    }
}

/* ------------------------------------------------------------------ linear */

/* y[t, n] = sum_k x[t, k] * W[n, k]  (+ b[n]); x [T, K], W [N, K], y [T, N].
 * The query up-projection GEMM (forward), bias added after the sum. */
void oracle_linear(int64_t T, int64_t K, int64_t N, const double *x, const double *W,
                   const double *b, double *y)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t n = 0; n < N; ++n) {
            double s = 0.0;
            for (int64_t k = 0; k < K; ++k) s += x[t * K + k] * W[n * K + k];
            if (b) s += b[n];
            y[t * N + n] = s;
        }
    }
}

/* ------------------------------------------------------------------- RoPE */

static int rope_check(int64_t T, int32_t H, int32_t Dn, int32_t Dr, int64_t cs_rows,
                      int64_t cs_width, const int32_t *pos)
{
    if (T < 0 || H <= 0 || Dn < 0 || Dr <= 0 || (Dr & 1)) return ORACLE_ERR_ARG;
    if (cs_width < Dr) return ORACLE_ERR_ROPE_WIDTH; /* never read past the table row */
    for (int64_t t = 0; t < T; ++t) {
        int64_t p = pos ? pos[t] : t;
        if (p < 0 || p >= cs_rows) return ORACLE_ERR_POS_RANGE;
    }
    return ORACLE_OK;
}

/* Forward rotate-half RoPE on y [T, H, Dn+Dr] into a fresh q (never in place).
 * For each token t (position p = pos[t], or t when pos is NULL), head h and
 * i < Dr/2, with a = y[Dn+i] and c = y[Dn+i+Dr/2]:
 *   q[Dn+i]      = a * cos[p, i]      - c * sin[p, i]
 *   q[Dn+i+Dr/2] = c * cos[p, i+Dr/2] + a * sin[p, i+Dr/2]
 * and q[c] = y[c] for the first Dn channels. Returns a status. */
int oracle_rope_fwd(int64_t T, int32_t H, int32_t Dn, int32_t Dr, const double *y,
                    const float *cos_tab, const float *sin_tab, int64_t cs_rows, int64_t cs_width,
                    const int32_t *pos, double *q)
{
    int st = rope_check(T, H, Dn, Dr, cs_rows, cs_width, pos);
    int64_t D = (int64_t)Dn + Dr, hh = Dr / 2;
    if (st != ORACLE_OK) return st;
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t) {
        int64_t p = pos ? pos[t] : t;
        const float *cs = cos_tab + p * cs_width, *sn = sin_tab + p * cs_width;
        for (int64_t h = 0; h < H; ++h) {
            const double *yi = y + (t * H + h) * D;
            double *qo = q + (t * H + h) * D;
            for (int64_t c = 0; c < Dn; ++c) qo[c] = yi[c];
            for (int64_t i = 0; i < hh; ++i) {
                double a = yi[Dn + i], c = yi[Dn + i + hh];
                qo[Dn + i] = a * (double)cs[i] - c * (double)sn[i];
                qo[Dn + i + hh] = c * (double)cs[i + hh] + a * (double)sn[i + hh];
            }
        }
    }
    return ORACLE_OK;
}

/* RoPE backward: dq_pre = J^T dq, J the Jacobian of oracle_rope_fwd at the
 * same positions. With g = dq[Dn + .]:
 *   dq_pre[Dn+i]      =  g[i] * cos[p, i] + g[i+Dr/2] * sin[p, i+Dr/2]
 *   dq_pre[Dn+i+Dr/2] = -g[i] * sin[p, i] + g[i+Dr/2] * cos[p, i+Dr/2]
 * and the first Dn channels are copied. This is the exact gradient for any
 * table; it is the inverse rotation when the table has unit amplitude and
 * equal columns i and i+Dr/2. */
int oracle_rope_bwd(int64_t T, int32_t H, int32_t Dn, int32_t Dr, const double *dq,
                    const float *cos_tab, const float *sin_tab, int64_t cs_rows, int64_t cs_width,
                    const int32_t *pos, double *dq_pre)
{
    int st = rope_check(T, H, Dn, Dr, cs_rows, cs_width, pos);
    int64_t D = (int64_t)Dn + Dr, hh = Dr / 2;
    if (st != ORACLE_OK) return st;
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t) {
        int64_t p = pos ? pos[t] : t;
        const float *cs = cos_tab + p * cs_width, *sn = sin_tab + p * cs_width;
        for (int64_t h = 0; h < H; ++h) {
            const double *g = dq + (t * H + h) * D;
            double *o = dq_pre + (t * H + h) * D;
            for (int64_t c = 0; c < Dn; ++c) o[c] = g[c];
            for (int64_t i = 0; i < hh; ++i) {
                double gi = g[Dn + i], gj = g[Dn + i + hh];
                o[Dn + i] = gi * (double)cs[i] + gj * (double)sn[i + hh];
                o[Dn + i + hh] = -gi * (double)sn[i] + gj * (double)cs[i + hh];
            }
        }
    }
    return ORACLE_OK;
}

/* -------------------------------------------------------------- gradients */

/* dx[t, k] = sum_n dq_pre[t, n] * W[n, k]; dq_pre [T, N], W [N, K], dx [T, K].
 * Each dx[t, k] is summed over n in index order; the k loop is innermost only
 * so that W is read row by row. */
void oracle_dgrad(int64_t T, int64_t K, int64_t N, const double *dq_pre, const double *W,
                  double *dx)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t t = 0; t < T; ++t) {
        double *o = dx + t * K;
        for (int64_t k = 0; k < K; ++k) o[k] = 0.0;
        for (int64_t n = 0; n < N; ++n) {
            double g = dq_pre[t * N + n];
            const double *w = W + n * K;
            for (int64_t k = 0; k < K; ++k) o[k] += g * w[k];
        }
    }
}

/* dW[n, k] = sum_t dq_pre[t, n] * x[t, k]; dq_pre [T, N], x [T, K], dW [N, K].
 * Each dW[n, k] is summed over t in index order. Only the rows n listed in
 * rows[0..nrows) are computed (all rows when rows is NULL; then nrows = N);
 * output row i of dW is channel rows[i]. */
void oracle_wgrad(int64_t T, int64_t K, int64_t N, const double *dq_pre, const double *x,
                  const int64_t *rows, int64_t nrows, double *dW)
{
    if (!rows) nrows = N;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < nrows; ++i) {
        int64_t n = rows ? rows[i] : i;
        double *o = dW + i * K;
        for (int64_t k = 0; k < K; ++k) o[k] = 0.0;
        for (int64_t t = 0; t < T; ++t) {
            double g = dq_pre[t * N + n];
            const double *xr = x + t * K;
            for (int64_t k = 0; k < K; ++k) o[k] += g * xr[k];
        }
    }
}

/* db[n] = sum_t dq_pre[t, n], in index order of t. */
void oracle_bgrad(int64_t T, int64_t N, const double *dq_pre, double *db)
{
#pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; ++n) {
        double s = 0.0;
        for (int64_t t = 0; t < T; ++t) s += dq_pre[t * N + n];
        db[n] = s;
    }
}
