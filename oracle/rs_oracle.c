/*
 * Plain CPU oracle for residue-compensated block-scaled FP4 linear layers.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may call, link or
 * load this file; only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no code, header or table with the CUDA
 * library.
 *
 * Source: "ResServe: Accurate and Efficient FP4 LLM Inference with Residue
 * Compensation" (arXiv 2611.08713).
 *   - Sec. 2 (Background) and Fig. 1: NVFP4 = E2M1 elements, one E4M3 scale per
 *     16 consecutive elements plus one FP32 tensor scale; MXFP4 = E2M1
 *     elements, one E8M0 power-of-two scale per 32 consecutive elements, no
 *     tensor scale.  Sec. 2 also defines QDQ and the residue r = x - QDQ(x).
 *   - App. B.2, Eq. 8-10: block amax, s_i = Max_i / 6, alpha = max_i s_i / 448,
 *     s_i,FP8 = round_E4M3(s_i / alpha), s~_i = alpha * s_i,FP8,
 *     x_FP4 = round_E2M1(x / s~_i), x^ = s~_i * x_FP4.
 *   - App. B.2, Algorithm 1 ("Residue NVFP4 quantization: eight inputs per
 *     thread"): the quantizer receives a precomputed tensor scale, forms the
 *     block scale and an fp32 multiplier scale, quantizes, forms the residue
 *     in fp32 and quantizes the residue with its own block scales and the
 *     same tensor scale.
 *   - Sec. 4.2, Eq. 1 and Sec. 4.3, Eq. 2: Y ~ X^ W^ + R^ W^ (full
 *     compensation), computed as a stacked GEMM followed by the Fold
 *     Y_j = Z_j + Z_{M+j}.
 *
 * Readings taken where the paper leaves a step open (each one is also listed
 * in the design notes):
 *   R1  The tensor scale is an input (Alg. 1 "receives a precomputed tensor
 *       scale").  When it is computed here it is fl(amax / 2688.0f), i.e. the
 *       6 * 448 of Eq. 8 folded into one fp32 division.
 *   R2  Block scale: s = fl(Max / 6), t = fl(s / alpha) (0 when alpha == 0),
 *       sf = round-to-nearest-even onto the E4M3 grid, values above 448
 *       clamped to 448, never NaN.  s~ = fl(alpha * dec(sf)).
 *   R3  Element scaling follows Alg. 1's "fp32 multiplier scale":
 *       mul = fl(1 / s~) (0 when s~ == 0), v = fl(x * mul).
 *   R4  E2M1 rounding is round-to-nearest, ties to the even code, magnitudes
 *       above 6 saturate to 6, and the sign is kept (a negative value that
 *       rounds to zero gives code 0x8).
 *   R5  Reconstruction uses Eq. 10's product x^ = fl(s~ * dec(q)); the
 *       residue is r = fl(x - x^) in fp32.
 *   R6  MXFP4 scale (the paper only cites the OCP MX format): the shared
 *       exponent is e = floor(log2(Max)) - 2 (2 = emax of E2M1), clamped to
 *       [-127, 127]; Max == 0 gives e = -127.  Stored byte = e + 127.
 *       v = fl(x * 2^-e); x^ = dec(q) * 2^e.  The residue gets its own scale.
 *   R7  Logical layouts: codes are packed two per byte along K, element 2j in
 *       the low nibble of byte j; scale bytes are [rows][K / block].
 *   R8  The GEMM is the plain definition: every product of decoded values is
 *       exact in double and the sum is taken in double; the tensor scales
 *       multiply the double result.
 *
 * All quantizer arithmetic is IEEE fp32 (the precision Alg. 1 names) and the
 * file must be compiled with -ffp-contract=off and without fast-math.
 *
 * Parity pins live in the test suite; every function below is pinned there
 * against format facts, library casts, brute force or closed forms.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* E2M1 (Sec. 2; max magnitude 6 per App. B.2).  1 sign, 2 exponent, 1       */
/* mantissa bit, exponent bias 1, one subnormal step 0.5.                     */
/* ------------------------------------------------------------------------ */

/* Decoded magnitude of the 3-bit magnitude field: exponent field E, mantissa
 * bit m.  E == 0: m * 0.5 (subnormal).  E > 0: (1 + m/2) * 2^(E-1). */
static double e2m1_magnitude(unsigned mag3)
{
    unsigned E = (mag3 >> 1) & 3u;
    unsigned m = mag3 & 1u;
    if (E == 0)
        return 0.5 * (double)m;
    return (1.0 + 0.5 * (double)m) * ldexp(1.0, (int)E - 1);
}

double or_e2m1_decode(uint8_t code)
{
    double mag = e2m1_magnitude(code & 7u);
    return (code & 8u) ? -mag : mag;
}

/* Decoded magnitudes of the 8 magnitude codes, filled once on first use. */
static double g_e2m1_mag[8];
static int g_e2m1_ready = 0;

static void e2m1_table_init(void)
{
    if (g_e2m1_ready)
        return;
    for (unsigned c = 0; c < 8; ++c)
        g_e2m1_mag[c] = e2m1_magnitude(c);
    g_e2m1_ready = 1;
}

/* Nearest of the 8 magnitudes; a tie goes to the code whose mantissa bit is
 * 0 (the even code).  Anything above the largest magnitude saturates to it.
 * The sign bit follows the sign of v, including -0 and negative values that
 * round to zero.  Input must be finite. */
uint8_t or_e2m1_encode(float v)
{
    double a = fabs((double)v);
    unsigned best = 0;
    double best_d;
    e2m1_table_init();
    if (a > g_e2m1_mag[7])                    /* saturate above 6 */
        return (uint8_t)((signbit(v) ? 8u : 0u) | 7u);
    best_d = fabs(a - g_e2m1_mag[0]);
    for (unsigned c = 1; c < 8; ++c) {
        double d = fabs(a - g_e2m1_mag[c]);
        if (d < best_d || (d == best_d && (c & 1u) == 0 && (best & 1u) == 1)) {
            best = c;
            best_d = d;
        }
    }
    return (uint8_t)((signbit(v) ? 8u : 0u) | best);
}

/* ------------------------------------------------------------------------ */
/* E4M3 (OCP FP8 "fn" variant: bias 7, no infinities, 0x7F / 0xFF are NaN,  */
/* max finite 448 as App. B.2 states).                                        */
/* ------------------------------------------------------------------------ */

double or_e4m3_decode(uint8_t b)
{
    unsigned E = (b >> 3) & 15u;
    unsigned m = b & 7u;
    double mag;
    if (E == 15 && m == 7)
        return NAN;
    if (E == 0)
        mag = ((double)m / 8.0) * ldexp(1.0, -6);
    else
        mag = (1.0 + (double)m / 8.0) * ldexp(1.0, (int)E - 7);
    return (b & 0x80u) ? -mag : mag;
}

/* Decoded values of the 127 finite non-negative codes, filled once. */
static double g_e4m3_val[0x7F];
static int g_e4m3_ready = 0;

static void e4m3_table_init(void)
{
    if (g_e4m3_ready)
        return;
    for (unsigned c = 0; c < 0x7Fu; ++c)
        g_e4m3_val[c] = or_e4m3_decode((uint8_t)c);
    g_e4m3_ready = 1;
}

/* Round-to-nearest-even onto the finite E4M3 grid, saturating to +-448.
 * Implemented as a search over the 127 finite non-negative codes: the
 * nearest value wins, a tie goes to the code with mantissa LSB 0. */
uint8_t or_e4m3_encode_satfinite(float t)
{
    double a = fabs((double)t);
    unsigned sign = signbit(t) ? 0x80u : 0u;
    unsigned best = 0;
    double best_d;
    if (a > 448.0)
        return (uint8_t)(sign | 0x7Eu);
    e4m3_table_init();
    best_d = fabs(a - g_e4m3_val[0]);
    for (unsigned c = 1; c <= 0x7Eu; ++c) {
        double d = fabs(a - g_e4m3_val[c]);
        if (d < best_d || (d == best_d && (c & 1u) == 0 && (best & 1u) == 1)) {
            best = c;
            best_d = d;
        }
    }
    return (uint8_t)(sign | best);
}

/* E8M0: unsigned power of two 2^(b - 127); 0xFF is NaN. */
double or_e8m0_decode(uint8_t b)
{
    if (b == 0xFF)
        return NAN;
    return ldexp(1.0, (int)b - 127);
}

/* ------------------------------------------------------------------------ */
/* bf16 input (Alg. 1 line 1: on-lane bf16 -> fp32 cast, exact).             */
/* ------------------------------------------------------------------------ */

static float bf16_to_float(uint16_t h)
{
    uint32_t bits = (uint32_t)h << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return f;
}

/* Tensor scale, reading R1: alpha = fl(amax / 2688), amax over all elements. */
float or_tensor_scale(const uint16_t *x, int64_t n)
{
    float amax = 0.0f;
    for (int64_t i = 0; i < n; ++i) {
        float a = fabsf(bf16_to_float(x[i]));
        if (a > amax)
            amax = a;
    }
    return amax / 2688.0f;
}

/* ------------------------------------------------------------------------ */
/* One NVFP4 block (App. B.2, Eq. 8-10; Alg. 1 lines 2-6).                    */
/* ------------------------------------------------------------------------ */

static void nvfp4_block(const float *xf, int n, float alpha,
                        uint8_t *sf_out, uint8_t *codes, float *xhat)
{
    float amax = 0.0f, s, t, st, mul;
    uint8_t sf;
    for (int i = 0; i < n; ++i)
        if (fabsf(xf[i]) > amax)
            amax = fabsf(xf[i]);
    s = amax / 6.0f;                          /* Eq. 8: s_i = Max_i / 6   */
    t = (alpha > 0.0f) ? s / alpha : 0.0f;    /* Eq. 9: s_i / alpha       */
    sf = or_e4m3_encode_satfinite(t);         /* Eq. 9: round_E4M3        */
    st = alpha * (float)or_e4m3_decode(sf);   /* Eq. 9: s~_i = alpha*sFP8 */
    mul = (st == 0.0f) ? 0.0f : 1.0f / st;    /* Alg. 1: fp32 multiplier  */
    for (int i = 0; i < n; ++i) {
        float v = xf[i] * mul;                /* Eq. 10: x / s~_i         */
        uint8_t q = or_e2m1_encode(v);        /* Eq. 10: round_E2M1       */
        codes[i] = q;
        xhat[i] = st * (float)or_e2m1_decode(q); /* Eq. 10: x^ = s~ x_FP4 */
    }
    *sf_out = sf;
}

/* The same block with Eq. 10's true division v = fl(x / s~) in place of
 * Alg. 1's multiplier (the alternative to reading R3; parity is defined on
 * the multiplier).  Codes and scale byte only. */
static void nvfp4_block_div(const float *xf, int n, float alpha, uint8_t *sf_out, uint8_t *codes)
{
    float amax = 0.0f, s, t, st;
    uint8_t sf;
    for (int i = 0; i < n; ++i)
        if (fabsf(xf[i]) > amax)
            amax = fabsf(xf[i]);
    s = amax / 6.0f;
    t = (alpha > 0.0f) ? s / alpha : 0.0f;
    sf = or_e4m3_encode_satfinite(t);
    st = alpha * (float)or_e4m3_decode(sf);
    for (int i = 0; i < n; ++i)
        codes[i] = or_e2m1_encode(st == 0.0f ? 0.0f * xf[i] : xf[i] / st);   /* Eq. 10: x / s~_i */
    *sf_out = sf;
}

/* ------------------------------------------------------------------------ */
/* One MXFP4 block (Sec. 2: E8M0 power-of-two scale per 32 elements;         */
/* reading R6 for the exponent).                                              */
/* ------------------------------------------------------------------------ */

static void mxfp4_block(const float *xf, int n,
                        uint8_t *sf_out, uint8_t *codes, float *xhat)
{
    float amax = 0.0f, scale, inv;
    int e, ex;
    for (int i = 0; i < n; ++i)
        if (fabsf(xf[i]) > amax)
            amax = fabsf(xf[i]);
    if (amax == 0.0f) {
        e = -127;
    } else {
        (void)frexpf(amax, &ex);   /* amax = f * 2^ex, f in [0.5, 1)   */
        e = (ex - 1) - 2;          /* floor(log2 amax) - emax(E2M1)    */
        if (e < -127)
            e = -127;
        if (e > 127)
            e = 127;
    }
    scale = ldexpf(1.0f, e);
    inv = ldexpf(1.0f, -e);
    for (int i = 0; i < n; ++i) {
        float v = xf[i] * inv;
        uint8_t q = or_e2m1_encode(v);
        codes[i] = q;
        xhat[i] = (float)or_e2m1_decode(q) * scale;
    }
    *sf_out = (uint8_t)(e + 127);
}

/* ------------------------------------------------------------------------ */
/* Row quantizers on logical layouts (reading R7).                            */
/* fmt: 0 = NVFP4 (block 16, alpha used), 1 = MXFP4 (block 32, alpha unused). */
/* ------------------------------------------------------------------------ */

int or_block_size(int fmt) { return fmt == 0 ? 16 : 32; }

static void put_nibble(uint8_t *row_codes, int k, uint8_t q)
{
    if ((k & 1) == 0)
        row_codes[k >> 1] = (uint8_t)((row_codes[k >> 1] & 0xF0u) | (q & 0xFu));
    else
        row_codes[k >> 1] = (uint8_t)((row_codes[k >> 1] & 0x0Fu) | ((q & 0xFu) << 4));
}

/* Quantize fp32 rows [rows][K] (K a multiple of the block size).
 * codes: [rows][K/2] bytes, sf: [rows][K/bs] bytes, xhat: [rows][K] (QDQ). */
static void quantize_f32_rows(int fmt, int rows, int K, const float *xf, float alpha,
                              uint8_t *codes, uint8_t *sf, float *xhat)
{
    int bs = or_block_size(fmt);
    uint8_t q[32];
    for (int r = 0; r < rows; ++r) {
        const float *xr = xf + (int64_t)r * K;
        uint8_t *cr = codes + (int64_t)r * (K / 2);
        float *hr = xhat + (int64_t)r * K;
        for (int b = 0; b < K / bs; ++b) {
            uint8_t s;
            if (fmt == 0)
                nvfp4_block(xr + b * bs, bs, alpha, &s, q, hr + b * bs);
            else
                mxfp4_block(xr + b * bs, bs, &s, q, hr + b * bs);
            sf[(int64_t)r * (K / bs) + b] = s;
            for (int i = 0; i < bs; ++i)
                put_nibble(cr, b * bs + i, q[i]);
        }
    }
}

/* Base quantization of bf16 rows: X^ = QDQ(X).  Returns 0 on success. */
int or_quantize(int fmt, int rows, int K, const uint16_t *x, float alpha,
                uint8_t *codes, uint8_t *sf, float *xhat /* may be NULL */)
{
    int64_t n = (int64_t)rows * K;
    float *xf, *h;
    if (rows < 0 || K <= 0 || K % or_block_size(fmt) != 0)
        return 1;
    xf = (float *)malloc(sizeof(float) * (size_t)(n > 0 ? n : 1));
    h = xhat ? xhat : (float *)malloc(sizeof(float) * (size_t)(n > 0 ? n : 1));
    for (int64_t i = 0; i < n; ++i)
        xf[i] = bf16_to_float(x[i]);
    quantize_f32_rows(fmt, rows, K, xf, alpha, codes, sf, h);
    if (!xhat)
        free(h);
    free(xf);
    return 0;
}

/* NVFP4 base quantization of bf16 rows with Eq. 10's division (see
 * nvfp4_block_div).  Returns 0 on success. */
int or_quantize_nvfp4_div(int rows, int K, const uint16_t *x, float alpha, uint8_t *codes, uint8_t *sf)
{
    uint8_t q[16];
    float xf[16];
    if (rows < 0 || K <= 0 || K % 16 != 0)
        return 1;
    for (int r = 0; r < rows; ++r) {
        for (int b = 0; b < K / 16; ++b) {
            for (int i = 0; i < 16; ++i)
                xf[i] = bf16_to_float(x[(int64_t)r * K + b * 16 + i]);
            nvfp4_block_div(xf, 16, alpha, &sf[(int64_t)r * (K / 16) + b], q);
            for (int i = 0; i < 16; ++i)
                put_nibble(codes + (int64_t)r * (K / 2), b * 16 + i, q[i]);
        }
    }
    return 0;
}

/* NVFP4 base plus residue with Alg. 1's form of the reconstruction in place
 * of Eq. 10's (the alternative to reading R5; parity is defined on Eq. 10).
 * Alg. 1 line 5 forms x_q = QDQ(scale * x), i.e. dec(q) in the scaled
 * domain, with `scale` the fp32 multiplier fl(1/s~); line 6 writes the
 * residue as x - x_q / scale.  So x^ = fl(dec(q) / fl(1/s~)) (0 when the
 * multiplier is 0), r = fl(x - x^), and r is quantized by the same rule as
 * the base (its own block scale, the same alpha).  Codes and scale bytes of
 * both operands, logical layout. */
int or_quantize_residue_nvfp4_recon_div(int rows, int K, const uint16_t *x, float alpha,
                                        uint8_t *codes_x, uint8_t *sf_x, uint8_t *codes_r, uint8_t *sf_r)
{
    float xf[16], r[16], xh_unused[16];
    uint8_t q[16];
    if (rows < 0 || K <= 0 || K % 16 != 0)
        return 1;
    for (int row = 0; row < rows; ++row) {
        for (int b = 0; b < K / 16; ++b) {
            float amax = 0.0f, s, t, st, mul;
            uint8_t sf;
            for (int i = 0; i < 16; ++i) {
                xf[i] = bf16_to_float(x[(int64_t)row * K + b * 16 + i]);
                if (fabsf(xf[i]) > amax)
                    amax = fabsf(xf[i]);
            }
            s = amax / 6.0f;
            t = (alpha > 0.0f) ? s / alpha : 0.0f;
            sf = or_e4m3_encode_satfinite(t);
            st = alpha * (float)or_e4m3_decode(sf);
            mul = (st == 0.0f) ? 0.0f : 1.0f / st;           /* Alg. 1 line 3: multiplier */
            for (int i = 0; i < 16; ++i) {
                float xq;
                q[i] = or_e2m1_encode(xf[i] * mul);           /* line 5: q of scale * x    */
                xq = (float)or_e2m1_decode(q[i]);             /* line 5: x_q = dec(q)      */
                r[i] = xf[i] - (mul == 0.0f ? 0.0f : xq / mul); /* line 6: x - x_q / scale */
                put_nibble(codes_x + (int64_t)row * (K / 2), b * 16 + i, q[i]);
            }
            sf_x[(int64_t)row * (K / 16) + b] = sf;
            nvfp4_block(r, 16, alpha, &sf_r[(int64_t)row * (K / 16) + b], q, xh_unused);
            for (int i = 0; i < 16; ++i)
                put_nibble(codes_r + (int64_t)row * (K / 2), b * 16 + i, q[i]);
        }
    }
    return 0;
}

/* Base plus residue (Sec. 2 "r = x - x^"; Sec. 4.2 R = X - X^; App. B.2: the
 * residue is a separate operand with its own block scales and the same tensor
 * scale).  Outputs the two operands separately in logical layout.
 * resid (optional): the fp32 residue R = X - X^. */
int or_quantize_residue(int fmt, int rows, int K, const uint16_t *x, float alpha,
                        uint8_t *codes_x, uint8_t *sf_x,
                        uint8_t *codes_r, uint8_t *sf_r,
                        float *resid /* may be NULL */,
                        float *rhat /* may be NULL */)
{
    int64_t n = (int64_t)rows * K;
    size_t bytes = sizeof(float) * (size_t)(n > 0 ? n : 1);
    float *xf, *xh, *r, *rh;
    if (rows < 0 || K <= 0 || K % or_block_size(fmt) != 0)
        return 1;
    xf = (float *)malloc(bytes);
    xh = (float *)malloc(bytes);
    r = resid ? resid : (float *)malloc(bytes);
    rh = rhat ? rhat : (float *)malloc(bytes);
    for (int64_t i = 0; i < n; ++i)
        xf[i] = bf16_to_float(x[i]);
    quantize_f32_rows(fmt, rows, K, xf, alpha, codes_x, sf_x, xh);
    for (int64_t i = 0; i < n; ++i)
        r[i] = xf[i] - xh[i];
    quantize_f32_rows(fmt, rows, K, r, alpha, codes_r, sf_r, rh);
    if (!resid)
        free(r);
    if (!rhat)
        free(rh);
    free(xh);
    free(xf);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Dequantization and the block-scaled GEMM (reading R8).                     */
/* ------------------------------------------------------------------------ */

static double decode_sf(int fmt, uint8_t b)
{
    return fmt == 0 ? or_e4m3_decode(b) : or_e8m0_decode(b);
}

/* Values represented by the codes and block scales, without the tensor scale:
 * out[r][k] = dec(code[r][k]) * dec(sf[r][k / bs]). */
/* Threads for the dequantization and the GEMM loops (1 unless the caller
 * asks for more: the all-core timing of the CPU baseline). */
static int or_threads = 1;

void or_set_threads(int n) { or_threads = n > 0 ? n : 1; }

void or_dequantize(int fmt, int rows, int K, const uint8_t *codes, const uint8_t *sf,
                   double *out)
{
    int bs = or_block_size(fmt);
#pragma omp parallel for schedule(static) num_threads(or_threads)
    for (int r = 0; r < rows; ++r) {
        for (int k = 0; k < K; ++k) {
            uint8_t byte = codes[(int64_t)r * (K / 2) + k / 2];
            uint8_t q = (k & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 0xF);
            out[(int64_t)r * K + k] =
                or_e2m1_decode(q) * decode_sf(fmt, sf[(int64_t)r * (K / bs) + k / bs]);
        }
    }
}

/* Z[m][n] = sum_k A[m][k] * B[n][k] with A, B the dequantized operands (a
 * linear layer with B in nn.Linear [N][K] layout).  Plain double loops. */
int or_block_gemm(int fmt, int M, int N, int K,
                  const uint8_t *codes_a, const uint8_t *sf_a,
                  const uint8_t *codes_b, const uint8_t *sf_b, double *Z)
{
    double *A, *B;
    if (M < 0 || N < 0 || K <= 0 || K % or_block_size(fmt) != 0)
        return 1;
    A = (double *)malloc(sizeof(double) * (size_t)((int64_t)M * K + 1));
    B = (double *)malloc(sizeof(double) * (size_t)((int64_t)N * K + 1));
    or_dequantize(fmt, M, K, codes_a, sf_a, A);
    or_dequantize(fmt, N, K, codes_b, sf_b, B);
    /* each output is the same k-ordered double sum whatever the thread count */
#pragma omp parallel for collapse(2) schedule(static) num_threads(or_threads)
    for (int m = 0; m < M; ++m) {
        for (int n = 0; n < N; ++n) {
            const double *a = A + (int64_t)m * K;
            const double *b = B + (int64_t)n * K;
            double acc = 0.0;
            for (int k = 0; k < K; ++k)
                acc += a[k] * b[k];
            Z[(int64_t)m * N + n] = acc;
        }
    }
    free(B);
    free(A);
    return 0;
}

/* The whole linear layer for one call (Sec. 4.2 Eq. 1 with full compensation,
 * Sec. 4.3 Eq. 2):
 *   compensated == 0 (W4A4):  Y = a_x a_w * (X^ W^T)
 *   compensated == 1:         Y = a_x a_w * (X^ W^T + R^ W^T)
 * where X^, R^ come from or_quantize_residue on x with tensor scale alpha_x
 * and W^ is given as codes/scales.  For MXFP4 the tensor scales are taken
 * as 1 (the format has none).  Y is [M][N] double. */
int or_linear(int fmt, int compensated, int M, int N, int K,
              const uint16_t *x, float alpha_x,
              const uint8_t *codes_w, const uint8_t *sf_w, float alpha_w,
              double *Y)
{
    int bs = or_block_size(fmt);
    int64_t nc = (int64_t)M * (K / 2), ns = (int64_t)M * (K / bs), ny = (int64_t)M * N;
    uint8_t *cx, *sx, *cr, *sr;
    double *Zx, *Zr, g;
    if (M < 0 || N < 0 || K <= 0 || K % bs != 0)
        return 1;
    cx = (uint8_t *)malloc((size_t)nc + 1);
    sx = (uint8_t *)malloc((size_t)ns + 1);
    cr = (uint8_t *)malloc((size_t)nc + 1);
    sr = (uint8_t *)malloc((size_t)ns + 1);
    Zx = (double *)malloc(sizeof(double) * (size_t)(ny + 1));
    Zr = (double *)malloc(sizeof(double) * (size_t)(ny + 1));
    or_quantize_residue(fmt, M, K, x, alpha_x, cx, sx, cr, sr, NULL, NULL);
    or_block_gemm(fmt, M, N, K, cx, sx, codes_w, sf_w, Zx);
    if (compensated)
        or_block_gemm(fmt, M, N, K, cr, sr, codes_w, sf_w, Zr);
    g = (fmt == 0) ? (double)alpha_x * (double)alpha_w : 1.0;
    for (int64_t i = 0; i < ny; ++i)
        Y[i] = g * (Zx[i] + (compensated ? Zr[i] : 0.0));
    free(Zr);
    free(Zx);
    free(sr);
    free(cr);
    free(sx);
    free(cx);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Array helpers for the codec pins (element-wise loops, nothing more).       */
/* ------------------------------------------------------------------------ */

void or_e2m1_encode_array(const float *v, int64_t n, uint8_t *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = or_e2m1_encode(v[i]);
}

void or_e4m3_encode_array(const float *v, int64_t n, uint8_t *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = or_e4m3_encode_satfinite(v[i]);
}

/* ------------------------------------------------------------------------ */
/* Selective prefill compensation, K-Ext (Sec. 5.3 and Eq. 6; App. A Eq. 7;  */
/* App. B.2 Alg. 1 for the partial residues).                                 */
/*                                                                            */
/* Readings (also in the design notes):                                       */
/*   R11 Eq. 7's TopK within a group of 8 channels keeps the channels with    */
/*       the larger calibration score; equal scores keep the lower channel.   */
/*   R12 The extension lists, group by group, the selected channels of each   */
/*       group in increasing channel order (Alg. 1 line 7 SELECT(r, mask)):  */
/*       extension element e = g*k + j is the j-th selected channel of group  */
/*       g.  Its residues are quantized as their own blocks of 16 (NVFP4) or  */
/*       32 (MXFP4) consecutive extension elements with the base operand's    */
/*       tensor scale (Sec. 5.3: "a separate NVFP4 operand with its own block  */
/*       scales and share the base operand's tensor scale").                  */
/*   R13 The weight side of Eq. 6 is [W | W[:, S]] in bf16 (the selected     */
/*       floating-point weight columns appended in extension order),          */
/*       quantized as one tensor in the extended block layout with the        */
/*       weight's tensor scale.                                               */
/* k = 8 * rho channels per group of 8; K_eff = K + K*k/8 (Eq. after 6).      */
/* ------------------------------------------------------------------------ */

int or_kext_width(int K, int k) { return K / 8 * k; }

/* Eq. 7: per group of 8 channels, the k channels with the largest score.
 * mask[g] bit t is set when channel 8g + t is selected. */
int or_kext_select(int K, int k, const float *score, uint8_t *mask)
{
    if (K <= 0 || K % 8 != 0 || k < 0 || k > 8)
        return 1;
    for (int g = 0; g < K / 8; ++g) {
        uint8_t m = 0;
        for (int j = 0; j < k; ++j) {
            int best = -1;
            for (int t = 0; t < 8; ++t) {
                if (m & (1u << t))
                    continue;
                if (best < 0 || score[8 * g + t] > score[8 * g + best])
                    best = t;
            }
            m = (uint8_t)(m | (1u << best));
        }
        mask[g] = m;
    }
    return 0;
}

/* Extension element e -> channel (reading R12).  Returns 1 when a group does
 * not have exactly k selected channels. */
static int kext_index(int K, int k, const uint8_t *mask, int *ext)
{
    for (int g = 0; g < K / 8; ++g) {
        int j = 0;
        for (int t = 0; t < 8; ++t)
            if (mask[g] & (1u << t))
                ext[g * k + j++] = 8 * g + t;
        if (j != k)
            return 1;
    }
    return 0;
}

static int kext_shape_ok(int fmt, int K, int k)
{
    int bs = or_block_size(fmt);
    return K > 0 && K % bs == 0 && k >= 1 && k <= 8 && (K / 8 * k) % bs == 0;
}

/* Extended activation operand [X^ | R^_S] (Eq. 6), logical layout with K_eff
 * columns: codes [rows][K_eff/2], scales [rows][K_eff/bs].  The base part is
 * exactly or_quantize's; R = X - X^ in fp32 (Alg. 1 line 6). */
int or_quantize_kext(int fmt, int rows, int K, int k, const uint16_t *x, float alpha, const uint8_t *mask,
                     uint8_t *codes, uint8_t *sf)
{
    int bs = or_block_size(fmt), Kx = or_kext_width(K, k), Ke = K + or_kext_width(K, k);
    int64_t n = (int64_t)rows * K, nx = (int64_t)rows * Kx;
    int *ext;
    float *xf, *xh, *rs, *rh;
    uint8_t *cb, *sb, *ce, *se;
    if (rows < 0 || !kext_shape_ok(fmt, K, k))
        return 1;
    ext = (int *)malloc(sizeof(int) * (size_t)Kx);
    if (kext_index(K, k, mask, ext)) {
        free(ext);
        return 1;
    }
    xf = (float *)malloc(sizeof(float) * (size_t)(n + 1));
    xh = (float *)malloc(sizeof(float) * (size_t)(n + 1));
    rs = (float *)malloc(sizeof(float) * (size_t)(nx + 1));
    rh = (float *)malloc(sizeof(float) * (size_t)(nx + 1));
    cb = (uint8_t *)malloc((size_t)(n / 2 + 1));
    sb = (uint8_t *)malloc((size_t)(n / bs + 1));
    ce = (uint8_t *)malloc((size_t)(nx / 2 + 1));
    se = (uint8_t *)malloc((size_t)(nx / bs + 1));
    for (int64_t i = 0; i < n; ++i)
        xf[i] = bf16_to_float(x[i]);
    quantize_f32_rows(fmt, rows, K, xf, alpha, cb, sb, xh);
    for (int r = 0; r < rows; ++r)
        for (int e = 0; e < Kx; ++e) {
            int64_t i = (int64_t)r * K + ext[e];
            rs[(int64_t)r * Kx + e] = xf[i] - xh[i];          /* selected residues */
        }
    quantize_f32_rows(fmt, rows, Kx, rs, alpha, ce, se, rh);
    for (int r = 0; r < rows; ++r) {
        memcpy(codes + (int64_t)r * (Ke / 2), cb + (int64_t)r * (K / 2), (size_t)(K / 2));
        memcpy(codes + (int64_t)r * (Ke / 2) + K / 2, ce + (int64_t)r * (Kx / 2), (size_t)(Kx / 2));
        memcpy(sf + (int64_t)r * (Ke / bs), sb + (int64_t)r * (K / bs), (size_t)(K / bs));
        memcpy(sf + (int64_t)r * (Ke / bs) + K / bs, se + (int64_t)r * (Kx / bs), (size_t)(Kx / bs));
    }
    free(se); free(ce); free(sb); free(cb); free(rh); free(rs); free(xh); free(xf); free(ext);
    return 0;
}

/* Extended weight (reading R13): [W | W[:, S]] bf16 [N][K_eff], quantized as
 * one tensor with tensor scale alpha_w. */
int or_quantize_weight_kext(int fmt, int N, int K, int k, const uint16_t *w, float alpha_w, const uint8_t *mask,
                            uint8_t *codes, uint8_t *sf)
{
    int Kx = or_kext_width(K, k), Ke = K + or_kext_width(K, k), rc;
    int *ext;
    uint16_t *we;
    if (N < 0 || !kext_shape_ok(fmt, K, k))
        return 1;
    ext = (int *)malloc(sizeof(int) * (size_t)Kx);
    if (kext_index(K, k, mask, ext)) {
        free(ext);
        return 1;
    }
    we = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)((int64_t)N * Ke + 1));
    for (int nn = 0; nn < N; ++nn) {
        memcpy(we + (int64_t)nn * Ke, w + (int64_t)nn * K, sizeof(uint16_t) * (size_t)K);
        for (int e = 0; e < Kx; ++e)
            we[(int64_t)nn * Ke + K + e] = w[(int64_t)nn * K + ext[e]];
    }
    rc = or_quantize(fmt, N, Ke, we, alpha_w, codes, sf, NULL);
    free(we);
    free(ext);
    return rc;
}

/* The K-Ext linear layer (Eq. 6): one GEMM over K_eff,
 *   Y = a_x a_w * [X^ | R^_S] [W^ | W^_S]^T   (MXFP4: tensor scales 1). */
int or_linear_kext(int fmt, int M, int N, int K, int k, const uint16_t *x, float alpha_x, const uint8_t *mask,
                   const uint8_t *codes_w, const uint8_t *sf_w, float alpha_w, double *Y)
{
    int bs = or_block_size(fmt), Ke = K + or_kext_width(K, k), rc;
    uint8_t *ca, *sa;
    double g;
    if (M < 0 || N < 0 || !kext_shape_ok(fmt, K, k))
        return 1;
    ca = (uint8_t *)malloc((size_t)((int64_t)M * (Ke / 2) + 1));
    sa = (uint8_t *)malloc((size_t)((int64_t)M * (Ke / bs) + 1));
    rc = or_quantize_kext(fmt, M, K, k, x, alpha_x, mask, ca, sa);
    if (rc == 0)
        rc = or_block_gemm(fmt, M, N, Ke, ca, sa, codes_w, sf_w, Y);
    g = (fmt == 0) ? (double)alpha_x * (double)alpha_w : 1.0;
    if (rc == 0)
        for (int64_t i = 0; i < (int64_t)M * N; ++i)
            Y[i] *= g;
    free(sa);
    free(ca);
    return rc;
}
