/*
 * mxoracle.c -- plain, slow CPU oracle for the MXFP4 A4W4 and FP8 PTPC A8W8
 * hot path.  TEST INFRASTRUCTURE ONLY: it exists so that the CUDA library can
 * be checked against an independent statement of what it must compute.  Only
 * tests/, the smoke entry and the benchmark's CPU-baseline leg may load it.
 * It shares no code, header, table or constant generator with the CUDA path.
 *
 * Sources (page title, section):
 *  [P1] "Kimi-K3 DSpark O-Proj-only MXFP4", section "Exact quantization
 *       coverage": MXFP4 E2M1 weight codes, E8M0 scales, 32 consecutive
 *       input-channel values per scale, stored weight (7168, 8192) and scale
 *       (7168, 256); runtime path "dynamic MXFP4 activations with A4W4
 *       dispatch"; the other projections FP8 E4M3 with FP32
 *       per-output-channel scales and dynamic per-token FP8 activations.
 *  [P2] "Kimi-K3-DSpark-FP8-PTPC", section "Phase 1 FP8 PTPC Quantization":
 *       weight dtype torch.float8_e4m3fn, per-output-channel scheme, FP32
 *       scale of shape (out_features, 1), activation scheme dynamic
 *       per-token FP8 computed online; activation scales are never stored.
 *  [P3] "Kimi-K3-Quark-MXFP4-AttnFP8", section "Model Overview" / "Model
 *       Quantization": the MX scheme is "OCP MXFP4"; attention is PTPC-FP8.
 *  [OCP] OCP Microscaling Formats (MX) v1.0, the standard [P3] names: E2M1
 *       element encoding, E8M0 shared scale, block size 32, shared exponent
 *       = floor(log2(amax)) - emax_elem with emax_elem = 2 for E2M1.
 *  [OFP8] OCP 8-bit Floating Point (E4M3, bias 7, no infinities, 0x7F/0xFF
 *       NaN, max finite 448) -- the format torch.float8_e4m3fn implements.
 *
 * Readings taken where the pages are silent (each one is a choice, listed
 * again in the design notes):
 *  R1 shared exponent uses the OCP floor rule, e = clamp(floor(log2 amax) - 2,
 *     -127, 127); an all-zero group gets e = -127 (scale code 0) because
 *     floor(log2 0) = -inf clamps to the bottom of the range.
 *  R2 element rounding is round-to-nearest, ties to the even code (mantissa
 *     bit 0), saturating to +-6 (E2M1) or +-448 (E4M3).
 *  R3 the sign is kept, including -0 and negative values that round to 0.
 *  R4 a group/row holding a NaN or infinity gets a NaN scale (E8M0 0xFF for
 *     MX, s = NaN for FP8) and all-zero codes.
 *  R5 packing: two E2M1 codes per byte, the lower k in the low nibble.
 *  R6 FP8 per-token scale s = amax / 448 (fp32 division, round to nearest);
 *     q = E4M3(x / s) with the division in fp32 first; an all-zero row gets
 *     s = 1.
 *  R7 GEMM is the Linear y = x . W^T with x (M, K) and W (N, K) both
 *     K-contiguous; the reference value is the exact dot product of the
 *     dequantized operands, accumulated in fp64.
 *
 * Portable C11 only: no intrinsics, no inline assembly, no reliance on the
 * signedness of char.  Build with -ffp-contract=off and without fast-math.
 */
#include <math.h>
#include <stdint.h>
#include <stddef.h>
#include <string.h>
#include <stdlib.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------ */
/* bf16 -> fp32: bf16 is the upper half of an IEEE binary32; widening is a  */
/* 16-bit left shift of the bit pattern and is exact.                       */
/* ------------------------------------------------------------------------ */
float orc_bf16_to_f32(uint16_t b)
{
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

static uint32_t f32_bits(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return u;
}

/* ------------------------------------------------------------------------ */
/* E2M1 [OCP]: 1 sign bit (bit 3), 2 exponent bits (bias 1), 1 mantissa bit. */
/* Exponent field 0 is subnormal: value = m * 2^(1-1) * 0.5.                  */
/* The eight magnitudes are listed directly.                                 */
/* ------------------------------------------------------------------------ */
static const double E2M1_MAG[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

double orc_e2m1_value(uint8_t code)
{
    double m = E2M1_MAG[code & 7u];
    return (code & 8u) ? -m : m;
}

/* E8M0 [OCP]: an unsigned biased exponent, value 2^(c-127); 0xFF is NaN. */
double orc_e8m0_value(uint8_t c)
{
    if (c == 0xFFu)
        return NAN;
    return ldexp(1.0, (int)c - 127);
}

/* E4M3 [OFP8]: sign bit 7, exponent bits 6..3 (bias 7), mantissa bits 2..0.
 * Exponent field 0 is subnormal: m/8 * 2^-6.  S.1111.111 is NaN; there is
 * no infinity, so S.1111.110 = 448 is the largest finite magnitude. */
double orc_e4m3_value(uint8_t code)
{
    unsigned e = (code >> 3) & 0xFu;
    unsigned m = code & 7u;
    double mag;
    if (e == 0xFu && m == 7u)
        return NAN;
    if (e == 0)
        mag = ldexp((double)m / 8.0, -6);
    else
        mag = ldexp(1.0 + (double)m / 8.0, (int)e - 7);
    return (code & 0x80u) ? -mag : mag;
}

/* ------------------------------------------------------------------------ */
/* Rounding to a code by table search (R2, R3): scan every finite magnitude, */
/* keep the nearest; on an exact tie keep the code whose mantissa LSB is 0.  */
/* A magnitude beyond the largest entry is nearest to the largest entry,     */
/* which is exactly saturation.                                              */
/* ------------------------------------------------------------------------ */
uint8_t orc_e2m1_round(double v)
{
    double a = fabs(v);
    unsigned best = 0;
    double best_d = INFINITY;
    for (unsigned c = 0; c < 8; ++c) {
        double d = fabs(a - E2M1_MAG[c]);
        if (d < best_d || (d == best_d && (c & 1u) == 0u && (best & 1u) != 0u)) {
            best = c;
            best_d = d;
        }
    }
    return (uint8_t)(best | (signbit(v) ? 8u : 0u));
}

static double E4M3_MAG[0x7F]; /* magnitudes of codes 0x00..0x7E */
static int e4m3_mag_ready = 0;

static void e4m3_mag_init(void)
{
    if (e4m3_mag_ready)
        return;
    for (unsigned c = 0; c < 0x7Fu; ++c)
        E4M3_MAG[c] = orc_e4m3_value((uint8_t)c);
    e4m3_mag_ready = 1;
}

uint8_t orc_e4m3_round(float v)
{
    double a = fabs((double)v);
    unsigned best = 0;
    double best_d = INFINITY;
    e4m3_mag_init();
    for (unsigned c = 0; c < 0x7Fu; ++c) { /* 0x7F is NaN: not a candidate */
        double d = fabs(a - E4M3_MAG[c]);
        if (d < best_d || (d == best_d && (c & 1u) == 0u && (best & 1u) != 0u)) {
            best = c;
            best_d = d;
        }
    }
    return (uint8_t)(best | (signbit(v) ? 0x80u : 0u));
}

/* floor(log2 a) for a finite a > 0, read exactly off the binary32 fields.
 * Subnormals: a = m * 2^-149 with m the 23-bit field, so floor(log2 a) =
 * floor(log2 m) - 149. */
int orc_floor_log2(float a)
{
    uint32_t u = f32_bits(a) & 0x7FFFFFFFu;
    int ef = (int)(u >> 23);
    if (ef != 0)
        return ef - 127;
    {
        uint32_t m = u & 0x7FFFFFu;
        int p = -1;
        while (m) {
            ++p;
            m >>= 1;
        }
        return p - 149;
    }
}

/* ------------------------------------------------------------------------ */
/* MXFP4 quantization of one block of 32 values [OCP], [P1] ("32 consecutive */
/* input-channel values per scale"), readings R1-R4.                         */
/*   amax = max |x|; e = clamp(floor(log2 amax) - 2, -127, 127);             */
/*   scale code = e + 127;  code_i = E2M1(x_i * 2^-e).                       */
/* x_i * 2^-e is formed in fp64, where it is exact.                          */
/* ------------------------------------------------------------------------ */
void orc_mx_quantize_block(const uint16_t *x, uint8_t *codes32, uint8_t *scale)
{
    float xf[32];
    float amax = 0.0f;
    int nonfinite = 0;
    int e;
    for (int i = 0; i < 32; ++i) {
        xf[i] = orc_bf16_to_f32(x[i]);
        if (!isfinite(xf[i]))
            nonfinite = 1;
        else if (fabsf(xf[i]) > amax)
            amax = fabsf(xf[i]);
    }
    if (nonfinite) { /* R4 */
        *scale = 0xFFu;
        memset(codes32, 0, 32);
        return;
    }
    if (amax == 0.0f) {
        e = -127; /* R1: floor(log2 0) = -inf, clamped */
    } else {
        e = orc_floor_log2(amax) - 2;
        if (e < -127) e = -127;
        if (e > 127) e = 127;
    }
    *scale = (uint8_t)(e + 127);
    for (int i = 0; i < 32; ++i) {
        double v = ldexp((double)xf[i], -e); /* exact in binary64; |v| < 8 */
        codes32[i] = orc_e2m1_round(v);
    }
}

/* Quantize each row of a bf16 matrix x (rows x K, leading dimension ldx in
 * elements) into packed E2M1 codes (rows x K/2 bytes, R5) and row-major
 * E8M0 scales (rows x K/32).  This is both the offline weight conversion of
 * [P1] (per output row of W, groups along the input channels) and the
 * dynamic activation quantization (per token).  K must be a multiple of 32. */
void orc_mx_quantize_rows(const uint16_t *x, int rows, int K, long long ldx,
                          uint8_t *codes, uint8_t *sf)
{
    const int G = K / 32;
#pragma omp parallel for schedule(static)
    for (int r = 0; r < rows; ++r) {
        uint8_t c32[32];
        for (int g = 0; g < G; ++g) {
            orc_mx_quantize_block(x + (size_t)r * (size_t)ldx + (size_t)g * 32,
                                  c32, sf + (size_t)r * G + g);
            for (int j = 0; j < 16; ++j)
                codes[(size_t)r * (K / 2) + (size_t)g * 16 + j] =
                    (uint8_t)((c32[2 * j] & 0xFu) | ((c32[2 * j + 1] & 0xFu) << 4));
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Scale-factor tile layout used by the GEMM operands: 128 rows x 4 scales   */
/* per 512-byte tile; tiles ordered row-block-major.  Inside a tile the      */
/* scale of (row r, group g) sits at (r % 32) * 16 + ((r % 128) / 32) * 4 +  */
/* g % 4.  (NVIDIA's public description of the 1-D block-scaling-factor     */
/* layout; not on the pages.)  G = K/32 must be a multiple of 4.            */
/* ------------------------------------------------------------------------ */
size_t orc_sf_swizzled_offset(int r, int g, int G)
{
    size_t tile = (size_t)(r / 128) * (size_t)(G / 4) + (size_t)(g / 4);
    return tile * 512u + (size_t)(r % 32) * 16u + (size_t)((r % 128) / 32) * 4u +
           (size_t)(g % 4);
}

size_t orc_sf_swizzled_bytes(int rows, int G)
{
    return (size_t)((rows + 127) / 128) * 128u * (size_t)G;
}

void orc_sf_swizzle(const uint8_t *sf_rowmajor, int rows, int G, uint8_t *sf_swz)
{
    for (int r = 0; r < rows; ++r)
        for (int g = 0; g < G; ++g)
            sf_swz[orc_sf_swizzled_offset(r, g, G)] = sf_rowmajor[(size_t)r * G + g];
}

/* ------------------------------------------------------------------------ */
/* FP8 E4M3 per-row quantization [P1], [P2], readings R2-R4, R6.             */
/*   amax = max |x|, s = amax / 448 (fp32), q = E4M3(fp32(x / s)).           */
/* Used for dynamic per-token activations and for per-output-channel        */
/* weights (a row of W (N, K) is one output channel).                        */
/* ------------------------------------------------------------------------ */
void orc_fp8_quantize_rows(const uint16_t *x, int rows, int K, long long ldx,
                           uint8_t *q, float *s)
{
#pragma omp parallel for schedule(static)
    for (int r = 0; r < rows; ++r) {
        const uint16_t *xr = x + (size_t)r * (size_t)ldx;
        float amax = 0.0f;
        int nonfinite = 0;
        volatile float sv; /* keep the scale a true binary32 value */
        for (int k = 0; k < K; ++k) {
            float f = orc_bf16_to_f32(xr[k]);
            if (!isfinite(f))
                nonfinite = 1;
            else if (fabsf(f) > amax)
                amax = fabsf(f);
        }
        if (nonfinite) {
            s[r] = NAN;
            memset(q + (size_t)r * K, 0, (size_t)K);
            continue;
        }
        sv = (amax == 0.0f) ? 1.0f : amax / 448.0f;
        s[r] = sv;
        for (int k = 0; k < K; ++k) {
            volatile float t = orc_bf16_to_f32(xr[k]) / sv; /* fp32 division, RN */
            q[(size_t)r * K + k] = orc_e4m3_round(t);
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Reference GEMMs (R7).  ref[i][n] = sum_k a[m_i][k] * w[n][k] over the     */
/* dequantized operands; bound[i][n] = sum_k |a[m_i][k] * w[n][k]|.          */
/* Only the activation rows listed in row_idx[0..nrows) are computed (all    */
/* rows when row_idx is NULL and nrows == M); outputs are nrows x N.         */
/* ------------------------------------------------------------------------ */

/* A4W4 [P1]: a_codes (M, K/2), a_sf row-major (M, K/32); w_codes (N, K/2),
 * w_sf row-major (N, K/32).  For each block of 32 the code products are
 * summed (an exact sum of multiples of 1/4), then scaled by
 * 2^(ea-127) * 2^(ew-127) and accumulated in fp64. */
void orc_gemm_a4w4(const uint8_t *a_codes, const uint8_t *a_sf,
                   const uint8_t *w_codes, const uint8_t *w_sf,
                   int M, int N, int K, const int *row_idx, int nrows,
                   double *ref, double *bound)
{
    const int G = K / 32;
    double *av = (double *)malloc(sizeof(double) * (size_t)nrows * (size_t)K);
    (void)M;
    /* decode the requested activation rows once: av[i][k] = v(code) */
    for (int i = 0; i < nrows; ++i) {
        int m = row_idx ? row_idx[i] : i;
        for (int k = 0; k < K; ++k) {
            uint8_t byte = a_codes[(size_t)m * (K / 2) + k / 2];
            av[(size_t)i * K + k] =
                orc_e2m1_value((uint8_t)((k & 1) ? (byte >> 4) : (byte & 0xFu)));
        }
    }
#pragma omp parallel for schedule(dynamic, 4)
    for (int n = 0; n < N; ++n) {
        double *wv = (double *)malloc(sizeof(double) * (size_t)K);
        for (int k = 0; k < K; ++k) {
            uint8_t byte = w_codes[(size_t)n * (K / 2) + k / 2];
            wv[k] = orc_e2m1_value((uint8_t)((k & 1) ? (byte >> 4) : (byte & 0xFu)));
        }
        for (int i = 0; i < nrows; ++i) {
            int m = row_idx ? row_idx[i] : i;
            const double *ar = av + (size_t)i * K;
            double acc = 0.0, accabs = 0.0;
            for (int g = 0; g < G; ++g) {
                double s = orc_e8m0_value(a_sf[(size_t)m * G + g]) *
                           orc_e8m0_value(w_sf[(size_t)n * G + g]);
                double blk = 0.0, blkabs = 0.0;
                for (int j = g * 32; j < g * 32 + 32; ++j) {
                    blk += ar[j] * wv[j];
                    blkabs += fabs(ar[j] * wv[j]);
                }
                acc += blk * s;
                accabs += blkabs * fabs(s);
            }
            ref[(size_t)i * N + n] = acc;
            bound[(size_t)i * N + n] = accabs;
        }
        free(wv);
    }
    free(av);
}

/* PTPC A8W8 [P1], [P2]: qa (M, K) E4M3 with per-token scale sa (M);
 * qw (N, K) E4M3 with per-output-channel scale sw (N).
 * y = (sum_k v(qa) v(qw)) * sa[m] * sw[n]; the code-product sum is exact in
 * fp64 (multiples of 2^-18 bounded by K * 448^2). */
void orc_gemm_ptpc(const uint8_t *qa, const float *sa, const uint8_t *qw,
                   const float *sw, int M, int N, int K, const int *row_idx,
                   int nrows, double *ref, double *bound)
{
    double lut[256];
    (void)M;
    for (int c = 0; c < 256; ++c)
        lut[c] = orc_e4m3_value((uint8_t)c);
#pragma omp parallel for schedule(dynamic, 4)
    for (int n = 0; n < N; ++n) {
        const uint8_t *wr = qw + (size_t)n * K;
        for (int i = 0; i < nrows; ++i) {
            int m = row_idx ? row_idx[i] : i;
            const uint8_t *ar = qa + (size_t)m * K;
            double acc = 0.0, accabs = 0.0;
            for (int k = 0; k < K; ++k) {
                double p = lut[ar[k]] * lut[wr[k]];
                acc += p;
                accabs += fabs(p);
            }
            ref[(size_t)i * N + n] = acc * (double)sa[m] * (double)sw[n];
            bound[(size_t)i * N + n] = accabs * fabs((double)sa[m] * (double)sw[n]);
        }
    }
}

/* ------------------------------------------------------------------------ */
/* SwiGLU between the packed gate_up projection and the down projection.     */
/* [P2] packs gate_proj and up_proj into one runtime gate_up_proj; the      */
/* pages do not name the activation between it and down_proj.  Readings:    */
/*  R14 the activation is SwiGLU: h = silu(gate) * up, silu(g) = g/(1+e^-g). */
/*  R15 a gate_up output row is [gate (I values) | up (I values)]: the two   */
/*      projections concatenated along the output axis, gate first.          */
/*  R16 h is rounded to bf16 (round to nearest even), the dtype in which     */
/*      the draft layers pass activations between linears, and the down     */
/*      projection's input is then quantized per token exactly as any other  */
/*      activation (orc_fp8_quantize_rows).                                  */
/*  R17 silu and the product are formed in binary32, one IEEE operation at   */
/*      a time, in the order written below, so that any IEEE machine gets    */
/*      the same h (and therefore the same FP8 codes).  e^t comes from the   */
/*      method of W. J. Cody and W. Waite (Software Manual for the           */
/*      Elementary Functions, 1980): n = nearest integer to t / ln2;         */
/*      r = (t - n*L1) - n*L2 with ln2 = L1 + L2 split so that n*L1 is exact */
/*      (L1 has 15 significant bits, |n| <= 128); e^r from its Taylor series */
/*      through r^7/7! (|r| <= ln2/2, the first dropped term is below 1e-8   */
/*      relative), summed by Horner's rule, each step one fused multiply-   */
/*      add (an IEEE 754 operation: fmaf); then the exact scaling by 2^n.    */
/* ------------------------------------------------------------------------ */
static float f32_from_bits(uint32_t u)
{
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* e^t in binary32 for the SwiGLU (R17).  Below t = -87.3 the result would
 * be subnormal and is returned as 0; above ln(FLT_MAX) it is +inf. */
float orc_exp_f32(float t)
{
    const float log2e = 0x1.715476p+0f;   /* 1/ln2 rounded to binary32 */
    const float L1 = 0x1.62e4p-1f;        /* 0.693145751953125: 15 significant bits */
    const float L2 = 0x1.7f7d1cp-20f;     /* ln2 - L1 rounded to binary32 */
    const float c2 = 0.5f, c3 = 0x1.555556p-3f, c4 = 0x1.555556p-5f, c5 = 0x1.111112p-7f,
                c6 = 0x1.6c16c2p-10f, c7 = 0x1.a01a02p-13f; /* 1/k! rounded to binary32 */
    float nf, r, p;
    int n;
    if (t != t)
        return t;
    if (t > 88.72283f)
        return INFINITY;
    if (t < -87.3f)
        return 0.0f;
    nf = rintf(t * log2e);
    n = (int)nf;
    r = t - nf * L1;
    r = r - nf * L2;
    p = c7;
    p = fmaf(p, r, c6);
    p = fmaf(p, r, c5);
    p = fmaf(p, r, c4);
    p = fmaf(p, r, c3);
    p = fmaf(p, r, c2);
    p = fmaf(p, r, 1.0f);
    p = fmaf(p, r, 1.0f);
    if (n > 127)
        return (p * f32_from_bits((uint32_t)(127 + 127) << 23)) * 2.0f;
    return p * f32_from_bits((uint32_t)(n + 127) << 23);
}

/* silu(g) * u in binary32 (R14, R17): e = e^-g, d = 1 + e, s = g / d, s * u. */
float orc_silu_mul_f32(float g, float u)
{
    float e = orc_exp_f32(-g);
    float d = 1.0f + e;
    float s = g / d;
    return s * u;
}

/* binary32 -> bf16 bits, round to nearest even (a NaN stays a NaN). */
uint16_t orc_f32_to_bf16(float f)
{
    uint32_t u = f32_bits(f);
    if ((u & 0x7FFFFFFFu) > 0x7F800000u)
        return (uint16_t)((u >> 16) | 0x0040u);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

/* h (rows x I bf16 bits) = bf16(silu(gate) * up) for every row of the
 * gate_up output gu (rows x 2I bf16, leading dimension ldgu, R15, R16). */
void orc_swiglu_rows(const uint16_t *gu, int rows, int I, long long ldgu, uint16_t *h)
{
#pragma omp parallel for schedule(static)
    for (int r = 0; r < rows; ++r) {
        const uint16_t *row = gu + (size_t)r * (size_t)ldgu;
        for (int j = 0; j < I; ++j) {
            float g = orc_bf16_to_f32(row[j]);
            float u = orc_bf16_to_f32(row[I + j]);
            h[(size_t)r * I + j] = orc_f32_to_bf16(orc_silu_mul_f32(g, u));
        }
    }
}

/* Threads OpenMP will use (1 when built without OpenMP). */
int orc_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
