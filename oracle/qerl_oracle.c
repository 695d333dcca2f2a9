/*
 * qerl_oracle.c -- plain, slow, CPU reference ("oracle") for the NVFP4
 * weight-only linear layer with a LoRA branch and Adaptive Quantization Noise.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, includes or
 * calls this file; only the tests, the smoke check and the CPU-baseline leg of
 * the benchmark load it.  It shares no code, header, table or constant
 * generator with the CUDA path.
 *
 * Sources (cited by page title and section/equation):
 *   [QeRL]  "QeRL: Beyond Efficiency -- Quantization-enhanced Reinforcement
 *           Learning for LLMs" (paper-graph-ui digest of arXiv 2510.11696),
 *           section 3.4, subsections "NVFP4 Quantization" (E2M1 level set,
 *           Eq. 6), "Low-Rank Adaptation (LoRA) Within Quantized Layers"
 *           (Eq. 2), "Adaptive Quantization Noise (AQN)" (Eq. 7, Eq. 8),
 *           "Noise Merging" (Eq. 9-12), "Algorithm 1" (stage mapping).
 *   [OCP]   OCP 8-bit / 4-bit floating point formats (E4M3, E2M1 bit layout);
 *           the digest only names the formats.
 *   [SC11]  Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy as
 *           1, 2, 3", SC'11 (Philox4x32-10).
 *
 * Precision: fp64 everywhere the method leaves it open.  Where a floating
 * point value decides a discrete result (an E2M1 code, an E4M3 scale, the
 * bf16 rounding of the noisy activation) the decision is taken in fp32, the
 * precision the kernels use.  Build with -ffp-contract=off and without
 * fast-math so every float operation is one IEEE operation.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_OK 0
#define ORC_ERR_ARG 1
#define ORC_ERR_SHAPE 2
#define ORC_ERR_NONFINITE 6

/* ------------------------------------------------------------------------ */
/* Generic "round a non-negative value to a small float format".            */
/* A format with `mant_bits` explicit significand bits whose smallest normal */
/* binade is [2^emin, 2^(emin+1)): subnormals share the quantum of that      */
/* binade.  Round to nearest, ties to even significand, then clamp at        */
/* `maxval` (saturation).  a/q and n*q are exact in double because q is a    */
/* power of two and a comes from an fp32 value.                              */
/* ------------------------------------------------------------------------ */
static double round_to_small_float(double a, int mant_bits, int emin, double maxval)
{
    if (a == 0.0) return 0.0;
    if (a > 2.0 * maxval) return maxval; /* far above the top: saturate */
    int e2;
    (void)frexp(a, &e2);     /* a = f * 2^e2, f in [0.5, 1) */
    int E = e2 - 1;          /* a in [2^E, 2^(E+1)) */
    if (E < emin) E = emin;  /* subnormal range keeps the quantum of emin */
    double q = ldexp(1.0, E - mant_bits);
    double n = nearbyint(a / q); /* default rounding mode: ties to even */
    double v = n * q;
    return v > maxval ? maxval : v;
}

/* ------------------------------------------------------------------------ */
/* E2M1: sign bit 3, exponent bits 2..1 (bias 1), mantissa bit 0.            */
/* Levels 0, 0.5, 1, 1.5, 2, 3, 4, 6 ([QeRL] "NVFP4 Quantization").          */
/* ------------------------------------------------------------------------ */
double orc_e2m1_decode(uint8_t code)
{
    int s = (code >> 3) & 1, e = (code >> 1) & 3, m = code & 1;
    double mag = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
    return s ? -mag : mag;
}

static uint8_t e2m1_code_of_magnitude(double v)
{
    if (v < 1.0) return (uint8_t)(v * 2.0); /* 0 -> 0, 0.5 -> 1 (subnormal) */
    int e2;
    (void)frexp(v, &e2);
    int E = e2 - 1;                                  /* 0, 1 or 2 */
    int m = (int)((v / ldexp(1.0, E) - 1.0) * 2.0);  /* 0 or 1 */
    return (uint8_t)(((E + 1) << 1) | m);
}

/* Encode one fp32 value: nearest level, ties to the even code, saturating at
 * 6.  A value that rounds to zero is encoded as +0 (code 0x0) whatever its
 * sign (reading: the digest gives no sign rule for zero). */
uint8_t orc_e2m1_encode(float v)
{
    double a = fabs((double)v);
    double mag = round_to_small_float(a, 1, 0, 6.0);
    uint8_t c = e2m1_code_of_magnitude(mag);
    if (c != 0 && signbit(v)) c |= 0x8;
    return c;
}

/* ------------------------------------------------------------------------ */
/* E4M3 ([OCP]): bias 7, 0x7F / 0xFF are NaN, no infinity, max 448,          */
/* min normal 2^-6, subnormal step 2^-9.                                     */
/* ------------------------------------------------------------------------ */
double orc_e4m3_decode(uint8_t code)
{
    int s = (code >> 7) & 1, e = (code >> 3) & 15, m = code & 7;
    double mag;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) mag = ldexp((double)m, -9);
    else mag = ldexp(1.0 + m / 8.0, e - 7);
    return s ? -mag : mag;
}

/* Encode a non-negative fp32 value: nearest, ties to even, saturate at 448. */
uint8_t orc_e4m3_encode_pos(float v)
{
    double v2 = round_to_small_float((double)v, 3, -6, 448.0);
    if (v2 < ldexp(1.0, -6)) return (uint8_t)(v2 * 512.0); /* subnormal: m * 2^-9 */
    int e2;
    (void)frexp(v2, &e2);
    int E = e2 - 1;
    int m = (int)((v2 / ldexp(1.0, E) - 1.0) * 8.0);
    return (uint8_t)(((E + 7) << 3) | m);
}

/* ------------------------------------------------------------------------ */
/* bf16 helpers                                                              */
/* ------------------------------------------------------------------------ */
static float bf16_bits_to_f32(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* fp32 -> bf16, round to nearest even (NaN stays NaN). */
static uint16_t f32_to_bf16_rn(float f)
{
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return (uint16_t)((u >> 16) | 0x40);
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7FFFu + lsb;
    return (uint16_t)(u >> 16);
}

/* fp64 -> bf16 with ONE rounding (no detour through fp32): nearest, ties to
 * even, overflow to infinity.  Used to round the exact oracle output. */
uint16_t orc_f64_to_bf16(double d)
{
    uint16_t sign = signbit(d) ? 0x8000 : 0;
    double a = fabs(d);
    if (isnan(d)) return 0x7FC0;
    if (a == 0.0) return sign;
    int e2;
    (void)frexp(a, &e2);
    int E = e2 - 1;
    if (E < -126) E = -126;             /* bf16 subnormals: quantum 2^-133 */
    double q = ldexp(1.0, E - 7);
    double v = nearbyint(a / q) * q;
    if (v >= ldexp(1.0, 128)) return (uint16_t)(sign | 0x7F80);
    float fv = (float)v;                /* exact: v has <= 8 significant bits */
    uint32_t u;
    memcpy(&u, &fv, 4);
    return (uint16_t)(sign | ((u >> 16) & 0x7FFF));
}

void orc_f64_to_bf16_array(const double* d, int64_t n, uint16_t* out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = orc_f64_to_bf16(d[i]);
}

/* ------------------------------------------------------------------------ */
/* NVFP4 quantizer.  Dequantization is [QeRL] Eq. 6:                         */
/*     W_hat = S_FP32 * (S_E4M3 (.) W_tilde),  one E4M3 scale per 16         */
/* contiguous elements along K.  The digest gives no encoder; the reading    */
/* implemented here (all fp32, in this order):                               */
/*   S   = amax(|W|) / (6 * 448)        (q_max of E2M1 times max of E4M3)    */
/*   r_b = (amax_b / 6) / S             per 16-element block b               */
/*   s_b = E4M3(r_b)  nearest-even, saturating                               */
/*   sc  = S * dec(s_b)                                                      */
/*   c   = E2M1(w / sc)  nearest-even-code, saturating (0 if sc == 0)        */
/* If S is 0 (all-zero tensor or underflow) S is set to 1.  Codes: row-major */
/* [n][k/2], element 2j in the low nibble, 2j+1 in the high nibble.  Scales: */
/* row-major [n][k/16].                                                      */
/* ------------------------------------------------------------------------ */
int orc_nvfp4_tensor_scale(const float* W, int64_t n, int64_t k, int64_t ldw, float* S_out)
{
    float amax = 0.0f;
    for (int64_t i = 0; i < n; ++i)
        for (int64_t j = 0; j < k; ++j) {
            float w = W[i * ldw + j];
            if (!isfinite(w)) return ORC_ERR_NONFINITE;
            float a = fabsf(w);
            if (a > amax) amax = a;
        }
    float S = amax / 2688.0f;
    if (S == 0.0f) S = 1.0f;
    *S_out = S;
    return ORC_OK;
}

int orc_nvfp4_quantize_with_scale(const float* W, int64_t n, int64_t k, int64_t ldw, float S,
                                  uint8_t* codes, uint8_t* scales)
{
    if (n < 0 || k < 0 || ldw < k) return ORC_ERR_ARG;
    if (k % 32 != 0) return ORC_ERR_SHAPE;
    for (int64_t i = 0; i < n; ++i) {
        for (int64_t b = 0; b < k / 16; ++b) {
            const float* wb = W + i * ldw + b * 16;
            float amax_b = 0.0f;
            for (int t = 0; t < 16; ++t) {
                if (!isfinite(wb[t])) return ORC_ERR_NONFINITE;
                float a = fabsf(wb[t]);
                if (a > amax_b) amax_b = a;
            }
            float r = (amax_b / 6.0f) / S;
            uint8_t s = orc_e4m3_encode_pos(r);
            float sc = S * (float)orc_e4m3_decode(s);
            scales[i * (k / 16) + b] = s;
            for (int t = 0; t < 16; t += 2) {
                uint8_t c0 = 0, c1 = 0;
                if (sc != 0.0f) {
                    c0 = orc_e2m1_encode(wb[t] / sc);
                    c1 = orc_e2m1_encode(wb[t + 1] / sc);
                }
                codes[i * (k / 2) + (b * 16 + t) / 2] = (uint8_t)(c0 | (c1 << 4));
            }
        }
    }
    return ORC_OK;
}

int orc_nvfp4_quantize(const float* W, int64_t n, int64_t k, int64_t ldw,
                       uint8_t* codes, uint8_t* scales, float* S_out)
{
    if (n < 0 || k < 0 || ldw < k) return ORC_ERR_ARG;
    if (k % 32 != 0) return ORC_ERR_SHAPE;
    float S;
    int st = orc_nvfp4_tensor_scale(W, n, k, ldw, &S);
    if (st != ORC_OK) return st;
    *S_out = S;
    return orc_nvfp4_quantize_with_scale(W, n, k, ldw, S, codes, scales);
}

/* Eq. 6 in fp64: W_hat[i][j] = S * dec(scale[i][j/16]) * e2m1(code[i][j]). */
void orc_nvfp4_dequant(const uint8_t* codes, const uint8_t* scales, float S, int64_t n, int64_t k,
                       double* W_hat)
{
    for (int64_t i = 0; i < n; ++i)
        for (int64_t j = 0; j < k; ++j) {
            uint8_t byte = codes[i * (k / 2) + j / 2];
            uint8_t c = (j & 1) ? (byte >> 4) : (byte & 0xF);
            double s = orc_e4m3_decode(scales[i * (k / 16) + j / 16]);
            W_hat[i * k + j] = (double)S * (s * orc_e2m1_decode(c));
        }
}

/* ------------------------------------------------------------------------ */
/* MXFP4, the format the digest compares with NVFP4 ([QeRL] "NVFP4           */
/* Quantization", other 4-bit formats): E2M1 elements with one shared E8M0   */
/* scale (a power of two) per block of 32 along K; no tensor scale.  The     */
/* digest does not say how the scale is chosen.  Reading: the OCP MX rule,   */
/* X = 2^(floor(log2(amax_b)) - 2), 2 being the largest E2M1 exponent, so    */
/* the block max lands in [4, 8) * X (values above 6 X saturate); E8M0 code  */
/* = log2(X) + 127, clamped to [0, 254]; an all-zero block gets code 0.      */
/* Elements: the E2M1 encoder above on w / X (exact: X is a power of two).   */
/* Layout: codes [n][k/2] (element 2j low nibble), scales [n][k/32].         */
/* ------------------------------------------------------------------------ */
double orc_e8m0_decode(uint8_t code)
{
    if (code == 0xFF) return NAN;
    return ldexp(1.0, (int)code - 127);
}

int orc_mxfp4_quantize(const float* W, int64_t n, int64_t k, int64_t ldw, uint8_t* codes, uint8_t* scales)
{
    if (n < 0 || k < 0 || ldw < k) return ORC_ERR_ARG;
    if (k % 32 != 0) return ORC_ERR_SHAPE;
    for (int64_t i = 0; i < n; ++i)
        for (int64_t b = 0; b < k / 32; ++b) {
            const float* blk = W + i * ldw + b * 32;
            float amax = 0.0f;
            for (int j = 0; j < 32; ++j) {
                if (!isfinite(blk[j])) return ORC_ERR_NONFINITE;
                if (fabsf(blk[j]) > amax) amax = fabsf(blk[j]);
            }
            int e = -127;
            if (amax > 0.0f) {
                int ex;
                frexp((double)amax, &ex); /* amax in [2^(ex-1), 2^ex): floor(log2(amax)) = ex - 1 */
                e = ex - 1 - 2;
                if (e < -127) e = -127;
                if (e > 127) e = 127;
            }
            scales[i * (k / 32) + b] = (uint8_t)(e + 127);
            const double X = ldexp(1.0, e);
            for (int j = 0; j < 32; j += 2) {
                const uint8_t lo = orc_e2m1_encode((float)((double)blk[j] / X));
                const uint8_t hi = orc_e2m1_encode((float)((double)blk[j + 1] / X));
                codes[i * (k / 2) + (b * 32 + j) / 2] = (uint8_t)(lo | (hi << 4));
            }
        }
    return ORC_OK;
}

void orc_mxfp4_dequant(const uint8_t* codes, const uint8_t* scales, int64_t n, int64_t k, double* W_hat)
{
    for (int64_t i = 0; i < n; ++i)
        for (int64_t j = 0; j < k; ++j) {
            const uint8_t byte = codes[i * (k / 2) + j / 2];
            const uint8_t c = (j & 1) ? (byte >> 4) : (byte & 0xF);
            W_hat[i * k + j] = orc_e8m0_decode(scales[i * (k / 32) + j / 32]) * orc_e2m1_decode(c);
        }
}

/* ------------------------------------------------------------------------ */
/* NF4, the QLoRA format the digest sets against NVFP4 ([QeRL] "NVFP4      */
/* Quantization", comparison to other 4-bit formats; "QLoRA's 4-bit          */
/* Quantization Addresses Memory but Degrades Speed": levels at quantiles of */
/* the Gaussian, recovered through a lookup table).  The digest             */
/* gives no construction; reading (the QLoRA one): 16 levels, ascending, are */
/* standard-normal quantiles at evenly spaced probabilities with an exact    */
/* zero -- 8 positive levels Phi^-1(1/2 + (i/8)(p - 1/2)), i = 1..8, 7       */
/* negative levels -Phi^-1(1/2 + (i/7)(p - 1/2)), i = 1..7, and 0, with      */
/* p = ((1 - 1/32) + (1 - 1/30)) / 2 -- each divided by the largest, so they */
/* span [-1, 1]; code c (0..15) is the c-th level (code 7 = 0).  Scaling     */
/* (reading): NVFP4's dual scaling with a level range of 1 instead of 6:     */
/* S = amax_t / 448 (1 if 0), block scale s = E4M3_RNE_SAT(amax_b / S) per   */
/* 16, element code = the level nearest to q = w / (S dec(s)) (one fp32     */
/* division), decided against the fp32-rounded midpoints m_c of adjacent    */
/* levels: c = #{ m_c <= q } (a quotient on a midpoint goes up).             */
/* Phi^-1 here: bisection of Phi(x) = erfc(-x / sqrt 2) / 2 to the last bit. */
/* ------------------------------------------------------------------------ */
static double norm_ppf_bisect(double prob)
{
    double lo = -40.0, hi = 40.0;
    for (int it = 0; it < 4000; ++it) {
        const double mid = 0.5 * (lo + hi);
        if (mid == lo || mid == hi) break;
        if (0.5 * erfc(-mid / sqrt(2.0)) < prob) lo = mid; else hi = mid;
    }
    return 0.5 * (lo + hi);
}

void orc_nf4_levels(double* out16)
{
    const double p = ((1.0 - 1.0 / 32.0) + (1.0 - 1.0 / 30.0)) / 2.0;
    const double top = norm_ppf_bisect(p);
    for (int i = 1; i <= 7; ++i) out16[7 - i] = -norm_ppf_bisect(0.5 + (i / 7.0) * (p - 0.5)) / top;
    out16[7] = 0.0;
    for (int i = 1; i <= 8; ++i) out16[7 + i] = norm_ppf_bisect(0.5 + (i / 8.0) * (p - 0.5)) / top;
}

uint8_t orc_nf4_encode(float q)
{
    double lv[16];
    orc_nf4_levels(lv);
    uint8_t c = 0;
    for (int i = 0; i < 15; ++i) {
        const float mid = (float)((lv[i] + lv[i + 1]) / 2.0);
        if (mid <= q) c = (uint8_t)(i + 1);
    }
    return c;
}

int orc_nf4_quantize(const float* W, int64_t n, int64_t k, int64_t ldw, uint8_t* codes, uint8_t* scales,
                     float* S_out)
{
    if (n < 0 || k < 0 || ldw < k) return ORC_ERR_ARG;
    if (k % 32 != 0) return ORC_ERR_SHAPE;
    float amax = 0.0f;
    for (int64_t i = 0; i < n; ++i)
        for (int64_t j = 0; j < k; ++j) {
            if (!isfinite(W[i * ldw + j])) return ORC_ERR_NONFINITE;
            if (fabsf(W[i * ldw + j]) > amax) amax = fabsf(W[i * ldw + j]);
        }
    float S = amax / 448.0f;
    if (S == 0.0f) S = 1.0f;
    *S_out = S;
    double lv[16];
    orc_nf4_levels(lv);
    float mids[15];
    for (int i = 0; i < 15; ++i) mids[i] = (float)((lv[i] + lv[i + 1]) / 2.0);
    for (int64_t i = 0; i < n; ++i)
        for (int64_t b = 0; b < k / 16; ++b) {
            const float* wb = W + i * ldw + b * 16;
            float amax_b = 0.0f;
            for (int t = 0; t < 16; ++t)
                if (fabsf(wb[t]) > amax_b) amax_b = fabsf(wb[t]);
            const uint8_t s = orc_e4m3_encode_pos(amax_b / S);
            const float sc = S * (float)orc_e4m3_decode(s);
            scales[i * (k / 16) + b] = s;
            for (int t = 0; t < 16; t += 2) {
                uint8_t cc[2] = {7, 7};
                for (int u = 0; u < 2; ++u) {
                    if (sc == 0.0f) continue;
                    const float q = wb[t + u] / sc;
                    uint8_t c = 0;
                    for (int m = 0; m < 15; ++m)
                        if (mids[m] <= q) c = (uint8_t)(m + 1);
                    cc[u] = c;
                }
                codes[i * (k / 2) + (b * 16 + t) / 2] = (uint8_t)(cc[0] | (cc[1] << 4));
            }
        }
    return ORC_OK;
}

/* W_hat[i][j] = S * dec(scale[i][j/16]) * level(code[i][j]), fp64. */
void orc_nf4_dequant(const uint8_t* codes, const uint8_t* scales, float S, int64_t n, int64_t k, double* W_hat)
{
    double lv[16];
    orc_nf4_levels(lv);
    for (int64_t i = 0; i < n; ++i)
        for (int64_t j = 0; j < k; ++j) {
            const uint8_t byte = codes[i * (k / 2) + j / 2];
            const uint8_t c = (j & 1) ? (byte >> 4) : (byte & 0xF);
            W_hat[i * k + j] = (double)S * (orc_e4m3_decode(scales[i * (k / 16) + j / 16]) * lv[c]);
        }
}

/* ------------------------------------------------------------------------ */
/* AQN schedule: [QeRL] Eq. 8, sigma(k) = s0 * (s1/s0)^((k-1)/(K-1)),        */
/* k = 1..K.  Library stage index `stage` = k - 1 (0..K-1); a negative stage */
/* is the warm-up stage of Algorithm 1 with sigma = 0; stages past the last  */
/* clamp to it; K == 1 gives s0.                                             */
/* ------------------------------------------------------------------------ */
double orc_aqn_sigma(int stage, int num_stages, double sigma_start, double sigma_end)
{
    if (stage < 0) return 0.0;
    if (num_stages <= 1) return sigma_start;
    if (stage > num_stages - 1) stage = num_stages - 1;
    return sigma_start * pow(sigma_end / sigma_start, (double)stage / (double)(num_stages - 1));
}

/* The digest's four decay schedules (AQN section, "Why exponential decay";
   ablation Figures 9 and 15), stage k = 1..K (library stage + 1):
   0 exponential: Eq. 8;
   1 linear:      s_start - (s_start - s_end) (k-1)/(K-1);
   2 cosine:      s_end + 1/2 (s_start - s_end) (1 + cos(pi (k-1)/(K-1)));
   3 logarithmic: s_start - (s_start - s_end) log(k) / log(K).
   Same special stages as Eq. 8 above; an unknown schedule gives NaN. */
double orc_aqn_sigma_schedule(int schedule, int stage, int num_stages, double s_start, double s_end)
{
    if (schedule < 0 || schedule > 3) return NAN;
    if (stage < 0) return 0.0;
    if (num_stages <= 1) return s_start;
    if (stage > num_stages - 1) stage = num_stages - 1;
    const int k = stage + 1, K = num_stages;
    const double frac = (double)(k - 1) / (double)(K - 1);
    switch (schedule) {
    case 0:
        return orc_aqn_sigma(stage, num_stages, s_start, s_end);
    case 1:
        return s_start - (s_start - s_end) * frac;
    case 2:
        return s_end + 0.5 * (s_start - s_end) * (1.0 + cos(acos(-1.0) * frac));
    default:
        return s_start - (s_start - s_end) * log((double)k) / log((double)K);
    }
}

/* Algorithm 1: total steps split into K stages of floor(total/K) steps. */
int orc_aqn_stage(int64_t step, int64_t total_steps, int num_stages)
{
    if (num_stages <= 0) return -1;
    if (step < 0) return -1;
    int64_t per = total_steps / num_stages;
    if (per < 1) per = 1;
    int64_t s = step / per;
    if (s > num_stages - 1) s = num_stages - 1;
    return (int)s;
}

/* ------------------------------------------------------------------------ */
/* Philox4x32-10 [SC11]: ten rounds of two 32x32->64 multiplies, key bumped  */
/* by the Weyl constants between rounds.                                     */
/* ------------------------------------------------------------------------ */
void orc_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2], uint32_t out[4])
{
    uint32_t c0 = ctr_in[0], c1 = ctr_in[1], c2 = ctr_in[2], c3 = ctr_in[3];
    uint32_t k0 = key_in[0], k1 = key_in[1];
    for (int round = 0; round < 10; ++round) {
        if (round > 0) {
            k0 += 0x9E3779B9u;
            k1 += 0xBB67AE85u;
        }
        uint64_t p0 = (uint64_t)0xD2511F53u * c0;
        uint64_t p1 = (uint64_t)0xCD9E8D57u * c2;
        uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
        uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
        uint32_t n0 = hi1 ^ c1 ^ k0;
        uint32_t n1 = lo1;
        uint32_t n2 = hi0 ^ c3 ^ k1;
        uint32_t n3 = lo0;
        c0 = n0; c1 = n1; c2 = n2; c3 = n3;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* AQN noise vector ([QeRL] Eq. 7: Z ~ N(0, sigma^2 I), one value per input
 * channel).  Generator (reading; the digest only says Gaussian): channels
 * 4i..4i+3 take Philox4x32-10 with counter (i, stream_id, counter_lo,
 * counter_hi) and key (seed_lo, seed_hi); u = (x + 0.5) * 2^-32 in fp64;
 * Box-Muller pairs (u0,u1) and (u2,u3): rho = sqrt(-2 ln u_a),
 * n = rho * cos(2 pi u_b), rho * sin(2 pi u_b); z = (float)(sigma * n). */
void orc_aqn_sample(float* z, int64_t k, float sigma, uint64_t seed, uint32_t stream_id, uint64_t counter)
{
    const double two_pi = 6.283185307179586476925286766559;
    const double inv32 = 1.0 / 4294967296.0;
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    for (int64_t i = 0; 4 * i < k; ++i) {
        uint32_t ctr[4] = {(uint32_t)i, stream_id, (uint32_t)counter, (uint32_t)(counter >> 32)};
        uint32_t r[4];
        orc_philox4x32_10(ctr, key, r);
        double u[4];
        for (int j = 0; j < 4; ++j) u[j] = ((double)r[j] + 0.5) * inv32;
        double rho0 = sqrt(-2.0 * log(u[0]));
        double rho1 = sqrt(-2.0 * log(u[2]));
        double nv[4] = {rho0 * cos(two_pi * u[1]), rho0 * sin(two_pi * u[1]),
                        rho1 * cos(two_pi * u[3]), rho1 * sin(two_pi * u[3])};
        for (int j = 0; j < 4 && 4 * i + j < k; ++j) z[4 * i + j] = (float)((double)sigma * nv[j]);
    }
}

/* ------------------------------------------------------------------------ */
/* Noisy activation.  [QeRL] "Noise Merging", Eq. 10-12: the noise folded    */
/* into the RMSNorm scale acts as a per-input-channel factor (1 + z) on the  */
/* activations, which the quantized kernel receives as bf16.  Reading:       */
/*   x_tilde = bf16_RN( float(x) * (1.0f + z) )   (fp32 ops)                 */
/* z == NULL means no noise (x_tilde = x).  Row i uses z + i * ldz: ldz = 0  */
/* is one vector for every row (the broadcast of Eq. 9), ldz = k one vector  */
/* per row (per rollout).                                                    */
/* ------------------------------------------------------------------------ */
void orc_noise_apply(const uint16_t* x, int64_t m, int64_t k, int64_t ldx, const float* z, int64_t ldz,
                     uint16_t* xt)
{
    for (int64_t i = 0; i < m; ++i)
        for (int64_t j = 0; j < k; ++j) {
            uint16_t h = x[i * ldx + j];
            if (z) {
                float f = bf16_bits_to_f32(h) * (1.0f + z[i * ldz + j]);
                h = f32_to_bf16_rn(f);
            }
            xt[i * k + j] = h;
        }
}

/* ------------------------------------------------------------------------ */
/* RMSNorm with the noise merged into its scale.  [QeRL] "Noise Merging",    */
/* Eq. 10:                                                                   */
/*   out[i][j] = (w_j + Z_j) * h[i][j] / sqrt((1/k) sum_l h[i][l]^2 + delta) */
/* h bf16 [m][k] (row stride ldh), w bf16 [k], Z fp32 [k] or NULL (plain     */
/* RMSNorm, Z = 0).  Everything in fp64; out64 (if not NULL) receives the    */
/* values, out_bits (if not NULL) their single rounding to bf16 (reading:    */
/* the digest leaves the output precision open; the linear consumes bf16).   */
/* delta is the caller's (the digest: "a small constant").  A zero row with  */
/* delta == 0 gives NaN (0 / 0), as the definition does.                     */
/* ------------------------------------------------------------------------ */
void orc_rmsnorm_noise(const uint16_t* h, int64_t m, int64_t k, int64_t ldh, const uint16_t* w, const float* Z,
                       double delta, double* out64, uint16_t* out_bits)
{
    for (int64_t i = 0; i < m; ++i) {
        const uint16_t* row = h + i * ldh;
        double ss = 0.0;
        for (int64_t j = 0; j < k; ++j) {
            const double v = (double)bf16_bits_to_f32(row[j]);
            ss += v * v;
        }
        const double denom = sqrt(ss / (double)k + delta);
        for (int64_t j = 0; j < k; ++j) {
            const double w_noise = (double)bf16_bits_to_f32(w[j]) + (Z ? (double)Z[j] : 0.0);
            const double v = w_noise * ((double)bf16_bits_to_f32(row[j]) / denom);
            if (out64) out64[i * k + j] = v;
            if (out_bits) out_bits[i * k + j] = orc_f64_to_bf16(v);
        }
    }
}

/* ------------------------------------------------------------------------ */
/* The linear layer, fp64 accumulation:                                      */
/*   y[m][c] = sum_k xt[m][k] * W_hat[c][k]                                  */
/*           + (alpha / r) * sum_j (sum_k xt[m][k] * A[j][k]) * B[c][j]      */
/* ([QeRL] Eq. 2: W + BA with B in R^{d x r}, A in R^{r x k}; for an input   */
/* row x the forward is x W^T + x A^T B^T.  A is r x k, B is n x r.)  Both   */
/* branches see the same noisy activation ([QeRL] "LoRA", interaction with   */
/* AQN).                                                                     */
/* round_xt = 1: xt is the bf16 noisy activation (the reading above);        */
/* round_xt = 0: xt = x * (1 + z) exactly in fp64 (used to check Eq. 12).    */
/* Row i of x uses noise row z + i * ldz (ldz = 0: one vector for all rows).  */
/* Output columns are the ncols indices in cols[] (all n if cols == NULL).   */
/* A or B NULL, or r == 0: no LoRA term.                                     */
/* ------------------------------------------------------------------------ */
/* One dequantized weight row c (k values) of a 4-bit format, for the linear. */
typedef void (*orc_row_dequant)(const uint8_t* codes, const uint8_t* scales, float S, int64_t k, int64_t c,
                                double* wrow);

/* Eq. 6: W_hat[c][j] = S * dec_E4M3(scale[c][j/16]) * e2m1(code[c][j]). */
static void nvfp4_row(const uint8_t* codes, const uint8_t* scales, float S, int64_t k, int64_t c, double* wrow)
{
    for (int64_t kk = 0; kk < k; ++kk) {
        uint8_t byte = codes[c * (k / 2) + kk / 2];
        uint8_t code = (kk & 1) ? (byte >> 4) : (byte & 0xF);
        wrow[kk] = (double)S * (orc_e4m3_decode(scales[c * (k / 16) + kk / 16]) * orc_e2m1_decode(code));
    }
}

/* MXFP4: W_hat[c][j] = dec_E8M0(scale[c][j/32]) * e2m1(code[c][j]) (no tensor scale). */
static void mxfp4_row(const uint8_t* codes, const uint8_t* scales, float S, int64_t k, int64_t c, double* wrow)
{
    (void)S;
    for (int64_t kk = 0; kk < k; ++kk) {
        uint8_t byte = codes[c * (k / 2) + kk / 2];
        uint8_t code = (kk & 1) ? (byte >> 4) : (byte & 0xF);
        wrow[kk] = orc_e8m0_decode(scales[c * (k / 32) + kk / 32]) * orc_e2m1_decode(code);
    }
}

/* NF4: W_hat[c][j] = S * dec_E4M3(scale[c][j/16]) * level(code[c][j]). */
static void nf4_row(const uint8_t* codes, const uint8_t* scales, float S, int64_t k, int64_t c, double* wrow)
{
    double lv[16];
    orc_nf4_levels(lv);
    for (int64_t kk = 0; kk < k; ++kk) {
        uint8_t byte = codes[c * (k / 2) + kk / 2];
        uint8_t code = (kk & 1) ? (byte >> 4) : (byte & 0xF);
        wrow[kk] = (double)S * (orc_e4m3_decode(scales[c * (k / 16) + kk / 16]) * lv[code]);
    }
}

static int lora_linear_core(const uint16_t* x, int64_t m, int64_t k, int64_t ldx,
                            const uint8_t* codes, const uint8_t* scales, float S, orc_row_dequant deq, int64_t n,
                            const float* z, int64_t ldz, const uint16_t* A, const uint16_t* B, int r, float alpha,
                            int round_xt, const int64_t* cols, int64_t ncols, double* y)
{
    if (m < 0 || k < 0 || n < 0 || ldx < k || r < 0 || ldz < 0) return ORC_ERR_ARG;
    if (k % 32 != 0) return ORC_ERR_SHAPE;
    int use_lora = (A != NULL && B != NULL && r > 0);
    if (cols == NULL) ncols = n;

    double* xt = (double*)malloc(sizeof(double) * (size_t)(m * k + 1));
    double* t = (double*)malloc(sizeof(double) * (size_t)(m * (r > 0 ? r : 1) + 1));
    double* wrow = (double*)malloc(sizeof(double) * (size_t)(k + 1));
    if (!xt || !t || !wrow) { free(xt); free(t); free(wrow); return ORC_ERR_ARG; }

    for (int64_t i = 0; i < m; ++i)
        for (int64_t j = 0; j < k; ++j) {
            uint16_t h = x[i * ldx + j];
            double v;
            if (z == NULL) v = (double)bf16_bits_to_f32(h);
            else if (round_xt) v = (double)bf16_bits_to_f32(f32_to_bf16_rn(bf16_bits_to_f32(h) * (1.0f + z[i * ldz + j])));
            else v = (double)bf16_bits_to_f32(h) * (1.0 + (double)z[i * ldz + j]);
            xt[i * k + j] = v;
        }

    if (use_lora)
        for (int64_t i = 0; i < m; ++i)
            for (int j = 0; j < r; ++j) {
                double acc = 0.0;
                for (int64_t kk = 0; kk < k; ++kk) acc += xt[i * k + kk] * (double)bf16_bits_to_f32(A[(int64_t)j * k + kk]);
                t[i * r + j] = acc;
            }

    double lora_scale = use_lora ? (double)alpha / (double)r : 0.0;
    for (int64_t ci = 0; ci < ncols; ++ci) {
        int64_t c = cols ? cols[ci] : ci;
        if (c < 0 || c >= n) { free(xt); free(t); free(wrow); return ORC_ERR_ARG; }
        deq(codes, scales, S, k, c, wrow);
        for (int64_t i = 0; i < m; ++i) {
            double acc = 0.0;
            for (int64_t kk = 0; kk < k; ++kk) acc += xt[i * k + kk] * wrow[kk];
            if (use_lora) {
                double l = 0.0;
                for (int j = 0; j < r; ++j) l += t[i * r + j] * (double)bf16_bits_to_f32(B[c * r + j]);
                acc += lora_scale * l;
            }
            y[i * ncols + ci] = acc;
        }
    }
    free(xt); free(t); free(wrow);
    return ORC_OK;
}

int orc_lora_linear(const uint16_t* x, int64_t m, int64_t k, int64_t ldx,
                    const uint8_t* codes, const uint8_t* scales, float S, int64_t n,
                    const float* z, int64_t ldz, const uint16_t* A, const uint16_t* B, int r, float alpha,
                    int round_xt, const int64_t* cols, int64_t ncols, double* y)
{
    return lora_linear_core(x, m, k, ldx, codes, scales, S, nvfp4_row, n, z, ldz, A, B, r, alpha, round_xt,
                            cols, ncols, y);
}

/* The same linear over an MXFP4 weight (codes [n][k/2], E8M0 scales        */
/* [n][k/32], as orc_mxfp4_quantize writes them): the format variant of the */
/* digest's 4-bit format comparison, with every other step unchanged.       */
int orc_mxfp4_lora_linear(const uint16_t* x, int64_t m, int64_t k, int64_t ldx,
                          const uint8_t* codes, const uint8_t* scales, int64_t n,
                          const float* z, int64_t ldz, const uint16_t* A, const uint16_t* B, int r, float alpha,
                          int round_xt, const int64_t* cols, int64_t ncols, double* y)
{
    return lora_linear_core(x, m, k, ldx, codes, scales, 1.0f, mxfp4_row, n, z, ldz, A, B, r, alpha, round_xt,
                            cols, ncols, y);
}

/* The same linear over an NF4 weight (codes [n][k/2], E4M3 scales [n][k/16], */
/* tensor scale S, as orc_nf4_quantize writes them).                          */
int orc_nf4_lora_linear(const uint16_t* x, int64_t m, int64_t k, int64_t ldx,
                        const uint8_t* codes, const uint8_t* scales, float S, int64_t n,
                        const float* z, int64_t ldz, const uint16_t* A, const uint16_t* B, int r, float alpha,
                        int round_xt, const int64_t* cols, int64_t ncols, double* y)
{
    return lora_linear_core(x, m, k, ldx, codes, scales, S, nf4_row, n, z, ldz, A, B, r, alpha, round_xt,
                            cols, ncols, y);
}

/* ------------------------------------------------------------------------ */
/* LoRA backward through the frozen NVFP4 weight ([QeRL] "Low-Rank          */
/* Adaptation (LoRA) Within Quantized Layers", gradient flow: only A and B  */
/* are trained, the quantized base weight is frozen and only passes the     */
/* input gradient).  For the forward above with the noisy activation xt,    */
/*   y = xt W_hat^T + s (xt A^T) B^T,   s = alpha / r,   t = xt A^T:         */
/*   d_xt = dy W_hat + s (dy B) A      [m][k]                                */
/*   dA   = s (dy B)^T xt              [r][k]                                */
/*   dB   = s dy^T t                   [n][r]                                */
/* fp64 throughout.  xt: [m][k] bf16 bits (the forward's input to both      */
/* branches); dy: [m][n] fp64.  A or B NULL, or r == 0: no LoRA term (dA    */
/* and dB untouched).                                                        */
/* ------------------------------------------------------------------------ */
int orc_lora_linear_backward(const uint16_t* xt, int64_t m, int64_t k, const uint8_t* codes, const uint8_t* scales,
                             float S, int64_t n, const uint16_t* A, const uint16_t* B, int r, float alpha,
                             const double* dy, double* dxt, double* dA, double* dB)
{
    if (m < 0 || k < 0 || n < 0 || r < 0) return ORC_ERR_ARG;
    if (k % 32 != 0) return ORC_ERR_SHAPE;
    const int use_lora = (A != NULL && B != NULL && r > 0);
    const double s = use_lora ? (double)alpha / (double)r : 0.0;
    double* W_hat = dxt != NULL ? (double*)malloc(sizeof(double) * (size_t)(n * k + 1)) : NULL;
    double* dyB = (double*)malloc(sizeof(double) * (size_t)(m * (r > 0 ? r : 1) + 1));
    double* t = (double*)malloc(sizeof(double) * (size_t)(m * (r > 0 ? r : 1) + 1));
    if ((dxt != NULL && !W_hat) || !dyB || !t) { free(W_hat); free(dyB); free(t); return ORC_ERR_ARG; }

    /* d_xt = dy W_hat (skipped when dxt is NULL: only the adapters' gradients) */
    if (dxt != NULL) {
        orc_nvfp4_dequant(codes, scales, S, n, k, W_hat);
        for (int64_t i = 0; i < m; ++i)
            for (int64_t kk = 0; kk < k; ++kk) {
                double acc = 0.0;
                for (int64_t c = 0; c < n; ++c) acc += dy[i * n + c] * W_hat[c * k + kk];
                dxt[i * k + kk] = acc;
            }
    }
    if (use_lora) {
        /* dy B and t = xt A^T */
        for (int64_t i = 0; i < m; ++i)
            for (int j = 0; j < r; ++j) {
                double a = 0.0, b = 0.0;
                for (int64_t c = 0; c < n; ++c) a += dy[i * n + c] * (double)bf16_bits_to_f32(B[c * r + j]);
                for (int64_t kk = 0; kk < k; ++kk)
                    b += (double)bf16_bits_to_f32(xt[i * k + kk]) * (double)bf16_bits_to_f32(A[(int64_t)j * k + kk]);
                dyB[i * r + j] = a;
                t[i * r + j] = b;
            }
        /* d_xt += s (dy B) A */
        for (int64_t i = 0; i < (dxt != NULL ? m : 0); ++i)
            for (int64_t kk = 0; kk < k; ++kk) {
                double acc = 0.0;
                for (int j = 0; j < r; ++j) acc += dyB[i * r + j] * (double)bf16_bits_to_f32(A[(int64_t)j * k + kk]);
                dxt[i * k + kk] += s * acc;
            }
        /* dA = s (dy B)^T xt */
        for (int j = 0; j < r; ++j)
            for (int64_t kk = 0; kk < k; ++kk) {
                double acc = 0.0;
                for (int64_t i = 0; i < m; ++i) acc += dyB[i * r + j] * (double)bf16_bits_to_f32(xt[i * k + kk]);
                dA[(int64_t)j * k + kk] = s * acc;
            }
        /* dB = s dy^T t */
        for (int64_t c = 0; c < n; ++c)
            for (int j = 0; j < r; ++j) {
                double acc = 0.0;
                for (int64_t i = 0; i < m; ++i) acc += dy[i * n + c] * t[i * r + j];
                dB[c * r + j] = s * acc;
            }
    }
    free(W_hat);
    free(dyB);
    free(t);
    return ORC_OK;
}
