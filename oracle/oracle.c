/*
 * oracle.c -- plain, slow CPU reference for the dense and block-scaled GEMM
 *             D = alpha * A * B^T  (A is M x K, B is N x K, both K-major).
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * bench's CPU-baseline leg may load this library.  It shares no code, header,
 * table or constant with the CUDA library under dense_block_scaled_gb300/.
 *
 * What it follows:
 *  - The GEMM and the three operand formats (BF16; MXFP8 = E4M3 values with
 *    one E8M0 scale per 1x32 K-block; NVFP4 = E2M1 values with one E4M3 scale
 *    per 1x16 K-block plus one FP32 per-tensor scale) are the ones named by
 *    "ThunderKittens 2.0 GPU Kernel优化" (yunpan.plus write-up of the
 *    HazyResearch TK 2.0 release), opening section and table of updates
 *    ("支持 MXFP8/NVFP4 低精度格式", and the BF16/MXFP8/NVFP4 GEMM kernels).
 *    The pages name the formats but give no bit layouts; the layouts used
 *    here are the standard ones for these type names (the tile types
 *    fp8e4m3, fp8e8m0 and the packed fp4e2m1_2 listed in "剖析 ThunderKittens",
 *    section "Tile 抽象").
 *  - The output is the plain definition
 *        ref[i][j] = alpha * sum_k dec(A[i][k]) * sA(i,k/bs) * dec(B[j][k]) * sB(j,k/bs)
 *    accumulated in FP64 in increasing k, together with
 *        S[i][j]   = sum_k |alpha * a_ik * b_jk|
 *    which sizes the tolerance of a comparison.
 *  - Quantisers turn FP32 inputs into codes by the rules of the workload
 *    definition (MXFP8: scale 2^ceil(log2(amax/448)), E4M3 RNE saturating;
 *    NVFP4: tensor scale amax/(6*448), block scale blockamax/(6*tensor scale)
 *    RNE to E4M3, values RNE to E2M1).  Every operation the pages leave open
 *    is taken in FP32, one correctly rounded IEEE operation at a time, in the
 *    order the rule is written.
 *
 * Every floating-point operation here is a single IEEE operation; the library
 * is compiled with -ffp-contract=off so that no multiply-add is fused.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORC_BF16 = 0, ORC_MXFP8 = 1, ORC_NVFP4 = 2 };

/* ------------------------------------------------------------------------ */
/* Decoders, written from the bit fields of each format.                     */
/* ------------------------------------------------------------------------ */

/* BF16: 1 sign, 8 exponent (bias 127), 7 mantissa bits; the upper half of an
 * IEEE binary32. */
static double dec_bf16_bits(uint16_t c) {
    int s = (c >> 15) & 1, e = (c >> 7) & 0xFF, m = c & 0x7F;
    double v;
    if (e == 0xFF) v = (m == 0) ? INFINITY : NAN;
    else if (e == 0) v = ldexp((double)m, -126 - 7);           /* subnormal */
    else v = ldexp(1.0 + m / 128.0, e - 127);
    return s ? -v : v;
}

/* E4M3 ("fn" variant): 1 sign, 4 exponent (bias 7), 3 mantissa bits, no
 * infinities; exponent 15 with mantissa 7 is NaN. Largest finite is 448. */
static double dec_e4m3_bits(uint8_t c) {
    int s = (c >> 7) & 1, e = (c >> 3) & 0xF, m = c & 0x7;
    double v;
    if (e == 0xF && m == 0x7) v = NAN;
    else if (e == 0) v = ldexp((double)m, -6 - 3);              /* subnormal */
    else v = ldexp(1.0 + m / 8.0, e - 7);
    return s ? -v : v;
}

/* E2M1: 1 sign, 2 exponent (bias 1), 1 mantissa bit. Magnitudes
 * 0, 0.5, 1, 1.5, 2, 3, 4, 6. */
static double dec_e2m1_bits(uint8_t c) {
    int s = (c >> 3) & 1, e = (c >> 1) & 0x3, m = c & 0x1;
    double v;
    if (e == 0) v = 0.5 * m;                                     /* subnormal */
    else v = ldexp(1.0 + m / 2.0, e - 1);
    return s ? -v : v;
}

/* E8M0: an unsigned power of two 2^(c-127); 0xFF is NaN. */
static double dec_e8m0_bits(uint8_t c) {
    if (c == 0xFF) return NAN;
    return ldexp(1.0, (int)c - 127);
}

/* Lookup tables, filled once from the functions above. */
static double T_BF16[65536], T_E4M3[256], T_E2M1[16], T_E8M0[256];
static int tables_ready = 0;

static void build_tables(void) {
    if (tables_ready) return;
    for (int c = 0; c < 65536; ++c) T_BF16[c] = dec_bf16_bits((uint16_t)c);
    for (int c = 0; c < 256; ++c) T_E4M3[c] = dec_e4m3_bits((uint8_t)c);
    for (int c = 0; c < 16; ++c) T_E2M1[c] = dec_e2m1_bits((uint8_t)c);
    for (int c = 0; c < 256; ++c) T_E8M0[c] = dec_e8m0_bits((uint8_t)c);
    tables_ready = 1;
}

void orc_decode_table(int which, double *out) {
    build_tables();
    switch (which) {
    case 0: memcpy(out, T_BF16, sizeof T_BF16); break;
    case 1: memcpy(out, T_E4M3, sizeof T_E4M3); break;
    case 2: memcpy(out, T_E2M1, sizeof T_E2M1); break;
    case 3: memcpy(out, T_E8M0, sizeof T_E8M0); break;
    default: break;
    }
}

/* ------------------------------------------------------------------------ */
/* GEMM                                                                      */
/* ------------------------------------------------------------------------ */

/* Decoded value of element (r, k) of an operand with K columns, scale
 * applied.  Row-major scales: sf[r * ld_sf + k / bs].  For NVFP4, element
 * 2j of a row sits in the low nibble of byte j. */
static double elem(int fmt, const void *X, const uint8_t *sf, int64_t ld_sf,
                   int64_t K, int64_t r, int64_t k) {
    if (fmt == ORC_BF16) {
        const uint16_t *x = (const uint16_t *)X;
        return T_BF16[x[r * K + k]];
    } else if (fmt == ORC_MXFP8) {
        const uint8_t *x = (const uint8_t *)X;
        return T_E4M3[x[r * K + k]] * T_E8M0[sf[r * ld_sf + k / 32]];
    } else {
        const uint8_t *x = (const uint8_t *)X;
        uint8_t byte = x[r * (K / 2) + k / 2];
        uint8_t nib = (k & 1) ? (byte >> 4) : (byte & 0xF);
        return T_E2M1[nib] * T_E4M3[sf[r * ld_sf + k / 16]];
    }
}

/* Rows [row0, row0 + nrows) of ref and S (each nrows x N, row-major).
 * B is decoded once into FP64 (N x K); each A row is decoded once.  The
 * scale is applied to each value while decoding: the product of a decoded
 * value and a decoded scale has at most 8 significant bits here, so this is
 * exact in FP64 and changes nothing in the sum. */
int orc_gemm_rows(int fmt, int64_t M, int64_t N, int64_t K,
                  const void *A, const void *B,
                  const uint8_t *sfa, const uint8_t *sfb, int64_t ld_sf,
                  double alpha, int64_t row0, int64_t nrows,
                  double *ref, double *S) {
    build_tables();
    if (row0 < 0 || nrows < 0 || row0 + nrows > M) return -1;
    double *bd = (double *)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1) * (size_t)(K > 0 ? K : 1));
    if (!bd) return -2;
#pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < N; ++j)
        for (int64_t k = 0; k < K; ++k)
            bd[j * K + k] = elem(fmt, B, sfb, ld_sf, K, j, k);
    int err = 0;
#pragma omp parallel
    {
        double *ad = (double *)malloc(sizeof(double) * (size_t)(K > 0 ? K : 1));
        if (!ad) {
#pragma omp atomic write
            err = -2;
        }
#pragma omp for schedule(dynamic, 1)
        for (int64_t ii = 0; ii < nrows; ++ii) {
            if (!ad) continue;
            int64_t i = row0 + ii;
            for (int64_t k = 0; k < K; ++k) ad[k] = elem(fmt, A, sfa, ld_sf, K, i, k);
            for (int64_t j = 0; j < N; ++j) {
                const double *b = bd + j * K;
                double acc = 0.0, mag = 0.0;
                for (int64_t k = 0; k < K; ++k) {
                    double p = ad[k] * b[k];
                    acc += p;
                    mag += fabs(alpha * p);
                }
                ref[ii * N + j] = alpha * acc;
                S[ii * N + j] = mag;
            }
        }
        free(ad);
    }
    free(bd);
    return err;
}

/* Single elements (ii[e], jj[e]); decodes on the fly, for sampling outputs of
 * GEMMs too large to evaluate in full. */
int orc_gemm_elems(int fmt, int64_t M, int64_t N, int64_t K,
                   const void *A, const void *B,
                   const uint8_t *sfa, const uint8_t *sfb, int64_t ld_sf,
                   double alpha, int64_t n_el, const int64_t *ii, const int64_t *jj,
                   double *ref, double *S) {
    build_tables();
    for (int64_t e = 0; e < n_el; ++e)
        if (ii[e] < 0 || ii[e] >= M || jj[e] < 0 || jj[e] >= N) return -1;
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t e = 0; e < n_el; ++e) {
        double acc = 0.0, mag = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            double p = elem(fmt, A, sfa, ld_sf, K, ii[e], k) *
                       elem(fmt, B, sfb, ld_sf, K, jj[e], k);
            acc += p;
            mag += fabs(alpha * p);
        }
        ref[e] = alpha * acc;
        S[e] = mag;
    }
    return 0;
}

int orc_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ------------------------------------------------------------------------ */
/* Round-to-nearest-even into a small float format, saturating.             */
/* ------------------------------------------------------------------------ */

/* Rounds |v| (finite) to the grid of a format with `mbits` mantissa bits,
 * smallest normal exponent `emin` and largest finite value `maxf`, ties to
 * the even mantissa, then clamps to maxf.  The grid spacing in the binade of
 * v is 2^(E - mbits), where E = max(floor(log2 v), emin); below 2^emin the
 * spacing stays that of the subnormals.  Everything is exact in FP64. */
static double round_small(double a, int mbits, int emin, double maxf) {
    if (a == 0.0) return 0.0;
    int ex;
    frexp(a, &ex);            /* a = f * 2^ex, f in [0.5, 1) */
    int E = ex - 1;           /* floor(log2 a) */
    if (E < emin) E = emin;
    double q = ldexp(1.0, E - mbits);
    double n = nearbyint(a / q);   /* current rounding mode: nearest-even */
    double r = n * q;
    if (r > maxf) r = maxf;
    return r;
}

/* Encodes a grid value (already rounded, |r| <= max) into E4M3 bits. */
static uint8_t enc_e4m3(double r, int neg) {
    uint8_t s = neg ? 0x80 : 0x00;
    if (r == 0.0) return s;
    if (r < ldexp(1.0, -6)) {                  /* subnormal: m * 2^-9 */
        int m = (int)(r / ldexp(1.0, -9));
        return (uint8_t)(s | m);
    }
    int ex;
    frexp(r, &ex);
    int E = ex - 1;
    int m = (int)((r / ldexp(1.0, E) - 1.0) * 8.0);
    return (uint8_t)(s | ((E + 7) << 3) | m);
}

/* Encodes a grid value into E2M1 bits (a nibble). */
static uint8_t enc_e2m1(double r, int neg) {
    uint8_t s = neg ? 0x8 : 0x0;
    if (r == 0.0) return s;
    if (r < 1.0) return (uint8_t)(s | 0x1);    /* 0.5, the only subnormal */
    int ex;
    frexp(r, &ex);
    int E = ex - 1;
    int m = (int)((r / ldexp(1.0, E) - 1.0) * 2.0);
    return (uint8_t)(s | ((E + 1) << 1) | m);
}

uint8_t orc_f32_to_e4m3(float v) {
    double a = fabs((double)v);
    return enc_e4m3(round_small(a, 3, -6, 448.0), signbit(v) != 0);
}

uint8_t orc_f32_to_e2m1(float v) {
    double a = fabs((double)v);
    return enc_e2m1(round_small(a, 1, 0, 6.0), signbit(v) != 0);
}

/* ------------------------------------------------------------------------ */
/* Quantisers (input preparation)                                            */
/* ------------------------------------------------------------------------ */

/* MXFP8, per 1x32 block along K of each row:
 *   amax = max |x|;  e = ceil(log2(amax / 448)), i.e. the smallest integer e
 *   with 448 * 2^e >= amax, found by exact comparisons; clamped to
 *   [-127, 127] (an all-zero block gets -127); scale code = e + 127;
 *   q = RNE_sat_E4M3(x * 2^-e), the product taken in FP32 (exact here).
 * K must be a multiple of 32.  SF is row-major rows x ld_sf. */
int orc_quant_mxfp8(int64_t rows, int64_t K, const float *X, uint8_t *Q,
                    uint8_t *SF, int64_t ld_sf) {
    if (K % 32 != 0 || ld_sf < K / 32) return -1;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t b = 0; b < K / 32; ++b) {
            const float *x = X + r * K + b * 32;
            float amax = 0.0f;
            for (int i = 0; i < 32; ++i) {
                float a = fabsf(x[i]);
                if (a > amax) amax = a;
            }
            int e;
            if (amax == 0.0f) {
                e = -127;
            } else {
                int ex;
                frexp((double)amax, &ex);
                e = ex - 10;   /* 448 * 2^(ex-10) < 2^(ex-1) <= amax: too small */
                while (448.0 * ldexp(1.0, e) < (double)amax) ++e;
                if (e < -127) e = -127;
                if (e > 127) e = 127;
            }
            SF[r * ld_sf + b] = (uint8_t)(e + 127);
            float inv = (float)ldexp(1.0, -e);      /* 2^-e, exact in FP32 */
            for (int i = 0; i < 32; ++i)
                Q[r * K + b * 32 + i] = orc_f32_to_e4m3(x[i] * inv);
        }
    }
    return 0;
}

/* NVFP4 with the tensor scale t given (the rule below without its first step):
 *   per 1x16 block along K:
 *   d   = fp32(6 * t);  s = RNE_sat_E4M3(fp32(blockamax / d))
 *   den = fp32(dec(s) * t)
 *   q   = RNE_sat_E2M1(fp32(x / den))
 * t <= 0 (or NaN) gives s = 0 and q = 0 everywhere; a block whose scale
 * decodes to 0 gets q = 0 (no division by zero).  A block whose maximum is
 * above 6 * 448 * t saturates: s = 448, and codes of quotients above 6 are 6.
 * Element 2j of a row goes to the low nibble of byte j.  K must be a multiple
 * of 16.  Returns 0, or -1 for a bad K or ld_sf. */
int orc_quant_nvfp4_given(int64_t rows, int64_t K, const float *X, uint8_t *Q,
                          uint8_t *SF, int64_t ld_sf, float t) {
    build_tables();
    if (K % 16 != 0 || ld_sf < K / 16) return -1;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t b = 0; b < K / 16; ++b) {
            const float *x = X + r * K + b * 16;
            uint8_t s = 0;
            float den = 0.0f;
            if (t > 0.0f) {
                float bmax = 0.0f;
                for (int i = 0; i < 16; ++i) {
                    float a = fabsf(x[i]);
                    if (a > bmax) bmax = a;
                }
                volatile float d = 6.0f * t;
                volatile float ratio = bmax / d;
                s = orc_f32_to_e4m3(ratio);
                volatile float dn = (float)T_E4M3[s] * t;
                den = dn;
            }
            SF[r * ld_sf + b] = s;
            for (int i = 0; i < 16; i += 2) {
                uint8_t lo = 0, hi = 0;
                if (den > 0.0f) {
                    volatile float q0 = x[i] / den, q1 = x[i + 1] / den;
                    lo = orc_f32_to_e2m1(q0);
                    hi = orc_f32_to_e2m1(q1);
                }
                Q[r * (K / 2) + (b * 16 + i) / 2] = (uint8_t)(lo | (hi << 4));
            }
        }
    }
    return 0;
}

/* NVFP4:
 *   t   = fp32(amax_tensor / 2688)                     (2688 = 6 * 448)
 *   then the per-block steps of orc_quant_nvfp4_given with that t.
 * An all-zero tensor gives t = 0 (all codes 0).  Returns t, or -1 for a bad
 * K or ld_sf. */
float orc_quant_nvfp4(int64_t rows, int64_t K, const float *X, uint8_t *Q,
                      uint8_t *SF, int64_t ld_sf) {
    if (K % 16 != 0 || ld_sf < K / 16) return -1.0f;
    float amax = 0.0f;
    for (int64_t i = 0; i < rows * K; ++i) {
        float a = fabsf(X[i]);
        if (a > amax) amax = a;
    }
    volatile float amax_v = amax;
    float t = amax_v / 2688.0f;
    if (orc_quant_nvfp4_given(rows, K, X, Q, SF, ld_sf, t) != 0) return -1.0f;
    return t;
}
