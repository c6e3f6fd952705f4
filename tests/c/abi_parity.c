/* The C ABI used from plain C (no Python, no torch): for each format, inputs
 * drawn from a seeded generator are quantised by the CPU oracle's own C
 * quantisers, the row-major scales go to the device as they are and
 * tkg_scales_to_tiled converts them, the GEMM runs through include/tkg_gemm.h,
 * and every output is compared with the oracle's FP64 GEMM at the acceptance
 * tolerance |D - ref| <= 2^-7 |ref| + 1e-5 sum|alpha a b|.
 *
 * Test code: built and run by tests/test_c_abi.py.  Exit status 0 when every
 * format passes. */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "tkg_gemm.h"

/* the CPU oracle (oracle/oracle.c) */
int orc_gemm_rows(int fmt, int64_t M, int64_t N, int64_t K, const void *A, const void *B, const uint8_t *sfa,
                  const uint8_t *sfb, int64_t ld_sf, double alpha, int64_t row0, int64_t nrows, double *ref,
                  double *S);
int orc_quant_mxfp8(int64_t rows, int64_t K, const float *X, uint8_t *Q, uint8_t *SF, int64_t ld_sf);
float orc_quant_nvfp4(int64_t rows, int64_t K, const float *X, uint8_t *Q, uint8_t *SF, int64_t ld_sf);

/* seeded N(0,1) values: xorshift64* and the Box-Muller transform */
static uint64_t rng_state;
static double uniform01(void) {
  rng_state ^= rng_state >> 12;
  rng_state ^= rng_state << 25;
  rng_state ^= rng_state >> 27;
  return ((rng_state * 0x2545F4914F6CDD1DULL) >> 11) * (1.0 / 9007199254740992.0);
}
static void normals(float *x, size_t n, uint64_t seed) {
  rng_state = seed * 0x9E3779B97F4A7C15ULL + 1;
  for (size_t i = 0; i < n; i += 2) {
    double u1 = uniform01(), u2 = uniform01();
    if (u1 < 1e-300) u1 = 1e-300;
    const double r = sqrt(-2.0 * log(u1)), a = 6.283185307179586 * u2;
    x[i] = (float)(r * cos(a));
    if (i + 1 < n) x[i + 1] = (float)(r * sin(a));
  }
}

/* FP32 -> BF16 code, round to nearest even (finite inputs) */
static uint16_t to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}
static double from_bf16(uint16_t c) {
  uint32_t u = (uint32_t)c << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

#define CHECK_CUDA(x)                                                   \
  do {                                                                  \
    if ((x) != cudaSuccess) {                                           \
      fprintf(stderr, "%s:%d CUDA error in %s\n", __FILE__, __LINE__, #x); \
      return 1;                                                         \
    }                                                                   \
  } while (0)
#define CHECK_TKG(x)                                                                          \
  do {                                                                                        \
    tkg_status s_ = (x);                                                                      \
    if (s_ != TKG_OK) {                                                                       \
      fprintf(stderr, "%s:%d %s -> %s\n", __FILE__, __LINE__, #x, tkg_status_string(s_));    \
      return 1;                                                                               \
    }                                                                                         \
  } while (0)

static int compare(const char *what, int m, int n, const uint16_t *d, const double *ref, const double *S) {
  long bad = 0;
  double worst = 0.0;
  for (long i = 0; i < (long)m * n; ++i) {
    const double err = fabs(from_bf16(d[i]) - ref[i]);
    const double bound = ldexp(fabs(ref[i]), -7) + 1e-5 * S[i];
    if (!(err <= bound)) ++bad;
    if (err > worst) worst = err;
  }
  printf("%s %dx%d: %ld of %ld outside tolerance (max |err| %.3g)\n", what, m, n, bad, (long)m * n, worst);
  return bad == 0 ? 0 : 1;
}

/* fmt: 0 BF16, 1 MXFP8, 2 NVFP4 (the oracle's numbering) */
static int run(int fmt, int m, int n, int k, uint64_t seed) {
  const float alpha = 0.75f;
  float *a = (float *)malloc(sizeof(float) * (size_t)m * k), *b = (float *)malloc(sizeof(float) * (size_t)n * k);
  normals(a, (size_t)m * k, seed);
  normals(b, (size_t)n * k, seed + 1);
  const int bs = fmt == 1 ? 32 : 16;
  const int kb = fmt == 0 ? 0 : k / bs;
  const int ld_sf = fmt == 0 ? 0 : ((kb + 15) / 16) * 16;
  const size_t row_bytes = fmt == 0 ? (size_t)k * 2 : (fmt == 1 ? (size_t)k : (size_t)k / 2);
  uint8_t *qa = (uint8_t *)malloc(row_bytes * m), *qb = (uint8_t *)malloc(row_bytes * n);
  uint8_t *sa = (uint8_t *)calloc((size_t)m * (ld_sf ? ld_sf : 1), 1), *sb = (uint8_t *)calloc((size_t)n * (ld_sf ? ld_sf : 1), 1);
  float ta = 1.0f, tb = 1.0f;
  if (fmt == 0) {
    for (size_t i = 0; i < (size_t)m * k; ++i) ((uint16_t *)qa)[i] = to_bf16(a[i]);
    for (size_t i = 0; i < (size_t)n * k; ++i) ((uint16_t *)qb)[i] = to_bf16(b[i]);
  } else if (fmt == 1) {
    if (orc_quant_mxfp8(m, k, a, qa, sa, ld_sf) || orc_quant_mxfp8(n, k, b, qb, sb, ld_sf)) return 1;
  } else {
    ta = orc_quant_nvfp4(m, k, a, qa, sa, ld_sf);
    tb = orc_quant_nvfp4(n, k, b, qb, sb, ld_sf);
    if (ta < 0.0f || tb < 0.0f) return 1;
  }

  void *dA, *dB, *dD, *dSA = NULL, *dSB = NULL, *dSAr = NULL, *dSBr = NULL;
  float *dT = NULL;
  CHECK_CUDA(cudaMalloc(&dA, row_bytes * m));
  CHECK_CUDA(cudaMalloc(&dB, row_bytes * n));
  CHECK_CUDA(cudaMalloc(&dD, (size_t)m * n * 2));
  CHECK_CUDA(cudaMemcpy(dA, qa, row_bytes * m, cudaMemcpyHostToDevice));
  CHECK_CUDA(cudaMemcpy(dB, qb, row_bytes * n, cudaMemcpyHostToDevice));
  if (fmt != 0) {
    /* row-major scales as the oracle wrote them, converted by the library */
    CHECK_CUDA(cudaMalloc(&dSAr, (size_t)m * ld_sf));
    CHECK_CUDA(cudaMalloc(&dSBr, (size_t)n * ld_sf));
    CHECK_CUDA(cudaMemcpy(dSAr, sa, (size_t)m * ld_sf, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(dSBr, sb, (size_t)n * ld_sf, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMalloc(&dSA, tkg_scale_bytes(m, k, bs)));
    CHECK_CUDA(cudaMalloc(&dSB, tkg_scale_bytes(n, k, bs)));
    CHECK_TKG(tkg_scales_to_tiled(m, kb, dSAr, ld_sf, dSA, 0));
    CHECK_TKG(tkg_scales_to_tiled(n, kb, dSBr, ld_sf, dSB, 0));
  }
  if (fmt == 0) {
    CHECK_TKG(tkg_gemm_bf16(m, n, k, dA, dB, dD, alpha, 0));
  } else if (fmt == 1) {
    CHECK_TKG(tkg_gemm_mxfp8(m, n, k, dA, dB, dSA, dSB, dD, alpha, 0));
  } else {
    float t2[2] = {ta, tb};
    CHECK_CUDA(cudaMalloc((void **)&dT, sizeof t2));
    CHECK_CUDA(cudaMemcpy(dT, t2, sizeof t2, cudaMemcpyHostToDevice));
    CHECK_TKG(tkg_gemm_nvfp4(m, n, k, dA, dB, dSA, dSB, dT, dT + 1, dD, alpha, 0));
  }
  CHECK_TKG(tkg_get_device_status(0));
  uint16_t *d = (uint16_t *)malloc((size_t)m * n * 2);
  CHECK_CUDA(cudaMemcpy(d, dD, (size_t)m * n * 2, cudaMemcpyDeviceToHost));

  /* the oracle: alpha_eff = fp32(fp32(alpha * tA) * tB) for NVFP4 */
  volatile float at = alpha * ta;
  volatile float aeff = at * tb;
  double *ref = (double *)malloc(sizeof(double) * (size_t)m * n), *S = (double *)malloc(sizeof(double) * (size_t)m * n);
  if (orc_gemm_rows(fmt, m, n, k, qa, qb, sa, sb, ld_sf, (double)(fmt == 2 ? aeff : alpha), 0, m, ref, S)) return 1;
  const char *names[3] = {"bf16", "mxfp8", "nvfp4"};
  const int rc = compare(names[fmt], m, n, d, ref, S);

  cudaFree(dA);
  cudaFree(dB);
  cudaFree(dD);
  if (dSA) cudaFree(dSA);
  if (dSB) cudaFree(dSB);
  if (dSAr) cudaFree(dSAr);
  if (dSBr) cudaFree(dSBr);
  if (dT) cudaFree(dT);
  free(a); free(b); free(qa); free(qb); free(sa); free(sb); free(d); free(ref); free(S);
  return rc;
}

int main(void) {
  int rc = 0;
  rc |= run(0, 300, 264, 512, 11);
  rc |= run(1, 300, 264, 512, 12);
  rc |= run(2, 300, 264, 512, 13);
  rc |= run(0, 1024, 2048, 512, 14);
  rc |= run(2, 1024, 2048, 1024, 15);
  printf(rc == 0 ? "c abi parity: ok\n" : "c abi parity: FAILED\n");
  return rc;
}
