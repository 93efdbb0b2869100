/*
 * CPU oracle for the linear-layer hot path.  TEST INFRASTRUCTURE ONLY.
 *
 * Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline leg may load
 * this library.  It shares no code, header, table or helper with the CUDA path
 * in linear_layer_gb300/csrc; it is written from the definitions on the pages:
 *
 *   "Tensor Core" chapter (anrans ai-infra-handbooks), section "Tensor Core 做什么":
 *       D = A x B + C with low-precision inputs and an FP32 (here: wider) accumulator.
 *   same chapter, table "精度：FP16、BF16、TF32、FP8": bit splits FP16 1/5/10,
 *       BF16 1/8/7, FP8 E4M3 1/4/3; FP8 GEMMs need scaling factors per tensor,
 *       row or block (fine-grained block scaling as in DeepSeek-V3).
 *   "NVIDIA A100: chip to SIMT", section 5.1: symmetric W8A8, per-token activation
 *       scale s_x, per-output-channel weight scale s_W[o], zero point 0, integer dot
 *       product over the whole K into INT32, then dequantise once in the epilogue.
 *   same page, section 5.2 (kernel epilogue): y[o] = half(float(z) * s_x * s_W[o]),
 *       evaluated left to right in FP32, then rounded to FP16.
 *
 * Arithmetic: every floating-point input is decoded exactly to double from its bit
 * fields and every sum is a plain double loop (int64 for the integer path).  The
 * W8A8 dequantisation is the one place where the result is defined in FP32: it is
 * computed with C float multiplies (this file is compiled with -ffp-contract=off so
 * no fused multiply-add can change the rounding) and an FP16 encoder written here
 * from the IEEE binary16 definition (round to nearest, ties to even).
 *
 * The W8A8 GEMV path, the GEMM paths and the decoders are pinned by the CPU tests
 * (closed forms, brute force with exact rationals, library decoders, the printed
 * INT32 bound of the A100 page section 5.1).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ decoders */

/* IEEE binary16: sign 1, exponent 5 (bias 15), mantissa 10. */
double orc_decode_f16(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 10) & 0x1F;
  int m = h & 0x3FF;
  double v;
  if (e == 0) {
    v = ldexp((double)m, -24); /* subnormal: m * 2^(1-15-10) */
  } else if (e == 31) {
    v = (m == 0) ? INFINITY : NAN;
  } else {
    v = ldexp((double)(1024 + m), e - 25); /* (1 + m/2^10) * 2^(e-15) */
  }
  return sign ? -v : v;
}

/* bfloat16: sign 1, exponent 8 (bias 127), mantissa 7. */
double orc_decode_bf16(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 7) & 0xFF;
  int m = h & 0x7F;
  double v;
  if (e == 0) {
    v = ldexp((double)m, -133); /* m * 2^(1-127-7) */
  } else if (e == 255) {
    v = (m == 0) ? INFINITY : NAN;
  } else {
    v = ldexp((double)(128 + m), e - 134); /* (1 + m/2^7) * 2^(e-127) */
  }
  return sign ? -v : v;
}

/* FP8 E4M3 in its finite-only form: sign 1, exponent 4 (bias 7), mantissa 3; no
 * infinities; the only NaN codes are S.1111.111; largest finite value 448. */
double orc_decode_e4m3(uint8_t b) {
  int sign = (b >> 7) & 1;
  int e = (b >> 3) & 0xF;
  int m = b & 0x7;
  double v;
  if (e == 15 && m == 7) {
    v = NAN;
  } else if (e == 0) {
    v = ldexp((double)m, -9); /* m * 2^(1-7-3) */
  } else {
    v = ldexp((double)(8 + m), e - 10); /* (1 + m/8) * 2^(e-7) */
  }
  return sign ? -v : v;
}

/* FP8 E5M2: sign 1, exponent 5 (bias 15), mantissa 2, with infinities and NaNs as in
 * IEEE binary formats (exponent 31: mantissa 0 = inf, else NaN); largest finite 57344. */
double orc_decode_e5m2(uint8_t b) {
  int sign = (b >> 7) & 1;
  int e = (b >> 2) & 0x1F;
  int m = b & 0x3;
  double v;
  if (e == 31) {
    v = (m == 0) ? INFINITY : NAN;
  } else if (e == 0) {
    v = ldexp((double)m, -16); /* m * 2^(1-15-2) */
  } else {
    v = ldexp((double)(4 + m), e - 17); /* (1 + m/4) * 2^(e-15) */
  }
  return sign ? -v : v;
}

/* Round a double to the nearest binary16 (ties to even) and return its bits.
 * Written from the binary16 definition: quantum 2^-24 below 2^-14, otherwise
 * 2^(e-10) for |v| in [2^e, 2^(e+1)); magnitudes that round past 65504 become inf. */
uint16_t orc_encode_f16_rn(double v) {
  uint16_t sign = (uint16_t)(signbit(v) ? 0x8000 : 0);
  double a = fabs(v);
  if (isnan(v)) return (uint16_t)(sign | 0x7E00);
  if (isinf(a)) return (uint16_t)(sign | 0x7C00);
  if (a < ldexp(1.0, -14)) {
    double q = nearbyint(a / ldexp(1.0, -24)); /* exact division; ties to even */
    return (uint16_t)(sign | (uint16_t)q);      /* q == 1024 encodes 2^-14 itself */
  }
  int e2;
  (void)frexp(a, &e2); /* a = f * 2^e2, f in [0.5, 1) */
  int e = e2 - 1;      /* a in [2^e, 2^(e+1)) */
  double q = nearbyint(a / ldexp(1.0, e - 10));
  if (q == 2048.0) { q = 1024.0; e += 1; }
  if (e > 15) return (uint16_t)(sign | 0x7C00);
  return (uint16_t)(sign | (uint16_t)((e + 15) << 10) | (uint16_t)((int)q - 1024));
}

static double decode_in(int kind, const void* base, int64_t idx) {
  switch (kind) {
    case 0: return orc_decode_f16(((const uint16_t*)base)[idx]);
    case 1: return orc_decode_bf16(((const uint16_t*)base)[idx]);
    case 2: return orc_decode_e4m3(((const uint8_t*)base)[idx]);
    default: return NAN;
  }
}

/* ------------------------------------------------------------------ GEMM */

/*
 * D_ref[r][j] = alpha * sum_k dec(A[i][k]) * dec(B[k][j]) + beta * C[i][j],  i = rows[r]
 *
 * kind: 0 = FP16, 1 = BF16, 2 = FP8 E4M3 (unscaled).  A row-major M x K (lda),
 * B row-major K x N (ldb), C FP32 row-major (ldc), not read when beta == 0.
 * absab[r][j] = sum_k |dec A[i][k]| * |dec B[k][j]| (the tolerance scale).
 * D_ref and absab are nrows x N, row-major, double.  Either output may be NULL.
 */
int orc_gemm(int kind, int M, int N, int K, double alpha, const void* A, int64_t lda,
             const void* B, int64_t ldb, double beta, const float* C, int64_t ldc,
             const int32_t* rows, int nrows, double* D_ref, double* absab) {
  if (M < 0 || N < 0 || K < 0 || nrows < 0) return 1;
  for (int r = 0; r < nrows; ++r)
    if (rows[r] < 0 || rows[r] >= M) return 2;
  if (beta != 0.0 && C == NULL) return 3;
  /* decode B once: Bd[k][j] */
  double* Bd = (double*)malloc(sizeof(double) * ((size_t)K * (size_t)N + 1));
  if (!Bd) return 4;
  for (int64_t k = 0; k < K; ++k)
    for (int64_t j = 0; j < N; ++j) Bd[k * N + j] = decode_in(kind, B, k * ldb + j);

#pragma omp parallel for schedule(dynamic, 1)
  for (int r = 0; r < nrows; ++r) {
    const int64_t i = rows[r];
    double* acc = (double*)calloc((size_t)N + 1, sizeof(double));
    double* aab = (double*)calloc((size_t)N + 1, sizeof(double));
    for (int64_t k = 0; k < K; ++k) {
      const double a = decode_in(kind, A, i * lda + k);
      const double* brow = Bd + k * N;
      for (int64_t j = 0; j < N; ++j) {
        acc[j] += a * brow[j];
        aab[j] += fabs(a) * fabs(brow[j]);
      }
    }
    for (int64_t j = 0; j < N; ++j) {
      double d = alpha * acc[j];
      if (beta != 0.0) d += beta * (double)C[i * ldc + j];
      if (D_ref) D_ref[(int64_t)r * N + j] = d;
      if (absab) absab[(int64_t)r * N + j] = aab[j];
    }
    free(acc);
    free(aab);
  }
  free(Bd);
  return 0;
}

/*
 * FP8 E4M3 GEMM with FP32 block scales, following the block structure:
 *   D_ref[i][j] = alpha * sum_kb sA[i][kb] * sB[kb][j/128] * P_kb[i][j] + beta * C[i][j]
 *   P_kb[i][j]  = sum_{k in [128 kb, min(128 kb + 128, K))} dec8(A[i][k]) * dec8(B[k][j])
 * sA is M x ceil(K/128) (ld_sa), one scale per row and 128-wide K block;
 * sB is ceil(K/128) x ceil(N/128) (ld_sb), one scale per 128 x 128 block of B.
 * absab[i][j] = sum_k |dec8(A[i][k]) sA[i][k/128]| * |dec8(B[k][j]) sB[k/128][j/128]|.
 */
static double decode_f8(int fmt, uint8_t b) {
  return fmt == 1 ? orc_decode_e5m2(b) : orc_decode_e4m3(b);
}

/* As orc_gemm_fp8_blockscaled, with each operand's 8-bit format chosen separately
 * (fmt 0 = E4M3, 1 = E5M2). */
int orc_gemm_f8_blockscaled_mixed(int a_fmt, int b_fmt, int M, int N, int K, double alpha,
                                  const uint8_t* A, int64_t lda, const float* sA, int64_t ld_sa,
                                  const uint8_t* B, int64_t ldb, const float* sB, int64_t ld_sb,
                                  double beta, const float* C, int64_t ldc, const int32_t* rows,
                                  int nrows, double* D_ref, double* absab);

int orc_gemm_fp8_blockscaled(int M, int N, int K, double alpha, const uint8_t* A, int64_t lda,
                             const float* sA, int64_t ld_sa, const uint8_t* B, int64_t ldb,
                             const float* sB, int64_t ld_sb, double beta, const float* C,
                             int64_t ldc, const int32_t* rows, int nrows, double* D_ref,
                             double* absab) {
  return orc_gemm_f8_blockscaled_mixed(0, 0, M, N, K, alpha, A, lda, sA, ld_sa, B, ldb, sB, ld_sb,
                                       beta, C, ldc, rows, nrows, D_ref, absab);
}

int orc_gemm_f8_blockscaled_mixed(int a_fmt, int b_fmt, int M, int N, int K, double alpha,
                                  const uint8_t* A, int64_t lda, const float* sA, int64_t ld_sa,
                                  const uint8_t* B, int64_t ldb, const float* sB, int64_t ld_sb,
                                  double beta, const float* C, int64_t ldc, const int32_t* rows,
                                  int nrows, double* D_ref, double* absab) {
  if (M < 0 || N < 0 || K < 0 || nrows < 0) return 1;
  for (int r = 0; r < nrows; ++r)
    if (rows[r] < 0 || rows[r] >= M) return 2;
  if (beta != 0.0 && C == NULL) return 3;
  const int64_t KB = ((int64_t)K + 127) / 128;
  double* Bd = (double*)malloc(sizeof(double) * ((size_t)K * (size_t)N + 1));
  if (!Bd) return 4;
  for (int64_t k = 0; k < K; ++k)
    for (int64_t j = 0; j < N; ++j) Bd[k * N + j] = decode_f8(b_fmt, B[k * ldb + j]);

#pragma omp parallel for schedule(dynamic, 1)
  for (int r = 0; r < nrows; ++r) {
    const int64_t i = rows[r];
    double* acc = (double*)calloc((size_t)N + 1, sizeof(double));
    double* part = (double*)calloc((size_t)N + 1, sizeof(double));
    double* aab = (double*)calloc((size_t)N + 1, sizeof(double));
    for (int64_t kb = 0; kb < KB; ++kb) {
      const int64_t k_end = (kb + 1) * 128 < K ? (kb + 1) * 128 : K;
      for (int64_t j = 0; j < N; ++j) part[j] = 0.0;
      const double sa = (double)sA[i * ld_sa + kb];
      for (int64_t k = kb * 128; k < k_end; ++k) {
        const double a = decode_f8(a_fmt, A[i * lda + k]);
        const double* brow = Bd + k * N;
        for (int64_t j = 0; j < N; ++j) {
          part[j] += a * brow[j];
          aab[j] += fabs(a * sa) * fabs(brow[j] * (double)sB[kb * ld_sb + j / 128]);
        }
      }
      for (int64_t j = 0; j < N; ++j) acc[j] += sa * (double)sB[kb * ld_sb + j / 128] * part[j];
    }
    for (int64_t j = 0; j < N; ++j) {
      double d = alpha * acc[j];
      if (beta != 0.0) d += beta * (double)C[i * ldc + j];
      if (D_ref) D_ref[(int64_t)r * N + j] = d;
      if (absab) absab[(int64_t)r * N + j] = aab[j];
    }
    free(acc);
    free(part);
    free(aab);
  }
  free(Bd);
  return 0;
}

/* ------------------------------------------------------------------ MX block-scaled GEMM */

/*
 * OCP microscaling (MX) shared scale E8M0: an 8-bit biased exponent with no sign and no
 * mantissa, X = 2^(e - 127) for e = 0..254; the code 255 is NaN.  ("Tensor Core"
 * chapter, table of tensor-core formats per generation: Blackwell adds block-scaled
 * formats such as MXFP4 / NVFP4; the pages name the formats only.)
 */
double orc_decode_ue8m0(uint8_t e) {
  if (e == 255) return NAN;
  return ldexp(1.0, (int)e - 127);
}

/*
 * MX block-scaled 8-bit GEMM: every 32 consecutive elements along K of a row of A, and
 * of a column of B, share one E8M0 scale:
 *   D_ref[i][j] = alpha * sum_k (XA[i][k/32] * dec(A[i][k])) * (XB[j][k/32] * dec(B[k][j]))
 *                 + beta * C[i][j]
 * A row-major M x K (lda), element format a_fmt (0 = E4M3, 1 = E5M2); B row-major K x N
 * (ldb), format b_fmt; SA E8M0 codes M x ceil(K/32) (ld_sa), one per row of A and 32-wide
 * K block; SB E8M0 codes N x ceil(K/32) (ld_sb), one per column of B and 32-wide K block
 * (a last block shorter than 32 keeps its scale).  Scaled elements are exact in double and
 * every sum is a plain double loop.  absab[i][j] = sum_k |scaled a| * |scaled b|.
 */
int orc_gemm_mx_f8(int a_fmt, int b_fmt, int M, int N, int K, double alpha, const uint8_t* A, int64_t lda,
                   const uint8_t* SA, int64_t ld_sa, const uint8_t* B, int64_t ldb, const uint8_t* SB,
                   int64_t ld_sb, double beta, const float* C, int64_t ldc, const int32_t* rows, int nrows,
                   double* D_ref, double* absab) {
  if (M < 0 || N < 0 || K < 0 || nrows < 0) return 1;
  for (int r = 0; r < nrows; ++r)
    if (rows[r] < 0 || rows[r] >= M) return 2;
  if (beta != 0.0 && C == NULL) return 3;
  /* B scaled once: Bs[k][j] = XB[k/32][j] * dec(B[k][j]) */
  double* Bs = (double*)malloc(sizeof(double) * ((size_t)K * (size_t)N + 1));
  if (!Bs) return 4;
  for (int64_t k = 0; k < K; ++k)
    for (int64_t j = 0; j < N; ++j)
      Bs[k * N + j] = orc_decode_ue8m0(SB[j * ld_sb + k / 32]) * decode_f8(b_fmt, B[k * ldb + j]);

#pragma omp parallel for schedule(dynamic, 1)
  for (int r = 0; r < nrows; ++r) {
    const int64_t i = rows[r];
    double* acc = (double*)calloc((size_t)N + 1, sizeof(double));
    double* aab = (double*)calloc((size_t)N + 1, sizeof(double));
    for (int64_t k = 0; k < K; ++k) {
      const double a = orc_decode_ue8m0(SA[i * ld_sa + k / 32]) * decode_f8(a_fmt, A[i * lda + k]);
      const double* brow = Bs + k * N;
      for (int64_t j = 0; j < N; ++j) {
        acc[j] += a * brow[j];
        aab[j] += fabs(a) * fabs(brow[j]);
      }
    }
    for (int64_t j = 0; j < N; ++j) {
      double d = alpha * acc[j];
      if (beta != 0.0) d += beta * (double)C[i * ldc + j];
      if (D_ref) D_ref[(int64_t)r * N + j] = d;
      if (absab) absab[(int64_t)r * N + j] = aab[j];
    }
    free(acc);
    free(aab);
  }
  free(Bs);
  return 0;
}

/*
 * FP4 E2M1 (one sign bit, 2 exponent bits with bias 1, 1 mantissa bit; no infinities or
 * NaN): exponent 0 is subnormal, m * 0.5; otherwise (1 + m / 2) * 2^(e - 1).  The values are
 * 0, 0.5, 1, 1.5, 2, 3, 4, 6 and their negatives.  ("Tensor Core" chapter: Blackwell adds
 * FP4, including block-scaled NVFP4 / MXFP4.)
 */
double orc_decode_e2m1(uint8_t c) {
  const int sign = (c >> 3) & 1, e = (c >> 1) & 3, m = c & 1;
  const double v = e == 0 ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
  return sign ? -v : v;
}

/* NVFP4 block scale UE4M3: the E4M3 bit layout without a sign (codes 0..126; 127 is NaN). */
double orc_decode_ue4m3(uint8_t c) {
  if (c >= 128) return NAN;
  return orc_decode_e4m3(c);
}

/*
 * NVFP4 GEMM: FP4 E2M1 elements packed two per byte (element k of a row in byte k / 2, the
 * low nibble for even k), one UE4M3 scale per 16 consecutive K elements of a row of A and of
 * a column of B:
 *   D_ref[i][j] = alpha * sum_k (SA[i][k/16] * e2m1(A[i][k])) * (SB[j][k/16] * e2m1(Bt[j][k]))
 *                 + beta * C[i][j]
 * A is M x K with row pitch lda ELEMENTS (lda even); B is given transposed, Bt N x K (row j =
 * column j of B) with pitch ldbt elements; SA M x ceil(K/16) (ld_sa), SB N x ceil(K/16)
 * (ld_sb).  Scaled elements are exact in double; sums are plain double loops.
 */
int orc_gemm_nvf4(int M, int N, int K, double alpha, const uint8_t* A, int64_t lda, const uint8_t* SA,
                  int64_t ld_sa, const uint8_t* Bt, int64_t ldbt, const uint8_t* SB, int64_t ld_sb, double beta,
                  const float* C, int64_t ldc, const int32_t* rows, int nrows, double* D_ref, double* absab) {
  if (M < 0 || N < 0 || K < 0 || nrows < 0 || (lda & 1) || (ldbt & 1)) return 1;
  for (int r = 0; r < nrows; ++r)
    if (rows[r] < 0 || rows[r] >= M) return 2;
  if (beta != 0.0 && C == NULL) return 3;
  double* Bs = (double*)malloc(sizeof(double) * ((size_t)K * (size_t)N + 1));  /* Bs[j][k] */
  if (!Bs) return 4;
  for (int64_t j = 0; j < N; ++j)
    for (int64_t k = 0; k < K; ++k) {
      const uint8_t byte = Bt[(j * ldbt + k) / 2];
      const uint8_t code = (k & 1) ? (byte >> 4) : (byte & 15);
      Bs[j * K + k] = orc_decode_ue4m3(SB[j * ld_sb + k / 16]) * orc_decode_e2m1(code);
    }

#pragma omp parallel for schedule(dynamic, 1)
  for (int r = 0; r < nrows; ++r) {
    const int64_t i = rows[r];
    double* a = (double*)malloc(sizeof(double) * ((size_t)K + 1));
    for (int64_t k = 0; k < K; ++k) {
      const uint8_t byte = A[(i * lda + k) / 2];
      const uint8_t code = (k & 1) ? (byte >> 4) : (byte & 15);
      a[k] = orc_decode_ue4m3(SA[i * ld_sa + k / 16]) * orc_decode_e2m1(code);
    }
    for (int64_t j = 0; j < N; ++j) {
      double acc = 0.0, aab = 0.0;
      const double* b = Bs + j * K;
      for (int64_t k = 0; k < K; ++k) {
        acc += a[k] * b[k];
        aab += fabs(a[k]) * fabs(b[k]);
      }
      double d = alpha * acc;
      if (beta != 0.0) d += beta * (double)C[i * ldc + j];
      if (D_ref) D_ref[(int64_t)r * N + j] = d;
      if (absab) absab[(int64_t)r * N + j] = aab;
    }
    free(a);
  }
  free(Bs);
  return 0;
}

/* ------------------------------------------------------------------ W8A8 GEMV */

/*
 * Batch-1 symmetric W8A8 linear layer (A100 page, sections 5.1 and 5.2):
 *   z[o] = sum_k x[k] * W[o][k]                      (exact, int64; must fit INT32)
 *   y[o] = fp16_rn( (float(z[o]) * s_x) * s_W[o] )    (two FP32 products, left to right)
 * x int8 [K]; W int8 row-major qweight[N][ldw] (output channel o is row o); s_x is
 * one FP32 scalar; s_W FP32 [N].  z (int64 [N]) and y (FP16 bits [N]) may be NULL.
 * Returns 0, or 5 if some |z[o]| does not fit a signed 32-bit integer.
 */
int orc_gemv_w8a8(int N, int K, const int8_t* x, float s_x, const int8_t* W, int64_t ldw,
                  const float* s_W, int64_t* z, uint16_t* y) {
  if (N < 0 || K < 0) return 1;
  int bad = 0;
#pragma omp parallel for reduction(| : bad)
  for (int o = 0; o < N; ++o) {
    int64_t acc = 0;
    for (int64_t k = 0; k < K; ++k) acc += (int64_t)x[k] * (int64_t)W[(int64_t)o * ldw + k];
    if (acc > INT32_MAX || acc < INT32_MIN) bad = 1;
    if (z) z[o] = acc;
    if (y) {
      float f = (float)(int32_t)acc; /* int -> float, round to nearest even */
      float t = f * s_x;             /* FP32 product, rounded */
      float u = t * s_W[o];          /* FP32 product, rounded */
      y[o] = orc_encode_f16_rn((double)u);
    }
  }
  return bad ? 5 : 0;
}

/* ------------------------------------------------------------------ W8A8 neighbours */

/*
 * Symmetric per-token activation quantiser (A100 page, section 5.1: the activation is
 * quantised at run time by the preceding operator or a separate quantisation step,
 * per-token scale s_x, zero point 0).  Reading: for each row i of x (FP16 bits,
 * M x K, pitch ldx)
 *   s_x[i] = amax_k |x[i][k]| / 127            (FP32 division; 1 for an all-zero row)
 *   q[i][k] = clamp(rint(x[i][k] / s_x[i]), -127, 127)   (FP32 division, ties to even)
 * q is int8 M x K (pitch ldq); s is FP32 [M].
 */
int orc_quantize_per_token_f16(int M, int K, const uint16_t* x, int64_t ldx, int8_t* q, int64_t ldq,
                               float* s) {
  if (M < 0 || K < 0) return 1;
  for (int64_t i = 0; i < M; ++i) {
    double amax = 0.0;
    for (int64_t k = 0; k < K; ++k) {
      const double v = fabs(orc_decode_f16(x[i * ldx + k]));
      if (v > amax) amax = v;
    }
    const float si = (amax > 0.0) ? (float)amax / 127.0f : 1.0f;
    s[i] = si;
    for (int64_t k = 0; k < K; ++k) {
      const float v = (float)orc_decode_f16(x[i * ldx + k]);
      float r = nearbyintf(v / si);
      if (r > 127.0f) r = 127.0f;
      if (r < -127.0f) r = -127.0f;
      q[i * ldq + k] = (int8_t)r;
    }
  }
  return 0;
}

/*
 * W8A8 GEMV with the epilogue variants of the A100 page, section 5.1 (an optional bias
 * added in the floating-point epilogue after dequantisation; or requantisation to INT8
 * for a next layer that takes INT8 instead of writing FP16):
 *   v[o] = (float(z[o]) * s_x) * s_W[o]      (as orc_gemv_w8a8)
 *   v[o] = v[o] + bias[o]                     (FP32 add; only when bias != NULL)
 *   out_int8 == 0: y16[o] = fp16_rn(v[o])
 *   out_int8 != 0: y8[o]  = clamp(rint(v[o] / s_y), -127, 127)   (FP32 division, ties to even)
 */
int orc_gemv_w8a8_ex(int N, int K, const int8_t* x, float s_x, const int8_t* W, int64_t ldw,
                     const float* s_W, const float* bias, int out_int8, float s_y, int64_t* z,
                     uint16_t* y16, int8_t* y8) {
  if (N < 0 || K < 0) return 1;
  int bad = 0;
  for (int o = 0; o < N; ++o) {
    int64_t acc = 0;
    for (int64_t k = 0; k < K; ++k) acc += (int64_t)x[k] * (int64_t)W[(int64_t)o * ldw + k];
    if (acc > INT32_MAX || acc < INT32_MIN) bad = 1;
    if (z) z[o] = acc;
    float v = (float)(int32_t)acc;
    v = v * s_x;
    v = v * s_W[o];
    if (bias) v = v + bias[o];
    if (out_int8) {
      float r = nearbyintf(v / s_y);
      if (r > 127.0f) r = 127.0f;
      if (r < -127.0f) r = -127.0f;
      if (y8) y8[o] = (int8_t)r;
    } else if (y16) {
      y16[o] = orc_encode_f16_rn((double)v);
    }
  }
  return bad ? 5 : 0;
}

/* ------------------------------------------------------------------ W8A8, several tokens */

/*
 * The W8A8 linear layer for a batch of M tokens ("NVIDIA A100: chip to SIMT", section
 * 5.1: the activation scale is per token, the weight scale per output channel).  Each
 * token m is its own symmetric W8A8 product with its own s_x[m]:
 *   z[m][o] = sum_k X[m][k] * W[o][k]                 (int64; INT32 range checked)
 *   v       = (float(z[m][o]) * s_x[m]) * s_W[o]  (+ bias[o])
 *   Y[m][o] = fp16_rn(v), or clamp(rint(v / s_y), -127, 127) with out_int8
 * X is M x ldx, Y is M x ldy (2-byte or 1-byte elements), z is M x N.
 */
int orc_linear_w8a8(int M, int N, int K, const int8_t* X, int64_t ldx, const float* s_x,
                    const int8_t* W, int64_t ldw, const float* s_W, const float* bias, int out_int8,
                    float s_y, int64_t* z, uint16_t* y16, int8_t* y8, int64_t ldy) {
  if (M < 0 || N < 0 || K < 0) return 1;
  int bad = 0;
  for (int m = 0; m < M; ++m) {
    const int rc = orc_gemv_w8a8_ex(N, K, X + (int64_t)m * ldx, s_x[m], W, ldw, s_W, bias, out_int8,
                                    s_y, z ? z + (int64_t)m * N : NULL,
                                    y16 ? y16 + (int64_t)m * ldy : NULL, y8 ? y8 + (int64_t)m * ldy : NULL);
    if (rc == 5) bad = 1;
    else if (rc != 0) return rc;
  }
  return bad ? 5 : 0;
}

/* ------------------------------------------------------------------ weight-only INT8 */

/*
 * Weight-only linear layer (the Tensor Core chapter's mixed-precision GEMM with the
 * weights kept in INT8 and a per-output-channel scale, as in the A100 page section
 * 5.1's s_W[o]; the activation stays BF16):
 *   y[m][o] = s_W[o] * sum_k dec_bf16(X[m][k]) * W[o][k]  (+ bias[o])
 * in double; y is M x N (pitch N).  absab[m][o] = |s_W[o]| * sum_k |x| |W| bounds the
 * rounding of any FP32 evaluation.
 */
int orc_linear_w8a16(int M, int N, int K, const uint16_t* X, int64_t ldx, const int8_t* W, int64_t ldw,
                     const float* s_W, const float* bias, double* y, double* absab) {
  if (M < 0 || N < 0 || K < 0) return 1;
  for (int m = 0; m < M; ++m) {
    for (int o = 0; o < N; ++o) {
      double acc = 0.0, aab = 0.0;
      for (int64_t k = 0; k < K; ++k) {
        const double xv = orc_decode_bf16(X[(int64_t)m * ldx + k]);
        const double wv = (double)W[(int64_t)o * ldw + k];
        acc += xv * wv;
        aab += fabs(xv * wv);
      }
      double v = (double)s_W[o] * acc;
      if (bias) v += (double)bias[o];
      y[(int64_t)m * N + o] = v;
      if (absab) absab[(int64_t)m * N + o] = fabs((double)s_W[o]) * aab;
    }
  }
  return 0;
}
