// Pieces shared by the tcgen05 GEMM kernels (gemm_tc.cu, gemm_mx.cu): the kernel parameter
// block, the instruction-descriptor fields, the grouped tile order and the row epilogue
// that stores D straight from accumulator registers.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"

namespace ll {

struct GemmParams {
  int M, N, K;
  float alpha, beta;
  const float* C;
  int64_t ldc;
  void* D;
  int64_t ldd;
  int d_type;
  int c_vec, d_vec;  // rows of C / D may be accessed with 4-element vectors
  int d_row16;       // rows of D start on 16-byte boundaries
  int epi_tma;       // CTA-pair 16-bit epilogue through TMA (C and D rows 16-byte aligned)
  int epi_res;       // CTA-pair epilogue for FP32 D rows not 16-byte aligned: C by TMA row classes, D by sectors
  const float* sA;
  int64_t ld_sa;
  const float* sB;
  int64_t ld_sb;
  const uint8_t* xA;  // MX: E8M0 scale codes of A (M x ld_xa) and of B (N x ld_xb)
  int64_t ld_xa;
  const uint8_t* xB;
  int64_t ld_xb;
  uint32_t* status;
  uint64_t timeout_ns;
  int group_m;
};

// Operand formats of an MMA, packed as a | (b << 3): kind::f16 0 = FP16, 1 = BF16;
// kind::f8f6f4 0 = E4M3, 1 = E5M2.
__host__ __device__ constexpr uint32_t fmt_pair(uint32_t a, uint32_t b) { return a | (b << 3); }

// tcgen05 instruction descriptor (kind::f16 / kind::f8f6f4): D = F32 (bits 4-5 = 1),
// A/B format (bits 7-9 / 10-12), A K-major (bit 15 = 0), B MN-major (bit 16 = 1),
// N >> 3 (bits 17-22), M >> 4 (bits 24-28).
__host__ __device__ constexpr uint32_t make_idesc(uint32_t fmts, int n, int m) {
  return (1u << 4) | ((fmts & 7u) << 7) | (((fmts >> 3) & 7u) << 10) | (1u << 16) |
         (static_cast<uint32_t>(n >> 3) << 17) | (static_cast<uint32_t>(m >> 4) << 24);
}

__device__ __forceinline__ void tile_coords(int t, int num_m, int num_n, int group_m, int& mb,
                                            int& nb) {
  const int span = group_m * num_n;
  const int g = t / span;
  const int first_m = g * group_m;
  const int gsz = min(num_m - first_m, group_m);
  const int r = t - g * span;
  mb = first_m + r % gsz;
  nb = r / gsz;
}

// Row epilogue.  A chunk is 32 columns n .. n + 31 of one row m of D, held by one lane:
//   D[m][n] = alpha * acc[m][n] + beta * C[m][n]   (C not read when beta == 0)
// evaluated as fma(beta, C, alpha * acc) in FP32 and rounded once to the output type, as
// every other epilogue of the library does.  C may alias D only as the same matrix (same
// base and pitch): each element is read before it is written.
// a[j] = alpha * a[j] (+ beta * C[m][n + j]) for one 32-column chunk of row m (< M),
// C consumed four columns at a time as it arrives.
__device__ __forceinline__ void combine_c_row(const GemmParams& p, int m, int n, float (&a)[32]) {
#pragma unroll
  for (int j = 0; j < 32; ++j) a[j] *= p.alpha;
  if (p.beta == 0.0f) return;
  const float* crow = p.C + static_cast<int64_t>(m) * p.ldc + n;
  if (n + 32 <= p.N && p.c_vec) {
#pragma unroll
    for (int j = 0; j < 32; j += 4) {
      const float4 cv = *reinterpret_cast<const float4*>(crow + j);
      a[j] = fmaf(p.beta, cv.x, a[j]);
      a[j + 1] = fmaf(p.beta, cv.y, a[j + 1]);
      a[j + 2] = fmaf(p.beta, cv.z, a[j + 2]);
      a[j + 3] = fmaf(p.beta, cv.w, a[j + 3]);
    }
  } else {
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (n + j < p.N) a[j] = fmaf(p.beta, crow[j], a[j]);
  }
}

// Store final values (alpha and beta applied) of one chunk of row m, masked to N.
__device__ __forceinline__ void store_row_final(const GemmParams& p, int m, int n, const float (&o)[32]) {
  const int64_t off = static_cast<int64_t>(m) * p.ldd + n;
  const bool full = n + 32 <= p.N;
  if (p.d_type == LL_OUT_F32) {
    float* dp = static_cast<float*>(p.D) + off;
    if (full && p.d_row16) {
#pragma unroll
      for (int j = 0; j < 32; j += 4)
        *reinterpret_cast<float4*>(dp + j) = make_float4(o[j], o[j + 1], o[j + 2], o[j + 3]);
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (n + j < p.N) dp[j] = o[j];
    }
  } else {
    const bool bf = p.d_type == LL_OUT_BF16;
    uint16_t* dp = reinterpret_cast<uint16_t*>(p.D) + off;
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (n + j < p.N)
        dp[j] = bf ? __bfloat16_as_ushort(__float2bfloat16_rn(o[j])) : __half_as_ushort(__float2half_rn(o[j]));
  }
}

// Up to CH consecutive chunks of one row (lane = row m), read straight from the FP32
// accumulator registers (the FP8 promotion epilogue, which holds CH = 4 chunks).
template <int CH>
__device__ __forceinline__ void epilogue_rows(const GemmParams& p, int m, int n0,
                                              float (&acc)[CH][32]) {
  if (m >= p.M) return;
#pragma unroll
  for (int c = 0; c < CH; ++c) {
    const int n = n0 + 32 * c;
    if (n >= p.N) break;
    combine_c_row(p, m, n, acc[c]);
    if (p.d_type != LL_OUT_F32 && n + 32 <= p.N && p.d_row16) {  // 16-byte vector stores
      uint16_t* dp = reinterpret_cast<uint16_t*>(p.D) + static_cast<int64_t>(m) * p.ldd + n;
      const bool bf = p.d_type == LL_OUT_BF16;
#pragma unroll
      for (int j = 0; j < 32; j += 8) {
        uint32_t w4[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          if (bf) {
            __nv_bfloat162 h2 = __floats2bfloat162_rn(acc[c][j + 2 * i], acc[c][j + 2 * i + 1]);
            w4[i] = *reinterpret_cast<uint32_t*>(&h2);
          } else {
            __half2 h2 = __floats2half2_rn(acc[c][j + 2 * i], acc[c][j + 2 * i + 1]);
            w4[i] = *reinterpret_cast<uint32_t*>(&h2);
          }
        }
        *reinterpret_cast<uint4*>(dp + j) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
      }
    } else {
      store_row_final(p, m, n, acc[c]);
    }
  }
}

inline GemmParams make_gemm_params(const GemmArgs& a, const LaunchCtx& ctx) {
  GemmParams p;
  p.M = a.M;
  p.N = a.N;
  p.K = a.K;
  p.alpha = a.alpha;
  p.beta = a.beta;
  p.C = a.C;
  p.ldc = a.ldc;
  p.D = a.D;
  p.ldd = a.ldd;
  p.d_type = a.d_type;
  const int dsize = a.d_type == LL_OUT_F32 ? 4 : 2;
  p.c_vec = a.C != nullptr && (reinterpret_cast<uintptr_t>(a.C) % 16 == 0) && ((a.ldc * 4) % 16 == 0);
  // vector stores: 16 bytes (FP32) or 8 bytes (BF16 / FP16) per lane, at 4-column steps
  p.d_vec = (reinterpret_cast<uintptr_t>(a.D) % (4 * dsize) == 0) && ((a.ldd * dsize) % (4 * dsize) == 0);
  p.d_row16 = (reinterpret_cast<uintptr_t>(a.D) % 16 == 0) && ((a.ldd * dsize) % 16 == 0);
  p.epi_tma = 0;
  p.epi_res = 0;
  p.sA = a.scale_a;
  p.ld_sa = a.ld_sa;
  p.sB = a.scale_b;
  p.ld_sb = a.ld_sb;
  p.xA = a.mx_sa;
  p.ld_xa = a.ld_mx_sa;
  p.xB = a.mx_sb;
  p.ld_xb = a.ld_mx_sb;
  p.status = ctx.status;
  p.timeout_ns = ctx.timeout_ns;
  p.group_m = 8;

  return p;
}

}  // namespace ll
