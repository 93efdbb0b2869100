// Weight-only INT8 linear layer with BF16 activations for a few tokens (the Tensor Core
// chapter's mixed-precision GEMM with INT8-stored weights; the per-output-channel scale
// of the A100 page, section 5.1):
//
//   y[m][o] = cast_out( s_W[o] * sum_k x[m][k] * W[o][k]  (+ bias[o]) ),  FP32 accumulation
//
// Decode-sized batches stream every weight byte once for a few FMAs, so the layer is
// bound by HBM like the W8A8 GEMV; it runs on CUDA cores:
//   * the weight walk is the one of the W8A8 small-batch kernel: rows in groups of R, a
//     CTA gets whole groups, its 8 warps split the CTA's 512-byte columns evenly, each
//     lane keeps U 16-byte pieces of R rows in flight (non-caching loads, D steps ahead);
//   * int8 -> FP32 exactly: the byte (offset by 128) placed under the FP32 exponent of
//     2^23 reads 2^23 + 128 + w, one subtraction leaves w; the MT tokens' activations are
//     staged once per CTA in shared memory (BF16) and reused for the R rows; conversion
//     and FMAs run on packed FP32 pairs (sub / fma .f32x2), even and odd K accumulating in
//     the two halves;
//   * a group split between warps is combined deterministically: every warp writes its
//     reduced partial sums into its own shared-memory slot and the epilogue adds the 8
//     slots in a fixed order, so results do not depend on timing.
// Programmatic dependent launch: weights stream before griddepcontrol.wait, activations,
// scales and outputs are touched only after it.  Before the wait each warp of the
// several-token kernel also bulk-prefetches its next D steps into L2 (measured on the
// 11008 x 4096 layer: 2 tokens 14.19 -> 13.01 us, 4 tokens 18.74 -> 17.60 us; the same
// for the single-token row kernel changed nothing, it is bound by its instruction stream).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"

namespace ll {

namespace {

constexpr int kWoThreads = 256;
constexpr int kWoWarps = kWoThreads / 32;

struct WoParams {
  int M, N, K;
  const __nv_bfloat16* X;
  int64_t ldx;
  const int8_t* W;
  int64_t ldw;
  const float* w_scale;
  const float* bias;
  int y_type;  // ll_out_type
  void* Y;
  int64_t ldy;
  int gpc;     // row groups per CTA
};

__host__ __device__ constexpr int ilog2(int v) { return v <= 1 ? 0 : 1 + ilog2(v / 2); }

// Transposing butterfly (as in the W8A8 small-batch kernel), FP32: lane l ends with the
// warp totals of indices (l >> (5 - S)) * (V >> S) + i, S = min(log2 V, 5).
template <int V>
__device__ __forceinline__ void warp_transpose_sum(float (&v)[V], int lane) {
  constexpr int S = ilog2(V) < 5 ? ilog2(V) : 5;
#pragma unroll
  for (int st = 0; st < S; ++st) {
    const int off = 16 >> st;
    const int half = V >> (st + 1);
    const bool hi = (lane & off) != 0;
#pragma unroll
    for (int i = 0; i < half; ++i) {
      const float send = hi ? v[i] : v[i + half];
      const float keep = hi ? v[i + half] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
    }
  }
#pragma unroll
  for (int st = S; st < 5; ++st) v[0] += __shfl_xor_sync(0xffffffffu, v[0], 16 >> st);
}

// bytes j and j + 1 of the 32-bit word u (already offset by 128) as two exact FP32
// values packed in 64 bits: each byte set under the exponent of 2^23 reads
// 2^23 + 128 + w, one packed subtraction leaves w.
__device__ __forceinline__ uint64_t bytes_to_f32x2(uint32_t u, int j) {
  uint32_t b0, b1;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(b0) : "r"(u), "r"(0x4B000000u), "r"(0x7540u | static_cast<uint32_t>(j)));
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(b1) : "r"(u), "r"(0x4B000000u), "r"(0x7540u | static_cast<uint32_t>(j + 1)));
  uint64_t v, r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(v) : "r"(b0), "r"(b1));
  const uint64_t magic = 0x4B0000804B000080ull;  // (2^23 + 128, 2^23 + 128)
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(v), "l"(magic));
  return r;
}

// two BF16 (one 32-bit word) as two FP32 packed in 64 bits
__device__ __forceinline__ uint64_t bf16x2_to_f32x2(uint32_t xa) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(xa << 16), "r"(xa & 0xFFFF0000u));
  return r;
}

__device__ __forceinline__ void fma_f32x2(uint64_t& acc, uint64_t a, uint64_t b) {
  asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc) : "l"(a), "l"(b));
}

template <int MT, int R, int U, int D, int CTAS>
__global__ void __launch_bounds__(kWoThreads, CTAS) w8a16_kernel(const WoParams p) {
  extern __shared__ int4 smem[];
  const int nch = p.K >> 4;        // 16-byte weight pieces per row
  const int Lc = (nch + 31) >> 5;  // 512-byte columns per row
  const int gpcR = p.gpc * R;
  int4* xs = smem;                                                    // [MT][K] activations, BF16
  float* part = reinterpret_cast<float*>(smem + MT * (p.K >> 3));      // [8 warps][gpc * R][MT]
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int ngroups = (p.N + R - 1) / R;
  const int g0 = blockIdx.x * p.gpc;
  const int gcount = min(p.gpc, ngroups - g0);
  const int total = gcount * Lc;
  const int ce = static_cast<int>((static_cast<int64_t>(warp + 1) * total) / kWoWarps);
  const int cb = static_cast<int>((static_cast<int64_t>(warp) * total) / kWoWarps);

  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  int pl = cb, gl = cb / Lc, kl = cb - (cb / Lc) * Lc;  // next step to load
  auto load_next = [&](int4 (&w)[R][U]) {
    const int n = min(U, min(Lc - kl, ce - pl));
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const int row = (g0 + gl) * R + r;
      const int4* src = reinterpret_cast<const int4*>(p.W + static_cast<int64_t>(row) * p.ldw) + kl * 32 + lane;
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const bool ok = u < n && row < p.N && (kl + u) * 32 + lane < nch;
        w[r][u] = ok ? ld_stream(src + 32 * u) : make_int4(0, 0, 0, 0);
      }
    }
    if (n > 0) {
      pl += n;
      kl += n;
      if (kl == Lc) {
        kl = 0;
        ++gl;
      }
    }
  };

  int4 w[D][R][U];
#pragma unroll
  for (int j = 0; j < D; ++j) load_next(w[j]);
  // the D steps after those go to L2 (one bulk prefetch per row and step) while the
  // activations are staged
  if (lane == 0) {
    int ql = pl, qg = gl, qk = kl;
    for (int j = 0; j < D; ++j) {
      const int n = min(U, min(Lc - qk, ce - ql));
      if (n <= 0) break;
      const int kbytes = min(n * 512, p.K - qk * 512);
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const int row = (g0 + qg) * R + r;
        if (row < p.N && kbytes > 0)
          bulk_prefetch_l2(p.W + static_cast<int64_t>(row) * p.ldw + qk * 512, static_cast<uint32_t>(kbytes));
      }
      ql += n;
      qk += n;
      if (qk == Lc) {
        qk = 0;
        ++qg;
      }
    }
  }

  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int xp = p.K >> 3;  // 16-byte pieces (8 BF16) per token
  for (int i = threadIdx.x; i < MT * xp; i += kWoThreads) {
    const int m = i / xp, c = i - m * xp;
    xs[i] = m < p.M ? reinterpret_cast<const int4*>(p.X + static_cast<int64_t>(m) * p.ldx)[c] : make_int4(0, 0, 0, 0);
  }
  for (int i = threadIdx.x; i < kWoWarps * gpcR * MT; i += kWoThreads) part[i] = 0.0f;
  __syncthreads();

  // even and odd K of each (row, token) accumulate in the two halves of a packed pair
  uint64_t acc2[R * MT];
#pragma unroll
  for (int i = 0; i < R * MT; ++i) acc2[i] = 0ull;

  auto flush = [&](int g) {  // this warp's partial sums of local group g -> its slot
    float acc[R * MT];
#pragma unroll
    for (int i = 0; i < R * MT; ++i) {
      uint32_t lo, hi;
      asm("mov.b64 {%0, %1}, %2;" : "=r"(lo), "=r"(hi) : "l"(acc2[i]));
      acc[i] = __fadd_rn(__uint_as_float(lo), __uint_as_float(hi));
      acc2[i] = 0ull;
    }
    warp_transpose_sum<R * MT>(acc, lane);
    constexpr int S = ilog2(R * MT) < 5 ? ilog2(R * MT) : 5;
    constexpr int PER = (R * MT) >> S;
    if ((lane & ((1 << (5 - S)) - 1)) == 0) {
#pragma unroll
      for (int i = 0; i < PER; ++i) {
        const int idx = (lane >> (5 - S)) * PER + i;  // = r * MT + m
        const int r = idx / MT, m = idx - r * MT;
        part[(warp * gpcR + g * R + r) * MT + m] = acc[i];
      }
    }
  };

  int pc = cb, gc = cb / Lc, kc = cb - (cb / Lc) * Lc;
  while (pc < ce) {
#pragma unroll
    for (int j = 0; j < D; ++j) {
      if (pc < ce) {
        const int n = min(U, min(Lc - kc, ce - pc));
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int c = (kc + u) * 32 + lane;
          if (u < n && c < nch) {
            uint32_t xr[MT][8];  // the 16 activations of piece c for every token (BF16 pairs)
#pragma unroll
            for (int m = 0; m < MT; ++m) {
              const int4* xq = xs + m * (p.K >> 3) + 2 * c;
              const int4 lo = xq[0], hi = xq[1];
              xr[m][0] = lo.x; xr[m][1] = lo.y; xr[m][2] = lo.z; xr[m][3] = lo.w;
              xr[m][4] = hi.x; xr[m][5] = hi.y; xr[m][6] = hi.z; xr[m][7] = hi.w;
            }
#pragma unroll
            for (int e4 = 0; e4 < 4; ++e4) {  // one 32-bit word (4 weights) of each row at a time
              uint64_t w01[R], w23[R];
#pragma unroll
              for (int r = 0; r < R; ++r) {
                const uint32_t wd = e4 == 0 ? w[j][r][u].x : e4 == 1 ? w[j][r][u].y : e4 == 2 ? w[j][r][u].z : w[j][r][u].w;
                const uint32_t q = wd ^ 0x80808080u;
                w01[r] = bytes_to_f32x2(q, 0);
                w23[r] = bytes_to_f32x2(q, 2);
              }
#pragma unroll
              for (int m = 0; m < MT; ++m) {
                const uint64_t x01 = bf16x2_to_f32x2(xr[m][2 * e4]);
                const uint64_t x23 = bf16x2_to_f32x2(xr[m][2 * e4 + 1]);
#pragma unroll
                for (int r = 0; r < R; ++r) {
                  fma_f32x2(acc2[r * MT + m], x01, w01[r]);
                  fma_f32x2(acc2[r * MT + m], x23, w23[r]);
                }
              }
            }
          }
        }
        load_next(w[j]);
        pc += n;
        kc += n;
        if (kc == Lc || pc == ce) {
          flush(gc);
          if (kc == Lc) {
            kc = 0;
            ++gc;
          }
        }
      }
    }
  }
  __syncthreads();

  // epilogue: thread i -> (token m, local row q), rows consecutive per token
  const int rows = min(gcount * R, p.N - g0 * R);
  for (int i = threadIdx.x; i < p.M * rows; i += kWoThreads) {
    const int m = i / rows, q = i - m * rows;
    const int o = g0 * R + q;
    float s = 0.0f;
#pragma unroll
    for (int wp = 0; wp < kWoWarps; ++wp) s = __fadd_rn(s, part[(wp * gpcR + q) * MT + m]);
    float v = __fmul_rn(s, p.w_scale[o]);
    if (p.bias) v = __fadd_rn(v, p.bias[o]);
    const int64_t off = static_cast<int64_t>(m) * p.ldy + o;
    if (p.y_type == LL_OUT_F32)
      static_cast<float*>(p.Y)[off] = v;
    else if (p.y_type == LL_OUT_BF16)
      static_cast<__nv_bfloat16*>(p.Y)[off] = __float2bfloat16_rn(v);
    else
      static_cast<__half*>(p.Y)[off] = __float2half_rn(v);
  }
}

// One token, K a multiple of 4096 (exact rows, as the W8A8 GEMV's exact path): warp g of
// the grid owns rows g, g + G, ...; each lane streams 8 16-byte pieces of a row per batch
// (4 KB per warp in flight), with the activation staged once per CTA in shared memory.
// Measured 4491 vs 3798 GB/s on the 11008 x 4096 layer against the general walk; refilling
// each half-batch's registers as soon as that half is multiplied in took 10.48 -> 10.20 us.
__global__ void __launch_bounds__(256, 3) w8a16_row_kernel(const WoParams p) {
  extern __shared__ int4 smem[];  // the token's K activations, BF16
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int lane = threadIdx.x & 31;
  const int G = gridDim.x * 8;
  const int nb = p.K >> 12;  // 4096-element batches per row
  int r = blockIdx.x * 8 + (threadIdx.x >> 5);
  int4 w[8];
  auto ld_batch = [&](int rr, int b) {
#pragma unroll
    for (int j = 0; j < 8; ++j)
      w[j] = rr < p.N ? ld_stream(reinterpret_cast<const int4*>(p.W + static_cast<int64_t>(rr) * p.ldw) + b * 256 + lane + 32 * j)
                      : make_int4(0, 0, 0, 0);
  };
  ld_batch(r, 0);
  asm volatile("griddepcontrol.wait;" ::: "memory");
  for (int i = threadIdx.x; i < (p.K >> 3); i += 256) smem[i] = reinterpret_cast<const int4*>(p.X)[i];
  __syncthreads();
  // The registers hold one 4096-element batch (row r, batch b) as two halves of 4
  // pieces; each half's registers are refilled with the next batch's half as soon as the
  // half has been multiplied in, so the next weights are in flight during the other
  // half's work (the products and their order are unchanged).
  auto ld_half = [&](int rr, int bb, int j0) {
#pragma unroll
    for (int j = j0; j < j0 + 4; ++j)
      w[j] = rr < p.N ? ld_stream(reinterpret_cast<const int4*>(p.W + static_cast<int64_t>(rr) * p.ldw) + bb * 256 + lane + 32 * j)
                      : make_int4(0, 0, 0, 0);
  };
  auto mul_piece = [&](uint64_t& acc2, int bb, int j) {
    const int c = bb * 256 + lane + 32 * j;  // 16-byte weight piece: K 16 c .. 16 c + 15
    const int4 lo = smem[2 * c], hi = smem[2 * c + 1];
    const uint32_t xr[8] = {static_cast<uint32_t>(lo.x), static_cast<uint32_t>(lo.y), static_cast<uint32_t>(lo.z),
                            static_cast<uint32_t>(lo.w), static_cast<uint32_t>(hi.x), static_cast<uint32_t>(hi.y),
                            static_cast<uint32_t>(hi.z), static_cast<uint32_t>(hi.w)};
#pragma unroll
    for (int e4 = 0; e4 < 4; ++e4) {
      const uint32_t wd = e4 == 0 ? w[j].x : e4 == 1 ? w[j].y : e4 == 2 ? w[j].z : w[j].w;
      const uint32_t q = wd ^ 0x80808080u;
      fma_f32x2(acc2, bf16x2_to_f32x2(xr[2 * e4]), bytes_to_f32x2(q, 0));
      fma_f32x2(acc2, bf16x2_to_f32x2(xr[2 * e4 + 1]), bytes_to_f32x2(q, 2));
    }
  };
  uint64_t acc2 = 0ull;
  int b = 0;
  while (r < p.N) {
    int rn = r, bn = b + 1;  // the batch after this one
    if (bn == nb) {
      bn = 0;
      rn = r + G;
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) mul_piece(acc2, b, j);
    ld_half(rn, bn, 0);
#pragma unroll
    for (int j = 4; j < 8; ++j) mul_piece(acc2, b, j);
    ld_half(rn, bn, 4);
    if (bn == 0) {  // row r complete
      uint32_t lo, hi;
      asm("mov.b64 {%0, %1}, %2;" : "=r"(lo), "=r"(hi) : "l"(acc2));
      float v = __fadd_rn(__uint_as_float(lo), __uint_as_float(hi));
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
      if (lane == 0) {
        v = __fmul_rn(v, p.w_scale[r]);
        if (p.bias) v = __fadd_rn(v, p.bias[r]);
        if (p.y_type == LL_OUT_F32)
          static_cast<float*>(p.Y)[r] = v;
        else if (p.y_type == LL_OUT_BF16)
          static_cast<__nv_bfloat16*>(p.Y)[r] = __float2bfloat16_rn(v);
        else
          static_cast<__half*>(p.Y)[r] = __float2half_rn(v);
      }
      acc2 = 0ull;
    }
    r = rn;
    b = bn;
  }
}

// Any shape or alignment: one warp per (token, output row), scalar loads.
__global__ void __launch_bounds__(256) w8a16_plain_kernel(const WoParams p) {
  const int lane = threadIdx.x & 31;
  const int64_t id = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  if (id >= static_cast<int64_t>(p.M) * p.N) return;
  const int m = static_cast<int>(id / p.N), o = static_cast<int>(id - static_cast<int64_t>(m) * p.N);
  const int8_t* wrow = p.W + static_cast<int64_t>(o) * p.ldw;
  const __nv_bfloat16* xrow = p.X + static_cast<int64_t>(m) * p.ldx;
  float acc = 0.0f;
  for (int k = lane; k < p.K; k += 32) acc = __fmaf_rn(__bfloat162float(xrow[k]), static_cast<float>(wrow[k]), acc);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (lane == 0) {
    float v = __fmul_rn(acc, p.w_scale[o]);
    if (p.bias) v = __fadd_rn(v, p.bias[o]);
    const int64_t off = static_cast<int64_t>(m) * p.ldy + o;
    if (p.y_type == LL_OUT_F32)
      static_cast<float*>(p.Y)[off] = v;
    else if (p.y_type == LL_OUT_BF16)
      static_cast<__nv_bfloat16*>(p.Y)[off] = __float2bfloat16_rn(v);
    else
      static_cast<__half*>(p.Y)[off] = __float2half_rn(v);
  }
}

template <int MT, int R, int U, int D, int CTAS>
ll_status launch_wo(WoParams p, const LaunchCtx& ctx) {
  auto kern = w8a16_kernel<MT, R, U, D, CTAS>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024) != cudaSuccess) {
    cudaGetLastError();
    return LL_ERR_CUDA;
  }
  const int ngroups = (p.N + R - 1) / R;
  size_t smem = 0;
  for (int c = CTAS; c >= 1; --c) {  // the most CTAs per SM whose shared memory fits
    p.gpc = (ngroups + c * ctx.num_sms - 1) / (c * ctx.num_sms);
    smem = static_cast<size_t>(MT) * p.K * 2 + static_cast<size_t>(kWoWarps) * p.gpc * R * MT * 4;
    int occ = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kWoThreads, smem) != cudaSuccess) {
      cudaGetLastError();
      return LL_ERR_CUDA;
    }
    if (occ >= c) break;
  }
  const int grid = (ngroups + p.gpc - 1) / p.gpc;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kWoThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = ctx.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kern, p) != cudaSuccess) {
    cudaGetLastError();
    return LL_ERR_CUDA;
  }
  return LL_OK;
}

constexpr size_t kWoSmemLimit = 200 * 1024;

}  // namespace

ll_status launch_linear_w8a16(int M, int N, int K, const void* X, int64_t ldx, const int8_t* W, int64_t ldw,
                              const float* w_scale, const float* bias, int y_type, void* Y, int64_t ldy,
                              const LaunchCtx& ctx) {
  const size_t ysize = y_type == LL_OUT_F32 ? 4 : 2;
  const bool aligned = (reinterpret_cast<uintptr_t>(X) % 16 == 0) && (reinterpret_cast<uintptr_t>(W) % 16 == 0) &&
                       (K % 16 == 0) && (ldx % 8 == 0) && (ldw % 16 == 0) && K > 0;
  WoParams p;
  p.N = N;
  p.K = K;
  p.ldx = ldx;
  p.W = W;
  p.ldw = ldw;
  p.w_scale = w_scale;
  p.bias = bias;
  p.y_type = y_type;
  p.ldy = ldy;
  p.gpc = 1;
  if (!aligned) {
    p.M = M;
    p.X = static_cast<const __nv_bfloat16*>(X);
    p.Y = Y;
    const int64_t warps = static_cast<int64_t>(M) * N;
    w8a16_plain_kernel<<<static_cast<unsigned>((warps + 7) / 8), 256, 0, ctx.stream>>>(p);
    return cudaGetLastError() == cudaSuccess ? LL_OK : LL_ERR_CUDA;
  }
  int m0 = 0;
  while (m0 < M) {
    const int left = M - m0;
    int MT = left >= 4 ? 4 : left >= 2 ? 2 : 1;
    while (MT > 1 && static_cast<size_t>(MT) * K * 2 > kWoSmemLimit) MT >>= 1;
    if (static_cast<size_t>(MT) * K * 2 > kWoSmemLimit) {  // K too long to stage: plain kernel
      p.M = left;
      p.X = static_cast<const __nv_bfloat16*>(X) + static_cast<int64_t>(m0) * ldx;
      p.Y = static_cast<char*>(Y) + static_cast<int64_t>(m0) * ldy * ysize;
      const int64_t warps = static_cast<int64_t>(left) * N;
      w8a16_plain_kernel<<<static_cast<unsigned>((warps + 7) / 8), 256, 0, ctx.stream>>>(p);
      return cudaGetLastError() == cudaSuccess ? LL_OK : LL_ERR_CUDA;
    }
    p.M = MT;
    p.X = static_cast<const __nv_bfloat16*>(X) + static_cast<int64_t>(m0) * ldx;
    p.Y = static_cast<char*>(Y) + static_cast<int64_t>(m0) * ldy * ysize;
    if (MT == 1 && K % 4096 == 0) {  // one token, exact rows
      const int smem = K * 2;
      if (smem > 48 * 1024 &&
          cudaFuncSetAttribute(w8a16_row_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) {
        cudaGetLastError();
        return LL_ERR_CUDA;
      }
      int grid = 3 * ctx.num_sms;
      const int need = (N + 7) / 8;
      if (need < grid) grid = need;
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(grid);
      cfg.blockDim = dim3(256);
      cfg.dynamicSmemBytes = smem;
      cfg.stream = ctx.stream;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
      attr[0].val.programmaticStreamSerializationAllowed = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      if (cudaLaunchKernelEx(&cfg, w8a16_row_kernel, p) != cudaSuccess) {
        cudaGetLastError();
        return LL_ERR_CUDA;
      }
      m0 += 1;
      continue;
    }
    ll_status st;
    switch (MT) {
      // launch shapes (rows per group, pieces per step, steps in flight, CTAs per SM)
      // from a sweep on the 11008 x 4096 layer
      case 4: st = launch_wo<4, 4, 2, 1, 2>(p, ctx); break;
      case 2: st = launch_wo<2, 2, 4, 2, 2>(p, ctx); break;
      default: st = launch_wo<1, 4, 2, 2, 2>(p, ctx); break;
    }
    if (st != LL_OK) return st;
    m0 += MT;
  }
  return LL_OK;
}

}  // namespace ll
