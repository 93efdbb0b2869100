// W8A8 linear layer for a small batch of tokens on CUDA cores ("NVIDIA A100: chip to
// SIMT", section 5.1: per-token activation scale, per-output-channel weight scale, zero
// point 0; section 5.2: the FP32 dequantisation order):
//
//   z[m][o] = sum_k X[m][k] * W[o][k]                      (int8 x int8 -> int32, exact)
//   y[m][o] = fp16_rn((float(z[m][o]) * s_x[m]) * s_W[o])  (+ bias, or INT8 requantised)
//
// With a handful of tokens every weight byte still feeds only MT dot products, so the
// layer stays bound by the weight stream from HBM; sm_103a has no INT8 tensor-core MMA,
// and dp4a keeps up with HBM until MT reaches about a dozen tokens.
//
// Design (K % 16 == 0, ldx % 16 == 0, ldw % 16 == 0, 16-byte aligned X and W):
//   * the rows are cut into groups of R output channels; a "slab" is one group's
//     512-byte K slice (32 lanes x 16 bytes).  Every CTA gets the same number of whole
//     groups and its 8 warps split the CTA's slabs evenly, so all warps carry the same
//     number of weight bytes and finish together (a plain row-per-warp split of 11008
//     rows over the resident warps leaves a latency-bound last wave).
//   * per slab each lane loads its 16 bytes of the R rows straight into registers
//     (non-caching loads, D slabs in flight), reads the matching 16 bytes of every token
//     from shared memory once and reuses them for all R rows (R x MT x 4 dp4a).
//   * when a warp leaves a group (or its slab range ends) it reduces its R x MT partial
//     sums across the warp with a transposing butterfly (each step halves the values a
//     lane holds) and adds them into the CTA's shared int32 totals: a group split
//     between two warps is summed exactly, in any order.  After one barrier the CTA
//     dequantises its totals and stores y token-major (coalesced along o).
//   * programmatic dependent launch as in the batch-1 GEMV: weights stream before
//     griddepcontrol.wait; X, the scales and the outputs are touched only after it.
//     Before the wait each warp also bulk-prefetches the D steps after its first D into
//     L2 (measured on the 11008 x 4096 layer: 2 tokens 9.55 -> 8.18 us, 4 tokens
//     10.08 -> 8.53 us, 8 tokens 12.91 -> 12.21 us).
#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"

namespace ll {

namespace {

constexpr int kBtThreads = 256;
constexpr int kBtWarps = kBtThreads / 32;

struct BatchParams {
  int M, N, K;          // M <= MT tokens in this launch
  const int8_t* X;
  int64_t ldx;
  const float* x_scale;  // [M]
  const int8_t* W;
  int64_t ldw;
  const float* w_scale;  // [N]
  const float* bias;     // [N] or NULL
  int out_i8;
  const float* y_scale;
  void* Y;
  int64_t ldy;
  int32_t* Z;            // [M][ldz] or NULL
  int64_t ldz;
  int gpc;               // row groups per CTA
};

__host__ __device__ constexpr int ilog2(int v) { return v <= 1 ? 0 : 1 + ilog2(v / 2); }

// Transposing butterfly over the warp: on entry every lane holds V partial sums, on exit
// lane l holds the warp totals of indices (l >> (5 - S)) * (V >> S) + i, i < V >> S,
// where S = min(log2 V, 5); with S < 5 the 2^(5-S) lanes of a group hold equal values.
template <int V>
__device__ __forceinline__ void warp_transpose_sum(int (&v)[V], int lane) {
  constexpr int S = ilog2(V) < 5 ? ilog2(V) : 5;
#pragma unroll
  for (int st = 0; st < S; ++st) {
    const int off = 16 >> st;
    const int half = V >> (st + 1);
    const bool hi = (lane & off) != 0;
#pragma unroll
    for (int i = 0; i < half; ++i) {
      const int send = hi ? v[i] : v[i + half];
      const int keep = hi ? v[i + half] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
    }
  }
#pragma unroll
  for (int st = S; st < 5; ++st) v[0] += __shfl_xor_sync(0xffffffffu, v[0], 16 >> st);
}

template <int MT, int R, int U, int D, int CTAS>
__global__ void __launch_bounds__(kBtThreads, CTAS) w8a8_batch_kernel(const BatchParams p) {
  extern __shared__ int4 smem[];
  const int nch = p.K >> 4;               // 16-byte chunks per row
  const int Lc = (nch + 31) >> 5;         // 512-byte columns per row
  int4* xs = smem;                        // MT x nch chunks of X
  const int gpcR = p.gpc * R;
  int* tot = reinterpret_cast<int*>(smem + MT * nch);  // [MT][gpc * R] totals
  float* sws = reinterpret_cast<float*>(tot + MT * gpcR);  // [gpc * R] weight scales
  float* sbias = sws + gpcR;                                // [gpc * R] bias (0 without)
  float* sxs = sbias + gpcR;                                // [MT] token scales
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int ngroups = (p.N + R - 1) / R;
  const int g0 = blockIdx.x * p.gpc;
  const int gcount = min(p.gpc, ngroups - g0);
  const int total = gcount * Lc;  // columns of this CTA, group-major
  const int ce = static_cast<int>((static_cast<int64_t>(warp + 1) * total) / kBtWarps);
  const int cb = static_cast<int>((static_cast<int64_t>(warp) * total) / kBtWarps);

  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  // A step covers up to U consecutive columns of one group's R rows, stopping at the
  // group's end and at the warp's range end.  Positions advance without divisions.
  int pl = cb, gl = cb / Lc, kl = cb - (cb / Lc) * Lc;  // next step to load
  auto load_next = [&](int4 (&w)[R][U]) {
    const int n = min(U, min(Lc - kl, ce - pl));  // <= 0 once the range is exhausted
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
  // tokens are staged
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
  for (int i = threadIdx.x; i < MT * nch; i += kBtThreads) {
    const int m = i / nch, c = i - m * nch;
    xs[i] = m < p.M ? reinterpret_cast<const int4*>(p.X + static_cast<int64_t>(m) * p.ldx)[c]
                    : make_int4(0, 0, 0, 0);
  }
  const int rows = min(gcount * R, p.N - g0 * R);  // output channels of this CTA
  for (int i = threadIdx.x; i < MT * gpcR; i += kBtThreads) tot[i] = 0;
  for (int i = threadIdx.x; i < rows; i += kBtThreads) {  // epilogue operands, fetched early
    sws[i] = p.w_scale[g0 * R + i];
    sbias[i] = p.bias ? p.bias[g0 * R + i] : 0.0f;
  }
  if (threadIdx.x < MT) sxs[threadIdx.x] = threadIdx.x < p.M ? p.x_scale[threadIdx.x] : 0.0f;
  const float sy = p.out_i8 ? *p.y_scale : 1.0f;
  __syncthreads();

  int acc[R * MT];
#pragma unroll
  for (int i = 0; i < R * MT; ++i) acc[i] = 0;

  // reduce acc over the warp and add it into the CTA totals of local group g
  auto flush = [&](int g) {
    warp_transpose_sum<R * MT>(acc, lane);
    constexpr int S = ilog2(R * MT) < 5 ? ilog2(R * MT) : 5;
    constexpr int PER = (R * MT) >> S;
    if ((lane & ((1 << (5 - S)) - 1)) == 0) {
#pragma unroll
      for (int i = 0; i < PER; ++i) {
        const int idx = (lane >> (5 - S)) * PER + i;  // = r * MT + m
        const int r = idx / MT, m = idx - r * MT;
        if (m < p.M) atomicAdd(&tot[m * gpcR + g * R + r], acc[i]);
      }
    }
#pragma unroll
    for (int i = 0; i < R * MT; ++i) acc[i] = 0;
  };

  int pc = cb, gc = cb / Lc, kc = cb - (cb / Lc) * Lc;  // step being computed
  while (pc < ce) {
#pragma unroll
    for (int j = 0; j < D; ++j) {
      if (pc < ce) {
        const int n = min(U, min(Lc - kc, ce - pc));
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int c = (kc + u) * 32 + lane;
          if (u < n && c < nch) {
#pragma unroll
            for (int m = 0; m < MT; ++m) {
              const int4 a = xs[m * nch + c];
#pragma unroll
              for (int r = 0; r < R; ++r) {
                int t = acc[r * MT + m];
                t = __dp4a(w[j][r][u].x, a.x, t);
                t = __dp4a(w[j][r][u].y, a.y, t);
                t = __dp4a(w[j][r][u].z, a.z, t);
                t = __dp4a(w[j][r][u].w, a.w, t);
                acc[r * MT + m] = t;
              }
            }
          }
        }
        load_next(w[j]);
        pc += n;
        kc += n;
        if (kc == Lc || pc == ce) {  // leaving the group, or the range ends inside it
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

  // dequantise: thread i handles (token m, local row q), rows consecutive per token
  for (int i = threadIdx.x; i < p.M * rows; i += kBtThreads) {
    const int m = i / rows, q = i - m * rows;
    const int o = g0 * R + q;
    const int z = tot[m * gpcR + q];
    if (p.Z) p.Z[static_cast<int64_t>(m) * p.ldz + o] = z;
    const float t = __fmul_rn(__int2float_rn(z), sxs[m]);
    float u = __fmul_rn(t, sws[q]);
    if (p.bias) u = __fadd_rn(u, sbias[q]);
    if (p.out_i8) {
      const int rq = __float2int_rn(__fdiv_rn(u, sy));
      static_cast<int8_t*>(p.Y)[static_cast<int64_t>(m) * p.ldy + o] =
          static_cast<int8_t>(max(-127, min(127, rq)));
    } else {
      static_cast<__half*>(p.Y)[static_cast<int64_t>(m) * p.ldy + o] = __float2half_rn(u);
    }
  }
}

template <int MT, int R, int U, int D, int CTAS>
ll_status launch_batch(BatchParams p, const LaunchCtx& ctx) {
  auto kern = w8a8_batch_kernel<MT, R, U, D, CTAS>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024) != cudaSuccess) {
    cudaGetLastError();
    return LL_ERR_CUDA;
  }
  // the largest CTAs-per-SM count (<= CTAS) whose shared memory still lets that many
  // CTAs reside, so that the whole grid is resident at once
  const int ngroups = (p.N + R - 1) / R;
  size_t smem = 0;
  for (int c = CTAS; c >= 1; --c) {
    p.gpc = (ngroups + c * ctx.num_sms - 1) / (c * ctx.num_sms);
    smem = static_cast<size_t>(MT) * p.K + static_cast<size_t>(MT + 2) * p.gpc * R * 4 + MT * 4;
    int occ = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kBtThreads, smem) != cudaSuccess) {
      cudaGetLastError();
      return LL_ERR_CUDA;
    }
    if (occ >= c) break;
  }
  const int grid = (ngroups + p.gpc - 1) / p.gpc;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kBtThreads);
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

// Launch shapes per token-group size, from a sweep of rows per group R, 512-byte
// columns per step U, steps in flight D and CTAs per SM on the 11008 x 4096 layer.
template <int MT> struct BtTune;
template <> struct BtTune<2> { static constexpr int R = 4, U = 2, D = 2, CTAS = 2; };
template <> struct BtTune<4> { static constexpr int R = 2, U = 4, D = 1, CTAS = 3; };
template <> struct BtTune<8> { static constexpr int R = 2, U = 4, D = 1, CTAS = 2; };
template <> struct BtTune<16> { static constexpr int R = 2, U = 2, D = 2, CTAS = 2; };

template <int MT>
ll_status launch_tuned(const BatchParams& p, const LaunchCtx& ctx) {
  using T = BtTune<MT>;
  return launch_batch<MT, T::R, T::U, T::D, T::CTAS>(p, ctx);
}

// shared memory a launch of MT tokens needs at one CTA per SM (the most it can take)
template <int MT>
size_t tuned_smem(int N, int K, int num_sms) {
  using T = BtTune<MT>;
  const int ngroups = (N + T::R - 1) / T::R;
  const int gpc = (ngroups + num_sms - 1) / num_sms;  // one CTA per SM: the largest case
  return static_cast<size_t>(MT) * K + static_cast<size_t>(MT + 2) * gpc * T::R * 4 + MT * 4;
}

size_t batch_smem(int MT, int N, int K, int num_sms) {
  switch (MT) {
    case 16: return tuned_smem<16>(N, K, num_sms);
    case 8: return tuned_smem<8>(N, K, num_sms);
    case 4: return tuned_smem<4>(N, K, num_sms);
    default: return tuned_smem<2>(N, K, num_sms);
  }
}

constexpr size_t kBtSmemLimit = 200 * 1024;

// From this many tokens on, weight passes of up to 32 tokens run on the tensor cores
// (w8a8_tc.cu); below it the dp4a kernel is as fast or faster (measured on the
// 11008 x 4096 layer: equal at 16 tokens, 1.8x slower at 32 in two 16-token passes).
constexpr int kTcMinTokens = 17;

}  // namespace

ll_status launch_linear_w8a8(int M, int N, int K, const int8_t* X, int64_t ldx, const float* x_scale,
                             const int8_t* W, int64_t ldw, const float* w_scale, const float* bias,
                             int out_i8, const float* y_scale, void* Y, int64_t ldy, int32_t* Z,
                             int64_t ldz, const LaunchCtx& ctx) {
  const size_t ysize = out_i8 ? 1 : 2;
  const bool aligned = (reinterpret_cast<uintptr_t>(X) % 16 == 0) && (reinterpret_cast<uintptr_t>(W) % 16 == 0) &&
                       (K % 16 == 0) && (ldx % 16 == 0) && (ldw % 16 == 0) && K > 0;
  int m0 = 0;
  while (m0 < M) {
    const int left = M - m0;
    if (aligned && left >= kTcMinTokens) {  // tensor cores: up to 32 tokens per weight pass
      const int mt = left < 32 ? left : 32;
      const ll_status st = launch_w8a8_tc(
          mt, N, K, X + static_cast<int64_t>(m0) * ldx, ldx, x_scale + m0, W, ldw, w_scale, bias, out_i8, y_scale,
          static_cast<char*>(Y) + static_cast<int64_t>(m0) * ldy * ysize, ldy,
          Z ? Z + static_cast<int64_t>(m0) * ldz : nullptr, ldz, ctx);
      if (st != LL_OK) return st;
      m0 += mt;
      continue;
    }
    int MT = left > 8 ? 16 : left > 4 ? 8 : left > 2 ? 4 : left;
    while (MT > 1 && batch_smem(MT, N, K, ctx.num_sms) > kBtSmemLimit) MT >>= 1;
    if (!aligned || MT == 1) {  // one token at a time through the batch-1 GEMV
      const ll_status st = launch_gemv_w8a8_ex(
          N, K, X + static_cast<int64_t>(m0) * ldx, x_scale + m0, nullptr, nullptr, nullptr, W, ldw, w_scale, bias,
          out_i8, y_scale, static_cast<char*>(Y) + static_cast<int64_t>(m0) * ldy * ysize,
          Z ? Z + static_cast<int64_t>(m0) * ldz : nullptr, ctx);
      if (st != LL_OK) return st;
      m0 += 1;
      continue;
    }
    const int mt = left < MT ? left : MT;
    BatchParams p;
    p.M = mt;
    p.N = N;
    p.K = K;
    p.X = X + static_cast<int64_t>(m0) * ldx;
    p.ldx = ldx;
    p.x_scale = x_scale + m0;
    p.W = W;
    p.ldw = ldw;
    p.w_scale = w_scale;
    p.bias = bias;
    p.out_i8 = out_i8;
    p.y_scale = y_scale;
    p.Y = static_cast<char*>(Y) + static_cast<int64_t>(m0) * ldy * ysize;
    p.ldy = ldy;
    p.Z = Z ? Z + static_cast<int64_t>(m0) * ldz : nullptr;
    p.ldz = ldz;
    p.gpc = 1;
    ll_status st;
    switch (MT) {
      case 16: st = launch_tuned<16>(p, ctx); break;
      case 8: st = launch_tuned<8>(p, ctx); break;
      case 4: st = launch_tuned<4>(p, ctx); break;
      default: st = launch_tuned<2>(p, ctx); break;
    }
    if (st != LL_OK) return st;
    m0 += mt;
  }
  return LL_OK;
}

}  // namespace ll
