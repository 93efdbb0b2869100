// Batch-1 W8A8 linear layer on CUDA cores ("NVIDIA A100: chip to SIMT", sections 5.1,
// 5.2 and 5.5):
//
//   z[o] = sum_k x[k] * W[o][k]   (int8 x int8 -> int32, exact)
//   y[o] = fp16_rn((float(z[o]) * s_x) * s_W[o])
//
// At batch 1 every weight byte is used once, so the kernel is bound by HBM bandwidth
// and does not use tensor cores (an M = 1 tile would leave 15/16 of an MMA idle).
//
// Design (fast path: K % 16 == 0, ldw % 16 == 0, 16-byte aligned x and W):
//   * 3 CTAs of 8 warps per SM (the fused FP16-activation kernel: one CTA of 24 warps,
//     since every CTA quantises the whole activation, a correctly rounded divide per
//     element; 8.01 -> 7.66 us against 3 CTAs); warp g of the grid owns rows g, g + G, ...
//   * each lane streams 16-byte chunks of its warp's row (lane-strided, 8 chunks =
//     4 KB per warp in flight) with non-caching loads straight into registers, and
//     multiplies them with the matching 16 bytes of x (staged once per CTA in shared
//     memory) with four dp4a;  the next row's first chunks are requested before the
//     warp reduces and dequantises the current row, so loads stay in flight.
//   * programmatic dependent launch: the kernel lets the next kernel of the stream be
//     scheduled as soon as SMs free up, and itself starts streaming weights before the
//     preceding kernel has finished; x and x_scale are read, and y / z written, only
//     after griddepcontrol.wait, i.e. after all preceding work on the stream is done.
//     Before the wait each warp also sends its second row to L2 with one bulk prefetch,
//     so DRAM stays busy while x is staged (or quantised); measured 7.40 -> 7.12 us on
//     the 11008 x 4096 layer (8.41 -> 7.95 us with the fused quantiser).  Prefetching
//     more rows ahead was slower (9.4 us).
//   Measured on GB300 against a TMA bulk-copy ring and a cp.async ring (one CTA per
//   SM): direct loads sustained the highest bandwidth for this 45 MB stream.
// Any other shape or alignment runs a plain warp-per-row kernel with scalar loads.
#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"

namespace ll {

constexpr int kGvThreads = 256;
constexpr int kGvCtasPerSm = 3;
// The fused FP16-activation kernel runs the same 24 warps per SM as one CTA: every CTA
// quantises the whole activation (a correctly rounded divide per element), so one CTA
// per SM does a third of that work.
__host__ __device__ constexpr int gv_threads(bool xf16) { return xf16 ? 3 * kGvThreads : kGvThreads; }
__host__ __device__ constexpr int gv_ctas_per_sm(bool xf16) { return xf16 ? 1 : kGvCtasPerSm; }
constexpr int kGvBatch = 8;  // 16-byte chunks per lane in flight (4 KB per warp)

struct GemvParams {
  int N, K;
  const int8_t* x;        // int8 activation (or NULL when xh is given)
  const float* x_scale;   // its scale (device, one float)
  const __half* xh;       // FP16 activation, quantised in the kernel (fused path)
  int8_t* xq_out;         // fused path: where CTA 0 stores the quantised activation
  float* xs_out;          //   and its scale (both optional)
  const int8_t* W;
  int64_t ldw;
  const float* w_scale;
  const float* bias;      // optional, added after dequantisation
  int out_i8;             // 0: FP16 y; 1: INT8 y requantised with *y_scale
  const float* y_scale;
  void* y;
  int32_t* z_out;
};

__device__ __forceinline__ int warp_sum(int v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}

// v = (float(z) * s_x) * s_W[o] (+ bias[o]); y = fp16_rn(v), or
// y = clamp(rint(v / s_y), -127, 127) for an INT8 next layer.
__device__ __forceinline__ void dequant_store(const GemvParams& p, int o, int z, float sx, float sw,
                                              float sy) {
  if (p.z_out) p.z_out[o] = z;
  const float f = __int2float_rn(z);
  const float t = __fmul_rn(f, sx);
  float u = __fmul_rn(t, sw);
  if (p.bias) u = __fadd_rn(u, p.bias[o]);
  if (p.out_i8) {
    const int r = __float2int_rn(__fdiv_rn(u, sy));
    static_cast<int8_t*>(p.y)[o] = static_cast<int8_t>(max(-127, min(127, r)));
  } else {
    static_cast<__half*>(p.y)[o] = __float2half_rn(u);
  }
}

// Symmetric per-token quantisation of one row of K FP16 values by the whole CTA:
// s = amax / 127 (1 for an all-zero row), q = clamp(rint(x / s), -127, 127), each
// step one FP32 operation rounded to nearest even.  q goes to shared memory `xq`;
// returns s.  `red` is 32 floats of shared scratch.  When x is 16-byte aligned, K is a
// multiple of 8 and the row fits VEC_MAX 8-element chunks per thread, each thread
// loads its chunks once (16-byte loads) and keeps them in registers for both passes.
template <int THREADS>
__device__ __forceinline__ float block_amax(float amax, float* red) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
  __syncthreads();
  if (threadIdx.x < 32) {
    float v = threadIdx.x < THREADS / 32 ? red[threadIdx.x] : 0.0f;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
    if (threadIdx.x == 0) red[0] = v;
  }
  __syncthreads();
  return red[0];
}

__device__ __forceinline__ int8_t quant1(float v, float s) {
  const int r = __float2int_rn(__fdiv_rn(v, s));
  return static_cast<int8_t>(max(-127, min(127, r)));
}

template <int THREADS>
__device__ __forceinline__ float quantize_row_to_smem(const __half* x, int K, int8_t* xq, float* red) {
  constexpr int VEC_MAX = 4;
  if ((reinterpret_cast<uintptr_t>(x) % 16 == 0) && (K % 8 == 0) && K <= THREADS * 8 * VEC_MAX) {
    const int nvec = K / 8;
    uint4 v[VEC_MAX];
    float amax = 0.0f;
#pragma unroll
    for (int j = 0; j < VEC_MAX; ++j) {
      const int c = threadIdx.x + j * THREADS;
      v[j] = c < nvec ? reinterpret_cast<const uint4*>(x)[c] : make_uint4(0, 0, 0, 0);
      const __half2* h = reinterpret_cast<const __half2*>(&v[j]);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = __half22float2(h[e]);
        amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
      }
    }
    const float a = block_amax<THREADS>(amax, red);
    const float s = a > 0.0f ? __fdiv_rn(a, 127.0f) : 1.0f;
#pragma unroll
    for (int j = 0; j < VEC_MAX; ++j) {
      const int c = threadIdx.x + j * THREADS;
      if (c < nvec) {
        const __half2* h = reinterpret_cast<const __half2*>(&v[j]);
        uint32_t lo = 0, hi = 0;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 f = __half22float2(h[e]);
          const uint32_t pair = static_cast<uint8_t>(quant1(f.x, s)) | (static_cast<uint32_t>(static_cast<uint8_t>(quant1(f.y, s))) << 8);
          if (e < 2)
            lo |= pair << (16 * e);
          else
            hi |= pair << (16 * (e - 2));
        }
        reinterpret_cast<uint2*>(xq)[c] = make_uint2(lo, hi);
      }
    }
    return s;
  }
  float amax = 0.0f;
  for (int k = threadIdx.x; k < K; k += THREADS) amax = fmaxf(amax, fabsf(__half2float(x[k])));
  const float a = block_amax<THREADS>(amax, red);
  const float s = a > 0.0f ? __fdiv_rn(a, 127.0f) : 1.0f;
  for (int k = threadIdx.x; k < K; k += THREADS) xq[k] = quant1(__half2float(x[k]), s);
  return s;
}

// Request chunks base + lane + 32 j (j < kGvBatch) of row `row`; chunks past the row are zero.
__device__ __forceinline__ void load_batch(int4 (&w)[kGvBatch], const int4* row, int base,
                                           int nch, int lane) {
#pragma unroll
  for (int j = 0; j < kGvBatch; ++j) {
    const int c = base + lane + 32 * j;
    w[j] = (c < nch) ? ld_stream(row + c) : make_int4(0, 0, 0, 0);
  }
}

// EXACT: K is a multiple of 32 lanes x kGvBatch x 16 bytes (4096), so every batch is
// whole and the row loop runs without per-chunk bounds checks (measured ~8% faster on
// the 11008 x 4096 layer than the general loop).
template <bool XF16, bool EXACT>
__global__ void __launch_bounds__(gv_threads(XF16), gv_ctas_per_sm(XF16)) gemv_w8a8_kernel(const GemvParams p) {
  constexpr int THREADS = gv_threads(XF16);
  extern __shared__ int4 xs[];  // x, K bytes
  __shared__ float red[32];
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int lane = threadIdx.x & 31;
  const int G = gridDim.x * (THREADS / 32);
  const int nch = p.K / 16;  // 16-byte chunks per row
  int r = blockIdx.x * (THREADS / 32) + (threadIdx.x >> 5);
  int4 w[kGvBatch];
  if (r < p.N) load_batch(w, reinterpret_cast<const int4*>(p.W + static_cast<int64_t>(r) * p.ldw), 0, nch, lane);
  // the warp's next row goes to L2 while the activation is staged (or quantised)
  if (lane == 0 && r + G < p.N) bulk_prefetch_l2(p.W + static_cast<int64_t>(r + G) * p.ldw, static_cast<uint32_t>(p.K));

  asm volatile("griddepcontrol.wait;" ::: "memory");  // x / outputs: after preceding work
  float sx;
  if (XF16) {  // fused upstream quantiser: every CTA quantises x into its shared memory
    sx = quantize_row_to_smem<THREADS>(p.xh, p.K, reinterpret_cast<int8_t*>(xs), red);
    __syncthreads();
    if (blockIdx.x == 0) {
      if (p.xq_out)
        for (int i = threadIdx.x; i < nch; i += THREADS) reinterpret_cast<int4*>(p.xq_out)[i] = xs[i];
      if (p.xs_out && threadIdx.x == 0) *p.xs_out = sx;
    }
  } else {
    for (int i = threadIdx.x; i < nch; i += THREADS) xs[i] = reinterpret_cast<const int4*>(p.x)[i];
    __syncthreads();
    sx = *p.x_scale;
  }
  const float sy = p.out_i8 ? *p.y_scale : 1.0f;

  while (r < p.N) {
    const int4* row = reinterpret_cast<const int4*>(p.W + static_cast<int64_t>(r) * p.ldw);
    int acc0 = 0, acc1 = 0;
    for (int base = 0;;) {
#pragma unroll
      for (int j = 0; j < kGvBatch; ++j) {
        const int c = base + lane + 32 * j;
        if (EXACT || c < nch) {
          const int4 a = xs[c];
          acc0 = __dp4a(w[j].x, a.x, acc0);
          acc1 = __dp4a(w[j].y, a.y, acc1);
          acc0 = __dp4a(w[j].z, a.z, acc0);
          acc1 = __dp4a(w[j].w, a.w, acc1);
        }
      }
      base += 32 * kGvBatch;
      if (base >= nch) break;
      if (EXACT) {
#pragma unroll
        for (int j = 0; j < kGvBatch; ++j) w[j] = ld_stream(row + base + lane + 32 * j);
      } else {
        load_batch(w, row, base, nch, lane);
      }
    }
    const int rn = r + G;
    if (rn < p.N)  // next row in flight while this one is reduced and stored
      load_batch(w, reinterpret_cast<const int4*>(p.W + static_cast<int64_t>(rn) * p.ldw), 0, nch, lane);
    const int z = warp_sum(acc0 + acc1);
    if (lane == 0) dequant_store(p, r, z, sx, p.w_scale[r], sy);
    r = rn;
  }
}

// Any shape or alignment: one warp per output row, scalar loads.
__global__ void __launch_bounds__(256) gemv_w8a8_plain_kernel(const GemvParams p) {
  const int lane = threadIdx.x & 31;
  const int o = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (o >= p.N) return;
  const int8_t* wrow = p.W + static_cast<int64_t>(o) * p.ldw;
  int acc = 0;
  for (int k = lane; k < p.K; k += 32) acc += static_cast<int>(p.x[k]) * static_cast<int>(wrow[k]);
  const int z = warp_sum(acc);
  if (lane == 0) dequant_store(p, o, z, *p.x_scale, p.w_scale[o], p.out_i8 ? *p.y_scale : 1.0f);
}

// Per-token quantiser, one CTA per row (x FP16 M x ldx -> q int8 M x ldq, s FP32 [M]).
__global__ void __launch_bounds__(256) quantize_per_token_kernel(int M, int K, const __half* x,
                                                                 int64_t ldx, int8_t* q, int64_t ldq,
                                                                 float* scale) {
  extern __shared__ int8_t qrow[];
  __shared__ float red[32];
  for (int i = blockIdx.x; i < M; i += gridDim.x) {
    const float s = quantize_row_to_smem<256>(x + static_cast<int64_t>(i) * ldx, K, qrow, red);
    __syncthreads();
    for (int k = threadIdx.x; k < K; k += 256) q[static_cast<int64_t>(i) * ldq + k] = qrow[k];
    if (threadIdx.x == 0) scale[i] = s;
    __syncthreads();
  }
}

static ll_status launch_gemv(const GemvParams& p0, const LaunchCtx& ctx) {
  GemvParams p = p0;
  const int N = p.N, K = p.K;
  const bool xh = p.xh != nullptr;
  const bool x_aligned = xh ? (reinterpret_cast<uintptr_t>(p.xh) % 16 == 0)
                            : (reinterpret_cast<uintptr_t>(p.x) % 16 == 0);
  const bool aligned = x_aligned && (reinterpret_cast<uintptr_t>(p.W) % 16 == 0) && (K % 16 == 0) &&
                       (p.ldw % 16 == 0) && (!p.xq_out || reinterpret_cast<uintptr_t>(p.xq_out) % 16 == 0);
  if (aligned && K > 0) {
    const int smem = K;  // x staged (as int8) in shared memory (K is a multiple of 16)
    const bool exact = (K / 16) % (32 * kGvBatch) == 0;
    auto kern = xh ? (exact ? gemv_w8a8_kernel<true, true> : gemv_w8a8_kernel<true, false>)
                   : (exact ? gemv_w8a8_kernel<false, true> : gemv_w8a8_kernel<false, false>);
    if (smem > 48 * 1024 &&
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
      return LL_ERR_CUDA;
    const int threads = gv_threads(xh);
    int grid = gv_ctas_per_sm(xh) * ctx.num_sms;
    const int need = (N + threads / 32 - 1) / (threads / 32);  // one warp per row at most
    if (need < grid) grid = need;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(threads);
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
  if (xh) {  // unaligned fused request: quantise into the caller's outputs, then the plain GEMV
    quantize_per_token_kernel<<<1, 256, K > 0 ? K : 1, ctx.stream>>>(1, K, p.xh, K, p.xq_out, K, p.xs_out);
    if (cudaGetLastError() != cudaSuccess) return LL_ERR_CUDA;
    p.x = p.xq_out;
    p.x_scale = p.xs_out;
    p.xh = nullptr;
  }
  gemv_w8a8_plain_kernel<<<(N + 7) / 8, 256, 0, ctx.stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? LL_OK : LL_ERR_CUDA;
}

static GemvParams gemv_params(int N, int K, const int8_t* x, const float* x_scale, const int8_t* W,
                              int64_t ldw, const float* w_scale, void* y, int32_t* z_out) {
  GemvParams p;
  p.N = N;
  p.K = K;
  p.x = x;
  p.x_scale = x_scale;
  p.xh = nullptr;
  p.xq_out = nullptr;
  p.xs_out = nullptr;
  p.W = W;
  p.ldw = ldw;
  p.w_scale = w_scale;
  p.bias = nullptr;
  p.out_i8 = 0;
  p.y_scale = nullptr;
  p.y = y;
  p.z_out = z_out;
  return p;
}

ll_status launch_gemv_w8a8(int N, int K, const int8_t* x, const float* x_scale, const int8_t* W,
                           int64_t ldw, const float* w_scale, void* y, int32_t* z_out,
                           const LaunchCtx& ctx) {
  return launch_gemv(gemv_params(N, K, x, x_scale, W, ldw, w_scale, y, z_out), ctx);
}

ll_status launch_gemv_w8a8_ex(int N, int K, const int8_t* x, const float* x_scale, const void* xh,
                              int8_t* xq_out, float* xs_out, const int8_t* W, int64_t ldw,
                              const float* w_scale, const float* bias, int out_i8,
                              const float* y_scale, void* y, int32_t* z_out, const LaunchCtx& ctx) {
  GemvParams p = gemv_params(N, K, x, x_scale, W, ldw, w_scale, y, z_out);
  p.xh = static_cast<const __half*>(xh);
  p.xq_out = xq_out;
  p.xs_out = xs_out;
  p.bias = bias;
  p.out_i8 = out_i8;
  p.y_scale = y_scale;
  return launch_gemv(p, ctx);
}

ll_status launch_quantize_per_token(int M, int K, const void* x, int64_t ldx, int8_t* q, int64_t ldq,
                                    float* scale, const LaunchCtx& ctx) {
  const int smem = K > 0 ? K : 1;
  if (smem > 48 * 1024 &&
      cudaFuncSetAttribute(quantize_per_token_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           smem) != cudaSuccess)
    return LL_ERR_CUDA;
  int grid = M < 8 * ctx.num_sms ? M : 8 * ctx.num_sms;
  quantize_per_token_kernel<<<grid, 256, smem, ctx.stream>>>(M, K, static_cast<const __half*>(x), ldx, q,
                                                             ldq, scale);
  return cudaGetLastError() == cudaSuccess ? LL_OK : LL_ERR_CUDA;
}

}  // namespace ll
