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
//   * 3 CTAs of 8 warps per SM; warp g of the grid owns rows g, g + G, g + 2G, ...
//   * each lane streams 16-byte chunks of its warp's row (lane-strided, 8 chunks =
//     4 KB per warp in flight) with non-caching loads straight into registers, and
//     multiplies them with the matching 16 bytes of x (staged once per CTA in shared
//     memory) with four dp4a;  the next row's first chunks are requested before the
//     warp reduces and dequantises the current row, so loads stay in flight.
//   * programmatic dependent launch: the kernel lets the next kernel of the stream be
//     scheduled as soon as SMs free up, and itself starts streaming weights before the
//     preceding kernel has finished; x and x_scale are read, and y / z written, only
//     after griddepcontrol.wait, i.e. after all preceding work on the stream is done.
//   Measured on GB300 against a TMA bulk-copy ring and a cp.async ring (one CTA per
//   SM): direct loads sustained the highest bandwidth for this 45 MB stream.
// Any other shape or alignment runs a plain warp-per-row kernel with scalar loads.
#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"

namespace ll {

constexpr int kGvThreads = 256;
constexpr int kGvCtasPerSm = 3;
constexpr int kGvBatch = 8;  // 16-byte chunks per lane in flight (4 KB per warp)

struct GemvParams {
  int N, K;
  const int8_t* x;
  const float* x_scale;
  const int8_t* W;
  int64_t ldw;
  const float* w_scale;
  __half* y;
  int32_t* z_out;
};

__device__ __forceinline__ int warp_sum(int v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}

__device__ __forceinline__ void dequant_store(const GemvParams& p, int o, int z, float sx) {
  if (p.z_out) p.z_out[o] = z;
  const float f = __int2float_rn(z);
  const float t = __fmul_rn(f, sx);
  const float u = __fmul_rn(t, p.w_scale[o]);
  p.y[o] = __float2half_rn(u);
}

__device__ __forceinline__ int4 ld_stream(const int4* p) {
  int4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.s32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
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

__global__ void __launch_bounds__(kGvThreads, kGvCtasPerSm) gemv_w8a8_kernel(const GemvParams p) {
  extern __shared__ int4 xs[];  // x, K bytes
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int lane = threadIdx.x & 31;
  const int G = gridDim.x * (kGvThreads / 32);
  const int nch = p.K / 16;  // 16-byte chunks per row
  int r = blockIdx.x * (kGvThreads / 32) + (threadIdx.x >> 5);
  int4 w[kGvBatch];
  if (r < p.N) load_batch(w, reinterpret_cast<const int4*>(p.W + static_cast<int64_t>(r) * p.ldw), 0, nch, lane);

  asm volatile("griddepcontrol.wait;" ::: "memory");  // x / outputs: after preceding work
  for (int i = threadIdx.x; i < nch; i += kGvThreads) xs[i] = reinterpret_cast<const int4*>(p.x)[i];
  __syncthreads();
  const float sx = *p.x_scale;

  while (r < p.N) {
    const int4* row = reinterpret_cast<const int4*>(p.W + static_cast<int64_t>(r) * p.ldw);
    int acc0 = 0, acc1 = 0;
    for (int base = 0;;) {
#pragma unroll
      for (int j = 0; j < kGvBatch; ++j) {
        const int c = base + lane + 32 * j;
        if (c < nch) {
          const int4 a = xs[c];
          acc0 = __dp4a(w[j].x, a.x, acc0);
          acc1 = __dp4a(w[j].y, a.y, acc1);
          acc0 = __dp4a(w[j].z, a.z, acc0);
          acc1 = __dp4a(w[j].w, a.w, acc1);
        }
      }
      base += 32 * kGvBatch;
      if (base >= nch) break;
      load_batch(w, row, base, nch, lane);
    }
    const int rn = r + G;
    if (rn < p.N)  // next row in flight while this one is reduced and stored
      load_batch(w, reinterpret_cast<const int4*>(p.W + static_cast<int64_t>(rn) * p.ldw), 0, nch, lane);
    const int z = warp_sum(acc0 + acc1);
    if (lane == 0) dequant_store(p, r, z, sx);
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
  if (lane == 0) dequant_store(p, o, z, *p.x_scale);
}

ll_status launch_gemv_w8a8(int N, int K, const int8_t* x, const float* x_scale, const int8_t* W,
                           int64_t ldw, const float* w_scale, void* y, int32_t* z_out,
                           const LaunchCtx& ctx) {
  GemvParams p;
  p.N = N;
  p.K = K;
  p.x = x;
  p.x_scale = x_scale;
  p.W = W;
  p.ldw = ldw;
  p.w_scale = w_scale;
  p.y = static_cast<__half*>(y);
  p.z_out = z_out;
  const bool aligned = (reinterpret_cast<uintptr_t>(x) % 16 == 0) &&
                       (reinterpret_cast<uintptr_t>(W) % 16 == 0) && (K % 16 == 0) &&
                       (ldw % 16 == 0);
  if (aligned && K > 0) {
    const int smem = K;  // x staged in shared memory (K is a multiple of 16)
    if (smem > 48 * 1024 &&
        cudaFuncSetAttribute(gemv_w8a8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smem) != cudaSuccess)
      return LL_ERR_CUDA;
    int grid = kGvCtasPerSm * ctx.num_sms;
    const int need = (N + kGvThreads / 32 - 1) / (kGvThreads / 32);  // one warp per row at most
    if (need < grid) grid = need;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kGvThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = ctx.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, gemv_w8a8_kernel, p) != cudaSuccess) {
      cudaGetLastError();
      return LL_ERR_CUDA;
    }
    return LL_OK;
  }
  gemv_w8a8_plain_kernel<<<(N + 7) / 8, 256, 0, ctx.stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? LL_OK : LL_ERR_CUDA;
}

}  // namespace ll
