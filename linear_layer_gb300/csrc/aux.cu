// Small kernels around the GEMM:
//   * operand repack into a 16-byte row pitch, for operands whose pitch or base
//     address a TMA tensor map cannot describe;
//   * D = beta * C for K == 0 (an empty contraction);
//   * the bounded-wait probe used to test failure detection.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"

namespace ll {

// Each thread writes one 16-byte vector of a destination row (the destination pitch is a
// multiple of 16 bytes); columns past `cols` are the pad and are written as zero.
template <class T>
__global__ void repack_kernel(const T* __restrict__ src, int64_t ld_src, T* __restrict__ dst,
                              int64_t ld_dst, int rows, int cols) {
  constexpr int V = 16 / sizeof(T);
  const int64_t vec_per_row = ld_dst / V;
  const int64_t total = static_cast<int64_t>(rows) * vec_per_row;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t r = i / vec_per_row;
    const int64_t c0 = (i - r * vec_per_row) * V;
    const T* s = src + r * ld_src + c0;
    union {
      T e[V];
      uint4 u;
    } buf;
#pragma unroll
    for (int v = 0; v < V; ++v) buf.e[v] = (c0 + v < cols) ? s[v] : T(0);
    *reinterpret_cast<uint4*>(dst + r * ld_dst + c0) = buf.u;
  }
}

ll_status launch_repack(const void* src, int64_t ld_src, void* dst, int64_t ld_dst, int rows,
                        int cols, int esize, const LaunchCtx& ctx) {
  if (rows <= 0 || cols <= 0) return LL_OK;
  const int threads = 256;
  const int64_t vecs = static_cast<int64_t>(rows) * (ld_dst * esize / 16);
  int64_t blocks = (vecs + threads - 1) / threads;
  if (blocks > 16 * ctx.num_sms) blocks = 16 * ctx.num_sms;
  if (esize == 2)
    repack_kernel<uint16_t><<<static_cast<int>(blocks), threads, 0, ctx.stream>>>(
        static_cast<const uint16_t*>(src), ld_src, static_cast<uint16_t*>(dst), ld_dst, rows, cols);
  else
    repack_kernel<uint8_t><<<static_cast<int>(blocks), threads, 0, ctx.stream>>>(
        static_cast<const uint8_t*>(src), ld_src, static_cast<uint8_t*>(dst), ld_dst, rows, cols);
  return cudaGetLastError() == cudaSuccess ? LL_OK : LL_ERR_CUDA;
}

__global__ void scale_c_kernel(int M, int N, float beta, const float* __restrict__ C, int64_t ldc,
                               void* D, int64_t ldd, int d_type) {
  for (int m = blockIdx.y; m < M; m += gridDim.y) {
    for (int n = blockIdx.x * blockDim.x + threadIdx.x; n < N; n += gridDim.x * blockDim.x) {
      const float v = (beta != 0.0f) ? beta * C[static_cast<int64_t>(m) * ldc + n] : 0.0f;
      const int64_t o = static_cast<int64_t>(m) * ldd + n;
      if (d_type == LL_OUT_F32)
        static_cast<float*>(D)[o] = v;
      else if (d_type == LL_OUT_BF16)
        static_cast<__nv_bfloat16*>(D)[o] = __float2bfloat16_rn(v);
      else
        static_cast<__half*>(D)[o] = __float2half_rn(v);
    }
  }
}

ll_status launch_scale_c(const GemmArgs& a, const LaunchCtx& ctx) {
  const int threads = 256;
  int gx = (a.N + threads - 1) / threads;
  if (gx > 64) gx = 64;
  const int gy = a.M < 65535 ? a.M : 65535;
  scale_c_kernel<<<dim3(gx, gy), threads, 0, ctx.stream>>>(a.M, a.N, a.beta, a.C, a.ldc, a.D,
                                                           a.ldd, a.d_type);
  return cudaGetLastError() == cudaSuccess ? LL_OK : LL_ERR_CUDA;
}

// One thread waits on a barrier phase nothing will complete; the bounded wait gives up
// after the configured limit and records the timeout.
__global__ void timeout_probe_kernel(uint32_t* status, uint64_t timeout_ns) {
  __shared__ uint64_t bar;
  __shared__ uint32_t abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_addr(&bar), 1);
    abort_flag = 0u;
    fence_mbar_init();
    WaitCtx ctx{status, timeout_ns, &abort_flag};
    (void)wait_bounded(smem_addr(&bar), 0u, ctx, kRoleProbe);
  }
}

ll_status launch_timeout_probe(const LaunchCtx& ctx) {
  timeout_probe_kernel<<<1, 32, 0, ctx.stream>>>(ctx.status, ctx.timeout_ns);
  return cudaGetLastError() == cudaSuccess ? LL_OK : LL_ERR_CUDA;
}

}  // namespace ll
