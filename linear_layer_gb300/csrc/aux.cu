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

// Each thread writes one 16-byte vector of a destination row (the destination pitch is
// a multiple of 16 bytes); bytes past the source row's `row_bytes` are the pad and are
// written as zero.  The source row may start at any element boundary: the thread reads
// the two aligned 16-byte words that cover its 16 source bytes and funnel-shifts them
// into place, so every global access is a full 16-byte vector.  A word is read only if
// it holds at least one byte of the row, and an aligned 16-byte word never crosses a
// page, so no read leaves the source allocation's pages.  The kernel is itself launched
// programmatically: its blocks may be scheduled while the previous kernel of the stream
// finishes, and touch memory only after the dependency wait.  It lets the GEMM behind it
// start its prologue at once; the GEMM's dependency wait still covers every write made here.
__global__ void repack_kernel(const uint8_t* __restrict__ src, int64_t ld_src, uint8_t* __restrict__ dst,
                              int64_t ld_dst, int rows, int64_t row_bytes) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int64_t vec_per_row = ld_dst / 16;
  const int64_t total = static_cast<int64_t>(rows) * vec_per_row;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t r = i / vec_per_row;
    const int64_t b0 = (i - r * vec_per_row) * 16;  // first byte of this vector in the row
    uint4 out = make_uint4(0u, 0u, 0u, 0u);
    if (b0 < row_bytes) {
      const uintptr_t sa = reinterpret_cast<uintptr_t>(src + r * ld_src + b0);
      const uintptr_t row_end = reinterpret_cast<uintptr_t>(src + r * ld_src + row_bytes);
      const uint32_t off = static_cast<uint32_t>(sa & 15u);
      const uint4* base = reinterpret_cast<const uint4*>(sa - off);
      const uint4 lo = __ldg(base);
      const uint4 hi = (sa - off + 16 < row_end) ? __ldg(base + 1) : make_uint4(0u, 0u, 0u, 0u);
      const uint32_t w[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
      // t[k] = w[off / 4 + k] through two fixed-index selections
      const uint32_t ws = off >> 2, bs = (off & 3u) * 8u;
      uint32_t s1[7], t[5];
#pragma unroll
      for (int k = 0; k < 7; ++k) s1[k] = (ws & 1u) ? w[k + 1] : w[k];
#pragma unroll
      for (int k = 0; k < 5; ++k) t[k] = (ws & 2u) ? s1[k + 2] : s1[k];
      uint32_t o[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) o[k] = __funnelshift_r(t[k], t[k + 1], bs);
      const int64_t valid = row_bytes - b0;  // >= 1
      if (valid < 16) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int64_t keep = valid - 4 * k;  // bytes of word k inside the row
          if (keep <= 0)
            o[k] = 0u;
          else if (keep < 4)
            o[k] &= (1u << (8 * keep)) - 1u;
        }
      }
      out = make_uint4(o[0], o[1], o[2], o[3]);
    }
    *reinterpret_cast<uint4*>(dst + r * ld_dst + b0) = out;
  }
}

ll_status launch_repack(const void* src, int64_t ld_src, void* dst, int64_t ld_dst, int rows,
                        int cols, int esize, const LaunchCtx& ctx) {
  if (rows <= 0 || cols <= 0) return LL_OK;
  const int threads = 256;
  const int64_t vecs = static_cast<int64_t>(rows) * (ld_dst * esize / 16);
  int64_t blocks = (vecs + threads - 1) / threads;
  if (blocks > 8 * ctx.num_sms) blocks = 8 * ctx.num_sms;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks));
  cfg.blockDim = dim3(threads);
  cfg.stream = ctx.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e =
      cudaLaunchKernelEx(&cfg, repack_kernel, static_cast<const uint8_t*>(src), ld_src * esize,
                         static_cast<uint8_t*>(dst), ld_dst * esize, rows, static_cast<int64_t>(cols) * esize);
  return e == cudaSuccess ? LL_OK : LL_ERR_CUDA;
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
