// Batch-1 W8A8 linear layer on CUDA cores ("NVIDIA A100: chip to SIMT", sections 5.1,
// 5.2 and 5.5):
//
//   z[o] = sum_k x[k] * W[o][k]   (int8 x int8 -> int32, exact)
//   y[o] = fp16_rn((float(z[o]) * s_x) * s_W[o])
//
// At batch 1 every weight byte is used once, so the kernel is bound by HBM bandwidth
// and does not use tensor cores (an M = 1 tile would leave 15/16 of an MMA idle).
//
// Design (fast path: K % 16 == 0, ldw % 16 == 0, 16-byte aligned x and W, 1024 <= K <= 32768):
//   * grid = one CTA per SM; CTA b owns the contiguous rows [b*N/G, (b+1)*N/G), so the
//     weight stream is split evenly over the SMs.
//   * one producer thread streams the CTA's rows into a ring of 32 KB shared-memory
//     stages with cp.async.bulk (one copy per stage when rows are contiguous), so
//     ~190 KB per SM are in flight from the first cycle.
//   * 8 consumer warps stage x and the CTA's w_scale values in shared memory while the
//     first weights are in flight.  Warp w takes rows w, w+8, ... of a stage; each lane
//     reads 16-byte chunks (lane-strided, conflict-free), multiplies them with the
//     matching 16 bytes of x with four dp4a, and releases the stage to the producer as
//     soon as its reads are done; then the warp reduces its 32 partial sums with
//     shuffles and lane 0 dequantises and stores.
// Any other shape runs a plain warp-per-row kernel with scalar loads (same results).
#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"

namespace ll {

constexpr int kGvWarps = 8;
constexpr int kGvThreads = 32 * (kGvWarps + 1);
constexpr int kGvStageBytes = 32768;
constexpr int kGvMaxRowsPerWarp = 4;  // rows of one stage per consumer warp (K >= 1024)

struct GemvParams {
  int N, K;
  const int8_t* x;
  const float* x_scale;
  const int8_t* W;
  int64_t ldw;
  const float* w_scale;
  __half* y;
  int32_t* z_out;
  int rows_per_stage;
  int stages;
  int contiguous;  // ldw == K: a stage is one contiguous copy
  int max_rows_per_cta;
  uint32_t* status;
  uint64_t timeout_ns;
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

__global__ void __launch_bounds__(kGvThreads, 1) gemv_w8a8_bulk_kernel(const GemvParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~static_cast<uintptr_t>(127));
  const int S = p.stages;
  const int kpad = (p.K + 127) & ~127;
  uint8_t* xs = smem + S * kGvStageBytes;
  float* sws = reinterpret_cast<float*>(xs + kpad);  // w_scale of this CTA's rows
  const int G = gridDim.x;
  const int r0 = static_cast<int>(static_cast<int64_t>(blockIdx.x) * p.N / G);
  const int r1 = static_cast<int>(static_cast<int64_t>(blockIdx.x + 1) * p.N / G);
  const int nrows = r1 - r0;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sws + ((p.max_rows_per_cta + 1) & ~1));
  uint32_t* abort_flag = reinterpret_cast<uint32_t*>(bars + 2 * S);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int RS = p.rows_per_stage;
  const int nchunks = (nrows + RS - 1) / RS;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_addr(bars + s), 1);
      mbar_init(smem_addr(bars + S + s), kGvWarps);
    }
    *abort_flag = 0u;
    fence_mbar_init();
  }
  __syncthreads();
  WaitCtx wctx{p.status, p.timeout_ns, abort_flag};

  if (warp == kGvWarps) {
    // ---------------------------------------------------------------- producer
    // starts streaming weights at once; the consumers stage x and the scales meanwhile
    if (lane == 0) {
      int issued = 0;
      for (int i = 0; i < nchunks; ++i) {
        const int s = i % S;
        if (!wait_bounded(smem_addr(bars + S + s), ((i / S) & 1) ^ 1, wctx, kRoleProducer)) break;
        const int rows = min(RS, nrows - i * RS);
        const uint32_t bar = smem_addr(bars + s);
        const uint32_t dst = smem_addr(smem + s * kGvStageBytes);
        const int row0 = r0 + i * RS;
        mbar_arrive_expect_tx(bar, static_cast<uint32_t>(rows * p.K));
        if (p.contiguous) {
          bulk_load(dst, p.W + static_cast<int64_t>(row0) * p.K, static_cast<uint32_t>(rows * p.K), bar);
        } else {
          for (int r = 0; r < rows; ++r)
            bulk_load(dst + r * p.K, p.W + static_cast<int64_t>(row0 + r) * p.ldw,
                      static_cast<uint32_t>(p.K), bar);
        }
        issued = i + 1;
      }
      if (*abort_flag) {
        for (int j = (issued > S ? issued - S : 0); j < issued; ++j)
          wait_drain(smem_addr(bars + (j % S)), (j / S) & 1, p.timeout_ns);
      }
    }
  } else {
    // ---------------------------------------------------------------- consumers
    const int ct = threadIdx.x;  // 0 .. 32 * kGvWarps - 1
    for (int i = ct; i < p.K / 16; i += 32 * kGvWarps)
      reinterpret_cast<int4*>(xs)[i] = __ldg(reinterpret_cast<const int4*>(p.x) + i);
    for (int i = ct; i < nrows; i += 32 * kGvWarps) sws[i] = __ldg(p.w_scale + r0 + i);
    const float sx = __ldg(p.x_scale);
    asm volatile("bar.sync 1, %0;" ::"r"(32 * kGvWarps) : "memory");  // consumer warps only

    const int kc = p.K / 16;
    const int4* xv = reinterpret_cast<const int4*>(xs);
    for (int i = 0; i < nchunks; ++i) {
      const int s = i % S;
      bool ok = wait_bounded(smem_addr(bars + s), (i / S) & 1, wctx, kRoleEpilogue);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      const int rows = min(RS, nrows - i * RS);
      const uint8_t* stage = smem + s * kGvStageBytes;
      // dot products of this warp's rows of the stage, then release the stage at once
      int part[kGvMaxRowsPerWarp];
      int nr = 0;
#pragma unroll
      for (int j = 0; j < kGvMaxRowsPerWarp; ++j) {
        const int r = warp + j * kGvWarps;
        part[j] = 0;
        if (r < rows) {
          const int4* wrow = reinterpret_cast<const int4*>(stage + r * p.K);
          int acc0 = 0, acc1 = 0;
#pragma unroll 4
          for (int c = lane; c < kc; c += 32) {
            const int4 w = wrow[c];
            const int4 a = xv[c];
            acc0 = __dp4a(w.x, a.x, acc0);
            acc1 = __dp4a(w.y, a.y, acc1);
            acc0 = __dp4a(w.z, a.z, acc0);
            acc1 = __dp4a(w.w, a.w, acc1);
          }
          part[j] = acc0 + acc1;
          nr = j + 1;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(bars + S + s));
#pragma unroll
      for (int j = 0; j < kGvMaxRowsPerWarp; ++j) {
        if (j < nr) {
          const int z = warp_sum(part[j]);
          const int rl = i * RS + warp + j * kGvWarps;  // row within this CTA
          if (lane == 0) {
            const int o = r0 + rl;
            if (p.z_out) p.z_out[o] = z;
            const float t = __fmul_rn(__int2float_rn(z), sx);
            p.y[o] = __float2half_rn(__fmul_rn(t, sws[rl]));
          }
        }
      }
    }
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
  p.status = ctx.status;
  p.timeout_ns = ctx.timeout_ns;
  p.contiguous = (ldw == K);
  const bool aligned = (reinterpret_cast<uintptr_t>(x) % 16 == 0) &&
                       (reinterpret_cast<uintptr_t>(W) % 16 == 0) && (K % 16 == 0) &&
                       (ldw % 16 == 0);
  if (aligned && K >= 1024 && K <= 32768) {
    const int kpad = (K + 127) & ~127;
    p.rows_per_stage = kGvStageBytes / K;  // <= kGvWarps * kGvMaxRowsPerWarp for K >= 1024
    const int chunks = (N + p.rows_per_stage - 1) / p.rows_per_stage;
    const int grid = chunks < ctx.num_sms ? chunks : ctx.num_sms;
    p.max_rows_per_cta = (N + grid - 1) / grid;
    const int scale_bytes = ((p.max_rows_per_cta + 1) & ~1) * 4;
    int stages = (220 * 1024 - kpad - scale_bytes) / kGvStageBytes;
    if (stages > 6) stages = 6;
    if (stages < 2) {
      p.stages = 0;
      gemv_w8a8_plain_kernel<<<(N + 7) / 8, 256, 0, ctx.stream>>>(p);
      return cudaGetLastError() == cudaSuccess ? LL_OK : LL_ERR_CUDA;
    }
    p.stages = stages;
    const int smem = stages * kGvStageBytes + kpad + scale_bytes + 2 * stages * 8 + 16 + 128;
    if (cudaFuncSetAttribute(gemv_w8a8_bulk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smem) != cudaSuccess)
      return LL_ERR_CUDA;
    gemv_w8a8_bulk_kernel<<<grid, kGvThreads, smem, ctx.stream>>>(p);
  } else {
    p.stages = 0;
    p.rows_per_stage = 0;
    gemv_w8a8_plain_kernel<<<(N + 7) / 8, 256, 0, ctx.stream>>>(p);
  }
  return cudaGetLastError() == cudaSuccess ? LL_OK : LL_ERR_CUDA;
}

}  // namespace ll
