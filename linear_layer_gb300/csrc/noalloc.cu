// ll_gemm_f16_noalloc: the FP16 GEMM for callers that cannot allocate device memory.
//
// ll_gemm_f16 needs caller-provided workspace when an operand's row pitch (or base
// address) is not a multiple of 16 bytes, because such an operand is first repacked
// into a 16-byte pitch that the TMA tensor maps can describe.  Some callers have no
// way to provide it: a runtime whose allocator owns all device memory and gives none
// to a library per call, a plugin interface that passes neither an allocator nor a
// workspace, or a latency-critical path where allocating is not allowed.  This
// variant repacks into a fixed scratch array that lives in the library itself:
// kNoAllocScratchBytes (16 MiB) of device memory, held on every GPU that loads the
// library until the process exits.  It calls no cudaMalloc / cudaFree and no
// allocating library routine.
#include <cuda_runtime.h>

#include <mutex>

#include "internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;

// The scratch itself.  In host code this name is only a host-side stand-in for the
// device array: its device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices] = {};
std::mutex g_scratch_mu;

// Device address of the scratch on the current device, looked up once per device
// (with that device current) on the first call that needs it.
ll_status scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return LL_ERR_NO_DEVICE;
  }
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return LL_ERR_CUDA;
    }
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return LL_OK;
}

int64_t round_up(int64_t v, int64_t m) { return (v + m - 1) / m * m; }

bool pitch_ok(const void* p, int64_t ld) {
  return (reinterpret_cast<uintptr_t>(p) % 16 == 0) && ((ld * 2) % 16 == 0);
}

}  // namespace

extern "C" ll_status ll_gemm_f16_noalloc(int M, int N, int K, float alpha, const void* A,
                                         int64_t lda, const void* B, int64_t ldb, float beta,
                                         const float* C, int64_t ldc, void* D, int64_t ldd,
                                         int d_type, ll_stream_t stream) {
  // the same argument rules as ll_gemm_f16
  if (M < 0 || N < 0 || K < 0) return LL_ERR_INVALID_ARG;
  if (d_type != LL_OUT_F32 && d_type != LL_OUT_BF16 && d_type != LL_OUT_F16)
    return LL_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return LL_OK;
  if (D == nullptr || ldd < N) return LL_ERR_INVALID_ARG;
  if (beta != 0.0f && (C == nullptr || ldc < N)) return LL_ERR_INVALID_ARG;
  if (beta != 0.0f && static_cast<const void*>(C) == D && (d_type != LL_OUT_F32 || ldc != ldd))
    return LL_ERR_INVALID_ARG;
  if (K > 0 && (A == nullptr || B == nullptr || lda < K || ldb < N)) return LL_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(D) % (d_type == LL_OUT_F32 ? 4 : 2) != 0) return LL_ERR_MISALIGNED;
  if (beta != 0.0f && reinterpret_cast<uintptr_t>(C) % 4 != 0) return LL_ERR_MISALIGNED;

  ll::GemmArgs a;
  a.in_type = LL_IN_F16;
  a.b_type = LL_IN_F16;
  a.M = M;
  a.N = N;
  a.K = K;
  a.alpha = alpha;
  a.beta = beta;
  a.A = A;
  a.lda = lda;
  a.B = B;
  a.ldb = ldb;
  a.C = C;
  a.ldc = ldc;
  a.D = D;
  a.ldd = ldd;
  a.d_type = d_type;
  a.scale_a = nullptr;
  a.ld_sa = 0;
  a.scale_b = nullptr;
  a.ld_sb = 0;

  ll::LaunchCtx ctx;
  ll_status st = ll::current_launch_ctx(stream, ctx);
  if (st != LL_OK) return st;
  if (K == 0) return ll::launch_scale_c(a, ctx);

  const bool repack_a = !pitch_ok(A, lda);
  const bool repack_b = !pitch_ok(B, ldb);
  const int64_t lda_p = round_up(K, 8), ldb_p = round_up(N, 8);  // 16-byte FP16 pitches
  const size_t a_bytes = repack_a ? static_cast<size_t>(round_up(int64_t(M) * lda_p * 2, 256)) : 0;
  const size_t b_bytes = repack_b ? static_cast<size_t>(int64_t(K) * ldb_p * 2) : 0;
  if (a_bytes + b_bytes > kNoAllocScratchBytes) return LL_ERR_WORKSPACE;  // beyond the fixed scratch
  if (repack_a || repack_b) {
    void* base = nullptr;
    st = scratch_address(&base);
    if (st != LL_OK) return st;
    unsigned char* w = static_cast<unsigned char*>(base);  // 256-byte aligned
    // every byte the GEMM reads from the scratch is rewritten here first (the pad
    // columns are zeroed), so nothing left by an earlier call can leak into this one
    if (repack_a) {
      st = ll::launch_repack(A, lda, w, lda_p, M, K, 2, ctx);
      if (st != LL_OK) return st;
      a.A = w;
      a.lda = lda_p;
    }
    if (repack_b) {
      st = ll::launch_repack(B, ldb, w + a_bytes, ldb_p, K, N, 2, ctx);
      if (st != LL_OK) return st;
      a.B = w + a_bytes;
      a.ldb = ldb_p;
    }
  }
  return ll::launch_gemm_tc(a, ctx);
}
