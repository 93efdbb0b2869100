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
struct ScratchAddr {
  void* ptr = nullptr;
  unsigned long long context_id = 0;  // the context `ptr` belongs to
};
ScratchAddr g_scratch_addr[kMaxDevices];
std::mutex g_scratch_mu;

// Device address of the scratch in the current context of the current device, looked up
// (with that device current) on the first call that needs it, and again only if the
// current CUDA context has changed since.
ll_status scratch_address(const ll::LaunchCtx& ctx, void** out) {
  if (ctx.device < 0 || ctx.device >= kMaxDevices) return LL_ERR_NO_DEVICE;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  ScratchAddr& sa = g_scratch_addr[ctx.device];
  if (sa.ptr == nullptr || sa.context_id != ctx.context_id) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return LL_ERR_CUDA;
    }
    sa.ptr = p;
    sa.context_id = ctx.context_id;
  }
  *out = sa.ptr;
  return LL_OK;
}

}  // namespace

extern "C" ll_status ll_gemm_f16_noalloc(int M, int N, int K, float alpha, const void* A,
                                         int64_t lda, const void* B, int64_t ldb, float beta,
                                         const float* C, int64_t ldc, void* D, int64_t ldd,
                                         int d_type, ll_stream_t stream) {
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
  a.mx = 0;
  a.nvf4 = 0;
  a.sk_ws = nullptr;
  a.sk_bytes = 0;
  a.mx_sa = nullptr;
  a.ld_mx_sa = 0;
  a.mx_sb = nullptr;
  a.ld_mx_sb = 0;
  a.mx_sat = nullptr;
  a.mx_sbt = nullptr;

  // the same argument rules as ll_gemm_f16 (the scratch cannot alias caller memory)
  ll_status st = ll::validate_gemm(a, nullptr, 0);
  if (st != LL_OK || M == 0 || N == 0) return st;
  ll::LaunchCtx ctx;
  st = ll::current_launch_ctx(stream, ctx);
  if (st != LL_OK) return st;
  if (K == 0) return ll::launch_scale_c(a, ctx);

  // the same repack layout as ll_gemm_f16, placed in the fixed scratch
  const ll::RepackPlan plan = ll::plan_repack(a);
  if (plan.a_bytes + plan.b_bytes > kNoAllocScratchBytes) return LL_ERR_WORKSPACE;  // beyond the scratch
  void* base = nullptr;  // 256-byte aligned
  if (plan.a || plan.b) {
    st = scratch_address(ctx, &base);
    if (st != LL_OK) return st;
  }
  return ll::launch_gemm_planned(a, plan, base, ctx);
}
