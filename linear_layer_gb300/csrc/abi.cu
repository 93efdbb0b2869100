// The C ABI (include/ll.h): argument validation, operand repack decisions, per-device
// state (status word, SM count, wait limit) and dispatch to the kernels.
#include <cuda_runtime.h>

#include <mutex>

#include "internal.h"

// The device status word: written by kernels whose bounded wait ran out.
__device__ uint32_t g_ll_status_word;

namespace {

struct DeviceState {
  bool ready = false;
  bool supported = false;
  uint32_t* status = nullptr;
  int num_sms = 0;
  uint64_t timeout_ns = 2000000000ull;
};

constexpr int kMaxDevices = 64;
DeviceState g_dev[kMaxDevices];
std::mutex g_mu;

ll_status current_ctx(ll_stream_t stream, ll::LaunchCtx& ctx) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return LL_ERR_NO_DEVICE;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState& st = g_dev[dev];
  if (!st.ready) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return LL_ERR_CUDA;
    }
    st.supported = (major == 10 && minor == 3);
    if (st.supported) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_ll_status_word) != cudaSuccess) {
        cudaGetLastError();
        return LL_ERR_CUDA;
      }
      st.status = static_cast<uint32_t*>(p);
    }
    st.num_sms = sms;
    st.ready = true;
  }
  if (!st.supported) return LL_ERR_NO_DEVICE;
  ctx.stream = reinterpret_cast<cudaStream_t>(stream);
  ctx.status = st.status;
  ctx.timeout_ns = st.timeout_ns;
  ctx.num_sms = st.num_sms;
  return LL_OK;
}

int in_esize(int in_type) { return (in_type == LL_IN_E4M3 || in_type == LL_IN_E5M2) ? 1 : 2; }

int64_t round_up(int64_t v, int64_t m) { return (v + m - 1) / m * m; }

bool pitch_ok(const void* p, int64_t ld, int esize) {
  return (reinterpret_cast<uintptr_t>(p) % 16 == 0) && ((ld * esize) % 16 == 0);
}

size_t repack_bytes(int rows, int cols, int esize) {
  return static_cast<size_t>(rows) * static_cast<size_t>(round_up(static_cast<int64_t>(cols) * esize, 16)) + 256;
}

ll_status gemm_common(ll::GemmArgs a, void* workspace, size_t ws_bytes, ll_stream_t stream) {
  if (a.M < 0 || a.N < 0 || a.K < 0) return LL_ERR_INVALID_ARG;
  if (a.d_type != LL_OUT_F32 && a.d_type != LL_OUT_BF16 && a.d_type != LL_OUT_F16)
    return LL_ERR_INVALID_ARG;
  if (a.M == 0 || a.N == 0) return LL_OK;
  if (a.D == nullptr || a.ldd < a.N) return LL_ERR_INVALID_ARG;
  if (a.beta != 0.0f && (a.C == nullptr || a.ldc < a.N)) return LL_ERR_INVALID_ARG;
  if (a.d_type != LL_OUT_F32 && a.C != nullptr && a.beta != 0.0f &&
      static_cast<const void*>(a.C) == a.D)
    return LL_ERR_INVALID_ARG;  // in place only for FP32 output
  if (a.beta != 0.0f && static_cast<const void*>(a.C) == a.D && a.ldc != a.ldd)
    return LL_ERR_INVALID_ARG;
  // C, D and the scales are read and written element by element: each must be aligned
  // to its element size (A and B are repacked from any address)
  const uintptr_t dsz = a.d_type == LL_OUT_F32 ? 4 : 2;
  if (reinterpret_cast<uintptr_t>(a.D) % dsz != 0) return LL_ERR_MISALIGNED;
  if (a.beta != 0.0f && reinterpret_cast<uintptr_t>(a.C) % 4 != 0) return LL_ERR_MISALIGNED;
  if ((a.scale_a && reinterpret_cast<uintptr_t>(a.scale_a) % 4 != 0) ||
      (a.scale_b && reinterpret_cast<uintptr_t>(a.scale_b) % 4 != 0))
    return LL_ERR_MISALIGNED;
  if (a.K > 0) {
    if (a.A == nullptr || a.B == nullptr || a.lda < a.K || a.ldb < a.N) return LL_ERR_INVALID_ARG;
    if (a.in_type == LL_IN_E4M3 || a.in_type == LL_IN_E5M2) {
      const int64_t kb = (a.K + 127) / 128, nb = (a.N + 127) / 128;
      if (a.scale_a == nullptr || a.scale_b == nullptr || a.ld_sa < kb || a.ld_sb < nb)
        return LL_ERR_INVALID_ARG;
    }
  }
  ll::LaunchCtx ctx;
  ll_status st = current_ctx(stream, ctx);
  if (st != LL_OK) return st;
  if (a.K == 0) return ll::launch_scale_c(a, ctx);

  const int es = in_esize(a.in_type);
  const bool repack_a = !pitch_ok(a.A, a.lda, es);
  const bool repack_b = !pitch_ok(a.B, a.ldb, es);
  size_t need = 0;
  if (repack_a) need += repack_bytes(a.M, a.K, es);
  if (repack_b) need += repack_bytes(a.K, a.N, es);
  if (need > 0) {
    if (workspace == nullptr || ws_bytes < need) return LL_ERR_WORKSPACE;
    uintptr_t w = (reinterpret_cast<uintptr_t>(workspace) + 255) & ~static_cast<uintptr_t>(255);
    if (repack_a) {
      const int64_t ld = round_up(a.K, 16 / es);
      st = ll::launch_repack(a.A, a.lda, reinterpret_cast<void*>(w), ld, a.M, a.K, es, ctx);
      if (st != LL_OK) return st;
      a.A = reinterpret_cast<void*>(w);
      a.lda = ld;
      w += static_cast<uintptr_t>(round_up(static_cast<int64_t>(a.M) * ld * es, 256));
    }
    if (repack_b) {
      const int64_t ld = round_up(a.N, 16 / es);
      st = ll::launch_repack(a.B, a.ldb, reinterpret_cast<void*>(w), ld, a.K, a.N, es, ctx);
      if (st != LL_OK) return st;
      a.B = reinterpret_cast<void*>(w);
      a.ldb = ld;
    }
  }
  return ll::launch_gemm_tc(a, ctx);
}

}  // namespace

ll_status ll::current_launch_ctx(ll_stream_t stream, ll::LaunchCtx& ctx) {
  return current_ctx(stream, ctx);
}

extern "C" {

size_t ll_gemm_workspace_size(int M, int N, int K, int64_t lda, int64_t ldb, int in_type) {
  if (M <= 0 || N <= 0 || K <= 0) return 0;
  const int es = in_esize(in_type);
  size_t need = 0;
  if ((lda * es) % 16 != 0) need += repack_bytes(M, K, es);
  if ((ldb * es) % 16 != 0) need += repack_bytes(K, N, es);
  return need;
}

static ll::GemmArgs dense_args(int in_type, int M, int N, int K, float alpha, const void* A,
                               int64_t lda, const void* B, int64_t ldb, float beta, const float* C,
                               int64_t ldc, void* D, int64_t ldd, int d_type) {
  ll::GemmArgs a;
  a.in_type = in_type;
  a.b_type = in_type;
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
  return a;
}

ll_status ll_gemm_f16(int M, int N, int K, float alpha, const void* A, int64_t lda, const void* B,
                      int64_t ldb, float beta, const float* C, int64_t ldc, void* D, int64_t ldd,
                      int d_type, void* workspace, size_t ws_bytes, ll_stream_t stream) {
  return gemm_common(dense_args(LL_IN_F16, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, D, ldd,
                                d_type),
                     workspace, ws_bytes, stream);
}

ll_status ll_gemm_bf16(int M, int N, int K, float alpha, const void* A, int64_t lda, const void* B,
                       int64_t ldb, float beta, const float* C, int64_t ldc, void* D, int64_t ldd,
                       int d_type, void* workspace, size_t ws_bytes, ll_stream_t stream) {
  return gemm_common(dense_args(LL_IN_BF16, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, D, ldd,
                                d_type),
                     workspace, ws_bytes, stream);
}

ll_status ll_gemm_fp8_blockscaled(int M, int N, int K, float alpha, const uint8_t* A, int64_t lda,
                                  const float* scale_a, int64_t ld_sa, const uint8_t* B,
                                  int64_t ldb, const float* scale_b, int64_t ld_sb, float beta,
                                  const float* C, int64_t ldc, void* D, int64_t ldd, int d_type,
                                  void* workspace, size_t ws_bytes, ll_stream_t stream) {
  ll::GemmArgs a = dense_args(LL_IN_E4M3, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, D, ldd,
                              d_type);
  a.scale_a = scale_a;
  a.ld_sa = ld_sa;
  a.scale_b = scale_b;
  a.ld_sb = ld_sb;
  return gemm_common(a, workspace, ws_bytes, stream);
}

ll_status ll_gemm_f8_blockscaled_mixed(int a_type, int b_type, int M, int N, int K, float alpha,
                                       const uint8_t* A, int64_t lda, const float* scale_a,
                                       int64_t ld_sa, const uint8_t* B, int64_t ldb,
                                       const float* scale_b, int64_t ld_sb, float beta,
                                       const float* C, int64_t ldc, void* D, int64_t ldd,
                                       int d_type, void* workspace, size_t ws_bytes,
                                       ll_stream_t stream) {
  auto f8 = [](int t) { return t == LL_IN_E4M3 || t == LL_IN_E5M2; };
  if (!f8(a_type) || !f8(b_type)) return LL_ERR_INVALID_ARG;
  ll::GemmArgs a = dense_args(a_type, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, D, ldd, d_type);
  a.b_type = b_type;
  a.scale_a = scale_a;
  a.ld_sa = ld_sa;
  a.scale_b = scale_b;
  a.ld_sb = ld_sb;
  return gemm_common(a, workspace, ws_bytes, stream);
}

ll_status ll_linear_w8a8_gemv(int N, int K, const int8_t* x, const float* x_scale, const int8_t* W,
                              int64_t ldw, const float* w_scale, void* y, int32_t* z_out,
                              ll_stream_t stream) {
  if (N < 0 || K < 0 || K > 131071) return LL_ERR_INVALID_ARG;
  if (N == 0) return LL_OK;
  if (x_scale == nullptr || w_scale == nullptr || y == nullptr || ldw < K) return LL_ERR_INVALID_ARG;
  if (K > 0 && (x == nullptr || W == nullptr)) return LL_ERR_INVALID_ARG;
  ll::LaunchCtx ctx;
  ll_status st = current_ctx(stream, ctx);
  if (st != LL_OK) return st;
  return ll::launch_gemv_w8a8(N, K, x, x_scale, W, ldw, w_scale, y, z_out, ctx);
}

ll_status ll_linear_w8a8_gemv_ex(int N, int K, const int8_t* x, const float* x_scale,
                                 const int8_t* W, int64_t ldw, const float* w_scale,
                                 const float* bias, int y_type, const float* y_scale, void* y,
                                 int32_t* z_out, ll_stream_t stream) {
  if (N < 0 || K < 0 || K > 131071) return LL_ERR_INVALID_ARG;
  if (y_type != LL_GEMV_OUT_F16 && y_type != LL_GEMV_OUT_I8) return LL_ERR_INVALID_ARG;
  if (N == 0) return LL_OK;
  if (x_scale == nullptr || w_scale == nullptr || y == nullptr || ldw < K) return LL_ERR_INVALID_ARG;
  if (K > 0 && (x == nullptr || W == nullptr)) return LL_ERR_INVALID_ARG;
  if (y_type == LL_GEMV_OUT_I8 && y_scale == nullptr) return LL_ERR_INVALID_ARG;
  ll::LaunchCtx ctx;
  ll_status st = current_ctx(stream, ctx);
  if (st != LL_OK) return st;
  return ll::launch_gemv_w8a8_ex(N, K, x, x_scale, nullptr, nullptr, nullptr, W, ldw, w_scale, bias,
                                 y_type == LL_GEMV_OUT_I8, y_scale, y, z_out, ctx);
}

ll_status ll_linear_f16_w8a8_gemv(int N, int K, const void* x, int8_t* x_q, float* x_scale,
                                  const int8_t* W, int64_t ldw, const float* w_scale,
                                  const float* bias, int y_type, const float* y_scale, void* y,
                                  int32_t* z_out, ll_stream_t stream) {
  if (N < 0 || K < 0 || K > 131071) return LL_ERR_INVALID_ARG;
  if (y_type != LL_GEMV_OUT_F16 && y_type != LL_GEMV_OUT_I8) return LL_ERR_INVALID_ARG;
  if (N == 0) return LL_OK;
  if (x_q == nullptr || x_scale == nullptr || w_scale == nullptr || y == nullptr || ldw < K)
    return LL_ERR_INVALID_ARG;
  if (K > 0 && (x == nullptr || W == nullptr)) return LL_ERR_INVALID_ARG;
  if (y_type == LL_GEMV_OUT_I8 && y_scale == nullptr) return LL_ERR_INVALID_ARG;
  ll::LaunchCtx ctx;
  ll_status st = current_ctx(stream, ctx);
  if (st != LL_OK) return st;
  return ll::launch_gemv_w8a8_ex(N, K, nullptr, nullptr, x, x_q, x_scale, W, ldw, w_scale, bias,
                                 y_type == LL_GEMV_OUT_I8, y_scale, y, z_out, ctx);
}

ll_status ll_linear_w8a8(int M, int N, int K, const int8_t* X, int64_t ldx, const float* x_scale,
                         const int8_t* W, int64_t ldw, const float* w_scale, const float* bias,
                         int y_type, const float* y_scale, void* Y, int64_t ldy, int32_t* z_out,
                         int64_t ldz, ll_stream_t stream) {
  if (M < 0 || N < 0 || K < 0 || K > 131071) return LL_ERR_INVALID_ARG;
  if (y_type != LL_GEMV_OUT_F16 && y_type != LL_GEMV_OUT_I8) return LL_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return LL_OK;
  if (x_scale == nullptr || w_scale == nullptr || Y == nullptr || ldy < N || ldw < K || ldx < K)
    return LL_ERR_INVALID_ARG;
  if (K > 0 && (X == nullptr || W == nullptr)) return LL_ERR_INVALID_ARG;
  if (z_out != nullptr && ldz < N) return LL_ERR_INVALID_ARG;
  if (y_type == LL_GEMV_OUT_I8 && y_scale == nullptr) return LL_ERR_INVALID_ARG;
  ll::LaunchCtx ctx;
  ll_status st = current_ctx(stream, ctx);
  if (st != LL_OK) return st;
  return ll::launch_linear_w8a8(M, N, K, X, ldx, x_scale, W, ldw, w_scale, bias, y_type == LL_GEMV_OUT_I8,
                                y_scale, Y, ldy, z_out, ldz, ctx);
}

ll_status ll_linear_w8a16(int M, int N, int K, const void* X, int64_t ldx, const int8_t* W, int64_t ldw,
                          const float* w_scale, const float* bias, int y_type, void* Y, int64_t ldy,
                          ll_stream_t stream) {
  if (M < 0 || N < 0 || K < 0) return LL_ERR_INVALID_ARG;
  if (y_type != LL_OUT_F32 && y_type != LL_OUT_BF16 && y_type != LL_OUT_F16) return LL_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return LL_OK;
  if (w_scale == nullptr || Y == nullptr || ldy < N || ldw < K || ldx < K) return LL_ERR_INVALID_ARG;
  if (K > 0 && (X == nullptr || W == nullptr)) return LL_ERR_INVALID_ARG;
  ll::LaunchCtx ctx;
  ll_status st = current_ctx(stream, ctx);
  if (st != LL_OK) return st;
  return ll::launch_linear_w8a16(M, N, K, X, ldx, W, ldw, w_scale, bias, y_type, Y, ldy, ctx);
}

ll_status ll_quantize_per_token_f16(int M, int K, const void* x, int64_t ldx, int8_t* q,
                                    int64_t ldq, float* scale, ll_stream_t stream) {
  if (M < 0 || K < 0 || ldx < K || ldq < K) return LL_ERR_INVALID_ARG;
  if (M == 0) return LL_OK;
  if (scale == nullptr || (K > 0 && (x == nullptr || q == nullptr))) return LL_ERR_INVALID_ARG;
  ll::LaunchCtx ctx;
  ll_status st = current_ctx(stream, ctx);
  if (st != LL_OK) return st;
  return ll::launch_quantize_per_token(M, K, x, ldx, q, ldq, scale, ctx);
}

ll_status ll_get_device_status(ll_stream_t stream, uint32_t* detail) {
  ll::LaunchCtx ctx;
  ll_status st = current_ctx(stream, ctx);
  if (st != LL_OK) return st;
  uint32_t word = 0;
  if (cudaStreamSynchronize(ctx.stream) != cudaSuccess ||
      cudaMemcpyAsync(&word, ctx.status, sizeof(word), cudaMemcpyDeviceToHost, ctx.stream) !=
          cudaSuccess ||
      cudaMemsetAsync(ctx.status, 0, sizeof(word), ctx.stream) != cudaSuccess ||
      cudaStreamSynchronize(ctx.stream) != cudaSuccess) {
    cudaGetLastError();
    return LL_ERR_CUDA;
  }
  if (detail) *detail = word;
  return (word & 0xFFu) == 0 ? LL_OK : static_cast<ll_status>(word & 0xFFu);
}

ll_status ll_set_wait_timeout_ns(uint64_t ns) {
  ll::LaunchCtx ctx;
  ll_status st = current_ctx(nullptr, ctx);
  if (st != LL_OK) return st;
  if (ns == 0) return LL_ERR_INVALID_ARG;
  int dev = 0;
  cudaGetDevice(&dev);
  std::lock_guard<std::mutex> lock(g_mu);
  g_dev[dev].timeout_ns = ns;
  return LL_OK;
}

ll_status ll_debug_timeout_probe(ll_stream_t stream) {
  ll::LaunchCtx ctx;
  ll_status st = current_ctx(stream, ctx);
  if (st != LL_OK) return st;
  return ll::launch_timeout_probe(ctx);
}

const char* ll_status_string(ll_status s) {
  switch (s) {
    case LL_OK: return "LL_OK";
    case LL_ERR_INVALID_ARG: return "LL_ERR_INVALID_ARG";
    case LL_ERR_MISALIGNED: return "LL_ERR_MISALIGNED";
    case LL_ERR_UNSUPPORTED: return "LL_ERR_UNSUPPORTED";
    case LL_ERR_WORKSPACE: return "LL_ERR_WORKSPACE";
    case LL_ERR_CUDA: return "LL_ERR_CUDA";
    case LL_ERR_DEVICE_TIMEOUT: return "LL_ERR_DEVICE_TIMEOUT";
    case LL_ERR_NO_DEVICE: return "LL_ERR_NO_DEVICE";
  }
  return "LL_ERR_UNKNOWN";
}

const char* ll_version(void) { return "linear_layer_gb300 0.1 sm_103a"; }

}  // extern "C"
