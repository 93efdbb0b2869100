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
  unsigned long long context_id = 0;  // context the cached addresses belong to
  uint32_t* status = nullptr;
  int num_sms = 0;
  uint64_t timeout_ns = 2000000000ull;
};

constexpr int kMaxDevices = 64;
DeviceState g_dev[kMaxDevices];
std::mutex g_mu;

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

// Unique ID of the calling thread's current CUDA context, 0 when there is none (or the
// driver cannot tell).  IDs are never reused within a process, so a new context (a
// device reset, or another context made current) never matches a cached one.
unsigned long long current_context_id() {
  static CtxGetCurrentFn get_cur = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_cur = reinterpret_cast<CtxGetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(p);
    cudaGetLastError();
  });
  if (!get_cur || !get_id) return 0;
  CUcontext c = nullptr;
  if (get_cur(&c) != CUDA_SUCCESS || c == nullptr) return 0;
  unsigned long long id = 0;
  return get_id(c, &id) == CUDA_SUCCESS ? id : 0;
}

ll_status current_ctx(ll_stream_t stream, ll::LaunchCtx& ctx) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return LL_ERR_NO_DEVICE;
  }
  unsigned long long cid = current_context_id();
  if (cid == 0) {
    // no context bound to this thread yet: cudaSetDevice makes the device's primary
    // context current (it initialises it if needed)
    if (cudaSetDevice(dev) != cudaSuccess) {
      cudaGetLastError();
      return LL_ERR_NO_DEVICE;
    }
    cid = current_context_id();
  }
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState& st = g_dev[dev];
  if (!st.ready || st.context_id != cid) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return LL_ERR_CUDA;
    }
    st.supported = (major == 10 && minor == 3);
    st.status = nullptr;
    if (st.supported) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_ll_status_word) != cudaSuccess) {
        cudaGetLastError();
        return LL_ERR_CUDA;
      }
      st.status = static_cast<uint32_t*>(p);
    }
    st.num_sms = sms;
    st.context_id = cid;
    st.ready = true;
  }
  if (!st.supported) return LL_ERR_NO_DEVICE;
  ctx.stream = reinterpret_cast<cudaStream_t>(stream);
  ctx.status = st.status;
  ctx.timeout_ns = st.timeout_ns;
  ctx.num_sms = st.num_sms;
  ctx.device = dev;
  ctx.context_id = cid;
  return LL_OK;
}

int in_esize(int in_type) { return (in_type == LL_IN_E4M3 || in_type == LL_IN_E5M2) ? 1 : 2; }

int64_t round_up(int64_t v, int64_t m) { return (v + m - 1) / m * m; }

bool pitch_ok(const void* p, int64_t ld, int esize) {
  return (reinterpret_cast<uintptr_t>(p) % 16 == 0) && ((ld * esize) % 16 == 0);
}

// Workspace bytes for one repacked operand, with room to align the workspace start.
size_t repack_bytes(int rows, int cols, int esize) {
  return static_cast<size_t>(rows) * static_cast<size_t>(round_up(static_cast<int64_t>(cols) * esize, 16)) + 256;
}

// floor(a / b) for b > 0
int64_t floor_div(int64_t a, int64_t b) { return a >= 0 ? a / b : -((-a + b - 1) / b); }

// last byte offset + 1 of an extent, saturating
uint64_t extent_span(const ll::Extent& e) {
  const uint64_t rows1 = static_cast<uint64_t>(e.rows - 1), pitch = static_cast<uint64_t>(e.pitch);
  const uint64_t width = static_cast<uint64_t>(e.width);
  if (rows1 != 0 && pitch > (UINT64_MAX - width) / rows1) return UINT64_MAX;
  return rows1 * pitch + width;
}

bool extent_empty(const ll::Extent& e) { return e.base == nullptr || e.rows <= 0 || e.width <= 0; }

}  // namespace

bool ll::extents_overlap(const Extent& x0, const Extent& y0) {
  if (extent_empty(x0) || extent_empty(y0)) return false;
  Extent x = x0, y = y0;
  if (x.rows == 1) x.pitch = y.rows == 1 ? x.width : y.pitch;
  if (y.rows == 1) y.pitch = x.pitch;
  const uint64_t xb = reinterpret_cast<uintptr_t>(x.base), yb = reinterpret_cast<uintptr_t>(y.base);
  const uint64_t xs = extent_span(x), ys = extent_span(y);
  const bool x_before = xs <= UINT64_MAX - xb ? xb + xs <= yb : false;
  const bool y_before = ys <= UINT64_MAX - yb ? yb + ys <= xb : false;
  if (x_before || y_before) return false;  // disjoint spans
  if (x.pitch != y.pitch || x.pitch <= 0) return true;
  // same pitch p: row r2 of y starts d + (r2 - r1) * p bytes after row r1 of x; the two
  // rows share a byte when -y.width < d + t * p < x.width for t = r2 - r1
  const int64_t p = x.pitch;
  const int64_t d = static_cast<int64_t>(yb - xb);
  int64_t t_lo = floor_div(-y.width - d, p) + 1;
  int64_t t_hi = -floor_div(d - x.width, p) - 1;
  if (t_lo < -(x.rows - 1)) t_lo = -(x.rows - 1);
  if (t_hi > y.rows - 1) t_hi = y.rows - 1;
  return t_lo <= t_hi;
}

bool ll::outputs_overlap(const Extent* outs, int n_out, const Extent* ins, int n_in) {
  for (int i = 0; i < n_out; ++i) {
    for (int j = i + 1; j < n_out; ++j)
      if (extents_overlap(outs[i], outs[j])) return true;
    for (int j = 0; j < n_in; ++j)
      if (extents_overlap(outs[i], ins[j])) return true;
  }
  return false;
}

ll_status ll::validate_gemm(const GemmArgs& a, const void* ws, size_t ws_bytes) {
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
  const int64_t dsz = a.d_type == LL_OUT_F32 ? 4 : 2;
  if (reinterpret_cast<uintptr_t>(a.D) % dsz != 0) return LL_ERR_MISALIGNED;
  if (a.beta != 0.0f && reinterpret_cast<uintptr_t>(a.C) % 4 != 0) return LL_ERR_MISALIGNED;
  if ((a.scale_a && reinterpret_cast<uintptr_t>(a.scale_a) % 4 != 0) ||
      (a.scale_b && reinterpret_cast<uintptr_t>(a.scale_b) % 4 != 0))
    return LL_ERR_MISALIGNED;
  const bool f8 = (a.in_type == LL_IN_E4M3 || a.in_type == LL_IN_E5M2) && !a.mx;  // FP32 128-blocks
  const int64_t kb = (a.K + 127) / 128, nb = (a.N + 127) / 128;
  const int64_t kb32 = a.nvf4 ? (a.K + 15) / 16 : (a.K + 31) / 32;  // scale codes per row (MX / NVFP4)
  const int64_t kbytes = a.K / 2;                                     // NVFP4 row bytes
  if (a.K > 0) {
    if (a.A == nullptr || a.B == nullptr) return LL_ERR_INVALID_ARG;
    if (a.nvf4 ? (a.K % 2 != 0 || a.lda < kbytes || a.ldb < kbytes) : (a.lda < a.K || a.ldb < a.N))
      return LL_ERR_INVALID_ARG;
    if (f8 && (a.scale_a == nullptr || a.scale_b == nullptr || a.ld_sa < kb || a.ld_sb < nb))
      return LL_ERR_INVALID_ARG;
    if (a.mx && (a.mx_sa == nullptr || a.mx_sb == nullptr || a.ld_mx_sa < kb32 || a.ld_mx_sb < kb32))
      return LL_ERR_INVALID_ARG;
  }
  // D may share bytes with no input other than itself as C (in place, checked above);
  // a workspace that a repack or the stream-K tail (16-bit inputs, 8-bit inputs with
  // FP32 block scales) may write shares bytes with nothing
  const int64_t es = in_esize(a.in_type);
  const bool c_read = a.beta != 0.0f;
  const bool in_place = c_read && static_cast<const void*>(a.C) == a.D;
  const Extent D{a.D, a.M, a.N * dsz, a.ldd * dsz};
  Extent ins[5] = {
      {a.K > 0 ? a.A : nullptr, a.M, a.K * es, a.lda * es},
      {a.K > 0 ? a.B : nullptr, a.K, a.N * es, a.ldb * es},
      {c_read && !in_place ? a.C : nullptr, a.M, a.N * 4, a.ldc * 4},
      {a.K > 0 && f8 ? a.scale_a : nullptr, a.M, kb * 4, a.ld_sa * 4},
      {a.K > 0 && f8 ? a.scale_b : nullptr, kb, nb * 4, a.ld_sb * 4},
  };
  if (a.mx) {
    ins[3] = Extent{a.K > 0 ? a.mx_sa : nullptr, a.M, kb32, a.ld_mx_sa};
    ins[4] = Extent{a.K > 0 ? a.mx_sb : nullptr, a.N, kb32, a.ld_mx_sb};
  }
  if (a.nvf4) {  // A: M x K/2 bytes; B^T: N x K/2 bytes
    ins[0] = Extent{a.K > 0 ? a.A : nullptr, a.M, kbytes, a.lda};
    ins[1] = Extent{a.K > 0 ? a.B : nullptr, a.N, kbytes, a.ldb};
  }
  if (outputs_overlap(&D, 1, ins, 5)) return LL_ERR_INVALID_ARG;
  if (a.K > 0 && ws != nullptr && ws_bytes > 0) {
    const RepackPlan plan = plan_repack(a);
    if (plan.a || plan.b || plan.mx || sk_capable(a)) {
      const Extent W{ws, 1, static_cast<int64_t>(ws_bytes), static_cast<int64_t>(ws_bytes)};
      Extent all[6] = {D, ins[0], ins[1], ins[2], ins[3], ins[4]};
      if (in_place) all[3] = Extent{a.C, a.M, a.N * 4, a.ldc * 4};
      if (outputs_overlap(&W, 1, all, 6)) return LL_ERR_INVALID_ARG;
    }
  }
  return LL_OK;
}

ll::RepackPlan ll::plan_repack(const GemmArgs& a) {
  const int es = in_esize(a.in_type);
  RepackPlan pl;
  pl.a = !pitch_ok(a.A, a.lda, es);
  pl.b = !pitch_ok(a.B, a.ldb, es);
  if (a.nvf4) {  // byte rows: A M x K/2, B^T N x K/2
    pl.lda_p = pl.ldb_p = round_up(a.K / 2, 16);
    pl.a_bytes = pl.a ? static_cast<size_t>(round_up(static_cast<int64_t>(a.M) * pl.lda_p, 256)) : 0;
    pl.b_bytes = pl.b ? static_cast<size_t>(static_cast<int64_t>(a.N) * pl.ldb_p) : 0;
  } else {
    pl.lda_p = round_up(a.K, 16 / es);
    pl.ldb_p = round_up(a.N, 16 / es);
    pl.a_bytes = pl.a ? static_cast<size_t>(round_up(static_cast<int64_t>(a.M) * pl.lda_p * es, 256)) : 0;
    pl.b_bytes = pl.b ? static_cast<size_t>(static_cast<int64_t>(a.K) * pl.ldb_p * es) : 0;
  }
  pl.mx = a.mx != 0;
  pl.xa_bytes = pl.xb_bytes = 0;
  if (pl.mx) pl.xb_bytes = mx_scale_block_bytes(a.M, a.N, a.K, a.nvf4 != 0, &pl.xa_bytes) - pl.xa_bytes;
  return pl;
}

ll_status ll::launch_gemm_planned(GemmArgs a, const RepackPlan& plan, void* scratch, const LaunchCtx& ctx) {
  const int es = in_esize(a.in_type);
  unsigned char* w = static_cast<unsigned char*>(scratch);
  // every byte the GEMM reads from the scratch is written here first (pad columns are
  // zeroed), so nothing an earlier call left there reaches this one
  const int arow = a.nvf4 ? a.K / 2 : a.K;    // row widths: elements (bytes for NVFP4)
  const int brows = a.nvf4 ? a.N : a.K, brow = a.nvf4 ? a.K / 2 : a.N;
  if (plan.a) {
    const ll_status st = launch_repack(a.A, a.lda, w, plan.lda_p, a.M, arow, es, ctx);
    if (st != LL_OK) return st;
    a.A = w;
    a.lda = plan.lda_p;
  }
  if (plan.b) {
    const ll_status st = launch_repack(a.B, a.ldb, w + plan.a_bytes, plan.ldb_p, brows, brow, es, ctx);
    if (st != LL_OK) return st;
    a.B = w + plan.a_bytes;
    a.ldb = plan.ldb_p;
  }
  if (plan.mx) {  // the scale codes, rearranged into the blocks the MX kernels fetch
    unsigned char* xa = w + plan.a_bytes + static_cast<size_t>(round_up(static_cast<int64_t>(plan.b_bytes), 256));
    const ll_status st = launch_mx_scale_tiles(a, xa, xa + plan.xa_bytes, ctx);
    if (st != LL_OK) return st;
    a.mx_sat = xa;
    a.mx_sbt = xa + plan.xa_bytes;
  }
  return launch_gemm_tc(a, ctx);
}

namespace {

ll_status gemm_common(const ll::GemmArgs& a, void* workspace, size_t ws_bytes, ll_stream_t stream) {
  ll_status st = ll::validate_gemm(a, workspace, ws_bytes);
  if (st != LL_OK || a.M == 0 || a.N == 0) return st;
  ll::LaunchCtx ctx;
  st = current_ctx(stream, ctx);
  if (st != LL_OK) return st;
  if (a.K == 0) return ll::launch_scale_c(a, ctx);
  const ll::RepackPlan plan = ll::plan_repack(a);
  void* base = nullptr;
  size_t need = 0;
  if (plan.a || plan.b || plan.mx) {
    const int es = in_esize(a.in_type);
    if (plan.a) need += repack_bytes(a.M, a.nvf4 ? a.K / 2 : a.K, es);
    if (plan.b) need += a.nvf4 ? repack_bytes(a.N, a.K / 2, es) : repack_bytes(a.K, a.N, es);
    if (plan.mx) need += plan.xa_bytes + plan.xb_bytes + 512;
    if (workspace == nullptr || ws_bytes < need) return LL_ERR_WORKSPACE;
  }
  if (workspace != nullptr)
    base = reinterpret_cast<void*>((reinterpret_cast<uintptr_t>(workspace) + 255) & ~static_cast<uintptr_t>(255));
  ll::GemmArgs b = a;
  if (base != nullptr && ll::sk_capable(a)) {
    // what the repacks leave, past the 256 bytes ll_gemm_workspace_size reserves for
    // alignment: the stream-K partial tiles, so the split runs exactly when ws_bytes
    // reaches the figure ll_gemm_workspace_size reports
    const size_t rep = static_cast<size_t>(round_up(static_cast<int64_t>(need), 256));
    if (ws_bytes > rep + 256) {
      b.sk_ws = static_cast<unsigned char*>(base) + rep;
      b.sk_bytes = ws_bytes - rep - 256;
    }
  }
  return ll::launch_gemm_planned(b, plan, base, ctx);
}

}  // namespace

ll_status ll::current_launch_ctx(ll_stream_t stream, ll::LaunchCtx& ctx) {
  return current_ctx(stream, ctx);
}

namespace {

// Outputs of a batch-1 W8A8 GEMV call (y, z_out, and for the fused quantiser x_q and its
// scale) against each other and against every input.
bool gemv_outputs_overlap(int N, int K, const void* x, int x_esize, const float* x_scale, const int8_t* W,
                          int64_t ldw, const float* w_scale, const float* bias, const float* y_scale, const void* y,
                          int y_esize, const int32_t* z_out, const int8_t* x_q, const float* xs_out) {
  const int64_t n = N, k = K;
  const ll::Extent outs[4] = {{y, 1, n * y_esize, n * y_esize},
                              {z_out, 1, n * 4, n * 4},
                              {K > 0 ? x_q : nullptr, 1, k, k},
                              {xs_out, 1, 4, 4}};
  const ll::Extent ins[6] = {{K > 0 ? x : nullptr, 1, k * x_esize, k * x_esize},
                             {x_scale, 1, 4, 4},
                             {K > 0 ? W : nullptr, n, k, ldw},
                             {w_scale, 1, n * 4, n * 4},
                             {bias, 1, n * 4, n * 4},
                             {y_scale, 1, 4, 4}};
  return ll::outputs_overlap(outs, 4, ins, 6);
}

}  // namespace

extern "C" {

// operand repacks only
static size_t gemm_repack_need(int M, int N, int K, int64_t lda, int64_t ldb, int in_type) {
  const int es = in_esize(in_type);
  size_t need = 0;
  if ((lda * es) % 16 != 0) need += repack_bytes(M, K, es);
  if ((ldb * es) % 16 != 0) need += repack_bytes(K, N, es);
  return need;
}

size_t ll_gemm_workspace_size(int M, int N, int K, int64_t lda, int64_t ldb, int in_type) {
  if (M <= 0 || N <= 0 || K <= 0) return 0;
  size_t need = gemm_repack_need(M, N, K, lda, ldb, in_type);
  // the optional stream-K tail of the CTA-pair 16-bit kernel or the one-CTA FP8 kernel
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) == cudaSuccess &&
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess) {
    const bool f16 = in_type == LL_IN_F16 || in_type == LL_IN_BF16;
    const size_t sk = f16 ? ll::pair_sk_workspace(M, N, K, sms) : ll::fp8_sk_workspace(M, N, K, sms);
    if (sk) need = static_cast<size_t>(round_up(static_cast<int64_t>(need), 256)) + 256 + sk;
  } else {
    cudaGetLastError();
  }
  return need;
}

size_t ll_gemm_mxf8_workspace_size(int M, int N, int K, int64_t lda, int64_t ldb) {
  if (M <= 0 || N <= 0 || K <= 0) return 0;
  return gemm_repack_need(M, N, K, lda, ldb, LL_IN_E4M3) + ll::mx_scale_block_bytes(M, N, K, false, nullptr) + 512;
}

size_t ll_gemm_nvf4_workspace_size(int M, int N, int K, int64_t lda, int64_t ldbt) {
  if (M <= 0 || N <= 0 || K <= 0) return 0;
  size_t need = ll::mx_scale_block_bytes(M, N, K, true, nullptr) + 512;
  if ((lda / 2) % 16 != 0) need += repack_bytes(M, K / 2, 1);
  if ((ldbt / 2) % 16 != 0) need += repack_bytes(N, K / 2, 1);
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

ll_status ll_gemm_mxf8(int a_type, int b_type, int M, int N, int K, float alpha, const uint8_t* A, int64_t lda,
                       const uint8_t* scale_a, int64_t ld_sa, const uint8_t* B, int64_t ldb, const uint8_t* scale_b,
                       int64_t ld_sb, float beta, const float* C, int64_t ldc, void* D, int64_t ldd, int d_type,
                       void* workspace, size_t ws_bytes, ll_stream_t stream) {
  auto f8 = [](int t) { return t == LL_IN_E4M3 || t == LL_IN_E5M2; };
  if (!f8(a_type) || !f8(b_type)) return LL_ERR_INVALID_ARG;
  ll::GemmArgs a = dense_args(a_type, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, D, ldd, d_type);
  a.b_type = b_type;
  a.mx = 1;
  a.mx_sa = scale_a;
  a.ld_mx_sa = ld_sa;
  a.mx_sb = scale_b;
  a.ld_mx_sb = ld_sb;
  return gemm_common(a, workspace, ws_bytes, stream);
}

ll_status ll_gemm_nvf4(int M, int N, int K, float alpha, const uint8_t* A, int64_t lda, const uint8_t* scale_a,
                       int64_t ld_sa, const uint8_t* Bt, int64_t ldbt, const uint8_t* scale_b, int64_t ld_sb,
                       float beta, const float* C, int64_t ldc, void* D, int64_t ldd, int d_type, void* workspace,
                       size_t ws_bytes, ll_stream_t stream) {
  if ((lda & 1) || (ldbt & 1)) return LL_ERR_INVALID_ARG;  // rows start on byte boundaries
  ll::GemmArgs a = dense_args(LL_IN_E4M3, M, N, K, alpha, A, lda / 2, Bt, ldbt / 2, beta, C, ldc, D, ldd, d_type);
  a.mx = 1;
  a.nvf4 = 1;
  a.mx_sa = scale_a;
  a.ld_mx_sa = ld_sa;
  a.mx_sb = scale_b;
  a.ld_mx_sb = ld_sb;
  return gemm_common(a, workspace, ws_bytes, stream);
}

ll_status ll_linear_w8a8_gemv(int N, int K, const int8_t* x, const float* x_scale, const int8_t* W,
                              int64_t ldw, const float* w_scale, void* y, int32_t* z_out,
                              ll_stream_t stream) {
  if (N < 0 || K < 0 || K > 131071) return LL_ERR_INVALID_ARG;
  if (N == 0) return LL_OK;
  if (x_scale == nullptr || w_scale == nullptr || y == nullptr || ldw < K) return LL_ERR_INVALID_ARG;
  if (K > 0 && (x == nullptr || W == nullptr)) return LL_ERR_INVALID_ARG;
  if (gemv_outputs_overlap(N, K, x, 1, x_scale, W, ldw, w_scale, nullptr, nullptr, y, 2, z_out, nullptr,
                           nullptr))
    return LL_ERR_INVALID_ARG;
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
  if (gemv_outputs_overlap(N, K, x, 1, x_scale, W, ldw, w_scale, bias, y_type == LL_GEMV_OUT_I8 ? y_scale : nullptr,
                           y, y_type == LL_GEMV_OUT_I8 ? 1 : 2, z_out, nullptr, nullptr))
    return LL_ERR_INVALID_ARG;
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
  if (gemv_outputs_overlap(N, K, x, 2, nullptr, W, ldw, w_scale, bias, y_type == LL_GEMV_OUT_I8 ? y_scale : nullptr,
                           y, y_type == LL_GEMV_OUT_I8 ? 1 : 2, z_out, x_q, x_scale))
    return LL_ERR_INVALID_ARG;
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
  {
    const int64_t ysz = y_type == LL_GEMV_OUT_I8 ? 1 : 2;
    const ll::Extent outs[2] = {{Y, M, N * ysz, ldy * ysz}, {z_out, M, N * 4, ldz * 4}};
    const ll::Extent ins[5] = {{K > 0 ? X : nullptr, M, K, ldx},
                               {x_scale, 1, int64_t(M) * 4, int64_t(M) * 4},
                               {K > 0 ? W : nullptr, N, K, ldw},
                               {w_scale, 1, int64_t(N) * 4, int64_t(N) * 4},
                               {bias, 1, int64_t(N) * 4, int64_t(N) * 4}};
    const ll::Extent ys{y_type == LL_GEMV_OUT_I8 ? y_scale : nullptr, 1, 4, 4};
    if (ll::outputs_overlap(outs, 2, ins, 5) || ll::outputs_overlap(outs, 2, &ys, 1)) return LL_ERR_INVALID_ARG;
  }
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
  {
    const int64_t ysz = y_type == LL_OUT_F32 ? 4 : 2;
    const ll::Extent out{Y, M, N * ysz, ldy * ysz};
    const ll::Extent ins[4] = {{K > 0 ? X : nullptr, M, int64_t(K) * 2, ldx * 2},
                               {K > 0 ? W : nullptr, N, K, ldw},
                               {w_scale, 1, int64_t(N) * 4, int64_t(N) * 4},
                               {bias, 1, int64_t(N) * 4, int64_t(N) * 4}};
    if (ll::outputs_overlap(&out, 1, ins, 4)) return LL_ERR_INVALID_ARG;
  }
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
  {
    const ll::Extent outs[2] = {{K > 0 ? q : nullptr, M, K, ldq}, {scale, 1, int64_t(M) * 4, int64_t(M) * 4}};
    const ll::Extent in{K > 0 ? x : nullptr, M, int64_t(K) * 2, ldx * 2};
    if (ll::outputs_overlap(outs, 2, &in, 1)) return LL_ERR_INVALID_ARG;
  }
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
