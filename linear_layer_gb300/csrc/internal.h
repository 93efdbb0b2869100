// Host-side interfaces shared between the C ABI (abi.cu) and the kernel files.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/ll.h"

namespace ll {

// Per-call context the ABI hands to every launcher.
struct LaunchCtx {
  cudaStream_t stream;
  uint32_t* status;     // device status word of the current device
  uint64_t timeout_ns;  // limit of one bounded wait
  int num_sms;          // SM count of the current device
  int device;           // ordinal of the current device
  unsigned long long context_id;  // unique ID of the current CUDA context (0 if unknown)
};

struct GemmArgs {
  int in_type;  // ll_in_type (of A; and of B unless b_type says otherwise)
  int b_type;   // ll_in_type of B (8-bit inputs may mix E4M3 and E5M2)
  int M, N, K;
  float alpha, beta;
  const void* A;
  int64_t lda;  // operand pitches as the kernel reads them (after any repack)
  const void* B;
  int64_t ldb;
  const float* C;
  int64_t ldc;
  void* D;
  int64_t ldd;
  int d_type;  // ll_out_type
  const float* scale_a;
  int64_t ld_sa;
  const float* scale_b;
  int64_t ld_sb;
  int mx;                 // hardware block scaling (MX or NVFP4) instead of FP32 128-blocks
  int nvf4;               // NVFP4: A is M x K/2 bytes and B holds B^T, N x K/2 bytes (pitches
                          // lda / ldb in bytes), scales UE4M3 per 16 K elements
  const uint8_t* mx_sa;   // MX: M x ld_mx_sa scale codes of A, one per row and 32-wide K block
  int64_t ld_mx_sa;
  const uint8_t* mx_sb;   // MX: N x ld_mx_sb scale codes of B, one per column and K block
  int64_t ld_mx_sb;
  const uint8_t* mx_sat;  // MX: the scale codes rearranged into tcgen05.cp blocks (workspace)
  const uint8_t* mx_sbt;
  void* sk_ws;            // workspace left after any repack (256-byte aligned), for the
  size_t sk_bytes;        //   stream-K partial tiles of the CTA-pair GEMM; NULL / 0: none
};

// Workspace bytes the CTA-pair 16-bit GEMM uses to split its last partial wave of tiles
// by K ranges (stream-K), for up to `pairs` CTA pairs (gemm_tc.cu).
size_t pair_sk_bytes(int pairs);
// Those bytes for an M x N x K 16-bit problem on a GPU with num_sms SMs, or 0 when its
// schedule has no such tail (gemm_tc.cu).
size_t pair_sk_workspace(int M, int N, int K, int num_sms);
// The same for the one-CTA FP8 kernel (FP32 block scales): bytes for up to `ctas` CTAs,
// and for an M x N x K problem (0 when its schedule has no such tail) (gemm_tc.cu).
size_t fp8_sk_bytes(int ctas);
size_t fp8_sk_workspace(int M, int N, int K, int num_sms);
// Whether the call may place stream-K partial tiles in its workspace: FP16 / BF16 inputs,
// and 8-bit inputs with FP32 block scales.
inline bool sk_capable(const GemmArgs& a) {
  return !a.mx && !a.nvf4;
}

// Launch context of the current device (status word, SM count, wait limit) for `stream`;
// LL_ERR_NO_DEVICE unless an sm_103 device is current (abi.cu).  Device addresses of the
// library's own __device__ variables are looked up again whenever the current CUDA
// context differs from the one they were found in (a context made current through the
// driver API, or a new primary context after a device reset).
ll_status current_launch_ctx(ll_stream_t stream, LaunchCtx& ctx);

// A matrix as a set of byte ranges: `rows` rows of `width` bytes, `pitch` bytes apart
// (pitch >= width), from `base`.  A NULL base or an empty shape is an empty set.
struct Extent {
  const void* base;
  int64_t rows, width, pitch;
};

// True when two extents may share a byte.  Exact when the extents have the same pitch
// (or one of them is a single row); otherwise any intersection of their first-to-last
// byte spans counts as shared.
bool extents_overlap(const Extent& x, const Extent& y);

// True when an output extent shares a byte with another output or with an input.
bool outputs_overlap(const Extent* outs, int n_out, const Extent* ins, int n_in);

// Host-side checks of a GEMM request that need no device (sizes, types, pitches,
// pointers, alignment, aliasing; the workspace only enters through ws/ws_bytes and is
// checked against the operands when it will be written).  LL_OK or the error to return.
ll_status validate_gemm(const GemmArgs& a, const void* ws, size_t ws_bytes);

// Where the operand repack of a GEMM puts A and B: A (when repacked) at the 256-byte-
// aligned start of the scratch, B after it.  a_bytes = roundup(M * lda_p * esize, 256)
// and b_bytes = K * ldb_p * esize with the pitches rounded up to 16 bytes; the MX scale
// blocks follow B (at a 256-byte boundary).
struct RepackPlan {
  bool a, b;
  int64_t lda_p, ldb_p;  // elements
  size_t a_bytes, b_bytes;
  // MX: the scale codes rearranged into the blocks tcgen05.cp copies (always), after B at a
  // 256-byte boundary: A's blocks (xa_bytes), then B's (xb_bytes)
  bool mx;
  size_t xa_bytes, xb_bytes;
};
RepackPlan plan_repack(const GemmArgs& a);

// Repack per `plan` into `scratch` (256-byte aligned, at least a_bytes + b_bytes), then
// launch the GEMM on the repacked operands.  `scratch` may be NULL when nothing is repacked.
ll_status launch_gemm_planned(GemmArgs a, const RepackPlan& plan, void* scratch, const LaunchCtx& ctx);

// tcgen05 GEMM (gemm_tc.cu).  Requires A, B 16-byte aligned with 16-byte-multiple pitches.
ll_status launch_gemm_tc(const GemmArgs& a, const LaunchCtx& ctx);

// MX block-scaled 8-bit GEMM on tcgen05 with hardware block scaling (gemm_mx.cu); the same
// operand requirements, and a.mx_sat / a.mx_sbt holding the scale blocks.
ll_status launch_gemm_mx(const GemmArgs& a, const LaunchCtx& ctx);

// Bytes of the MX scale blocks of an M x N x K problem (A's in *a_bytes when not NULL), and
// the kernel that writes them from a.mx_sa / a.mx_sb into xa / xb (gemm_mx.cu).
size_t mx_scale_block_bytes(int M, int N, int K, bool nv, size_t* a_bytes);
ll_status launch_mx_scale_tiles(const GemmArgs& a, uint8_t* xa, uint8_t* xb, const LaunchCtx& ctx);

// D = beta * C (or 0) for K == 0 (aux.cu).
ll_status launch_scale_c(const GemmArgs& a, const LaunchCtx& ctx);

// Row-pitch repack of a rows x cols matrix of esize-byte elements (aux.cu).
ll_status launch_repack(const void* src, int64_t ld_src, void* dst, int64_t ld_dst, int rows,
                        int cols, int esize, const LaunchCtx& ctx);

// Tensor map of a row-major rows x cols matrix (pitch in elements), tiles of box_cols x
// box_rows, 128-byte swizzle unless given, zero fill out of bounds (gemm_tc.cu).
bool make_tensor_map_2d(CUtensorMap* map, const void* base, CUtensorMapDataType dt, int esize,
                        int64_t rows, int64_t cols, int64_t pitch, int box_cols, int box_rows,
                        CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B);

// Bounded-wait probe (aux.cu).
ll_status launch_timeout_probe(const LaunchCtx& ctx);

// W8A8 GEMV (gemv_w8a8.cu).
ll_status launch_gemv_w8a8(int N, int K, const int8_t* x, const float* x_scale, const int8_t* W,
                           int64_t ldw, const float* w_scale, void* y, int32_t* z_out,
                           const LaunchCtx& ctx);

// W8A8 GEMV with epilogue variants and the optional fused FP16-activation quantiser
// (xh != NULL: x and x_scale are ignored; xq_out / xs_out receive the quantised
// activation and its scale when not NULL, and are required when xh is unaligned).
ll_status launch_gemv_w8a8_ex(int N, int K, const int8_t* x, const float* x_scale, const void* xh,
                              int8_t* xq_out, float* xs_out, const int8_t* W, int64_t ldw,
                              const float* w_scale, const float* bias, int out_i8,
                              const float* y_scale, void* y, int32_t* z_out, const LaunchCtx& ctx);

// W8A8 linear layer for M tokens (w8a8_batch.cu): X M x ldx int8, x_scale [M], Y M x ldy
// (FP16, or INT8 with out_i8), Z M x ldz int32 or NULL.
ll_status launch_linear_w8a8(int M, int N, int K, const int8_t* X, int64_t ldx, const float* x_scale,
                             const int8_t* W, int64_t ldw, const float* w_scale, const float* bias,
                             int out_i8, const float* y_scale, void* Y, int64_t ldy, int32_t* Z,
                             int64_t ldz, const LaunchCtx& ctx);

// The same for 1..64 tokens on the tensor cores (w8a8_tc.cu): K % 16 == 0, ldx and ldw
// multiples of 16, 16-byte aligned X and W.
ll_status launch_w8a8_tc(int M, int N, int K, const int8_t* X, int64_t ldx, const float* x_scale,
                         const int8_t* W, int64_t ldw, const float* w_scale, const float* bias, int out_i8,
                         const float* y_scale, void* Y, int64_t ldy, int32_t* Z, int64_t ldz,
                         const LaunchCtx& ctx);

// Weight-only INT8 layer with BF16 activations (w8a16.cu): X M x ldx BF16, W N x ldw
// int8, w_scale [N], bias [N] or NULL, Y M x ldy of ll_out_type y_type.
ll_status launch_linear_w8a16(int M, int N, int K, const void* X, int64_t ldx, const int8_t* W, int64_t ldw,
                              const float* w_scale, const float* bias, int y_type, void* Y, int64_t ldy,
                              const LaunchCtx& ctx);

// Per-token activation quantiser (gemv_w8a8.cu).
ll_status launch_quantize_per_token(int M, int K, const void* x, int64_t ldx, int8_t* q, int64_t ldq,
                                    float* scale, const LaunchCtx& ctx);

}  // namespace ll
