/*
 * linear_layer_gb300 -- C ABI of the GB300 (sm_103a) linear-layer hot path.
 *
 * The library computes, on one GPU, the tiled matrix multiply-accumulate
 *
 *     D = alpha * A x B + beta * C          (FP32 accumulation)
 *
 * for FP16, BF16 and block-scaled FP8 E4M3 inputs, and its batch-1 W8A8 special
 * case (int8 x int8 -> int32, per-token x per-channel dequantisation to FP16).
 *
 * Conventions shared by every entry point
 *   - All matrices are row-major.  A leading dimension (ld*) is the distance, in
 *     ELEMENTS, between the starts of consecutive rows; ld >= the row width.
 *   - Every pointer except the ones named "host" is caller-owned DEVICE memory on
 *     the current CUDA device.  The library allocates no device memory per call;
 *     its only device state is one status word per device (see ll_get_device_status)
 *     and the fixed scratch array of ll_gemm_f16_noalloc (16 MiB per device).  The
 *     device addresses of both are looked up in the calling thread's current CUDA
 *     context, again whenever that context differs from the one of the last lookup
 *     (a context made current through the driver API, or the new primary context
 *     after a device reset).
 *   - Outputs may not share memory with inputs or with each other: a request whose
 *     output byte ranges meet another operand's is rejected (LL_ERR_INVALID_ARG)
 *     before any launch.  Two matrices with the same row pitch are compared row by
 *     row (column blocks of one matrix are fine); matrices with different pitches
 *     count as overlapping when their first-to-last byte spans intersect.  The only
 *     exception is the in-place GEMM, D == C (see ll_gemm_f16).
 *   - Ordering with programmatic dependent launch.  Every kernel of this library lets
 *     the next kernel of its stream begin as soon as it has started, and waits for the
 *     work before it (griddepcontrol.wait) before it reads activations, C or scales or
 *     writes any output.  The W8A8 and weight-only layers (ll_linear_w8a8*,
 *     ll_linear_f16_w8a8_gemv, ll_linear_w8a16) read their weights W and w_scale
 *     BEFORE that wait, to stream them while earlier work drains.  So W and w_scale
 *     must not be written by any call of this library that may still be running when
 *     the layer is launched: every library call on the stream since the last kernel
 *     there that does not come from this library (such a kernel lets nothing after it
 *     start before it has finished), or since the last host synchronisation of the
 *     stream.
 *     Weights of a model are constants, which meets this; to use a library output
 *     (say the INT8 output of ll_linear_w8a8) as W, launch any other kernel on the
 *     stream in between, or synchronise.  The GEMMs read nothing before the wait
 *     (they only prefetch into L2, which is coherent), so they have no such rule.
 *   - Every entry point is asynchronous on `stream` (a cudaStream_t; NULL = the
 *     legacy default stream).  Argument errors are detected on the host and
 *     returned before anything is launched; nothing is written in that case.
 *   - Calls are deterministic: identical arguments (sizes, data and, for the FP16 /
 *     BF16 and FP8 block-scaled GEMMs, workspace size) on the same GPU give
 *     bit-identical outputs.
 *   - A wait inside a kernel that exceeds its time limit does not hang the GPU: the
 *     kernel records LL_ERR_DEVICE_TIMEOUT in the status word and exits.
 *
 * Scope: one GPU; no collective; no CPU fallback.
 */
#ifndef LINEAR_LAYER_GB300_LL_H
#define LINEAR_LAYER_GB300_LL_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st; /* the type behind cudaStream_t */
typedef struct CUstream_st* ll_stream_t;

typedef enum {
  LL_OK = 0,
  LL_ERR_INVALID_ARG = 1,    /* a size, leading dimension or pointer is invalid       */
  LL_ERR_MISALIGNED = 2,     /* C, D or a scale pointer not aligned to its element   */
  LL_ERR_UNSUPPORTED = 3,    /* a valid request this build does not implement         */
  LL_ERR_WORKSPACE = 4,      /* workspace too small for the operand repack it needs   */
  LL_ERR_CUDA = 5,           /* a CUDA runtime/driver call or a launch failed         */
  LL_ERR_DEVICE_TIMEOUT = 6, /* a kernel's bounded wait ran out (device status word)  */
  LL_ERR_NO_DEVICE = 7       /* no sm_103 device is current                            */
} ll_status;

/* Element type of the A and B operands. */
typedef enum { LL_IN_F16 = 0, LL_IN_BF16 = 1, LL_IN_E4M3 = 2, LL_IN_E5M2 = 3 } ll_in_type;

/* Element type of the output D. */
typedef enum { LL_OUT_F32 = 0, LL_OUT_BF16 = 1, LL_OUT_F16 = 2 } ll_out_type;

/* ------------------------------------------------------------------ dense GEMM */

/*
 * Bytes of workspace a GEMM with these sizes and leading dimensions needs
 * (0 when both operands can be read in place).  An operand is read in place when
 * its base pointer is 16-byte aligned and its row pitch (ld * element size) is a
 * multiple of 16 bytes; otherwise the call first repacks it into the workspace
 * (row pitch rounded up to 16 bytes) inside the same stream, and that copy is part
 * of the call.  The figure assumes 16-byte-aligned base pointers; a misaligned base
 * pointer is repacked too and needs at most ll_gemm_workspace_size(...,lda=1,ldb=1).
 * The figure also holds room for the partial accumulators of the stream-K tail (when a
 * CUDA device is current and the problem leaves a partial last wave of tiles: 256 x 256
 * tiles on SM pairs for FP16 / BF16 inputs, 128 x 256 tiles on single SMs for 8-bit
 * inputs with FP32 block scales): the K blocks of the last tiles are then split evenly
 * over all workers (SM pairs or SMs), and a worker whose range ends inside a tile leaves
 * its FP32 partial (for 8-bit inputs: block scales applied) and a ready flag in the
 * workspace for the worker that finishes the tile.  That room is optional: with less
 * workspace (or none) the call still succeeds and finishes the last wave with half-width
 * tiles (16-bit) or whole tiles (8-bit) instead.  The split changes only the order in
 * which FP32 partial sums over K are added (partials are added in a fixed order), so the
 * result is deterministic for a given problem and workspace size.  A workspace must
 * not be shared by calls that may run at the same time (other streams, other threads).
 * The worker that finishes a split tile waits (bounded) for workers of lower index, which
 * the hardware starts no later than it; if kernels on other streams keep part of the
 * grid from starting for longer than the wait limit (ll_set_wait_timeout_ns), the call
 * reports LL_ERR_DEVICE_TIMEOUT rather than hang.  A caller that runs other kernels
 * concurrently with large GEMMs can turn the split off by passing one byte less than
 * ll_gemm_workspace_size reports (the repacks still fit): the split runs exactly when
 * ws_bytes reaches that figure.
 */
size_t ll_gemm_workspace_size(int M, int N, int K, int64_t lda, int64_t ldb, int in_type);

/*
 * D = alpha * A x B + beta * C for FP16 (ll_gemm_f16) or BF16 (ll_gemm_bf16) A, B.
 *
 * Defined by: "Tensor Core" chapter (anrans ai-infra-handbooks), section
 * "Tensor Core 做什么" (D = A x B + C, low-precision inputs) and table
 * "精度：FP16、BF16、TF32、FP8" (FP16/BF16 inputs, FP32 accumulation), with the
 * BLAS alpha/beta scaling.
 *
 *   A : M x K, lda >= K (FP16 or BF16)          B : K x N, ldb >= N (same type as A)
 *   C : M x N FP32, ldc >= N; not read when beta == 0 (may then be NULL)
 *   D : M x N, ldd >= N, element type d_type; D may alias C only as the same matrix
 *       (D == C, d_type == LL_OUT_F32, ldd == ldc: each element is read before it is
 *       written); any other overlap of D with A, B or C is rejected (LL_ERR_INVALID_ARG).
 *       Nothing outside the M x N elements of D is written (padding columns included).
 *   workspace : device scratch of ws_bytes (see ll_gemm_workspace_size); may be NULL if 0.
 *       The call may write any of it (repacked operands, stream-K partial tiles), so it
 *       may overlap no operand (LL_ERR_INVALID_ARG).
 * Every product is accumulated in FP32 over the whole K; alpha * acc + beta * C is
 * evaluated in FP32 and rounded once to d_type (round to nearest even).
 * M == 0 or N == 0: nothing is done.  K == 0: D = beta * C (alpha is not used).
 * Errors: LL_ERR_INVALID_ARG for negative sizes, ld < width, NULL operands,
 * beta != 0 with C == NULL, or overlapping memory; LL_ERR_MISALIGNED if D (or C when read) is not aligned to
 * its element size; LL_ERR_WORKSPACE if a repack is needed and ws_bytes is smaller
 * than ll_gemm_workspace_size; LL_ERR_CUDA if a launch fails.
 */
ll_status ll_gemm_f16(int M, int N, int K, float alpha, const void* A, int64_t lda,
                      const void* B, int64_t ldb, float beta, const float* C, int64_t ldc,
                      void* D, int64_t ldd, int d_type, void* workspace, size_t ws_bytes,
                      ll_stream_t stream);
ll_status ll_gemm_bf16(int M, int N, int K, float alpha, const void* A, int64_t lda,
                       const void* B, int64_t ldb, float beta, const float* C, int64_t ldc,
                       void* D, int64_t ldd, int d_type, void* workspace, size_t ws_bytes,
                       ll_stream_t stream);

/*
 * FP8 E4M3 GEMM with FP32 block scales:
 *
 *   D[i][j] = alpha * sum_kb scale_a[i][kb] * scale_b[kb][j / 128]
 *                          * sum_{k in block kb} A[i][k] * B[k][j]  + beta * C[i][j]
 *
 * Defined by: "Tensor Core" chapter, table "精度：FP16、BF16、TF32、FP8" and the text
 * under it (FP8 E4M3 1/4/3; FP8 GEMMs need scaling factors per tensor, row or block;
 * fine-grained block scaling as used for DeepSeek-V3 training).
 *
 *   A       : M x K E4M3 codes (1 byte), lda >= K
 *   scale_a : M x ceil(K/128) FP32, ld_sa >= ceil(K/128); one scale per row and 128-wide K block
 *   B       : K x N E4M3 codes, ldb >= N
 *   scale_b : ceil(K/128) x ceil(N/128) FP32, ld_sb >= ceil(N/128); one per 128 x 128 block
 *   C, D, workspace, stream: as for ll_gemm_f16.
 * E4M3 is the finite-only form (bias 7, max 448, NaN = S.1111.111).  Each 128-K
 * block is accumulated in FP32 by the tensor cores, then scaled by
 * scale_a * scale_b and added into an FP32 accumulator (block-wise promotion).
 * Errors: as for ll_gemm_f16; scale pointers must be non-NULL when M, N, K > 0.
 */
ll_status ll_gemm_fp8_blockscaled(int M, int N, int K, float alpha, const uint8_t* A, int64_t lda,
                                  const float* scale_a, int64_t ld_sa, const uint8_t* B,
                                  int64_t ldb, const float* scale_b, int64_t ld_sb, float beta,
                                  const float* C, int64_t ldc, void* D, int64_t ldd, int d_type,
                                  void* workspace, size_t ws_bytes, ll_stream_t stream);

/*
 * ll_gemm_f16 for callers that cannot allocate device memory.  The pages have no
 * counterpart: this entry point exists for integration, not for the method.
 *
 * Some callers cannot provide the workspace ll_gemm_f16 needs for an operand whose
 * row pitch or base address is not a multiple of 16 bytes: a runtime whose allocator
 * owns all device memory and hands none to libraries, a plugin interface that passes
 * the library neither an allocator nor a workspace, or a latency-critical path where
 * allocating is not allowed.  This
 * variant takes the same arguments minus the workspace and repacks such operands
 * into a fixed scratch array inside the library: 16 MiB of device memory that every
 * GPU which loads the library holds until the process exits.  It calls no cudaMalloc,
 * cudaFree or allocating library routine.
 *   - Limit: the repacked operands must fit the 16 MiB scratch, i.e.
 *     (A repacked ? roundup(M * roundup(K, 8) * 2, 256) : 0)
 *       + (B repacked ? K * roundup(N, 8) * 2 : 0)  <=  16 MiB;
 *     larger requests return LL_ERR_WORKSPACE before anything is launched.
 *     Operands that are already 16-byte aligned use no scratch and have no limit.
 *   - The first call on a device that needs the scratch looks up its device address
 *     (once per device and CUDA context, with that device current); make that first
 *     call before any stream capture.
 *   - Every call shares the one scratch array and overwrites what it reads, so calls
 *     that overlap on the GPU (for instance on different streams) race: serialise
 *     them.
 * Results equal, bit for bit, those of ll_gemm_f16 given a workspace of exactly the
 * repack bytes; it never splits the last wave of tiles by K (that needs workspace), so
 * where ll_gemm_f16 with a larger workspace does, the FP32 partial sums are added in
 * another order and the results may differ in rounding.  Errors as for ll_gemm_f16.
 */
ll_status ll_gemm_f16_noalloc(int M, int N, int K, float alpha, const void* A, int64_t lda,
                              const void* B, int64_t ldb, float beta, const float* C,
                              int64_t ldc, void* D, int64_t ldd, int d_type, ll_stream_t stream);

/*
 * ll_gemm_fp8_blockscaled with each operand's 8-bit format chosen separately:
 * a_type, b_type in { LL_IN_E4M3, LL_IN_E5M2 }.
 *
 * Defined by: "Tensor Core" chapter, table "精度：FP16、BF16、TF32、FP8": FP8 E5M2
 * (1/5/2, wider range, used for gradients) beside E4M3 (1/4/3).  E5M2 follows the IEEE
 * conventions (bias 15, infinities and NaNs at exponent 31, largest finite 57344).
 * Scales, layouts, tails and errors as ll_gemm_fp8_blockscaled; LL_ERR_INVALID_ARG for
 * any other a_type / b_type.
 */
ll_status ll_gemm_f8_blockscaled_mixed(int a_type, int b_type, int M, int N, int K, float alpha,
                                       const uint8_t* A, int64_t lda, const float* scale_a,
                                       int64_t ld_sa, const uint8_t* B, int64_t ldb,
                                       const float* scale_b, int64_t ld_sb, float beta,
                                       const float* C, int64_t ldc, void* D, int64_t ldd,
                                       int d_type, void* workspace, size_t ws_bytes,
                                       ll_stream_t stream);

/*
 * MX block-scaled 8-bit GEMM (OCP microscaling): every 32 consecutive K elements of a row
 * of A, and of a column of B, share one E8M0 scale X = 2^(e - 127):
 *
 *   D[i][j] = alpha * sum_k (2^(scale_a[i][k/32] - 127) A[i][k])
 *                         * (2^(scale_b[j][k/32] - 127) B[k][j])  + beta * C[i][j]
 *
 * Defined by: "Tensor Core" chapter, the table of tensor-core formats per generation
 * (Blackwell adds block-scaled formats such as MXFP4 / NVFP4), with the MX layout of the
 * OCP microscaling format (32-element blocks, E8M0 shared exponent), applied here to
 * 8-bit elements (MXFP8).  The tensor cores apply the scales (no software promotion).
 *
 *   a_type, b_type : LL_IN_E4M3 or LL_IN_E5M2 (element formats of A and of B)
 *   A       : M x K codes, lda >= K          B : K x N codes, ldb >= N
 *   scale_a : M x ld_sa E8M0 codes (uint8), ld_sa >= ceil(K/32): row i holds the scales of
 *             row i of A, one per 32-wide K block (a shorter last block keeps its scale)
 *   scale_b : N x ld_sb E8M0 codes, ld_sb >= ceil(K/32): row j holds the scales of column j
 *             of B, one per 32-wide K block
 *   C, D, stream: as for ll_gemm_f16.  The code 255 (NaN) is not supported.
 *   workspace : required, sized by ll_gemm_mxf8_workspace_size: the call first rearranges
 *             the scale codes into the blocks the tensor cores' scale copies read (a few
 *             MB: 4 MiB at 8192^3), plus any operand repack as for ll_gemm_f16.  The
 *             scale matrices may start at any address and have any pitch >= ceil(K/32).
 * Accumulation is FP32 over the whole K; alpha / beta and the output cast as ll_gemm_f16.
 * Errors: as ll_gemm_fp8_blockscaled; LL_ERR_INVALID_ARG for other a_type / b_type or
 * scale pitches below ceil(K/32).
 */
/* Workspace bytes an ll_gemm_mxf8 call needs: the rearranged scale codes, plus the operand
 * repacks of ll_gemm_workspace_size (assuming 16-byte-aligned A and B; see there). */
size_t ll_gemm_mxf8_workspace_size(int M, int N, int K, int64_t lda, int64_t ldb);

ll_status ll_gemm_mxf8(int a_type, int b_type, int M, int N, int K, float alpha, const uint8_t* A, int64_t lda,
                       const uint8_t* scale_a, int64_t ld_sa, const uint8_t* B, int64_t ldb, const uint8_t* scale_b,
                       int64_t ld_sb, float beta, const float* C, int64_t ldc, void* D, int64_t ldd, int d_type,
                       void* workspace, size_t ws_bytes, ll_stream_t stream);

/*
 * NVFP4 block-scaled GEMM: FP4 E2M1 elements (values 0, 0.5, 1, 1.5, 2, 3, 4, 6 and their
 * negatives), every 16 consecutive K elements of a row of A, and of a column of B, sharing
 * one UE4M3 scale (the E4M3 bit pattern with the sign bit clear):
 *
 *   D[i][j] = alpha * sum_k (ue4m3(scale_a[i][k/16]) e2m1(A[i][k]))
 *                         * (ue4m3(scale_b[j][k/16]) e2m1(B[k][j]))  + beta * C[i][j]
 *
 * Defined by: "Tensor Core" chapter, the table of tensor-core formats per generation
 * (Blackwell adds block-scaled 4-bit formats, NVFP4 among them).  The tensor cores apply
 * the scales.
 *
 *   A      : M x K elements packed two per byte (element k of a row in byte k/2 of it, the
 *            low nibble for even k); lda = row pitch in ELEMENTS, even, >= K
 *   Bt     : B given transposed, N x K (row j holds column j of B), packed like A; ldbt =
 *            row pitch in elements, even, >= K
 *   K      : even (a row ends on a byte boundary); the last block may be shorter than 16
 *   scale_a: M x ld_sa UE4M3 codes, ld_sa >= ceil(K/16), row i for row i of A
 *   scale_b: N x ld_sb UE4M3 codes, ld_sb >= ceil(K/16), row j for column j of B
 *            scale codes 0..126 (127 is NaN and codes >= 128 carry a sign: not supported)
 *   C, D, stream: as for ll_gemm_f16.
 *   workspace : required, sized by ll_gemm_nvf4_workspace_size: the scale codes are first
 *            rearranged there (16 ceil(K/256) bytes for each of ceil(M/128) 128 rows and
 *            ceil(N/256) 256 columns: 8 MiB at 8192^3), plus a 16-byte-pitch copy of A or
 *            Bt when its byte pitch (lda/2, ldbt/2) is not a multiple of 16.
 * Accumulation is FP32 over the whole K; alpha / beta and the output cast as ll_gemm_f16.
 * Errors: LL_ERR_INVALID_ARG for odd K, lda or ldbt, pitches below K, scale pitches below
 * ceil(K/16), overlapping output; others as ll_gemm_f16.
 */
/* Workspace bytes an ll_gemm_nvf4 call needs (assuming 16-byte-aligned A and Bt). */
size_t ll_gemm_nvf4_workspace_size(int M, int N, int K, int64_t lda, int64_t ldbt);

ll_status ll_gemm_nvf4(int M, int N, int K, float alpha, const uint8_t* A, int64_t lda, const uint8_t* scale_a,
                       int64_t ld_sa, const uint8_t* Bt, int64_t ldbt, const uint8_t* scale_b, int64_t ld_sb,
                       float beta, const float* C, int64_t ldc, void* D, int64_t ldd, int d_type, void* workspace,
                       size_t ws_bytes, ll_stream_t stream);

/* ------------------------------------------------------------------ W8A8 GEMV */

/*
 * Batch-1 symmetric W8A8 linear layer:
 *
 *   z[o] = sum_k x[k] * W[o][k]                    (int32, exact)
 *   y[o] = fp16_rn( (float(z[o]) * x_scale) * w_scale[o] )   (two FP32 products, in order)
 *
 * Defined by: "NVIDIA A100: chip to SIMT", section 5.1 (symmetric W8A8: per-token
 * activation scale, per-output-channel weight scale, zero point 0, qweight[N,K]
 * stored output-channel-major; integer dot product over the whole K into INT32,
 * dequantised once in the epilogue) and section 5.2 (epilogue order).
 *
 *   x       : K int8 codes (the quantised activation of one token)
 *   x_scale : device pointer to ONE FP32 value (per-token scale s_x)
 *   W       : N x K int8, row o = output channel o, ldw >= K
 *   w_scale : N FP32 per-output-channel scales
 *   y       : N FP16 outputs (written)
 *   z_out   : N int32 raw dot products (written when not NULL)
 * |z| <= K * 128^2 must fit INT32, i.e. K <= 131071 (checked: LL_ERR_INVALID_ARG).
 * Ordering: the kernel is launched with programmatic dependent launch.  x, x_scale
 * are read and y, z_out written only after all preceding work on the stream has
 * finished; W and w_scale are read earlier, so they must not be written by a call of
 * this library that may still be running (the ordering rule at the top of this file).
 * N == 0: nothing is done.  K == 0: z = 0 and y = fp16(0 * s_x * s_W[o]).
 * Errors: LL_ERR_INVALID_ARG for negative sizes, ldw < K, NULL pointers, or outputs
 * that overlap an input or each other.
 */
ll_status ll_linear_w8a8_gemv(int N, int K, const int8_t* x, const float* x_scale,
                              const int8_t* W, int64_t ldw, const float* w_scale, void* y,
                              int32_t* z_out, ll_stream_t stream);

/* Output of the W8A8 GEMV variants. */
typedef enum { LL_GEMV_OUT_F16 = 0, LL_GEMV_OUT_I8 = 1 } ll_gemv_out_type;

/*
 * W8A8 GEMV with the epilogue variants of the A100 page, section 5.1 (an optional
 * bias is added in the floating-point epilogue after dequantisation; a next layer
 * that takes INT8 can receive a requantised INT8 output instead of FP16):
 *
 *   v[o] = (float(z[o]) * x_scale) * w_scale[o]          (as ll_linear_w8a8_gemv)
 *   v[o] = v[o] + bias[o]                                 (when bias != NULL; FP32 add)
 *   y_type == LL_GEMV_OUT_F16: y[o] = fp16_rn(v[o])                    (y FP16 [N])
 *   y_type == LL_GEMV_OUT_I8:  y[o] = clamp(rint(v[o] / *y_scale), -127, 127)   (y int8 [N])
 *
 *   bias    : N FP32 or NULL          y_scale : device pointer to one FP32 (INT8 output)
 * Other arguments, ordering and errors as ll_linear_w8a8_gemv; LL_ERR_INVALID_ARG also
 * for an unknown y_type or a NULL y_scale with INT8 output.
 */
ll_status ll_linear_w8a8_gemv_ex(int N, int K, const int8_t* x, const float* x_scale,
                                 const int8_t* W, int64_t ldw, const float* w_scale,
                                 const float* bias, int y_type, const float* y_scale, void* y,
                                 int32_t* z_out, ll_stream_t stream);

/*
 * W8A8 linear layer for a batch of M tokens (A100 page, section 5.1: the activation
 * scale is per token, the weight scale per output channel, zero point 0; section 5.2:
 * the dequantisation order).  Token m is the batch-1 layer with its own scale:
 *
 *   z[m][o] = sum_k X[m][k] * W[o][k]                           (exact INT32)
 *   v       = (float(z[m][o]) * x_scale[m]) * w_scale[o]  (+ bias[o])
 *   Y[m][o] = fp16_rn(v)  or  clamp(rint(v / *y_scale), -127, 127)   (as y_type)
 *
 *   X       : M x K int8 row-major, row pitch ldx >= K bytes (one token per row)
 *   x_scale : M FP32 (device)          W, ldw, w_scale, bias, y_type, y_scale: as
 *   Y       : M x N, pitch ldy >= N      ll_linear_w8a8_gemv_ex
 *             elements (FP16 or int8)
 *   z_out   : M x N INT32 with pitch ldz >= N, or NULL
 * Every weight byte is read from memory once per group of up to 16 tokens: larger M
 * runs as consecutive groups.  M == 1 is exactly ll_linear_w8a8_gemv_ex.  Results are
 * bit-identical to M calls of ll_linear_w8a8_gemv_ex, one per token.
 * Ordering: programmatic dependent launch as ll_linear_w8a8_gemv (W and w_scale are
 * read before the preceding work of the stream has finished; X, the other scales and
 * the outputs only after).
 * M == 0 or N == 0: nothing.  Errors: LL_ERR_INVALID_ARG for negative sizes,
 * K > 131071, ldx < K, ldw < K, ldy < N, ldz < N with z_out, NULL pointers, an unknown
 * y_type, a NULL y_scale with INT8 output, or outputs that overlap an input or each other.
 */
ll_status ll_linear_w8a8(int M, int N, int K, const int8_t* X, int64_t ldx, const float* x_scale,
                         const int8_t* W, int64_t ldw, const float* w_scale, const float* bias,
                         int y_type, const float* y_scale, void* Y, int64_t ldy, int32_t* z_out,
                         int64_t ldz, ll_stream_t stream);

/*
 * Weight-only INT8 linear layer with BF16 activations (the Tensor Core chapter's mixed
 * precision: low-precision storage, FP32 accumulation; weights stored as INT8 with the
 * per-output-channel scale s_W[o] of the A100 page, section 5.1; activations not
 * quantised):
 *
 *   y[m][o] = cast_out( w_scale[o] * sum_k X[m][k] * W[o][k]  (+ bias[o]) )
 *
 *   X       : M x K BF16 row-major, pitch ldx >= K elements (one token per row)
 *   W       : N x K int8, pitch ldw >= K bytes (qweight[N][K], output-channel-major)
 *   w_scale : N FP32                 bias : N FP32 or NULL
 *   Y       : M x N, pitch ldy >= N elements, of type y_type (ll_out_type: F32, BF16, F16;
 *             rounded to nearest even)
 * The dot product is accumulated in FP32 (any order; results are deterministic run to
 * run); the scale multiplies the sum, then the bias is added, in FP32.  Designed for
 * decode-sized M (up to 4 tokens per weight pass; larger M runs as several passes).
 * Ordering: programmatic dependent launch as ll_linear_w8a8_gemv.
 * M == 0 or N == 0: nothing.  Errors: LL_ERR_INVALID_ARG for negative sizes, ldx < K,
 * ldw < K, ldy < N, NULL pointers, an unknown y_type, or Y overlapping an input.
 */
ll_status ll_linear_w8a16(int M, int N, int K, const void* X, int64_t ldx, const int8_t* W, int64_t ldw,
                          const float* w_scale, const float* bias, int y_type, void* Y, int64_t ldy,
                          ll_stream_t stream);

/*
 * Symmetric per-token activation quantiser (A100 page, section 5.1: the activation is
 * quantised at run time by the preceding operator or a separate quantisation step):
 *
 *   scale[i] = amax_k |x[i][k]| / 127        (FP32; 1 for an all-zero row)
 *   q[i][k]  = clamp(rint(x[i][k] / scale[i]), -127, 127)   (FP32 division, ties to even)
 *
 *   x : M x K FP16 (ldx >= K)    q : M x K int8 (ldq >= K)    scale : M FP32
 * M == 0: nothing.  Errors: LL_ERR_INVALID_ARG for negative sizes, ld < K, NULL pointers,
 * or q / scale overlapping x or each other.
 */
ll_status ll_quantize_per_token_f16(int M, int K, const void* x, int64_t ldx, int8_t* q,
                                    int64_t ldq, float* scale, ll_stream_t stream);

/*
 * The batch-1 linear layer on an FP16 activation: the per-token quantiser fused into
 * the W8A8 GEMV (every CTA quantises x into its shared memory; the int8 activation
 * never goes through HBM on the way to the dot products).  Results are bit-identical to
 * ll_quantize_per_token_f16 (M = 1) followed by ll_linear_w8a8_gemv_ex.
 *
 *   x       : K FP16 (the activation of one token)
 *   x_q     : K int8, written with the quantised activation (required)
 *   x_scale : one FP32, written with its scale (required)
 *   other arguments, ordering and errors as ll_linear_w8a8_gemv_ex (x_q and x_scale
 *   are outputs and may overlap nothing else).
 */
ll_status ll_linear_f16_w8a8_gemv(int N, int K, const void* x, int8_t* x_q, float* x_scale,
                                  const int8_t* W, int64_t ldw, const float* w_scale,
                                  const float* bias, int y_type, const float* y_scale, void* y,
                                  int32_t* z_out, ll_stream_t stream);

/* ------------------------------------------------------------------ status */

/*
 * Synchronise `stream`, then read and clear the current device's status word.
 * Returns LL_OK, LL_ERR_DEVICE_TIMEOUT if a kernel's bounded wait ran out since the
 * last call, or LL_ERR_CUDA if the synchronisation itself failed.
 * `detail` (host, may be NULL) receives the raw word: bits 0-7 the status code,
 * bits 8-15 the kernel role that gave up (1 producer, 2 MMA, 3 epilogue, 4 test wait,
 * 5 block-scale staging).
 */
ll_status ll_get_device_status(ll_stream_t stream, uint32_t* detail);

/*
 * Set the time limit, in nanoseconds, of every bounded wait in this library's
 * kernels on the current device (default 2e9 = 2 s).  Applies to kernels launched
 * after this call returns (the limit travels with each launch as a parameter).
 * Returns LL_ERR_INVALID_ARG for ns == 0.
 */
ll_status ll_set_wait_timeout_ns(uint64_t ns);

/*
 * Launch one CTA that waits, with the bounded wait the GEMM kernels use, on an
 * mbarrier phase that nothing completes.  The wait runs out after the configured
 * limit, the kernel records LL_ERR_DEVICE_TIMEOUT (role 4) and returns.  Used to
 * test failure detection without a GPU fault; the paper has no counterpart.
 */
ll_status ll_debug_timeout_probe(ll_stream_t stream);

/* Human-readable name of a status code (static storage). */
const char* ll_status_string(ll_status s);

/* Library version string, e.g. "linear_layer_gb300 0.1 sm_103a". */
const char* ll_version(void);

#ifdef __cplusplus
}
#endif

#endif /* LINEAR_LAYER_GB300_LL_H */
