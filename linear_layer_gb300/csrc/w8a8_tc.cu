// W8A8 linear layer for 17..32 tokens per weight pass on the tensor cores ("NVIDIA
// A100: chip to SIMT", sections 5.1 and 5.2; section 5.5 asks when the tensor-core tile
// pays off for a handful of tokens):
//
//   z[m][o] = sum_k X[m][k] * W[o][k]                      (exact INT32)
//   y[m][o] = fp16_rn((float(z[m][o]) * s_x[m]) * s_W[o])  (+ bias, or INT8 requantised)
//
// sm_103a has no INT8 tensor-core MMA, and its dp4a rate (about 128 int8 MACs per clock
// per SM) falls behind the weight stream from about six tokens on.  This kernel runs the
// integer product exactly on the FP16 tensor-core path:
//   * int8 values are exact in FP16, a product of two (|p| <= 2^14) is exact in the FP32
//     accumulator, and so is every partial sum of at most 512 of them (|s| <= 2^23).
//     The MMAs accumulate each 512-K chunk into a fresh TMEM buffer; the epilogue turns
//     the chunk (an exact integer in FP32) into INT32 and adds it in registers, so z is
//     exact for any K.
//   * weights are the A operand: TMEM lane = output channel, M = 128; the tokens are the
//     B operand (N = tokens rounded up to 16, K-major, shared memory).  Each CTA (one
//     per SM) owns strips of at most 80 consecutive output channels, the strips split N
//     evenly, so every SM streams the same number of weight bytes.
//   * the weight stream needs well over 100 KB in flight per SM (the loaded latency is
//     about 3.5 us), so one producer thread fetches it with TMA into a deep int8 ring:
//     per 256-K stage one 128-byte-swizzled box of 80 rows x 128 bytes per 128-K half
//     (rows past the strip belong to the neighbour strip, which reads them at the same
//     time, or lie past N and arrive as zeros) plus the tokens; K past the end arrives as
//     zeros.  Its position advances without divisions: a stage costs a few instructions.
//   * CQ converter warps per TMEM lane quarter turn each stage into FP16: the weight rows
//     go from shared memory straight into TMEM (tcgen05.st; the MMA reads A from TMEM,
//     so FP16 weights cost no shared-memory bandwidth), the token rows into the swizzled
//     K-major B tile in shared memory.  int8 -> FP16 is two byte permutes and one packed
//     subtraction per four values.  A warp reaches only its lane quarter, so the strip's
//     rows are spread over the four quarters (rows q * hq .. q * hq + hq - 1 in quarter q).
//   * one thread issues the MMAs (kind::f16, A from TMEM, M = 128, N = NP, K = 16) and
//     commits each stage and each chunk; 4 epilogue warps read a chunk, add it, hand the
//     buffer back and finally dequantise and store.
// Measured limits on GB300 (11008 x 4096 layer): a tcgen05.mma with M = 128, K = 16 takes
// at least ~43 cycles whatever N <= 64 is, so the 256 MMAs of a 4096-K strip need ~6 us,
// and the conversion about as much again; this path reaches ~2.2 TB/s of weights, as
// fast as dp4a at 16 tokens and faster above, so it serves passes of 17..32 tokens.
// Every wait is bounded (a timeout records the role in the device status word and the
// CTA winds down, draining its copies and MMAs); programmatic dependent launch: the
// first weight stages are requested before griddepcontrol.wait, X, the scales and the
// outputs are touched only after it.
#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"

namespace ll {

namespace {

constexpr int kTcProducerWarp = 0;
constexpr int kTcMmaWarp = 1;
constexpr int kTcConvWarp0 = 2;
constexpr int kTcBK = 256;         // K per stage
constexpr int kTcChunkStages = 2;  // 512 K per exact FP32 partial
constexpr int kTcHR = 80;          // most strip rows a stage holds
constexpr int kTcACols = kTcBK / 2;  // TMEM columns of one A stage (FP16 pairs)
constexpr int kTcA0 = 128;           // first TMEM column of the A stages

struct TcParams {
  int M, N, K;
  const float* x_scale;
  const float* w_scale;
  const float* bias;
  int out_i8;
  const float* y_scale;
  void* Y;
  int64_t ldy;
  int32_t* Z;
  int64_t ldz;
  int strips;  // output-channel strips, split evenly over N
  uint32_t* status;
  uint64_t timeout_ns;
};

// tcgen05 instruction descriptor, kind::f16: FP16 A and B, FP32 D, both K-major.
__host__ __device__ constexpr uint32_t idesc_f16_kk(int n, int m) {
  return (1u << 4) | (static_cast<uint32_t>(n >> 3) << 17) | (static_cast<uint32_t>(m >> 4) << 24);
}

// four int8 (one 32-bit word) -> four FP16 (two 32-bit words), exactly: byte b + 128 set
// under the FP16 exponent of 1024 reads 1024 + b + 128; subtracting 1152 leaves b.
__device__ __forceinline__ void i8x4_to_f16x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t u = w ^ 0x80808080u;
  uint32_t a, b;
  asm("prmt.b32 %0, %1, %2, 0x7170;" : "=r"(a) : "r"(u), "r"(0x64646464u));
  asm("prmt.b32 %0, %1, %2, 0x7372;" : "=r"(b) : "r"(u), "r"(0x64646464u));
  const uint32_t bias = 0x64806480u;  // FP16 1152 in both halves
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(lo) : "r"(a), "r"(bias));
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(hi) : "r"(b), "r"(bias));
}

__device__ __forceinline__ int4 ld_shared_v4(uint32_t addr) {
  int4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
               : "memory");
}

__device__ __forceinline__ void tmem_st_x8(uint32_t taddr, const uint32_t (&r)[8]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
      : "memory");
}

__device__ __forceinline__ void tmem_st_x32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, "
      "%13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]),
      "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
      "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// D[tmem] (+)= A[tmem] x B[smem], FP16 inputs, FP32 accumulator.
__device__ __forceinline__ void mma_f16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                           uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

template <int NP, int S8, int SA, int BR, int CQ>
struct TcCfg {
  static constexpr int CONV_WARPS = 4 * CQ;         // CQ converter warps per TMEM lane quarter
  static constexpr int CONV_THREADS = CONV_WARPS * 32;
  static constexpr int EPI_WARP0 = kTcConvWarp0 + CONV_WARPS;
  static constexpr int THREADS = (EPI_WARP0 + 4) * 32;
  static constexpr int KQ = kTcBK / CQ;              // K of a stage per converter warp
  static constexpr int W_COL = kTcHR * 128;     // one 128-K column of the strip's rows
  static constexpr int X_COL = NP * 128;        // one 128-K column of the tokens
  static constexpr int I8_STAGE = 2 * W_COL + 2 * X_COL;
  static constexpr int B_ATOM = NP * 128;       // one 64-K swizzle-atom column of B
  static constexpr int B_STAGE = 4 * B_ATOM;    // FP16 tokens, 256 K
  static constexpr size_t SMEM = 1024 + static_cast<size_t>(S8) * I8_STAGE + static_cast<size_t>(SA) * B_STAGE + 1024;
  static_assert(NP % 16 == 0 && NP >= 16 && NP <= 32, "token tile");
  static_assert(kTcA0 + SA * kTcACols <= 512 && 2 * NP <= kTcA0, "TMEM columns");
  static_assert(I8_STAGE % 1024 == 0 && B_STAGE % 1024 == 0, "swizzle atoms stay 1024-byte aligned");
  static_assert(BR % 8 == 0 && kTcHR % BR == 0, "boxes tile the stage rows");
};

__device__ __forceinline__ void strip_rows(const TcParams& p, int t, int& row0, int& h) {
  row0 = static_cast<int>((static_cast<int64_t>(t) * p.N) / p.strips);
  h = static_cast<int>((static_cast<int64_t>(t + 1) * p.N) / p.strips) - row0;
}

template <int NP, int S8, int SA, int BR, int CQ>
__global__ void __launch_bounds__(TcCfg<NP, S8, SA, BR, CQ>::THREADS, 1)
    w8a8_tc_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                   const TcParams p) {
  using Cfg = TcCfg<NP, S8, SA, BR, CQ>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* i8_ring = smem;
  uint8_t* b_ring = smem + S8 * Cfg::I8_STAGE;
  uint64_t* bars = reinterpret_cast<uint64_t*>(b_ring + SA * Cfg::B_STAGE);
  // bars: i8full[S8], i8empty[S8], afull[SA], aempty[SA], cfull[2], cempty[2], drain
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * S8 + 2 * SA + 5);
  uint32_t* abort_flag = tmem_slot + 1;
  float* sxs = reinterpret_cast<float*>(tmem_slot + 2);  // [NP] token scales

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  auto i8full = [&](int s) { return smem_addr(bars + s); };
  auto i8empty = [&](int s) { return smem_addr(bars + S8 + s); };
  auto afull = [&](int s) { return smem_addr(bars + 2 * S8 + s); };
  auto aempty = [&](int s) { return smem_addr(bars + 2 * S8 + SA + s); };
  auto cfull = [&](int b) { return smem_addr(bars + 2 * S8 + 2 * SA + b); };
  auto cempty = [&](int b) { return smem_addr(bars + 2 * S8 + 2 * SA + 2 + b); };
  const uint32_t drain_bar = smem_addr(bars + 2 * S8 + 2 * SA + 4);

  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (threadIdx.x == 0) {
    for (int s = 0; s < S8; ++s) {
      mbar_init(i8full(s), 1);
      mbar_init(i8empty(s), Cfg::CONV_THREADS);
    }
    for (int s = 0; s < SA; ++s) {
      mbar_init(afull(s), Cfg::CONV_THREADS);
      mbar_init(aempty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(cfull(b), 1);
      mbar_init(cempty(b), 128);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0u;
    fence_mbar_init();
  }
  if (warp == kTcMmaWarp) {
    tmem_alloc(smem_addr(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(tmem_slot);

  WaitCtx wctx{p.status, p.timeout_ns, abort_flag};
  const int KBLK = (p.K + kTcBK - 1) / kTcBK;
  const int nstrips = blockIdx.x < p.strips ? (p.strips - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
  const int nstages = nstrips * KBLK;

  if (warp == kTcProducerWarp) {
    // ---------------------------------------------------------------- TMA producer
    // One thread keeps the ring full; its position (strip, K block) advances without
    // divisions, so issuing a stage costs a handful of instructions.
    if (lane == 0) {
      tma_prefetch_desc(&tmW);
      tma_prefetch_desc(&tmX);
      int t = blockIdx.x, kb = 0, row0, h;
      strip_rows(p, t, row0, h);
      auto next = [&]() {
        if (++kb == KBLK) {
          kb = 0;
          t += gridDim.x;
          strip_rows(p, t, row0, h);
        }
      };
      auto issue_w = [&](int s) {
        const uint32_t st = smem_addr(i8_ring + s * Cfg::I8_STAGE);
        const int boxes = (h + BR - 1) / BR;
        mbar_arrive_expect_tx(i8full(s), 2 * boxes * BR * 128 + 2 * Cfg::X_COL);
        for (int i = 0; i < boxes; ++i)
          for (int c = 0; c < 2; ++c)
            tma_load_2d(st + c * Cfg::W_COL + i * BR * 128, &tmW, i8full(s), kb * kTcBK + c * 128, row0 + BR * i);
      };
      auto issue_x = [&](int s, int kbx) {
        const uint32_t st = smem_addr(i8_ring + s * Cfg::I8_STAGE) + 2 * Cfg::W_COL;
        for (int c = 0; c < 2; ++c) tma_load_2d(st + c * Cfg::X_COL, &tmX, i8full(s), kbx * kTcBK + c * 128, 0);
      };
      // the ring starts empty: the weights of its first stages go out before the
      // dependency wait, their X after it
      const int early = nstages < S8 ? nstages : S8;
      for (int j = 0; j < early; ++j) {
        issue_w(j);
        next();
      }
      asm volatile("griddepcontrol.wait;" ::: "memory");
      for (int j = 0, kbx = 0; j < early; ++j) {
        issue_x(j, kbx);
        if (++kbx == KBLK) kbx = 0;
      }
      int it = early;
      bool ok = true;
      for (; it < nstages; ++it) {
        const int s = it % S8;
        if (!wait_bounded(i8empty(s), ((it / S8) & 1u) ^ 1u, wctx, kRoleProducer)) {
          ok = false;
          break;
        }
        issue_w(s);
        issue_x(s, kb);
        next();
      }
      if (!ok) {  // copies still in flight must land before the CTA exits
        for (int j = (it > S8 ? it - S8 : 0); j < it; ++j) wait_drain(i8full(j % S8), (j / S8) & 1u, p.timeout_ns);
      }
    }
  } else if (warp == kTcMmaWarp) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t IDESC = idesc_f16_kk(NP, 128);
      uint32_t chunk = 0, d_tmem = 0;
      bool ok = true;
      int kb = 0;
      for (int it = 0; it < nstages && ok; ++it) {
        const bool first = (kb % kTcChunkStages) == 0;
        const bool last = (kb % kTcChunkStages) == kTcChunkStages - 1 || kb == KBLK - 1;
        if (first) {
          const uint32_t cb = chunk & 1u;
          if (!wait_bounded(cempty(cb), ((chunk >> 1) & 1u) ^ 1u, wctx, kRoleMma)) {
            ok = false;
            break;
          }
          tc_fence_after();
          d_tmem = tmem_base + cb * NP;
        }
        const int sa = it % SA;
        if (!wait_bounded(afull(sa), (it / SA) & 1u, wctx, kRoleMma)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t a_tm = tmem_base + kTcA0 + sa * kTcACols;
        const uint32_t b_st = smem_addr(b_ring + sa * Cfg::B_STAGE);
#pragma unroll
        for (int kk = 0; kk < kTcBK / 16; ++kk) {
          const uint64_t bdesc = smem_desc_sw128(b_st + (kk >> 2) * Cfg::B_ATOM + (kk & 3) * 32, 16, 1024);
          mma_f16_ta(d_tmem, a_tm + kk * 8, bdesc, IDESC, (first && kk == 0) ? 0u : 1u);
        }
        mma_commit(aempty(sa));
        if (last) {
          mma_commit(cfull(chunk & 1u));
          ++chunk;
        }
        if (++kb == KBLK) kb = 0;
      }
      mma_commit(drain_bar);  // every MMA must finish before TMEM is freed
      wait_drain(drain_bar, 0u, p.timeout_ns);
    }
  } else if (warp < Cfg::EPI_WARP0) {
    // ---------------------------------------------------------------- converters
    const int qd = warp & 3;                       // TMEM lane quarter
    const int part = (warp - kTcConvWarp0) >> 2;   // which K part (of CQ) of the stage
    const int ct = threadIdx.x - kTcConvWarp0 * 32;
    const uint32_t lane_base = static_cast<uint32_t>(qd * 32) << 16;
    int t = blockIdx.x, kb = 0, row0, h;
    strip_rows(p, t, row0, h);
    for (int it = 0; it < nstages; ++it) {
      const int s8 = it % S8, sa = it % SA;
      bool w = wait_bounded(i8full(s8), (it / S8) & 1u, wctx, kRoleProducer);
      w = w && wait_bounded(aempty(sa), ((it / SA) & 1u) ^ 1u, wctx, kRoleProducer);
      if (!__all_sync(0xffffffffu, w)) break;
      tc_fence_after();
      const uint32_t st = smem_addr(i8_ring + s8 * Cfg::I8_STAGE);
      // weights: strip row r = qd * hq + lane -> TMEM lane qd * 32 + lane; this warp
      // converts K [part * KQ, +KQ) of the stage (16-byte pieces, 8 columns each)
      const int hq = (h + 3) >> 2;
      const int r = qd * hq + lane;
      const bool live = lane < hq && r < h;
      const uint32_t a_tm = tmem_base + lane_base + kTcA0 + sa * kTcACols + part * (Cfg::KQ / 2);
#pragma unroll
      for (int g4 = 0; g4 < Cfg::KQ / 64; ++g4) {  // 4 pieces (64 K) per 32-column TMEM store
        int4 v[4];
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          const int ch = part * (Cfg::KQ / 16) + g4 * 4 + cc;  // piece of the 256-K stage
          v[cc] = live ? ld_shared_v4(st + (ch >> 3) * Cfg::W_COL + r * 128 + (((ch & 7) ^ (r & 7)) << 4))
                       : make_int4(0, 0, 0, 0);
        }
        uint32_t f[32];
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          i8x4_to_f16x4(static_cast<uint32_t>(v[cc].x), f[8 * cc + 0], f[8 * cc + 1]);
          i8x4_to_f16x4(static_cast<uint32_t>(v[cc].y), f[8 * cc + 2], f[8 * cc + 3]);
          i8x4_to_f16x4(static_cast<uint32_t>(v[cc].z), f[8 * cc + 4], f[8 * cc + 5]);
          i8x4_to_f16x4(static_cast<uint32_t>(v[cc].w), f[8 * cc + 6], f[8 * cc + 7]);
        }
        tmem_st_x32(a_tm + g4 * 32, f);
      }
      // tokens: piece c (16 K) of token m -> the swizzled K-major B tile
      const uint32_t xs = st + 2 * Cfg::W_COL;
      const uint32_t bs = smem_addr(b_ring + sa * Cfg::B_STAGE);
      for (int pc = ct; pc < 16 * NP; pc += Cfg::CONV_THREADS) {
        const int m = pc >> 4, c = pc & 15;
        if (m >= p.M) break;
        const int4 v = ld_shared_v4(xs + (c >> 3) * Cfg::X_COL + m * 128 + (((c & 7) ^ (m & 7)) << 4));
        uint32_t f[8];
        i8x4_to_f16x4(static_cast<uint32_t>(v.x), f[0], f[1]);
        i8x4_to_f16x4(static_cast<uint32_t>(v.y), f[2], f[3]);
        i8x4_to_f16x4(static_cast<uint32_t>(v.z), f[4], f[5]);
        i8x4_to_f16x4(static_cast<uint32_t>(v.w), f[6], f[7]);
        const uint32_t rb = bs + (c >> 2) * Cfg::B_ATOM + m * 128;
        const int u = 2 * (c & 3);
        st_shared_v4(rb + ((u ^ (m & 7)) << 4), f[0], f[1], f[2], f[3]);
        st_shared_v4(rb + (((u + 1) ^ (m & 7)) << 4), f[4], f[5], f[6], f[7]);
      }
      tmem_st_wait();
      tc_fence_before();
      fence_proxy_async_smem();  // B tile stores -> tcgen05.mma reads
      mbar_arrive(afull(sa));
      mbar_arrive(i8empty(s8));
      if (++kb == KBLK) {
        kb = 0;
        t += gridDim.x;
        strip_rows(p, t, row0, h);
      }
    }
  } else {
    // ---------------------------------------------------------------- epilogue
    const int qd = warp & 3;
    const uint32_t lane_base = static_cast<uint32_t>(qd * 32) << 16;
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int et = threadIdx.x - Cfg::EPI_WARP0 * 32;
    if (et < NP) sxs[et] = et < p.M ? p.x_scale[et] : 0.0f;
    asm volatile("bar.sync 1, 128;" ::: "memory");  // the 4 epilogue warps only
    const float sy = p.out_i8 ? *p.y_scale : 1.0f;
    const int nchunks = (KBLK + kTcChunkStages - 1) / kTcChunkStages;
    uint32_t chunk = 0;
    bool ok = true;
    for (int i = 0; i < nstrips && ok; ++i) {
      int row0, h;
      strip_rows(p, blockIdx.x + i * gridDim.x, row0, h);
      int acc[NP];
#pragma unroll
      for (int j = 0; j < NP; ++j) acc[j] = 0;
      for (int c = 0; c < nchunks; ++c) {
        const uint32_t cb = chunk & 1u;
        bool w = wait_bounded(cfull(cb), (chunk >> 1) & 1u, wctx, kRoleEpilogue);
        w = __all_sync(0xffffffffu, w);
        if (!w) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int c16 = 0; c16 < NP / 16; ++c16) {
          uint32_t r[16];
          tmem_ld_x16(tmem_base + lane_base + cb * NP + c16 * 16, r);
          tmem_ld_wait(r);
#pragma unroll
          for (int j = 0; j < 16; ++j) acc[c16 * 16 + j] += __float2int_rn(__uint_as_float(r[j]));
        }
        tc_fence_before();
        mbar_arrive(cempty(cb));
        ++chunk;
      }
      if (!ok) break;
      const int hq = (h + 3) >> 2;
      const int r = qd * hq + lane;
      if (lane < hq && r < h) {
        const int o = row0 + r;
        const float sw = p.w_scale[o];
        const float b = p.bias ? p.bias[o] : 0.0f;
#pragma unroll
        for (int m = 0; m < NP; ++m) {
          if (m < p.M) {
            if (p.Z) p.Z[static_cast<int64_t>(m) * p.ldz + o] = acc[m];
            const float tt = __fmul_rn(__int2float_rn(acc[m]), sxs[m]);
            float u = __fmul_rn(tt, sw);
            if (p.bias) u = __fadd_rn(u, b);
            if (p.out_i8) {
              const int rq = __float2int_rn(__fdiv_rn(u, sy));
              static_cast<int8_t*>(p.Y)[static_cast<int64_t>(m) * p.ldy + o] =
                  static_cast<int8_t>(max(-127, min(127, rq)));
            } else {
              static_cast<__half*>(p.Y)[static_cast<int64_t>(m) * p.ldy + o] = __float2half_rn(u);
            }
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kTcMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 512);
  }
}

template <int NP, int S8, int SA, int BR, int CQ>
ll_status launch_tc(TcParams p, const int8_t* X, int64_t ldx, const int8_t* W, int64_t ldw,
                    const LaunchCtx& ctx) {
  using Cfg = TcCfg<NP, S8, SA, BR, CQ>;
  auto kern = w8a8_tc_kernel<NP, S8, SA, BR, CQ>;
  CUtensorMap tmW, tmX;
  if (!make_tensor_map_2d(&tmW, W, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, p.N, p.K, ldw, 128, BR)) return LL_ERR_CUDA;
  if (!make_tensor_map_2d(&tmX, X, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, p.M, p.K, ldx, 128, NP)) return LL_ERR_CUDA;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(Cfg::SMEM)) !=
      cudaSuccess) {
    cudaGetLastError();
    return LL_ERR_CUDA;
  }
  // strips of at most kTcHR rows, the same number for every CTA
  const int G = ctx.num_sms < p.N ? ctx.num_sms : p.N;
  const int per = (p.N + kTcHR * G - 1) / (kTcHR * G);
  p.strips = G * per;
  if (p.strips > p.N) p.strips = p.N;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(G);
  cfg.blockDim = dim3(Cfg::THREADS);
  cfg.dynamicSmemBytes = Cfg::SMEM;
  cfg.stream = ctx.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kern, tmW, tmX, p) != cudaSuccess) {
    cudaGetLastError();
    return LL_ERR_CUDA;
  }
  return LL_OK;
}

}  // namespace

// Up to 32 tokens of the W8A8 layer on the tensor cores (K % 16 == 0, ldx and ldw
// multiples of 16, 16-byte aligned X and W).
ll_status launch_w8a8_tc(int M, int N, int K, const int8_t* X, int64_t ldx, const float* x_scale,
                         const int8_t* W, int64_t ldw, const float* w_scale, const float* bias, int out_i8,
                         const float* y_scale, void* Y, int64_t ldy, int32_t* Z, int64_t ldz,
                         const LaunchCtx& ctx) {
  TcParams p;
  p.M = M;
  p.N = N;
  p.K = K;
  p.x_scale = x_scale;
  p.w_scale = w_scale;
  p.bias = bias;
  p.out_i8 = out_i8;
  p.y_scale = y_scale;
  p.Y = Y;
  p.ldy = ldy;
  p.Z = Z;
  p.ldz = ldz;
  p.strips = 1;
  p.status = ctx.status;
  p.timeout_ns = ctx.timeout_ns;
  return launch_tc<32, 6, 3, 80, 2>(p, X, ldx, W, ldw, ctx);
}

}  // namespace ll
