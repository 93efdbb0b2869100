// Dense GEMM on the 5th-generation tensor cores of sm_103a:
//
//   D = alpha * A x B + beta * C,   FP32 accumulation
//
// ("Tensor Core" chapter, section "Tensor Core 做什么" and table "精度": low-precision
// inputs, FP32 accumulator; FP8 with per-block scaling factors.)
//
// Two kernels: the one-CTA kernel below (small 16-bit problems, and FP8 at every size)
// and the CTA-pair kernel further down (large 16-bit problems); launch_gemm_tc at the
// end chooses.  In the one-CTA kernel one persistent CTA per SM walks a static list of
// 128 x BN output tiles in a grouped (L2-friendly) order.  Warp roles:
//   warp 0      TMA producer: A (128 x BK, K-major) and B (BK x BN, N-major) tiles,
//               128-byte swizzle, into a STAGES-deep shared-memory ring (mbarrier
//               full/empty pairs).  The K tail is zero-filled by TMA out-of-bounds fill.
//   warp 1      TMEM allocator and MMA issuer: one thread issues tcgen05.mma
//               (M = 128, N = BN) into a TMEM accumulator; tcgen05.commit releases
//               smem stages and hands finished accumulators to the epilogue.
//   warps 2..   epilogue.  16-bit inputs: 4 warps read the accumulator with
//               tcgen05.ld while the next tile's MMAs run into the other of two TMEM
//               accumulators, then apply alpha/beta, cast and store; each 32 x 32
//               chunk is transposed through shared memory so that global C loads and
//               D stores are row segments (coalesced for any leading dimension).
//               FP8 inputs: 8 warps promote each 128-K block: the MMAs accumulate one
//               block into a TMEM partial buffer (NACC of them in turn: two for
//               256-wide tiles, four for 128-wide ones), the warps read it and add
//               scale_a[m][kb] * scale_b[kb][n/128] * partial into FP32 registers; at
//               the end of the tile they apply alpha/beta and store.
// Every wait is bounded: on expiry the CTA records LL_ERR_DEVICE_TIMEOUT, drains the
// copies and MMAs it has in flight, frees TMEM and exits.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstring>
#include <mutex>

#include <atomic>
#include <chrono>

#include "gemm_common.cuh"

namespace ll {


template <int BN_, bool FP8_>
struct TileCfg {
  static constexpr int BN = BN_;
  static constexpr bool FP8 = FP8_;
  static constexpr int BM = 128;
  static constexpr int ELT = FP8 ? 1 : 2;
  static constexpr int BK = 128 / ELT;        // K elements per stage: one 128-byte swizzle row
  static constexpr int UMMA_K = 32 / ELT;     // K of one tcgen05.mma (32 bytes)
  static constexpr int KSTEPS = BK / UMMA_K;  // MMAs per stage
  static constexpr int A_BYTES = BM * 128;
  static constexpr int B_BOX_N = 128 / ELT;  // N elements in one 128-byte swizzle row
  static constexpr int B_BOXES = BN / B_BOX_N;
  static constexpr int B_BOX_BYTES = BK * 128;
  static constexpr int B_BYTES = B_BOXES * B_BOX_BYTES;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int STAGES = (196608 / STAGE_BYTES) < 8 ? (196608 / STAGE_BYTES) : 8;
  // accumulators (16-bit: tiles) or FP8 partial buffers (128-K blocks) in TMEM; FP8
  // uses all 512 columns, so a 128-column tile has four partial buffers
  static constexpr int TMEM_COLS = FP8 ? 512 : 2 * BN;
  static constexpr int NACC = TMEM_COLS / BN;
  static constexpr int EPI_WARPS = FP8 ? 8 : 4;
  static constexpr int EPI_THREADS = 32 * EPI_WARPS;
  static constexpr int EPI_WARP0 = 2;  // first epilogue warp
  static constexpr int THREADS = 32 * EPI_WARP0 + EPI_THREADS;
  static constexpr int EPI_STAGE_BYTES = FP8 ? 0 : EPI_WARPS * 32 * 32 * 4;  // 32x32 FP32 per warp
  static constexpr int SMEM = STAGES * STAGE_BYTES + EPI_STAGE_BYTES + 512 + 1024;
  static_assert(SMEM <= 227 * 1024, "shared memory budget");
  static_assert(B_BOXES >= 1 && BN % B_BOX_N == 0, "tile N must cover whole swizzle rows");
  static_assert(STAGE_BYTES % 1024 == 0, "stages must keep 1024-byte swizzle alignment");
  static_assert(TMEM_COLS >= 32 && TMEM_COLS <= 512 && (TMEM_COLS & (TMEM_COLS - 1)) == 0,
                "TMEM allocation must be a power of two in [32, 512]");
  static_assert(STAGES >= 2, "need at least two stages");
};


// One 32 x 32 chunk of 16-bit D into a 2 KB staging buffer in the layout of a TMA box
// of 64-byte rows with 64-byte swizzle: 16-byte slot j of row l (= lane) at
// j ^ ((l >> 1) & 3).  The buffer must be 512-byte aligned.
__device__ __forceinline__ void stage_row16(uint8_t* buf, int lane, const float (&o)[32], bool bf) {
  uint4* drow = reinterpret_cast<uint4*>(buf + lane * 64);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    uint32_t w4[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float lo = o[8 * j + 2 * i], hi = o[8 * j + 2 * i + 1];
      if (bf) {
        __nv_bfloat162 h2 = __floats2bfloat162_rn(lo, hi);
        w4[i] = *reinterpret_cast<uint32_t*>(&h2);
      } else {
        __half2 h2 = __floats2half2_rn(lo, hi);
        w4[i] = *reinterpret_cast<uint32_t*>(&h2);
      }
    }
    drow[j ^ ((lane >> 1) & 3)] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
  }
}

// Transposed layout (any pitch): the chunk goes through the warp's 32 x 32 FP32
// staging buffer; float4 slot c of row r is stored at slot c ^ (r & 7), which keeps
// the row-per-lane writes and the segment-per-8-lanes reads free of bank conflicts.
// Lane l then handles columns 4*(l%8) .. 4*(l%8)+3 of rows 4*g + l/8 (g = 0..7): each
// warp access is four 128-byte row segments (4-element vectors where the pitch allows,
// else scalars).  In this layout cv[4*g + i] is column 4*(l%8) + i of row 4*g + l/8.
// Measured alternatives that were slower: a column-per-lane pass for unaligned
// pitches, and prefetching the next tile's C rows into L2 (it evicted operand panels).
__device__ __forceinline__ void load_c_chunk(const GemmParams& p, int m_base, int n0, int lane,
                                             float (&cv)[32]) {
#pragma unroll
  for (int j = 0; j < 32; ++j) cv[j] = 0.0f;
  const int n = n0 + 4 * (lane & 7);
  const int ncols = min(4, p.N - n);  // valid columns of this lane (<= 0: none)
  if (p.beta == 0.0f || ncols <= 0) return;
#pragma unroll
  for (int g = 0; g < 8; ++g) {
    const int m = m_base + 4 * g + (lane >> 3);
    if (m < p.M) {
      const float* cp = p.C + static_cast<int64_t>(m) * p.ldc + n;
      if (ncols == 4 && p.c_vec) {
        const float4 t = *reinterpret_cast<const float4*>(cp);
        cv[4 * g] = t.x;
        cv[4 * g + 1] = t.y;
        cv[4 * g + 2] = t.z;
        cv[4 * g + 3] = t.w;
      } else {
        cv[4 * g] = cp[0];
        if (ncols > 1) cv[4 * g + 1] = cp[1];
        if (ncols > 2) cv[4 * g + 2] = cp[2];
        if (ncols > 3) cv[4 * g + 3] = cp[3];
      }
    }
  }
}

__device__ __forceinline__ void store_chunk(const GemmParams& p, float* st, int m_base, int n0,
                                            const float (&v)[32], const float (&cv)[32], int lane) {
  float4* st4 = reinterpret_cast<float4*>(st);
#pragma unroll
  for (int c = 0; c < 8; ++c)
    st4[lane * 8 + (c ^ (lane & 7))] = make_float4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
  __syncwarp();
  const int c4 = lane & 7;
  const int n = n0 + 4 * c4;
  const int ncols = min(4, p.N - n);
  const bool full_cols = ncols == 4;
#pragma unroll
  for (int g = 0; g < 8; ++g) {
    const int r = 4 * g + (lane >> 3);
    const int m = m_base + r;
    if (m >= p.M || ncols <= 0) continue;
    const float4 a = st4[r * 8 + (c4 ^ (r & 7))];
    float o[4] = {p.alpha * a.x, p.alpha * a.y, p.alpha * a.z, p.alpha * a.w};
    if (p.beta != 0.0f) {
#pragma unroll
      for (int i = 0; i < 4; ++i) o[i] = fmaf(p.beta, cv[4 * g + i], o[i]);
    }
    const int64_t off = static_cast<int64_t>(m) * p.ldd + n;
    if (p.d_type == LL_OUT_F32) {
      float* dp = static_cast<float*>(p.D) + off;
      if (full_cols && p.d_vec) {
        *reinterpret_cast<float4*>(dp) = make_float4(o[0], o[1], o[2], o[3]);
      } else {
        dp[0] = o[0];
        if (ncols > 1) dp[1] = o[1];
        if (ncols > 2) dp[2] = o[2];
        if (ncols > 3) dp[3] = o[3];
      }
    } else {
      uint32_t lo, hi;
      if (p.d_type == LL_OUT_BF16) {
        __nv_bfloat162 l2 = __floats2bfloat162_rn(o[0], o[1]), h2 = __floats2bfloat162_rn(o[2], o[3]);
        lo = *reinterpret_cast<uint32_t*>(&l2);
        hi = *reinterpret_cast<uint32_t*>(&h2);
      } else {
        __half2 l2 = __floats2half2_rn(o[0], o[1]), h2 = __floats2half2_rn(o[2], o[3]);
        lo = *reinterpret_cast<uint32_t*>(&l2);
        hi = *reinterpret_cast<uint32_t*>(&h2);
      }
      uint16_t* dp = reinterpret_cast<uint16_t*>(p.D) + off;
      if (full_cols && p.d_vec) {
        *reinterpret_cast<uint2*>(dp) = make_uint2(lo, hi);
      } else {
        dp[0] = static_cast<uint16_t>(lo);
        if (ncols > 1) dp[1] = static_cast<uint16_t>(lo >> 16);
        if (ncols > 2) dp[2] = static_cast<uint16_t>(hi);
        if (ncols > 3) dp[3] = static_cast<uint16_t>(hi >> 16);
      }
    }
  }
  __syncwarp();
}

// Row-contiguous variants for rows of C or D that need not start on 16-byte boundaries
// (the CTA-pair kernel's transposing epilogue): lane l handles column n0 + l of each of
// the chunk's 32 rows, so that every warp-wide access is 32 consecutive elements of one
// row (one contiguous 128-byte or 64-byte span whatever the row's alignment).  C goes to
// a 32 x 32 FP32 buffer in shared memory (row r at r * 32) by cp.async, each lane copying
// the elements it later reads itself.
__device__ __forceinline__ void issue_c_rows(const GemmParams& p, uint32_t cbuf, int m_base, int n0, int lane) {
  const int n = n0 + lane;
  if (p.beta == 0.0f || n >= p.N) return;
  const float* cp = p.C + static_cast<int64_t>(m_base) * p.ldc + n;
#pragma unroll 8
  for (int r = 0; r < 32; ++r)
    if (m_base + r < p.M) cp_async_4(cbuf + (r * 32 + lane) * 4, cp + static_cast<int64_t>(r) * p.ldc);
}

// st: the chunk's accumulator, row r (TMEM lane) holding its 32 columns as 8 float4 slots,
// slot j at position j ^ (r & 7).
__device__ __forceinline__ void store_rows(const GemmParams& p, const float* st, int m_base, int n0,
                                           const float* cbuf, int lane) {
  const int n = n0 + lane;
  if (n >= p.N) return;
  const bool use_c = p.beta != 0.0f;
#pragma unroll
  for (int r = 0; r < 32; ++r) {
    const int m = m_base + r;
    if (m >= p.M) break;
    float o = p.alpha * st[(r * 8 + ((lane >> 2) ^ (r & 7))) * 4 + (lane & 3)];
    if (use_c) o = fmaf(p.beta, cbuf[r * 32 + lane], o);
    const int64_t off = static_cast<int64_t>(m) * p.ldd + n;
    if (p.d_type == LL_OUT_F32)
      static_cast<float*>(p.D)[off] = o;
    else if (p.d_type == LL_OUT_BF16)
      static_cast<__nv_bfloat16*>(p.D)[off] = __float2bfloat16_rn(o);
    else
      static_cast<__half*>(p.D)[off] = __float2half_rn(o);
  }
}

// Schedule of the one-CTA kernel: whole tiles t = cta, cta + grid, ... below full_tiles;
// with an FP8 stream-K tail (sk_tiles > 0) the sk_tiles tiles after them are done by K
// ranges, one contiguous range of their K blocks per CTA.  A CTA whose range ends inside a
// tile writes that piece's promoted FP32 partial to its slot of sk_part (128 rows x 256
// columns) and sets its promotion warps' flags (sk_flag[cta * 8 + warp]) to `epoch`; the
// CTA whose range ends at a tile's end adds the partials of the CTAs before it, in CTA
// order, and stores the tile.
struct TileSched {
  int full_tiles;
  int sk_tiles;
  float* sk_part;
  unsigned long long* sk_flag;
  unsigned long long epoch;
};

template <class Cfg, uint32_t AB_FMT>
__global__ void __launch_bounds__(Cfg::THREADS, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const GemmParams p, const TileSched ts) {
  constexpr int S = Cfg::STAGES;
  constexpr int BN = Cfg::BN;
  constexpr uint32_t IDESC = make_idesc(AB_FMT, BN, 128);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  float* epi_stage = reinterpret_cast<float*>(smem + S * Cfg::STAGE_BYTES);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S * Cfg::STAGE_BYTES + Cfg::EPI_STAGE_BYTES);
  constexpr int NA = Cfg::NACC;
  // bars: full[S], empty[S], tfull[NA], tempty[NA], drain
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * S + 2 * NA + 1);
  uint32_t* abort_flag = tmem_slot + 1;
  // this CTA's stream-K items (at most two: a range of fewer K blocks than a tile meets at
  // most two tiles), written once by thread 0 and read by every role
  int4* sk_items = reinterpret_cast<int4*>((reinterpret_cast<uintptr_t>(abort_flag + 1) + 15) & ~static_cast<uintptr_t>(15));
  int* sk_count = reinterpret_cast<int*>(sk_items + 2);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  auto full_bar = [&](int s) { return smem_addr(bars + s); };
  auto empty_bar = [&](int s) { return smem_addr(bars + S + s); };
  auto tfull_bar = [&](int b) { return smem_addr(bars + 2 * S + b); };
  auto tempty_bar = [&](int b) { return smem_addr(bars + 2 * S + NA + b); };
  const uint32_t drain_bar = smem_addr(bars + 2 * S + 2 * NA);

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < NA; ++b) {
      mbar_init(tfull_bar(b), 1);
      mbar_init(tempty_bar(b), Cfg::EPI_THREADS);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0u;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(tmem_slot), Cfg::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(tmem_slot);

  WaitCtx wctx{p.status, p.timeout_ns, abort_flag};
  const int num_m = (p.M + 127) / 128;
  const int num_n = (p.N + BN - 1) / BN;
  const int KB = (p.K + Cfg::BK - 1) / Cfg::BK;
  // This CTA's work items, in order: its stream-K pieces first (the piece that ends inside
  // a tile, kind kSkPart; then the piece that ends at a tile's end, kSkOwner when CTAs
  // before this one hold the tile's first K blocks, otherwise kWhole), then its whole
  // tiles t = cta, cta + grid, ... below ts.full_tiles, as in the CTA-pair kernel.  The
  // stream-K items live in shared memory, so the roles' loops carry no extra state.
  enum { kWhole = 0, kSkPart = 1, kSkOwner = 2 };
  struct Item {
    int t, kb0, kb1, kind, pfirst;
  };
  if (threadIdx.x == 0) {
    const int cta = blockIdx.x, P = gridDim.x;
    const int64_t sk_total = static_cast<int64_t>(ts.sk_tiles) * KB;
    auto sk_begin = [&](int c2) { return static_cast<int64_t>(c2) * sk_total / P; };
    const int64_t sk_a = sk_begin(cta), sk_b = sk_begin(cta + 1);
    // the tiles the range [sk_a, sk_b) meets: the piece that ends inside a tile first
    const int t_first = static_cast<int>(sk_a / KB);
    const int t_last = sk_b > sk_a ? static_cast<int>((sk_b - 1) / KB) : t_first - 1;
    int n = 0;
    for (int pass = 0; pass < 2; ++pass)
      for (int t = t_first; t <= t_last && n < 2; ++t) {
        const int64_t t0 = static_cast<int64_t>(t) * KB;
        const int kb0 = static_cast<int>((sk_a > t0 ? sk_a : t0) - t0);
        const int kb1 = static_cast<int>((sk_b < t0 + KB ? sk_b : t0 + KB) - t0);
        const bool part = kb1 < KB;
        if (part != (pass == 0)) continue;
        const int kind = part ? kSkPart : (kb0 > 0 ? kSkOwner : kWhole);
        int pf = cta;
        if (kind == kSkOwner)  // the CTAs whose ranges end inside this tile
          while (pf > 0 && sk_begin(pf) > t0) --pf;
        sk_items[n] = make_int4(ts.full_tiles + t, kb0 | (kb1 << 16), kind, pf);
        ++n;
      }
    *sk_count = n;
  }
  __syncthreads();
  const int n_sk = *sk_count;
  const int n_items =
      n_sk + (static_cast<int>(blockIdx.x) < ts.full_tiles
                  ? (ts.full_tiles - 1 - static_cast<int>(blockIdx.x)) / static_cast<int>(gridDim.x) + 1
                  : 0);
  auto item = [&](int i) {
    Item it;
    if (i < n_sk) {
      const int4 v = sk_items[i];
      it.t = v.x;
      it.kb0 = v.y & 0xFFFF;
      it.kb1 = v.y >> 16;
      it.kind = v.z;
      it.pfirst = v.w;
    } else {
      it.t = static_cast<int>(blockIdx.x) + (i - n_sk) * static_cast<int>(gridDim.x);
      it.kb0 = 0;
      it.kb1 = KB;
      it.kind = kWhole;
      it.pfirst = blockIdx.x;
    }
    return it;
  };

  // programmatic dependent launch (as in the pair kernel): L2 prefetch of the first
  // ring of operand tiles, then the wait for the previous kernel of the stream
  if (warp == 0 && lane == 0 && n_items > 0) {
    const Item it0 = item(0);
    int mb, nb;
    tile_coords(it0.t, num_m, num_n, p.group_m, mb, nb);
    const int pre = it0.kb1 - it0.kb0 < S ? it0.kb1 - it0.kb0 : S;
    for (int kb = it0.kb0; kb < it0.kb0 + pre; ++kb) {
      tma_prefetch_l2(&tmA, kb * Cfg::BK, mb * 128);
      for (int j = 0; j < Cfg::B_BOXES; ++j) tma_prefetch_l2(&tmB, nb * BN + j * Cfg::B_BOX_N, kb * Cfg::BK);
    }
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");

  if (warp == 0) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      tma_prefetch_desc(&tmA);
      tma_prefetch_desc(&tmB);
      uint32_t it = 0;
      bool ok = true;
      for (int i = 0; i < n_items && ok; ++i) {
        const Item w = item(i);
        int mb, nb;
        tile_coords(w.t, num_m, num_n, p.group_m, mb, nb);
        for (int kb = w.kb0; kb < w.kb1; ++kb) {
          const int s = it % S;
          const uint32_t ph = (it / S) & 1u;
          if (!wait_bounded(empty_bar(s), ph ^ 1u, wctx, kRoleProducer)) {
            ok = false;
            break;
          }
          uint8_t* a_s = smem + s * Cfg::STAGE_BYTES;
          uint8_t* b_s = a_s + Cfg::A_BYTES;
          mbar_arrive_expect_tx(full_bar(s), Cfg::STAGE_BYTES);
          tma_load_2d(smem_addr(a_s), &tmA, full_bar(s), kb * Cfg::BK, mb * 128);
#pragma unroll
          for (int j = 0; j < Cfg::B_BOXES; ++j)
            tma_load_2d(smem_addr(b_s + j * Cfg::B_BOX_BYTES), &tmB, full_bar(s),
                        nb * BN + j * Cfg::B_BOX_N, kb * Cfg::BK);
          ++it;
        }
      }
      if (!ok) {
        // wait for the copies still in flight before the CTA can exit
        for (uint32_t j = (it > static_cast<uint32_t>(S) ? it - S : 0u); j < it; ++j)
          wait_drain(full_bar(j % S), (j / S) & 1u, p.timeout_ns);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      uint32_t it = 0, acc_it = 0;
      bool ok = true;
      for (int i = 0; i < n_items && ok; ++i) {
        const Item w = item(i);
        uint32_t d_tmem = 0;
        if (!Cfg::FP8) {
          const uint32_t ab = acc_it % NA;
          if (!wait_bounded(tempty_bar(ab), ((acc_it / NA) & 1u) ^ 1u, wctx, kRoleMma)) {
            ok = false;
            break;
          }
          tc_fence_after();
          d_tmem = tmem_base + ab * BN;
        }
        for (int kb = w.kb0; kb < w.kb1; ++kb) {
          if (Cfg::FP8) {  // one TMEM partial buffer per 128-K block, alternating
            const uint32_t pb = acc_it % NA;
            if (!wait_bounded(tempty_bar(pb), ((acc_it / NA) & 1u) ^ 1u, wctx, kRoleMma)) {
              ok = false;
              break;
            }
            tc_fence_after();
            d_tmem = tmem_base + pb * BN;
          }
          const int s = it % S;
          if (!wait_bounded(full_bar(s), (it / S) & 1u, wctx, kRoleMma)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_base = smem_addr(smem + s * Cfg::STAGE_BYTES);
          const uint32_t b_base = a_base + Cfg::A_BYTES;
#pragma unroll
          for (int kk = 0; kk < Cfg::KSTEPS; ++kk) {
            const uint64_t adesc = smem_desc_sw128(a_base + kk * 32, 16, 1024);
            const uint64_t bdesc =
                smem_desc_sw128(b_base + kk * Cfg::UMMA_K * 128, Cfg::B_BOX_BYTES, 1024);
            const uint32_t accum = Cfg::FP8 ? (kk > 0) : (kb > w.kb0 || kk > 0);
            if (Cfg::FP8)
              mma_f8(d_tmem, adesc, bdesc, IDESC, accum);
            else
              mma_f16(d_tmem, adesc, bdesc, IDESC, accum);
          }
          mma_commit(empty_bar(s));
          ++it;
          if (Cfg::FP8) {
            mma_commit(tfull_bar(acc_it % NA));
            ++acc_it;
          }
        }
        if (!ok) break;
        if (!Cfg::FP8) {
          mma_commit(tfull_bar(acc_it % NA));
          ++acc_it;
        }
      }
      // every MMA issued by this thread must finish before TMEM is freed
      mma_commit(drain_bar);
      wait_drain(drain_bar, 0u, p.timeout_ns);
    }
  } else if (!Cfg::FP8) {
    // ---------------------------------------------------------------- epilogue (16-bit)
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
    float* st = epi_stage + (warp - 2) * 32 * 32;
    uint32_t acc_it = 0;
    for (int i = 0; i < n_items; ++i) {  // whole tiles only (no stream-K for 16-bit here)
      int mb, nb;
      tile_coords(item(i).t, num_m, num_n, p.group_m, mb, nb);
      const uint32_t ab = acc_it % NA;
      bool ok = wait_bounded(tfull_bar(ab), (acc_it / NA) & 1u, wctx, kRoleEpilogue);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      const int m_base = mb * 128 + q * 32;
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t r[32];
        tmem_ld_x32(tmem_base + lane_base + ab * BN + c * 32, r);
        tmem_ld_wait(r);
        if (c == BN / 32 - 1) {  // the accumulator is in registers: hand TMEM back now
          tc_fence_before();
          mbar_arrive(tempty_bar(ab));
        }
        float v[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
        float cv[32];
        load_c_chunk(p, m_base, nb * BN + c * 32, lane, cv);
        store_chunk(p, st, m_base, nb * BN + c * 32, v, cv, lane);
      }
      ++acc_it;
    }
  } else {
    // ---------------------------------------------------------------- promotion + epilogue (FP8)
    constexpr int HALF = BN / 2;  // columns per thread
    constexpr int CH = HALF / 32;
    const int ew = warp - Cfg::EPI_WARP0;
    const int q = warp & 3;
    const int h = ew >> 2;
    const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
    uint32_t pit = 0;
    bool ok = true;
    // a stream-K slot holds the CTA's 128 rows x 256 columns as [warp][chunk][4-column
    // group][row within the warp's 32][4]: a warp's 32 lanes access 512 contiguous bytes
    auto sk_vec = [&](int slot, int c, int j) {
      return reinterpret_cast<float4*>(ts.sk_part + static_cast<size_t>(slot) * (128 * 256)) +
             (((ew * CH + c) * 8 + j) * 32 + lane);
    };
    auto sk_flag = [&](int slot) { return ts.sk_flag + static_cast<size_t>(slot) * 8 + ew; };
    for (int i = 0; i < n_items && ok; ++i) {
      const Item w = item(i);
      int mb, nb;
      tile_coords(w.t, num_m, num_n, p.group_m, mb, nb);
      const int m = mb * 128 + q * 32 + lane;
      const bool row_ok = m < p.M;
      const int ncol0 = nb * BN + h * HALF;
      const bool col_ok = ncol0 < p.N;
      const int nblk = ncol0 / 128;
      const float* sa_row = p.sA + static_cast<int64_t>(row_ok ? m : 0) * p.ld_sa;
      float acc[CH][32];
#pragma unroll
      for (int c = 0; c < CH; ++c)
#pragma unroll
        for (int j = 0; j < 32; ++j) acc[c][j] = 0.0f;
      float sa_next = row_ok ? __ldg(sa_row + w.kb0) : 0.0f;
      float sb_next = col_ok ? __ldg(p.sB + static_cast<int64_t>(w.kb0) * p.ld_sb + nblk) : 0.0f;
      for (int kb = w.kb0; kb < w.kb1; ++kb) {
        const float s = sa_next * sb_next;
        if (kb + 1 < w.kb1) {  // next block's scales travel while this block is promoted
          sa_next = row_ok ? __ldg(sa_row + kb + 1) : 0.0f;
          sb_next = col_ok ? __ldg(p.sB + static_cast<int64_t>(kb + 1) * p.ld_sb + nblk) : 0.0f;
        }
        const uint32_t pb = pit % NA;
        bool w = wait_bounded(tfull_bar(pb), (pit / NA) & 1u, wctx, kRoleEpilogue);
        w = __all_sync(0xffffffffu, w);
        if (!w) {
          ok = false;
          break;
        }
        tc_fence_after();
        // 16 columns per TMEM load keep 128 accumulators + staging within the
        // register budget of a 320-thread block
#pragma unroll
        for (int c = 0; c < 2 * CH; ++c) {
          uint32_t r[16];
          tmem_ld_x16(tmem_base + lane_base + pb * BN + h * HALF + c * 16, r);
          tmem_ld_wait(r);
          if (c == 2 * CH - 1) {  // partial fully read: the MMAs may reuse the buffer
            tc_fence_before();
            mbar_arrive(tempty_bar(pb));
          }
#pragma unroll
          for (int j = 0; j < 16; j += 2)
            ffma2(acc[c >> 1][(c & 1) * 16 + j], acc[c >> 1][(c & 1) * 16 + j + 1],
                  __uint_as_float(r[j]), __uint_as_float(r[j + 1]), s);
        }
        ++pit;
      }
      if (!ok) break;
      const Item wk = item(i);  // (shared memory) kind and first CTA of this item
      if (wk.kind == kSkPart) {
        // a piece that ends inside its tile: the promoted partial goes to this CTA's slot,
        // then the flag tells the CTA that completes the tile
#pragma unroll
        for (int c = 0; c < CH; ++c)
#pragma unroll
          for (int j = 0; j < 8; ++j)
            *sk_vec(blockIdx.x, c, j) = make_float4(acc[c][4 * j], acc[c][4 * j + 1], acc[c][4 * j + 2], acc[c][4 * j + 3]);
        __threadfence();
        __syncwarp();
        if (lane == 0) flag_release(sk_flag(blockIdx.x), ts.epoch);
        continue;
      }
      if (wk.kind == kSkOwner) {  // add the partials of the CTAs before this one, in order
        const int cta = blockIdx.x;
        bool fw = true;
        if (lane == 0)
          for (int c2 = wk.pfirst; c2 < cta && fw; ++c2) fw = flag_wait_bounded(sk_flag(c2), ts.epoch, wctx, kRoleEpilogue);
        fw = __shfl_sync(0xffffffffu, fw ? 1 : 0, 0) != 0;
        __syncwarp();  // lane 0's acquire, before every lane's reads of the partials
        if (!fw) {
          ok = false;
          break;
        }
        for (int c2 = wk.pfirst; c2 < cta; ++c2) {
#pragma unroll
          for (int c = 0; c < CH; ++c)
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const float4 v = __ldcg(sk_vec(c2, c, j));
              acc[c][4 * j] += v.x;
              acc[c][4 * j + 1] += v.y;
              acc[c][4 * j + 2] += v.z;
              acc[c][4 * j + 3] += v.w;
            }
        }
      }
      epilogue_rows<CH>(p, m, ncol0, acc);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
  }
}


// ------------------------------------------------------------------ CTA-pair kernel
//
// Large 16-bit problems run on CTA pairs (2-CTA clusters).  A pair owns a 256 x 256
// output tile: each CTA loads its 128 rows of A and its half (128 columns) of B into its
// own shared memory, the even CTA's single MMA thread issues tcgen05.mma with
// cta_group::2 (M = 256), and each CTA's TMEM receives its own 128 rows of the
// accumulator.  Per SM this halves the B traffic (TMA fill and shared-memory reads)
// of the one-CTA 128 x 256 tile.
//   full[s]   (even CTA)  count 1: the even CTA's producer arms it with both CTAs'
//                         transaction bytes; both CTAs' TMA copies complete on it
//                         (the odd CTA's bytes may land first: the transaction count
//                         then runs negative until the arrival, which is allowed).
//   empty[s]  (each CTA)  count 1: the MMA commit, multicast to both CTAs.
//   tfull[b]  (each CTA)  count 1: the MMA commit, multicast to both CTAs.
//   tempty[b] (even CTA)  one arrival per epilogue warp of each CTA.
// The accumulator of a tile is double buffered in TMEM (2 x 256 columns) and 4
// epilogue warps per CTA drain one while the MMAs fill the other (TMA epilogue for
// 16-byte-aligned C / D rows, a shared-memory transpose otherwise; see the epilogue).
// Output tiles past the last full wave are split into two 256 x 128 halves when that
// lets one half-wave finish the problem, and a problem whose halves all fit one wave
// runs as halves only.  (FP8 runs on the one-CTA kernel: a pair version of the block
// promotion, whose MMA waits for the partial-buffer hand-back of 16 warps in two CTAs,
// measured 3 to 17 % slower at every size from 1792^3 to 8192^3.)
template <int BN_>
struct PairCfg {
  static constexpr int BN = BN_;  // pair tile N
  static constexpr int ELT = 2;
  static constexpr int BK = 64;   // K per stage (one 128-byte row)
  static constexpr int UMMA_K = 16;
  static constexpr int KSTEPS = BK / UMMA_K;
  static constexpr int A_BYTES = 128 * 128;
  static constexpr int B_BOX_N = 64;
  static constexpr int B_BOX_BYTES = BK * 128;
  static constexpr int B_BOXES_MAX = BN / 2 / B_BOX_N;  // per CTA
  static constexpr int STAGE_BYTES = A_BYTES + B_BOXES_MAX * B_BOX_BYTES;
  // 5 operand stages leave room for the epilogue's C / D buffers
  static constexpr int STAGES = 163840 / STAGE_BYTES;
  static constexpr int TMEM_COLS = 2 * BN;
  static constexpr int EPI_WARP0 = 2;  // warps: producer, MMA, epilogue
  static constexpr int EPI_WARPS = 4;
  static constexpr int THREADS = 32 * (EPI_WARP0 + EPI_WARPS);
  // EPI_BUFS buffers of one 32 x 32 FP32 chunk per epilogue warp (the TMA path cycles
  // through them; the transposing path uses the first as its staging buffer)
  static constexpr int EPI_BUFS = 4;
  static constexpr int EPI_BUF_BYTES = 32 * 32 * 4;
  static constexpr int EPI_STAGE_BYTES = EPI_WARPS * EPI_BUFS * EPI_BUF_BYTES;
  static constexpr int NBARS = 2 * STAGES + 5 + EPI_WARPS * EPI_BUFS;
  static constexpr int SMEM = STAGES * STAGE_BYTES + EPI_STAGE_BYTES + NBARS * 8 + 16 + 1024;
  static_assert(SMEM <= 227 * 1024, "shared memory budget");
  static_assert(TMEM_COLS <= 512, "TMEM budget");
  static_assert(B_BOXES_MAX >= 1, "B half must cover a whole swizzle row");
};

struct PairSched {
  int num_m2, num_n;  // pair tiles in M (256 rows) and N (BN columns)
  int full_units;     // units that are whole tiles
  int num_units;      // full_units + 2 * split tiles
  // stream-K tail: the sk_tiles tiles after the num_units whole ones are done by K ranges,
  // one contiguous range of their K blocks per pair (0: none).  A pair whose range ends
  // inside a tile writes that piece's FP32 partial to its slot of sk_part (two CTAs x 128
  // rows x 256 columns) and sets its flags (sk_flag[(pair * 2 + rank) * 4 + warp quarter])
  // to `epoch`; the pair whose range ends at a tile's end adds the partials of the pairs
  // before it to its own, in pair order, and stores the tile.
  int sk_tiles;
  float* sk_part;
  unsigned long long* sk_flag;
  unsigned long long epoch;
};

// FP32 C whose rows do not start on 16-byte boundaries, as four row classes: class k holds
// rows k, k + 4, k + 8, ..., 16 * ldc bytes apart (a pitch a tensor map can describe), its
// map starting at the first 16-byte boundary of row k, off_k = 0..3 elements in; all rows of
// a class then have the same offset.  Column c of a row of class k is element c - off_k of
// that map's row.  Boxes of 36 x 8, loaded from x = n - 4, cover columns n .. n + 31 whatever
// off_k is.  (D of such rows is stored by the lanes in whole 32-byte sectors, see the kernel.)
struct EpiResMaps {
  CUtensorMap c[4];
};

// 32 bytes to a 32-byte-aligned global address in one store, with an L2 cache policy.
__device__ __forceinline__ void st_global_v8_hint(float* p, const float* v, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.v8.f32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8}, %9;" ::"l"(p), "f"(v[0]),
               "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]), "l"(pol)
               : "memory");
}

template <class Cfg, uint32_t AB_FMT>
__global__ void __launch_bounds__(Cfg::THREADS, 1)
    gemm_tc2_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmD,
                    const GemmParams p, const PairSched sc, const __grid_constant__ EpiResMaps rm) {
  constexpr int S = Cfg::STAGES;
  constexpr int BN = Cfg::BN;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  float* epi_stage = reinterpret_cast<float*>(smem + S * Cfg::STAGE_BYTES);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S * Cfg::STAGE_BYTES + Cfg::EPI_STAGE_BYTES);
  // bars: full[S], empty[S], tfull[2], tempty[2], drain,
  //       cfull[EPI_WARPS][EPI_BUFS] (TMA epilogue: a C chunk landed in a buffer)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + Cfg::NBARS);
  uint32_t* abort_flag = tmem_slot + 1;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const uint32_t rank = cluster_ctarank();
  const int pair = blockIdx.x >> 1;
  const int num_pairs = gridDim.x >> 1;
  auto full_bar = [&](int s) { return smem_addr(bars + s); };
  auto empty_bar = [&](int s) { return smem_addr(bars + S + s); };
  auto tfull_bar = [&](int b) { return smem_addr(bars + 2 * S + b); };
  auto tempty_bar = [&](int b) { return smem_addr(bars + 2 * S + 2 + b); };
  const uint32_t drain_bar = smem_addr(bars + 2 * S + 4);
  auto cfull_bar = [&](int w, int b) { return smem_addr(bars + 2 * S + 5 + w * Cfg::EPI_BUFS + b); };

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull_bar(b), 1);
      mbar_init(tempty_bar(b), 2 * Cfg::EPI_WARPS);
    }
    mbar_init(drain_bar, 1);
    for (int w = 0; w < Cfg::EPI_WARPS; ++w)
      for (int b = 0; b < Cfg::EPI_BUFS; ++b) mbar_init(cfull_bar(w, b), 1);
    *abort_flag = 0u;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_addr(tmem_slot), Cfg::TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync();  // barriers of both CTAs initialised, TMEM allocated
  tc_fence_after();
  const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(tmem_slot);

  WaitCtx wctx{p.status, p.timeout_ns, abort_flag};
  const int KB = (p.K + Cfg::BK - 1) / Cfg::BK;
  // unit -> (first row of the pair tile, first column, columns)
  auto unit = [&](int u, int& m0, int& n0, int& ncols) {
    int t = u, half = -1;
    if (u >= sc.full_units) {
      t = sc.full_units + ((u - sc.full_units) >> 1);
      half = (u - sc.full_units) & 1;
    }
    int mb, nb;
    tile_coords(t, sc.num_m2, sc.num_n, p.group_m, mb, nb);
    m0 = mb * 256;
    n0 = nb * BN + (half > 0 ? BN / 2 : 0);
    ncols = half < 0 ? BN : BN / 2;
  };
  // This pair's work items, in order: its stream-K pieces first — the piece that ends
  // inside a tile (kind kSkPart: its partial goes to the workspace), then the pieces that
  // end at a tile's end (kSkOwner when pairs before this one hold the tile's first K
  // blocks, whose partials it adds; otherwise kWhole) — then its units (u = pair,
  // pair + num_pairs, ...).  With the pieces first, every partial is written early, each
  // owner adds them while its next tile's MMAs run, and the grid ends on whole tiles.
  enum { kWhole = 0, kSkPart = 1, kSkOwner = 2 };
  struct Item {
    int m0, n0, ncols, kb0, kb1, kind, pfirst;
  };
  const int n_units = pair < sc.num_units ? (sc.num_units - 1 - pair) / num_pairs + 1 : 0;
  const int64_t sk_total = static_cast<int64_t>(sc.sk_tiles) * KB;
  auto sk_begin = [&](int q2) { return static_cast<int64_t>(q2) * sk_total / num_pairs; };
  const int64_t sk_a = sk_begin(pair), sk_b = sk_begin(pair + 1);
  const bool sk_has_part = sk_b > sk_a && sk_b % KB != 0;
  const int sk_t0 = static_cast<int>(sk_a / KB);
  const int sk_tend = sk_b > sk_a ? static_cast<int>((sk_b - 1) / KB) + (sk_has_part ? 0 : 1) : sk_t0;
  const int n_sk = (sk_has_part ? 1 : 0) + (sk_tend > sk_t0 ? sk_tend - sk_t0 : 0);
  const int n_items = n_sk + n_units;
  auto item = [&](int i) {
    Item it;
    it.pfirst = pair;
    if (i >= n_sk) {
      unit(pair + (i - n_sk) * num_pairs, it.m0, it.n0, it.ncols);
      it.kb0 = 0;
      it.kb1 = KB;
      it.kind = kWhole;
      return it;
    }
    const int j = i;
    int t;
    if (sk_has_part && j == 0) {
      t = static_cast<int>((sk_b - 1) / KB);
      it.kind = kSkPart;
      it.kb1 = static_cast<int>(sk_b - static_cast<int64_t>(t) * KB);
    } else {
      t = sk_t0 + j - (sk_has_part ? 1 : 0);
      it.kb1 = KB;
    }
    const int64_t t0 = static_cast<int64_t>(t) * KB;
    it.kb0 = static_cast<int>((sk_a > t0 ? sk_a : t0) - t0);
    if (!(sk_has_part && j == 0)) {
      it.kind = it.kb0 > 0 ? kSkOwner : kWhole;
      if (it.kind == kSkOwner) {  // the pairs whose ranges end inside this tile
        int pf = pair;
        while (pf > 0 && sk_begin(pf) > t0) --pf;
        it.pfirst = pf;
      }
    }
    int mb, nb;
    tile_coords(sc.num_units + t, sc.num_m2, sc.num_n, p.group_m, mb, nb);
    it.m0 = mb * 256;
    it.n0 = nb * BN;
    it.ncols = BN;
    return it;
  };

  // Programmatic dependent launch: everything above overlaps the previous kernel of
  // the stream; the producer also pulls its first ring of operand tiles into L2 (L2 is
  // coherent, so a prefetch may run ahead of the previous kernel's writes).  Operand
  // copies into shared memory, scale and C reads and D writes come after the wait.
  if (warp == 0 && lane == 0 && n_items > 0) {
    const Item it0 = item(0);
    const int boxes = it0.ncols / 2 / Cfg::B_BOX_N;
    const int pre = it0.kb1 - it0.kb0 < S ? it0.kb1 - it0.kb0 : S;
    for (int kb = it0.kb0; kb < it0.kb0 + pre; ++kb) {
      tma_prefetch_l2(&tmA, kb * Cfg::BK, it0.m0 + 128 * static_cast<int>(rank));
      for (int j = 0; j < boxes; ++j)
        tma_prefetch_l2(&tmB, it0.n0 + static_cast<int>(rank) * (it0.ncols / 2) + j * Cfg::B_BOX_N, kb * Cfg::BK);
    }
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");

  if (warp == 0) {
    // ---------------------------------------------------------------- producer (each CTA)
    if (lane == 0) {
      tma_prefetch_desc(&tmA);
      tma_prefetch_desc(&tmB);
      uint32_t it = 0;
      bool ok = true;
      for (int i = 0; i < n_items && ok; ++i) {
        const Item w = item(i);
        const int m0 = w.m0, n0 = w.n0, ncols = w.ncols;
        const int boxes = ncols / 2 / Cfg::B_BOX_N;
        const uint32_t bytes = Cfg::A_BYTES + boxes * Cfg::B_BOX_BYTES;
        for (int kb = w.kb0; kb < w.kb1; ++kb) {
          const int s = it % S;
          if (!wait_bounded(empty_bar(s), ((it / S) & 1u) ^ 1u, wctx, kRoleProducer)) {
            ok = false;
            break;
          }
          const uint32_t cfull = mapa_cluster(full_bar(s), 0);
          uint8_t* a_s = smem + s * Cfg::STAGE_BYTES;
          uint8_t* b_s = a_s + Cfg::A_BYTES;
          if (rank == 0) mbar_arrive_expect_tx(full_bar(s), 2 * bytes);
          tma_load_2d_pair(smem_addr(a_s), &tmA, cfull, kb * Cfg::BK, m0 + 128 * rank);
          for (int j = 0; j < boxes; ++j)
            tma_load_2d_pair(smem_addr(b_s + j * Cfg::B_BOX_BYTES), &tmB, cfull,
                             n0 + rank * (ncols / 2) + j * Cfg::B_BOX_N, kb * Cfg::BK);
          ++it;
        }
      }
      if (!ok && rank == 0) {  // the even CTA's full barriers see both CTAs' copies
        for (uint32_t j = (it > static_cast<uint32_t>(S) ? it - S : 0u); j < it; ++j)
          wait_drain(full_bar(j % S), (j / S) & 1u, p.timeout_ns);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer (even CTA)
    if (lane == 0 && rank == 0) {
      uint32_t it = 0, acc_it = 0;
      bool ok = true;
      for (int i = 0; i < n_items && ok; ++i) {
        const Item w = item(i);
        const uint32_t idesc = make_idesc(AB_FMT, w.ncols, 256);
        const uint32_t ab = acc_it & 1u;  // one accumulator per item
        if (!wait_bounded(tempty_bar(ab), ((acc_it >> 1) & 1u) ^ 1u, wctx, kRoleMma)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + ab * BN;
        for (int kb = w.kb0; kb < w.kb1; ++kb) {
          const int s = it % S;
          if (!wait_bounded(full_bar(s), (it / S) & 1u, wctx, kRoleMma)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_base = smem_addr(smem + s * Cfg::STAGE_BYTES);
          const uint32_t b_base = a_base + Cfg::A_BYTES;
#pragma unroll
          for (int kk = 0; kk < Cfg::KSTEPS; ++kk) {
            const uint64_t adesc = smem_desc_sw128(a_base + kk * 32, 16, 1024);
            const uint64_t bdesc =
                smem_desc_sw128(b_base + kk * Cfg::UMMA_K * 128, Cfg::B_BOX_BYTES, 1024);
            mma_f16_pair(d_tmem, adesc, bdesc, idesc, (kb > w.kb0 || kk > 0) ? 1u : 0u);
          }
          mma_commit_pair_mc(empty_bar(s), 0x3);
          ++it;
        }
        if (!ok) break;
        mma_commit_pair_mc(tfull_bar(ab), 0x3);
        ++acc_it;
      }
      mma_commit_pair(drain_bar);
      wait_drain(drain_bar, 0u, p.timeout_ns);
    }
  } else {
    // ---------------------------------------------------------------- epilogue (each CTA)
    const int q = warp & 3;
    const int ew = warp - Cfg::EPI_WARP0;
    const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
    uint8_t* ebuf = reinterpret_cast<uint8_t*>(epi_stage) + ew * Cfg::EPI_BUFS * Cfg::EPI_BUF_BYTES;
    const int row_off = 128 * static_cast<int>(rank) + q * 32;  // this warp's rows in a pair tile
    if (p.epi_tma) {
      // C and D rows on 16-byte boundaries: chunks of C arrive by TMA into this warp's
      // ring of EPI_BUFS buffers, PF chunks ahead of the one being stored (the first ones
      // before the accumulator is ready); each lane combines its accumulator row with
      // its C row in place, and one TMA store per chunk writes D.  Buffer b of chunk g
      // (b = g % EPI_BUFS) is refilled only after the store of chunk g - EPI_BUFS has
      // read it.  Chunks wholly outside the matrix are neither loaded nor stored; the
      // chunk that crosses column N is stored by the lanes themselves (a TMA store
      // writes whole 16-byte units and would reach into the columns past N).
      constexpr int R = Cfg::EPI_BUFS;
      constexpr int PF = R - 2;  // C loads in flight ahead; the latest store may still read
      const bool use_c = p.beta != 0.0f;
      const uint64_t pol_once = l2_evict_first_policy();
      const bool out32 = p.d_type == LL_OUT_F32;
      const bool bf = p.d_type == LL_OUT_BF16;
      // prefetch cursor: the chunk whose C load is issued next (items that end in a
      // stream-K partial store no D and read no C)
      int pu = 0, pc = 0, pchunks = 0, pm = 0, pn = 0;
      auto cursor_item = [&](int i) {
        while (i < n_items && item(i).kind == kSkPart) ++i;
        pu = i;
        pc = 0;
        if (i < n_items) {
          const Item w = item(i);
          pm = w.m0 + row_off;
          pn = w.n0;
          pchunks = w.ncols / 32;
        }
      };
      uint32_t issued = 0;  // C loads issued by this warp
      auto issue_c = [&]() {  // lane 0; call with the ring slot free
        if (pu >= n_items) return;
        const int b = static_cast<int>(issued % R);
        const int n = pn + 32 * pc;
        if (n < p.N && pm < p.M) {
          mbar_arrive_expect_tx(cfull_bar(ew, b), Cfg::EPI_BUF_BYTES);
          tma_load_2d_hint(smem_addr(ebuf + b * Cfg::EPI_BUF_BYTES), &tmC, cfull_bar(ew, b), n, pm, pol_once);
        } else {
          mbar_arrive(cfull_bar(ew, b));
        }
        ++issued;
        if (++pc == pchunks) cursor_item(pu + 1);
      };
      if (use_c) {
        cursor_item(0);
        if (lane == 0) {
          tma_prefetch_desc(&tmC);
          for (int i = 0; i < PF; ++i) issue_c();
        }
      }
      if (lane == 0) tma_prefetch_desc(&tmD);
      // a stream-K slot holds the CTA's 128 rows x 256 columns as [chunk c][4-column group
      // j][row][4]: the 32 lanes (rows) of a warp access 512 contiguous bytes at a time
      auto sk_vec = [&](int slot, int c, int j) {
        return reinterpret_cast<float4*>(sc.sk_part + (static_cast<size_t>(slot) * 2 + rank) * (128 * 256)) +
               ((c * 8 + j) * 128 + q * 32 + lane);
      };
      auto sk_flag = [&](int slot) { return sc.sk_flag + (static_cast<size_t>(slot) * 2 + rank) * 4 + q; };
      uint32_t acc_it = 0, g = 0;
      bool ok = true;
      for (int i = 0; i < n_items && ok; ++i) {
        const Item w = item(i);
        const int m0 = w.m0, n0 = w.n0, ncols = w.ncols;
        const uint32_t ab = acc_it & 1u;
        const int chunks = ncols / 32;
        if (w.kind == kSkOwner) {  // a tile this pair completes: the pairs before it are done
          bool fw = true;
          if (lane == 0)
            for (int pc2 = w.pfirst; pc2 < pair && fw; ++pc2) fw = flag_wait_bounded(sk_flag(pc2), sc.epoch, wctx, kRoleEpilogue);
          fw = __shfl_sync(0xffffffffu, fw ? 1 : 0, 0) != 0;
          __syncwarp();  // lane 0's acquire, before every lane's reads of the partials
          if (!fw) {
            ok = false;
            break;
          }
        }
        ok = wait_bounded(tfull_bar(ab), (acc_it >> 1) & 1u, wctx, kRoleEpilogue);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        if (w.kind == kSkPart) {
          // a stream-K piece that ends inside its tile: its FP32 partial goes to this pair's
          // slot, then the flag tells the pair that completes the tile
#pragma unroll 1
          for (int c = 0; c < chunks; ++c) {
            uint32_t r[32];
            tmem_ld_x32(tmem_base + lane_base + ab * BN + c * 32, r);
            tmem_ld_wait(r);
            if (c == chunks - 1) {
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive_cluster_relaxed(mapa_cluster(tempty_bar(ab), 0));
            }
#pragma unroll
            for (int j = 0; j < 8; ++j)
              *sk_vec(pair, c, j) = make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                                                __uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3]));
          }
          __threadfence();
          __syncwarp();
          if (lane == 0) flag_release(sk_flag(pair), sc.epoch);
          ++acc_it;
          continue;
        }
        const int m_w = m0 + row_off;
#pragma unroll 1
        for (int c = 0; c < chunks; ++c, ++g) {
          const int b = static_cast<int>(g % R);
          const uint32_t bsm = smem_addr(ebuf + b * Cfg::EPI_BUF_BYTES);
          if (lane == 0) {
            if (use_c) {
              bulk_wait_read<1>();  // the slot of chunk g + PF: its store (chunk g + PF - R) has read it
              if (static_cast<int>(issued - g) < PF + 1) issue_c();
            } else {
              bulk_wait_read<R - 1>();  // slot b: the store of chunk g - R has read it
            }
          }
          __syncwarp();
          uint32_t r[32];
          tmem_ld_x32(tmem_base + lane_base + ab * BN + c * 32, r);
          tmem_ld_wait(r);
          if (c == chunks - 1) {  // accumulator in registers: release it to the MMA
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster_relaxed(mapa_cluster(tempty_bar(ab), 0));
          }
          float o[32];
          if (w.kind == kSkOwner) {  // own partial, then the others' in pair order, then alpha
#pragma unroll
            for (int j = 0; j < 32; ++j) o[j] = __uint_as_float(r[j]);
            for (int pc2 = w.pfirst; pc2 < pair; ++pc2) {
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                const float4 v = __ldcg(sk_vec(pc2, c, j));
                o[4 * j] += v.x;
                o[4 * j + 1] += v.y;
                o[4 * j + 2] += v.z;
                o[4 * j + 3] += v.w;
              }
            }
#pragma unroll
            for (int j = 0; j < 32; ++j) o[j] *= p.alpha;
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) o[j] = p.alpha * __uint_as_float(r[j]);
          }
          const float4* row = reinterpret_cast<const float4*>(ebuf + b * Cfg::EPI_BUF_BYTES + lane * 128);
          if (use_c) {
            bool cw = wait_bounded(cfull_bar(ew, b), (g / R) & 1u, wctx, kRoleEpilogue);
            cw = __all_sync(0xffffffffu, cw);
            if (!cw) {
              ok = false;
              break;
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {  // 128-byte swizzle: 16-byte slot j of row l at j ^ (l & 7)
              const float4 cv = row[j ^ (lane & 7)];
              o[4 * j] = fmaf(p.beta, cv.x, o[4 * j]);
              o[4 * j + 1] = fmaf(p.beta, cv.y, o[4 * j + 1]);
              o[4 * j + 2] = fmaf(p.beta, cv.z, o[4 * j + 2]);
              o[4 * j + 3] = fmaf(p.beta, cv.w, o[4 * j + 3]);
            }
            __syncwarp();  // every C row read before a 16-bit D row overwrites it
          }
          const int n = n0 + 32 * c;
          if (n + 32 <= p.N) {  // whole chunk: through shared memory and one TMA store
            if (out32) {
              float4* drow = reinterpret_cast<float4*>(ebuf + b * Cfg::EPI_BUF_BYTES + lane * 128);
#pragma unroll
              for (int j = 0; j < 8; ++j)
                drow[j ^ (lane & 7)] = make_float4(o[4 * j], o[4 * j + 1], o[4 * j + 2], o[4 * j + 3]);
            } else {
              stage_row16(ebuf + b * Cfg::EPI_BUF_BYTES, lane, o, bf);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0 && m_w < p.M) tma_store_2d_hint(&tmD, bsm, n, m_w, pol_once);
          } else if (n < p.N && m_w + lane < p.M) {
            // the chunk that crosses column N: a TMA store may write whole 16-byte units
            // past N, so each lane stores its row's valid columns itself
            store_row_final(p, m_w + lane, n, o);
          }
          if (lane == 0) bulk_commit_group();  // one group per chunk (empty without a store)
        }
        ++acc_it;
      }
      if (lane == 0) {
        if (!ok) {  // C loads still in flight land before the CTA may exit
          for (uint32_t j = g; j < issued; ++j)
            wait_drain(cfull_bar(ew, static_cast<int>(j % R)), (j / R) & 1u, p.timeout_ns);
        }
        bulk_wait_all();
      }
      __syncwarp();
    } else if (p.epi_res) {
      // FP32 D rows that do not start on 16-byte boundaries.  Each lane keeps its own
      // accumulator row (no transpose): lane l is row m_w + l.  C arrives by TMA by row
      // classes (EpiResMaps) two chunks ahead, in a ring of two slots of four 36 x 8 boxes
      // (box k holds the warp's rows of class k); the lane reads its row's 32 values at box
      // column 4 - off + t (the columns left of a map's first element, only in the chunk at
      // column 0, are read by the lane itself).  D is stored by the lanes in whole 32-byte
      // sectors: a store that covers only part of a sector makes the memory system read
      // the rest of it first, which with rows off the sector grid would happen at every
      // chunk edge.  With od = 0..7 the offset of the row's first 32-byte boundary at or
      // after the tile's first column n0, chunk c writes the four sectors that start at
      // columns n0 + 32 c - 8 + od, ..., n0 + 32 c + 16 + od: the window of 32 values that
      // starts od values into (previous chunk's last 8 values, this chunk's 32).  Only the
      // sectors cut by the tile's edges or by column N are written element by element.
      // Every value is fma(beta, C, alpha * acc) in FP32, as on the other paths.
      constexpr int CBOX = 8 * 36 * 4;
      constexpr int CSLOT = 4 * CBOX;
      const bool use_c = p.beta != 0.0f;
      const uint64_t pol_once = l2_evict_first_policy();  // C read once, D written once
      const int rc = lane & 3, jr = lane >> 2;
      int pu = pair, pc = 0, pchunks = 0, pm = 0, pn = 0;
      auto cursor_unit = [&](int u) {
        pu = u;
        pc = 0;
        if (u < sc.num_units) {
          int m1, n1, nc1;
          unit(u, m1, n1, nc1);
          pm = m1 + row_off;
          pn = n1;
          pchunks = nc1 / 32;
        }
      };
      uint32_t issued = 0;
      auto issue_c = [&]() {  // lane 0; the ring slot is free
        if (pu >= sc.num_units) return;
        const int b = static_cast<int>(issued & 1u);
        const int n = pn + 32 * pc;
        if (n < p.N && pm < p.M) {
          mbar_arrive_expect_tx(cfull_bar(ew, b), CSLOT);
#pragma unroll
          for (int k = 0; k < 4; ++k)
            tma_load_2d_hint(smem_addr(ebuf + b * CSLOT + k * CBOX), &rm.c[k], cfull_bar(ew, b), n - 4, pm / 4,
                             pol_once);
        } else {
          mbar_arrive(cfull_bar(ew, b));
        }
        ++issued;
        if (++pc == pchunks) cursor_unit(pu + num_pairs);
      };
      if (use_c) {
        cursor_unit(pair);
        if (lane == 0) {
#pragma unroll
          for (int k = 0; k < 4; ++k) tma_prefetch_desc(&rm.c[k]);
          issue_c();
          issue_c();
        }
      }
      uint32_t acc_it = 0, g = 0;
      bool ok = true;
      for (int u = pair; u < sc.num_units && ok; u += num_pairs) {
        int m0, n0, ncols;
        unit(u, m0, n0, ncols);
        const uint32_t ab = acc_it & 1u;
        ok = wait_bounded(tfull_bar(ab), (acc_it >> 1) & 1u, wctx, kRoleEpilogue);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        const int m_w = m0 + row_off;
        const int m = m_w + lane;
        const bool row_ok = m < p.M;
        // this lane's row (the addresses are only formed, never used, for rows past M)
        const float* crow = p.C + static_cast<int64_t>(m) * p.ldc;
        float* dtile = static_cast<float*>(p.D) + static_cast<int64_t>(m) * p.ldd + n0;
        const int off_c = use_c ? static_cast<int>((4u - ((reinterpret_cast<uintptr_t>(crow) >> 2) & 3u)) & 3u) : 0;
        const int od = static_cast<int>((8u - ((reinterpret_cast<uintptr_t>(dtile) >> 2) & 7u)) & 7u);
        const int len = min(ncols, p.N - n0);  // valid columns of the unit
        // one sector of the window: columns a .. a + 7 of the unit, whole when it lies in
        // [0, len), element by element where it is cut
        auto put_sector = [&](int a, const float* v) {
          if (a >= 0 && a + 8 <= len) {
            st_global_v8_hint(dtile + a, v, pol_once);
          } else if (a < len && a + 8 > 0) {
#pragma unroll
            for (int t = 0; t < 8; ++t)
              if (a + t >= 0 && a + t < len) dtile[a + t] = v[t];
          }
        };
        float carry[8];  // the previous chunk's last 8 values
#pragma unroll
        for (int t = 0; t < 8; ++t) carry[t] = 0.0f;
        const int chunks = ncols / 32;
#pragma unroll 1
        for (int c = 0; c < chunks; ++c, ++g) {
          const int b = static_cast<int>(g & 1u);
          const int n = n0 + 32 * c;
          uint32_t r[32];
          tmem_ld_x32(tmem_base + lane_base + ab * BN + c * 32, r);
          tmem_ld_wait(r);
          if (c == chunks - 1) {  // accumulator in registers: release it to the MMA
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster_relaxed(mapa_cluster(tempty_bar(ab), 0));
          }
          float o[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) o[j] = p.alpha * __uint_as_float(r[j]);
          if (use_c) {
            bool w = wait_bounded(cfull_bar(ew, b), (g >> 1) & 1u, wctx, kRoleEpilogue);
            w = __all_sync(0xffffffffu, w);
            if (!w) {
              ok = false;
              break;
            }
            const float* cb = reinterpret_cast<const float*>(ebuf + b * CSLOT + rc * CBOX) + jr * 36 + 4 - off_c;
            const bool lead = n == 0 && row_ok;  // columns left of the class map's first element
#pragma unroll
            for (int t = 0; t < 32; ++t) {
              const float cv = (t < 3 && lead && t < off_c) ? crow[t] : cb[t];
              o[t] = fmaf(p.beta, cv, o[t]);
            }
            fence_proxy_async_smem();  // this lane's reads of the slot, before the TMA refills it
            __syncwarp();
            if (lane == 0 && static_cast<int>(issued - g) < 3) issue_c();  // chunk g + 2 into this slot
          }
          // window w[i] = (carry, o)[od + i]: three fixed-distance selections on od's bits
          float w1[39], w2[37], wv[32];
#pragma unroll
          for (int i = 0; i < 39; ++i) {
            const float x0 = i < 8 ? carry[i] : o[i - 8];
            const float x1 = i + 1 < 8 ? carry[i + 1] : o[i - 7];
            w1[i] = (od & 1) ? x1 : x0;
          }
#pragma unroll
          for (int i = 0; i < 37; ++i) w2[i] = (od & 2) ? w1[i + 2] : w1[i];
#pragma unroll
          for (int i = 0; i < 32; ++i) wv[i] = (od & 4) ? w2[i + 4] : w2[i];
          if (row_ok && 32 * c - 8 + od < len) {
#pragma unroll
            for (int k = 0; k < 4; ++k) put_sector(32 * c - 8 + od + 8 * k, wv + 8 * k);
          }
#pragma unroll
          for (int t = 0; t < 8; ++t) carry[t] = o[24 + t];
        }
        if (!ok) break;
        // the unit's last sector: columns 32 * chunks - 8 + od .. of the last chunk's values
        if (row_ok) {
          float last[8];
#pragma unroll
          for (int t = 0; t < 8; ++t) {
            float v = carry[t];
#pragma unroll
            for (int k = 1; k < 8; ++k)
              if (od == k) v = t + k < 8 ? carry[t + k] : 0.0f;
            last[t] = v;
          }
          put_sector(32 * chunks - 8 + od, last);
        }
        ++acc_it;
      }
      if (lane == 0 && !ok && use_c) {  // C loads still in flight land before the CTA may exit
        for (uint32_t j = g; j < issued; ++j) wait_drain(cfull_bar(ew, static_cast<int>(j & 1u)), (j >> 1) & 1u, p.timeout_ns);
      }
      __syncwarp();
    } else {
      // unaligned rows of C or D: each chunk is transposed through shared memory, and
      // every warp-wide load of C and store of D covers 32 consecutive elements of one
      // row.  C arrives by cp.async two chunks ahead, across unit boundaries, in a ring of
      // three 4 KB buffers (this warp's epilogue buffers 1-3; buffer 0 holds the
      // transposed accumulator), so that several chunks' loads are in flight while one is
      // stored.
      float* st = reinterpret_cast<float*>(ebuf);
      float4* st4 = reinterpret_cast<float4*>(ebuf);
      const uint32_t cring = smem_addr(ebuf + Cfg::EPI_BUF_BYTES);
      int lu = pair, lc = 0;  // the chunk whose C is requested next
      uint32_t k_req = 0;     // chunks requested (one cp.async group each)
      auto request_next = [&]() {
        if (lu < sc.num_units) {
          int m1, n1, nc1;
          unit(lu, m1, n1, nc1);
          issue_c_rows(p, cring + (k_req % 3) * Cfg::EPI_BUF_BYTES, m1 + row_off, n1 + 32 * lc, lane);
          if (++lc == nc1 / 32) {
            lc = 0;
            lu += num_pairs;
          }
        }
        cp_async_commit();
        ++k_req;
      };
      request_next();
      request_next();
      uint32_t acc_it = 0, k = 0;
      for (int u = pair; u < sc.num_units; u += num_pairs) {
        int m0, n0, ncols;
        unit(u, m0, n0, ncols);
        const uint32_t ab = acc_it & 1u;
        bool ok = wait_bounded(tfull_bar(ab), (acc_it >> 1) & 1u, wctx, kRoleEpilogue);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        const int m_base = m0 + row_off;
        const int chunks = ncols / 32;
#pragma unroll 1
        for (int c = 0; c < chunks; ++c, ++k) {
          request_next();       // chunk k + 2
          cp_async_wait<2>();   // chunk k's C has landed (this lane's elements)
          uint32_t r[32];
          tmem_ld_x32(tmem_base + lane_base + ab * BN + c * 32, r);
          tmem_ld_wait(r);
          if (c == chunks - 1) {  // accumulator in registers: release it to the MMA
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster_relaxed(mapa_cluster(tempty_bar(ab), 0));
          }
#pragma unroll
          for (int j = 0; j < 8; ++j)
            st4[lane * 8 + (j ^ (lane & 7))] = make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                                                           __uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3]));
          __syncwarp();
          store_rows(p, st, m_base, n0 + c * 32, st + (1 + k % 3) * (Cfg::EPI_BUF_BYTES / 4), lane);
          __syncwarp();
        }
        ++acc_it;
      }
      cp_async_wait<0>();  // no copy into shared memory outlives the loop
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();  // no CTA leaves while its peer may still touch its memory
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, Cfg::TMEM_COLS);
  }
}

// ------------------------------------------------------------------ host side

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

// 2-D row-major matrix rows x cols (pitch in elements) with a box of box_cols x box_rows.
bool make_tensor_map_2d(CUtensorMap* map, const void* base, CUtensorMapDataType dt, int esize,
                        int64_t rows, int64_t cols, int64_t pitch, int box_cols, int box_rows,
                        CUtensorMapSwizzle swizzle) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(pitch * esize)};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}


// stream-K tail: one 256 x 256 FP32 partial slot (two CTAs x 128 rows) and 8 flags per pair
size_t pair_sk_bytes(int pairs) {
  return static_cast<size_t>(pairs) * (2 * 128 * 256 * sizeof(float) + 8 * sizeof(unsigned long long));
}

// The schedule's tail: W whole waves of P workers (CTA pairs, or CTAs of the one-CTA FP8
// kernel) and R more tiles.  The R tiles are split by K ranges across all P workers when
// there are at least P / 4 of them and at least 8 K blocks a tile (so that no tile has
// more than ~5 pieces); otherwise the 16-bit pair kernel runs them as 256 x 128 halves and
// the FP8 kernel as whole tiles.
static bool sk_tail(int T, int P, int KB, int& W, int& R) {
  W = T / P;
  R = T - W * P;
  return W >= 1 && R > 0 && 4 * R >= P && KB >= 8;
}

size_t pair_sk_workspace(int M, int N, int K, int num_sms) {
  const int P = num_sms / 2;
  if (P <= 0) return 0;
  const int T = ((M + 255) / 256) * ((N + 255) / 256);
  const int KB = (K + PairCfg<256>::BK - 1) / PairCfg<256>::BK;
  int W, R;
  return sk_tail(T, P, KB, W, R) ? pair_sk_bytes(P) : 0;
}

// A value no flag of an earlier call holds: a per-process random high word over a call count.
static unsigned long long next_epoch() {
  static std::atomic<unsigned long long> seq{0};
  static const unsigned long long salt = [] {
    unsigned long long x = static_cast<unsigned long long>(std::chrono::steady_clock::now().time_since_epoch().count()) ^
                           static_cast<unsigned long long>(reinterpret_cast<uintptr_t>(&seq));
    x += 0x9E3779B97F4A7C15ull;  // splitmix64 finaliser
    x = (x ^ (x >> 30)) * 0xBF58476D1CE4E5B9ull;
    x = (x ^ (x >> 27)) * 0x94D049BB133111EBull;
    x ^= x >> 31;
    return (x | 1ull) << 32;
  }();
  return salt | ((seq.fetch_add(1) + 1) & 0xFFFFFFFFull);
}

// FP8 stream-K tail: one 128 x 256 FP32 partial slot and 8 flags (one per promotion
// warp) per CTA
size_t fp8_sk_bytes(int ctas) {
  return static_cast<size_t>(ctas) * (128 * 256 * sizeof(float) + 8 * sizeof(unsigned long long));
}

size_t fp8_sk_workspace(int M, int N, int K, int num_sms) {
  if (num_sms <= 0 || M <= 0 || N <= 0 || K <= 0) return 0;
  // the tile width run_fp8 picks
  const int tiles128 = ((M + 127) / 128) * ((N + 127) / 128);
  const int BN = (N > 128 && tiles128 > num_sms) ? 256 : 128;
  const int T = ((M + 127) / 128) * ((N + BN - 1) / BN);
  const int P = T < num_sms ? T : num_sms;
  const int KB = (K + 127) / 128;
  int W, R;
  return KB < 32768 && sk_tail(T, P, KB, W, R) ? fp8_sk_bytes(P) : 0;
}

constexpr int kMaxDev = 64;

template <class Cfg, uint32_t AB_FMT>
static ll_status run(const GemmArgs& a, const LaunchCtx& ctx) {
  auto kern = gemm_tc_kernel<Cfg, AB_FMT>;
  // the attribute is per device; setting it on every call is cheap and always correct
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM) !=
      cudaSuccess)
    return LL_ERR_CUDA;
  const CUtensorMapDataType dt =
      Cfg::FP8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
               : ((AB_FMT & 7u) == 1 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16);
  CUtensorMap tmA, tmB;
  if (!make_tensor_map_2d(&tmA, a.A, dt, Cfg::ELT, a.M, a.K, a.lda, Cfg::BK, 128)) return LL_ERR_CUDA;
  if (!make_tensor_map_2d(&tmB, a.B, dt, Cfg::ELT, a.K, a.N, a.ldb, Cfg::B_BOX_N, Cfg::BK)) return LL_ERR_CUDA;

  GemmParams p = make_gemm_params(a, ctx);

  const int num_tiles = ((a.M + 127) / 128) * ((a.N + Cfg::BN - 1) / Cfg::BN);
  const int grid = num_tiles < ctx.num_sms ? num_tiles : ctx.num_sms;
  TileSched ts;
  ts.full_tiles = num_tiles;
  ts.sk_tiles = 0;
  ts.sk_part = nullptr;
  ts.sk_flag = nullptr;
  ts.epoch = 0;
  if (Cfg::FP8) {  // stream-K tail, when the caller's workspace has room for it
    const int KB = (a.K + Cfg::BK - 1) / Cfg::BK;
    int W, R;
    // (K block indices are packed into 16 bits in the kernel's item table)
    if (KB < 32768 && sk_tail(num_tiles, grid, KB, W, R) && a.sk_ws != nullptr && a.sk_bytes >= fp8_sk_bytes(grid)) {
      ts.full_tiles = W * grid;
      ts.sk_tiles = R;
      ts.sk_part = static_cast<float*>(a.sk_ws);
      ts.sk_flag = reinterpret_cast<unsigned long long*>(static_cast<unsigned char*>(a.sk_ws) +
                                                         static_cast<size_t>(grid) * 128 * 256 * sizeof(float));
      ts.epoch = next_epoch();
    }
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(Cfg::THREADS);
  cfg.dynamicSmemBytes = Cfg::SMEM;
  cfg.stream = ctx.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kern, tmA, tmB, p, ts) != cudaSuccess) {
    cudaGetLastError();
    return LL_ERR_CUDA;
  }
  return LL_OK;
}


template <uint32_t AB_FMT>
static ll_status run_pair(const GemmArgs& a, const LaunchCtx& ctx) {
  using Cfg = PairCfg<256>;
  auto kern = gemm_tc2_kernel<Cfg, AB_FMT>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM) !=
      cudaSuccess)
    return LL_ERR_CUDA;
  const CUtensorMapDataType dt =
      (AB_FMT & 7u) == 1 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  CUtensorMap tmA, tmB, tmC, tmD;
  if (!make_tensor_map_2d(&tmA, a.A, dt, Cfg::ELT, a.M, a.K, a.lda, Cfg::BK, 128)) return LL_ERR_CUDA;
  if (!make_tensor_map_2d(&tmB, a.B, dt, Cfg::ELT, a.K, a.N, a.ldb, Cfg::B_BOX_N, Cfg::BK)) return LL_ERR_CUDA;
  GemmParams p = make_gemm_params(a, ctx);
  // 16-bit epilogue through TMA when the rows of D (and of C, if read) start on
  // 16-byte boundaries: 32 x 32 boxes, 128-byte rows (FP32) or 64-byte rows (16-bit)
  memset(&tmC, 0, sizeof(tmC));
  memset(&tmD, 0, sizeof(tmD));
  const bool o32 = a.d_type == LL_OUT_F32;
  p.epi_tma = p.d_row16 && (a.beta == 0.0f || p.c_vec);
  // FP32 D rows not on 16-byte boundaries: C through TMA by row classes (EpiResMaps), D by
  // whole 32-byte sectors from the lanes
  EpiResMaps rm;
  memset(&rm, 0, sizeof(rm));
  p.epi_res = !p.epi_tma && o32 && a.M >= 4 && a.N >= 4;
  if (p.epi_res) {
    for (int k = 0; k < 4; ++k) {
      if (a.beta != 0.0f) {
        const float* crow = a.C + static_cast<int64_t>(k) * a.ldc;
        const int off_c = static_cast<int>((4u - ((reinterpret_cast<uintptr_t>(crow) >> 2) & 3u)) & 3u);
        if (!make_tensor_map_2d(&rm.c[k], crow + off_c, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, (a.M - k + 3) / 4,
                                a.N - off_c, 4 * a.ldc, 36, 8, CU_TENSOR_MAP_SWIZZLE_NONE))
          return LL_ERR_CUDA;
      }
    }
  }
  if (p.epi_tma) {
    if (!make_tensor_map_2d(&tmD, a.D, o32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_UINT16,
                            o32 ? 4 : 2, a.M, a.N, a.ldd, 32, 32,
                            o32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B))
      return LL_ERR_CUDA;
    if (a.beta != 0.0f &&
        !make_tensor_map_2d(&tmC, a.C, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, a.M, a.N, a.ldc, 32, 32))
      return LL_ERR_CUDA;
  }

  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(Cfg::THREADS);
  cfg.dynamicSmemBytes = Cfg::SMEM;
  cfg.stream = ctx.stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  // co-resident CTA pairs (one CTA per SM): the persistent grid
  static int max_pairs[kMaxDev] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= kMaxDev) return LL_ERR_NO_DEVICE;
  if (max_pairs[dev] == 0) {
    cfg.gridDim = dim3(2 * (ctx.num_sms / 2));
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n <= 0) {
      cudaGetLastError();
      n = ctx.num_sms / 2;
    }
    max_pairs[dev] = n;
  }
  PairSched sc;
  sc.num_m2 = (a.M + 255) / 256;
  sc.num_n = (a.N + Cfg::BN - 1) / Cfg::BN;
  const int T = sc.num_m2 * sc.num_n;
  int P = T < max_pairs[dev] ? T : max_pairs[dev];
  const int waves = T / P, rem = T - waves * P;
  // finish with one half-wave of 256 x 128 halves when that is shorter; a problem whose
  // halves all fit one wave runs as halves only (twice the pairs at work)
  if (2 * T <= max_pairs[dev]) {
    sc.full_units = 0;
    sc.num_units = 2 * T;
    P = 2 * T;
  } else if (rem > 0 && 2 * rem <= P) {
    sc.full_units = waves * P;
    sc.num_units = sc.full_units + 2 * rem;
  } else {
    sc.full_units = T;
    sc.num_units = T;
  }
  sc.sk_tiles = 0;
  sc.sk_part = nullptr;
  sc.sk_flag = nullptr;
  sc.epoch = 0;
  {  // stream-K tail (TMA epilogue only), when the caller's workspace has room for it
    const int KB = (a.K + Cfg::BK - 1) / Cfg::BK;
    int W, R;
    if (p.epi_tma && T > max_pairs[dev] && sk_tail(T, max_pairs[dev], KB, W, R) && a.sk_ws != nullptr &&
        a.sk_bytes >= pair_sk_bytes(max_pairs[dev])) {
      P = max_pairs[dev];
      sc.full_units = W * P;
      sc.num_units = W * P;
      sc.sk_tiles = R;
      sc.sk_part = static_cast<float*>(a.sk_ws);
      sc.sk_flag = reinterpret_cast<unsigned long long*>(static_cast<unsigned char*>(a.sk_ws) +
                                                         static_cast<size_t>(P) * 2 * 128 * 256 * sizeof(float));
      sc.epoch = next_epoch();
    }
  }
  cfg.gridDim = dim3(2 * P);
  if (cudaLaunchKernelEx(&cfg, kern, tmA, tmB, tmC, tmD, p, sc, rm) != cudaSuccess) {
    cudaGetLastError();
    return LL_ERR_CUDA;
  }
  return LL_OK;
}

// 128 x 256 tiles, or 128 x 128 ones (four TMEM partial buffers) when N <= 128 or when
// the narrower tiles still fit one wave: measured 1536 x 1536 x 4096 923 -> 1105 TFLOPS,
// while at 2048^3 and above the 256-wide tile is 1.4-1.6x faster
template <uint32_t F>
static ll_status run_fp8(const GemmArgs& a, const LaunchCtx& ctx) {
  const int tiles128 = ((a.M + 127) / 128) * ((a.N + 127) / 128);
  if (a.N > 128 && tiles128 > ctx.num_sms) return run<TileCfg<256, true>, F>(a, ctx);
  return run<TileCfg<128, true>, F>(a, ctx);
}

ll_status launch_gemm_tc(const GemmArgs& a, const LaunchCtx& ctx) {
  if (a.mx) return launch_gemm_mx(a, ctx);  // hardware block scaling (gemm_mx.cu)
  // FP8: the one-CTA kernel at every size (it measured 3 to 17 % faster than a CTA-pair
  // version of the block promotion from 1792^3 to 8192^3)
  if (a.in_type == LL_IN_E4M3 || a.in_type == LL_IN_E5M2) {
    const bool a5 = a.in_type == LL_IN_E5M2, b5 = a.b_type == LL_IN_E5M2;
    if (!a5 && !b5) return run_fp8<fmt_pair(0, 0)>(a, ctx);
    if (a5 && b5) return run_fp8<fmt_pair(1, 1)>(a, ctx);
    if (!a5) return run_fp8<fmt_pair(0, 1)>(a, ctx);
    return run_fp8<fmt_pair(1, 0)>(a, ctx);
  }
  // 16-bit: CTA pairs from SMs/4 pair tiles on, or from SMs/8 when M and N both exceed
  // 128 (the problems with at most half a wave of tiles then running as 256 x 128
  // halves; measured on GB300: 1280^3 265 -> 343 TFLOPS, 1536^3 400 -> 532,
  // 1536 x 1536 x 4096 494 -> 777, 256 x 8192 x 4096 424 -> 684, while 1024^3 (16 pair
  // tiles) and M or N of 128 stay faster on the one-CTA kernel); the rest has fewer tiles
  // than SMs even at 128 x 64
  const int pair_tiles = ((a.M + 255) / 256) * ((a.N + 255) / 256);
  const bool pair = pair_tiles >= ctx.num_sms / 4 || (pair_tiles >= ctx.num_sms / 8 && a.M > 128 && a.N > 128);
  constexpr uint32_t F16 = fmt_pair(0, 0), BF16 = fmt_pair(1, 1);
  const bool bf = a.in_type == LL_IN_BF16;
  if (pair) return bf ? run_pair<BF16>(a, ctx) : run_pair<F16>(a, ctx);
  return bf ? run<TileCfg<64, false>, BF16>(a, ctx) : run<TileCfg<64, false>, F16>(a, ctx);
}

}  // namespace ll
