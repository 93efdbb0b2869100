// MX block-scaled 8-bit GEMM on the 5th-generation tensor cores of sm_103a:
//
//   D[i][j] = alpha * sum_k (XA[i][k/32] A[i][k]) (XB[j][k/32] B[k][j]) + beta * C[i][j]
//
// with FP32 accumulation, where every 32 consecutive K elements of a row of A (of a column
// of B) share one E8M0 scale 2^(e - 127): OCP microscaling, the block-scaled formats the
// "Tensor Core" chapter lists for Blackwell (table of tensor-core formats per generation).
// The tensor cores apply the scales themselves (tcgen05.mma kind::mxf8f6f4.block_scale),
// so unlike the FP32 128-block path there is no software promotion between K blocks.
//
// The scale codes are first rearranged (mx_scale_tile_kernel, into the caller's workspace)
// into the blocks tcgen05.cp copies into TMEM: for every 128 rows of A (128 columns of B)
// and every 128-K stage, 32 rows of 16 bytes where row r holds at byte 4j + b the code of
// item 32j + r for the stage's K block b.  The GEMM kernels then fetch each stage's blocks
// by TMA together with its operands, so scale codes reach shared memory the same way the
// operands do (asynchronously, completing on the stage's barrier).  TMEM then holds, per
// stage, A's codes with row m at lane m, column m / 32, and B's with column n at lanes
// 32 q + n % 32 of every lane quarter q, column 4 + n / 32; the scale-factor IDs of the
// instruction descriptor (B bits 4-5, A bits 29-30) pick K block kk's byte of those words.
//
// One-CTA kernel (gemm_mx_kernel): one persistent CTA per SM walks 128 x 256 output tiles
// in the grouped order.  Roles:
//   warp 0      producer: TMA copies of A (128 rows x 128 K, K-major) and B (128 K x 256
//               columns, N-major), 128-byte swizzle, and of the stage's three scale blocks
//               into a 4-stage ring.
//   warp 1      TMEM allocator and MMA issuer.  Per stage, three tcgen05.cp copies put the
//               scale blocks into TMEM (replicated over the four lane quarters), then four
//               K = 32 tcgen05.mma .kind::mxf8f6f4.block_scale.
//   warps 2-9   epilogue.  They drain the tile's 128 x 256 FP32 accumulator from TMEM into
//               registers (32 rows x 128 columns per warp), hand TMEM back at once so the
//               next tile's MMAs run, then apply alpha / beta and store D from registers.
// TMEM: the accumulator in columns 0-255; stage s's scales in columns 256 + 16 s (A's in
// the first 4, B's in the next 8).  Every wait is bounded; on expiry the CTA records
// LL_ERR_DEVICE_TIMEOUT, drains its copies and MMAs, frees TMEM and exits.
#include <cstring>

#include "gemm_common.cuh"

namespace ll {

namespace {

// NV = false: MXFP8 (8-bit elements, B N-major as K x N, one E8M0 scale per 32 K elements:
// one 4-byte scale word per row / column covers a 128-byte stage, its bytes picked by the
// scale-factor IDs).  NV = true: NVFP4 (E2M1 elements two per byte, B given K-major as N x K,
// one UE4M3 scale per 16 K elements: each K = 64 MMA reads a whole word, so a 128-byte stage
// of 256 elements carries four words per row / column).
template <bool NV>
struct MxCfg {
  static constexpr int BM = 128, BN = 256;
  static constexpr int BK = 128;                 // bytes of K per stage
  static constexpr int BK_ELEMS = NV ? 256 : 128;
  static constexpr int KSTEPS = 4;               // MMAs per stage (K = 64 FP4 or 32 FP8: 32 bytes)
  static constexpr int A_BYTES = BM * 128;
  static constexpr int B_BOX_N = NV ? BN : 128;  // B rows (NV: N rows of B^T) or columns per box
  static constexpr int B_BOXES = BN / B_BOX_N;
  static constexpr int B_BOX_BYTES = NV ? BN * 128 : BK * 128;
  static constexpr int STAGE_BYTES = A_BYTES + B_BOXES * B_BOX_BYTES;  // 48 KB
  static constexpr int SETS = NV ? 4 : 1;                                // scale words per row and stage
  static constexpr int SF_BLOCK = 512;                                   // 32 rows x 16 bytes
  static constexpr int SF_STAGE_BYTES = 3 * SETS * SF_BLOCK;             // A's blocks, then B's
  static constexpr int STAGES = 4;
  static constexpr int EPI_WARP0 = 2, EPI_WARPS = 8;
  static constexpr int EPI_THREADS = 32 * EPI_WARPS;
  static constexpr int THREADS = 32 * (EPI_WARP0 + EPI_WARPS);
  static constexpr int TMEM_COLS = 512;
  static constexpr int SF_COL0 = BN, SF_COLS = 12 * SETS;  // A: 4 per set, B: 8 per set
  static constexpr int NBARS = 2 * STAGES + 3;  // full, empty, tfull, tempty, drain
  static constexpr int SMEM = STAGES * (STAGE_BYTES + SF_STAGE_BYTES) + NBARS * 8 + 16 + 1024;
  static_assert(SF_COL0 + STAGES * SF_COLS <= TMEM_COLS, "TMEM budget");
  static_assert(SMEM <= 227 * 1024, "shared memory budget");
};

// Block-scaled instruction descriptor (kind::mxf8f6f4): A / B format (bits 7-9 / 10-12),
// A K-major, B MN-major (bit 16), N >> 3 (bits 17-22), scale type E8M0 (bit 23),
// M >> 4 (bits 24-28); the scale-factor IDs (B bits 4-5, A bits 29-30) are added per MMA.
__host__ __device__ constexpr uint32_t make_idesc_mx(uint32_t fmts, int n, int m) {
  return ((fmts & 7u) << 7) | (((fmts >> 3) & 7u) << 10) | (1u << 16) |
         (static_cast<uint32_t>(n >> 3) << 17) | (1u << 23) | (static_cast<uint32_t>(m >> 4) << 24);
}

__host__ __device__ constexpr uint32_t sf_ids(uint32_t kk) { return (kk << 4) | (kk << 29); }

// kind::mxf4nvf4 (NVFP4): A / B format E2M1 (1), both K-major, N >> 3, scale type UE4M3
// (bit 23 = 0), M >> 4; scale-factor IDs 0 (each K = 64 MMA reads all four bytes of a word).
__host__ __device__ constexpr uint32_t make_idesc_nv(int n, int m) {
  return (1u << 7) | (1u << 10) | (static_cast<uint32_t>(n >> 3) << 17) | (static_cast<uint32_t>(m >> 4) << 24);
}

template <bool NV>
__host__ __device__ constexpr uint32_t mx_idesc(uint32_t fmts, int n, int m) {
  return NV ? make_idesc_nv(n, m) : make_idesc_mx(fmts, n, m);
}

// MMA kk of a stage: its instruction descriptor and the TMEM columns (from the stage's base)
// of its A and B scale words
template <bool NV>
__device__ __forceinline__ uint32_t mma_idesc(uint32_t base, int kk) {
  return NV ? base : base | sf_ids(kk);
}
template <bool NV, int SETS>
__device__ __forceinline__ uint32_t sfa_col(int kk) { return NV ? 4 * kk : 0; }
template <bool NV, int SETS>
__device__ __forceinline__ uint32_t sfb_col(int kk) { return 4 * SETS + (NV ? 8 * kk : 0); }

// 4-code scale words per row of the rearranged scale blocks: one per 128-K stage (MX), four
// per 256-element stage (NVFP4; whole stages, the words past K holding neutral codes)
__host__ __device__ constexpr int mx_words(int K, bool nv) { return nv ? 4 * ((K + 255) / 256) : (K + 127) / 128; }

// ------------------------------------------------------------------ scale blocks
//
// Block (blk, kb) of a code matrix (rows of K-block-contiguous codes, `ld` bytes apart)
// holds rows 128 blk .. 128 blk + 127 and K blocks 4 kb .. 4 kb + 3: 512 bytes, 16-byte row r
// holding at byte 4j + b the code of row 128 blk + 32j + r for K block 4 kb + b.  Codes of
// rows past `rows` or K blocks past `nkb` are written as `neutral` (a finite scale: their
// operand elements are zero).  Blocks are stored in the order the kernels fetch them:
//   A (cols256 = 0): block (blk, kb) at ((blk * KB) + kb) * 512
//   B (cols256 = 1): block (blk, kb) at (((blk / 2) * KB + kb) * 2 + blk % 2) * 512
// so that the two blocks of a 256-column tile's stage are adjacent.  One CTA of 128
// threads per (blk, four stages): each thread loads one row's 16 codes, the block is
// transposed through shared memory, and each warp writes one 512-byte block.
__global__ void __launch_bounds__(128) mx_scale_tile_kernel(const uint8_t* __restrict__ src, int64_t ld, int rows,
                                                            int nkb, int KB, int cols256, uint32_t neutral,
                                                            uint8_t* __restrict__ dst) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  __shared__ __align__(16) uint8_t sm[128 * 16];
  const int t = threadIdx.x;
  const int blk = blockIdx.x, g = blockIdx.y;  // g: four stages, 16 K blocks
  const int row = blk * 128 + t;
  const int k0 = 16 * g;
  const uint32_t n4 = neutral * 0x01010101u;
  uint4 v = make_uint4(n4, n4, n4, n4);
  if (row < rows) {
    const uint8_t* q = src + static_cast<int64_t>(row) * ld + k0;
    if (k0 + 16 <= nkb && (reinterpret_cast<uintptr_t>(q) & 15u) == 0) {
      v = __ldg(reinterpret_cast<const uint4*>(q));
    } else {
      uint32_t w[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        uint32_t x = 0;
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          const int k = k0 + 4 * i + b;
          x |= (k < nkb ? static_cast<uint32_t>(__ldg(q + 4 * i + b)) : neutral) << (8 * b);
        }
        w[i] = x;
      }
      v = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
  *reinterpret_cast<uint4*>(sm + t * 16) = v;
  __syncthreads();
  const int c = t >> 5, r = t & 31;  // stage within the four, block row
  const int kb = 4 * g + c;
  if (kb >= KB) return;
  uint32_t o[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) o[j] = *reinterpret_cast<const uint32_t*>(sm + (32 * j + r) * 16 + 4 * c);
  const int64_t blk_off = cols256 ? ((static_cast<int64_t>(blk / 2) * KB + kb) * 2 + (blk & 1)) * 512
                                  : (static_cast<int64_t>(blk) * KB + kb) * 512;
  *reinterpret_cast<uint4*>(dst + blk_off + r * 16) = make_uint4(o[0], o[1], o[2], o[3]);
}

// ------------------------------------------------------------------ one-CTA kernel

template <uint32_t AB_FMT, bool NV>
__global__ void __launch_bounds__(MxCfg<NV>::THREADS, 1)
    gemm_mx_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmXA, const __grid_constant__ CUtensorMap tmXB,
                   const GemmParams p) {
  using Cfg = MxCfg<NV>;
  constexpr int S = Cfg::STAGES;
  constexpr uint32_t IDESC = mx_idesc<NV>(AB_FMT, Cfg::BN, Cfg::BM);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sf_base = smem + S * Cfg::STAGE_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sf_base + S * Cfg::SF_STAGE_BYTES);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + Cfg::NBARS);
  uint32_t* abort_flag = tmem_slot + 1;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  auto full_bar = [&](int s) { return smem_addr(bars + s); };
  auto empty_bar = [&](int s) { return smem_addr(bars + S + s); };
  const uint32_t tfull_bar = smem_addr(bars + 2 * S);
  const uint32_t tempty_bar = smem_addr(bars + 2 * S + 1);
  const uint32_t drain_bar = smem_addr(bars + 2 * S + 2);

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    mbar_init(tfull_bar, 1);
    mbar_init(tempty_bar, Cfg::EPI_THREADS);
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
  const int num_m = (p.M + Cfg::BM - 1) / Cfg::BM;
  const int num_n = (p.N + Cfg::BN - 1) / Cfg::BN;
  const int num_tiles = num_m * num_n;
  const int KB = (p.K + Cfg::BK_ELEMS - 1) / Cfg::BK_ELEMS;  // stages per tile
  const int KBw = mx_words(p.K, NV);                            // scale words per row

  // programmatic dependent launch: L2 prefetch of the first ring of operand tiles, then
  // the wait for the previous kernel of the stream (scale blocks, C and D come after it)
  if (warp == 0 && lane == 0 && static_cast<int>(blockIdx.x) < num_tiles) {
    int mb, nb;
    tile_coords(blockIdx.x, num_m, num_n, p.group_m, mb, nb);
    const int pre = KB < S ? KB : S;
    for (int kb = 0; kb < pre; ++kb) {
      tma_prefetch_l2(&tmA, kb * Cfg::BK, mb * Cfg::BM);
      if (NV)
        tma_prefetch_l2(&tmB, kb * Cfg::BK, nb * Cfg::BN);
      else
        for (int j = 0; j < Cfg::B_BOXES; ++j) tma_prefetch_l2(&tmB, nb * Cfg::BN + j * Cfg::B_BOX_N, kb * Cfg::BK);
    }
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");

  if (warp == 0) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      tma_prefetch_desc(&tmA);
      tma_prefetch_desc(&tmB);
      tma_prefetch_desc(&tmXA);
      tma_prefetch_desc(&tmXB);
      uint32_t it = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
        int mb, nb;
        tile_coords(t, num_m, num_n, p.group_m, mb, nb);
        for (int kb = 0; kb < KB; ++kb) {
          const int s = it % S;
          if (!wait_bounded(empty_bar(s), ((it / S) & 1u) ^ 1u, wctx, kRoleProducer)) {
            ok = false;
            break;
          }
          uint8_t* a_s = smem + s * Cfg::STAGE_BYTES;
          uint8_t* b_s = a_s + Cfg::A_BYTES;
          uint8_t* sf = sf_base + s * Cfg::SF_STAGE_BYTES;
          mbar_arrive_expect_tx(full_bar(s), Cfg::STAGE_BYTES + Cfg::SF_STAGE_BYTES);
          tma_load_2d(smem_addr(a_s), &tmA, full_bar(s), kb * Cfg::BK, mb * Cfg::BM);
          if (NV) {  // B^T: 256 rows x 128 bytes, K-major
            tma_load_2d(smem_addr(b_s), &tmB, full_bar(s), kb * Cfg::BK, nb * Cfg::BN);
          } else {
#pragma unroll
            for (int j = 0; j < Cfg::B_BOXES; ++j)
              tma_load_2d(smem_addr(b_s + j * Cfg::B_BOX_BYTES), &tmB, full_bar(s), nb * Cfg::BN + j * Cfg::B_BOX_N,
                          kb * Cfg::BK);
          }
          tma_load_2d(smem_addr(sf), &tmXA, full_bar(s), 0, (mb * KBw + Cfg::SETS * kb) * 2);
          tma_load_2d(smem_addr(sf + Cfg::SETS * Cfg::SF_BLOCK), &tmXB, full_bar(s), 0,
                      (nb * KBw + Cfg::SETS * kb) * 4);
          ++it;
        }
      }
      if (!ok) {  // wait for the copies still in flight before the CTA can exit
        for (uint32_t j = (it > static_cast<uint32_t>(S) ? it - S : 0u); j < it; ++j)
          wait_drain(full_bar(j % S), (j / S) & 1u, p.timeout_ns);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- scale copies + MMA issuer
    if (lane == 0) {
      uint32_t it = 0, tiles = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
        if (!wait_bounded(tempty_bar, (tiles & 1u) ^ 1u, wctx, kRoleMma)) break;
        tc_fence_after();
        for (int kb = 0; kb < KB; ++kb) {
          const int s = it % S;
          if (!wait_bounded(full_bar(s), (it / S) & 1u, wctx, kRoleMma)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sf_t = tmem_base + Cfg::SF_COL0 + s * Cfg::SF_COLS;
          const uint32_t sf_s = smem_addr(sf_base + s * Cfg::SF_STAGE_BYTES);
#pragma unroll
          for (int j = 0; j < 3 * Cfg::SETS; ++j)  // A's blocks, then B's (two per set)
            tmem_cp_32x128b_x4(sf_t + 4 * j, smem_desc_plain16(sf_s + j * Cfg::SF_BLOCK));
          const uint32_t a_base = smem_addr(smem + s * Cfg::STAGE_BYTES);
          const uint32_t b_base = a_base + Cfg::A_BYTES;
#pragma unroll
          for (int kk = 0; kk < Cfg::KSTEPS; ++kk) {
            const uint64_t adesc = smem_desc_sw128(a_base + kk * 32, 16, 1024);
            const uint64_t bdesc = NV ? smem_desc_sw128(b_base + kk * 32, 16, 1024)
                                      : smem_desc_sw128(b_base + kk * 32 * 128, Cfg::B_BOX_BYTES, 1024);
            const uint32_t acc = (kb > 0 || kk > 0) ? 1u : 0u;
            if (NV)
              mma_nvf4(tmem_base, adesc, bdesc, IDESC, sf_t + sfa_col<NV, Cfg::SETS>(kk),
                       sf_t + sfb_col<NV, Cfg::SETS>(kk), acc);
            else
              mma_mxf8(tmem_base, adesc, bdesc, mma_idesc<NV>(IDESC, kk), sf_t + sfa_col<NV, Cfg::SETS>(kk),
                       sf_t + sfb_col<NV, Cfg::SETS>(kk), acc);
          }
          mma_commit(empty_bar(s));  // the stage (operands and scale blocks) may be refilled
          ++it;
        }
        if (!ok) break;
        mma_commit(tfull_bar);
        ++tiles;
      }
      // every MMA and copy issued by this thread must finish before TMEM is freed
      mma_commit(drain_bar);
      wait_drain(drain_bar, 0u, p.timeout_ns);
    }
  } else {
    // ---------------------------------------------------------------- epilogue
    const int ew = warp - Cfg::EPI_WARP0;
    const int q = warp & 3;   // TMEM lane quarter this warp may access
    const int h = ew >> 2;    // column half of the tile
    const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
    uint32_t tiles = 0;
    for (int t = blockIdx.x; t < num_tiles; t += gridDim.x) {
      int mb, nb;
      tile_coords(t, num_m, num_n, p.group_m, mb, nb);
      const int m = mb * Cfg::BM + q * 32 + lane;
      const int ncol0 = nb * Cfg::BN + h * (Cfg::BN / 2);
      bool w = wait_bounded(tfull_bar, tiles & 1u, wctx, kRoleEpilogue);
      w = __all_sync(0xffffffffu, w);
      if (!w) break;
      tc_fence_after();
      uint32_t u[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld_x32(tmem_base + lane_base + h * (Cfg::BN / 2) + c * 32, u[c]);
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld_wait(u[c]);
      tc_fence_before();
      mbar_arrive(tempty_bar);  // the accumulator is in registers: the next tile's MMAs may start
      float acc[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int j = 0; j < 32; ++j) acc[c][j] = __uint_as_float(u[c][j]);
      epilogue_rows<4>(p, m, ncol0, acc);
      ++tiles;
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
// Large problems run on CTA pairs (2-CTA clusters): a pair owns a 256 x 256 output tile;
// CTA r loads rows 128 r .. 128 r + 127 of the tile's A and columns 128 r .. 128 r + 127
// of its B (one 128-byte-swizzled box per stage), and the even CTA's MMA thread issues
// tcgen05.mma.cta_group::2 (M = 256).  Per SM that halves the B bytes TMA writes into
// shared memory and the tensor cores read back (the one-CTA tile moves 96 KB through
// shared memory per 128-K stage, which bounds it).
//
// Scales.  Each CTA's TMEM must hold the scales of its own 128 rows of A and of all 256
// columns of B.  Copying them with tcgen05.cp (as the one-CTA kernel does) puts three
// copies per stage for MX, twelve for NVFP4, into the tensor pipe in front of the MMAs,
// which measured as the larger part of the NVFP4 kernel's time.  Here four scale warps per
// CTA, one per TMEM lane quarter, write the same TMEM contents with tcgen05.st instead:
// warp q reads row `lane` of each of the stage's scale blocks (fetched by TMA into its own
// CTA's shared memory) and stores it into lane 32 q + lane, so that every lane quarter
// holds what the replicating copy would have put there:
//   SFA: block kk (4 words: rows lane, 32 + lane, 64 + lane, 96 + lane) at column SFA + 4 kk,
//   SFB: block (kk, h) (columns 128 h + 32 j + lane, j < 4) at column SFB + 8 kk + 4 h.
// (The scale-factor TMEM addresses given to the MMA stay multiples of 4 columns, as the
// copy layout has them.)  Each warp then arrives on the even CTA's sf_ready[s] (8 arrivals:
// 4 warps x 2 CTAs).  The odd CTA's arrivals are relaxed: tcgen05.wait::st has completed the
// warp's TMEM writes before it, so the arrival publishes no outstanding memory writes (a
// release arrival at cluster scope waits on the whole memory system and measured 2x slower
// overall); tcgen05.fence::before_thread_sync orders the writes before it, and the MMA
// thread's acquire wait and tcgen05.fence::after_thread_sync order its MMAs after.
//
// Warps: 0 producer, 1 TMEM allocator and (even CTA) MMA issuer, 2-3 idle, 4-7 scale
// warps, 8-15 epilogue.  setmaxnreg gives the epilogue warpgroups 192 registers a thread
// and the others 48 / 72, within the 512 x 128 the block is launched with.
//   full[s]     (even CTA) count 1: the even producer arms it with both CTAs' operand bytes
//   sf_full[s]  (each CTA) count 1: its own producer arms it with its scale-block bytes
//   sf_ready[s] (even CTA) count 8: the scale warps of both CTAs
//   empty[s], tfull       (each CTA) count 1: the MMA commits, multicast to both CTAs
//   tempty    (even CTA)  one relaxed arrival per epilogue warp of each CTA (16)
template <bool NV>
struct Mx2Cfg {
  static constexpr int BM = 128;                 // rows per CTA (the pair tile has 256)
  static constexpr int BN = 256;                 // columns of the pair tile
  static constexpr int BK = 128;                 // bytes of K per stage
  static constexpr int BK_ELEMS = NV ? 256 : 128;
  static constexpr int KSTEPS = 4;
  static constexpr int A_BYTES = BM * 128;
  static constexpr int B_HALF = BN / 2;          // columns of B (NV: rows of B^T) in each CTA
  static constexpr int B_BYTES = 128 * 128;      // one box: 128 K x 128 columns, or 128 rows x 128 K bytes
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;  // 32 KB
  static constexpr int SETS = NV ? 4 : 1;
  static constexpr int SF_BLOCK = 512;
  static constexpr int SF_STAGE_BYTES = 3 * SETS * SF_BLOCK;
  static constexpr int STAGES = NV ? 5 : 6;
  static constexpr int SF_WARP0 = 4, EPI_WARP0 = 8, EPI_WARPS = 8;
  static constexpr int THREADS = 512;
  static constexpr int LAUNCH_REGS = 65536 / THREADS;  // 128
  static constexpr int REGS_CTRL = 48, REGS_SF = 72, REGS_EPI = 192;
  static constexpr int TMEM_COLS = 512;
  static constexpr int SFA_COLS = 4 * SETS;
  static constexpr int SF_COL0 = BN, SF_COLS = SFA_COLS + 8 * SETS;
  static constexpr int NBARS = 4 * STAGES + 3;   // full, empty, sf_full, sf_ready, tfull, tempty, drain
  static constexpr int SMEM = STAGES * (STAGE_BYTES + SF_STAGE_BYTES) + NBARS * 8 + 16 + 1024;
  static_assert(SF_COL0 + STAGES * SF_COLS <= TMEM_COLS, "TMEM budget");
  static_assert(SMEM <= 227 * 1024, "shared memory budget");
  static_assert(128 * REGS_CTRL + 128 * REGS_SF + 256 * REGS_EPI <= THREADS * LAUNCH_REGS, "register split");
};

template <uint32_t AB_FMT, bool NV>
__global__ void __launch_bounds__(Mx2Cfg<NV>::THREADS, 1)
    gemm_mx2_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmXA, const __grid_constant__ CUtensorMap tmXB,
                    const GemmParams p) {
  using Cfg = Mx2Cfg<NV>;
  constexpr int S = Cfg::STAGES;
  constexpr uint32_t IDESC = mx_idesc<NV>(AB_FMT, Cfg::BN, 2 * Cfg::BM);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sf_base = smem + S * Cfg::STAGE_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sf_base + S * Cfg::SF_STAGE_BYTES);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + Cfg::NBARS);
  uint32_t* abort_flag = tmem_slot + 1;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const uint32_t rank = cluster_ctarank();
  const int rank_i = static_cast<int>(rank);
  const int pair = blockIdx.x >> 1;
  const int num_pairs = gridDim.x >> 1;
  auto full_bar = [&](int s) { return smem_addr(bars + s); };
  auto empty_bar = [&](int s) { return smem_addr(bars + S + s); };
  auto sf_full_bar = [&](int s) { return smem_addr(bars + 2 * S + s); };
  auto sf_ready_bar = [&](int s) { return smem_addr(bars + 3 * S + s); };
  const uint32_t tfull_bar = smem_addr(bars + 4 * S);
  const uint32_t tempty_bar = smem_addr(bars + 4 * S + 1);
  const uint32_t drain_bar = smem_addr(bars + 4 * S + 2);

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
      mbar_init(sf_full_bar(s), 1);
      mbar_init(sf_ready_bar(s), 8);
    }
    mbar_init(tfull_bar, 1);
    mbar_init(tempty_bar, 2 * Cfg::EPI_WARPS);
    mbar_init(drain_bar, 1);
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
  const int num_m2 = (p.M + 2 * Cfg::BM - 1) / (2 * Cfg::BM);
  const int num_n = (p.N + Cfg::BN - 1) / Cfg::BN;
  const int num_tiles = num_m2 * num_n;
  const int KB = (p.K + Cfg::BK_ELEMS - 1) / Cfg::BK_ELEMS;
  const int KBw = mx_words(p.K, NV);  // scale words per row

  if (warp == 0 && lane == 0 && pair < num_tiles) {
    int mb, nb;
    tile_coords(pair, num_m2, num_n, p.group_m, mb, nb);
    const int pre = KB < S ? KB : S;
    for (int kb = 0; kb < pre; ++kb) {
      tma_prefetch_l2(&tmA, kb * Cfg::BK, mb * 2 * Cfg::BM + Cfg::BM * rank_i);
      if (NV)
        tma_prefetch_l2(&tmB, kb * Cfg::BK, nb * Cfg::BN + Cfg::B_HALF * rank_i);
      else
        tma_prefetch_l2(&tmB, nb * Cfg::BN + Cfg::B_HALF * rank_i, kb * Cfg::BK);
    }
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");

  if (warp < Cfg::SF_WARP0) {
    regs_dec<Cfg::REGS_CTRL>();  // warpgroup 0: producer, MMA issuer, two idle warps
  } else if (warp < Cfg::EPI_WARP0) {
    regs_dec<Cfg::REGS_SF>();
  } else {
    regs_inc<Cfg::REGS_EPI>();
  }

  if (warp < Cfg::SF_WARP0) {
  if (warp == 0) {
    // ---------------------------------------------------------------- producer (each CTA)
    if (lane == 0) {
      tma_prefetch_desc(&tmA);
      tma_prefetch_desc(&tmB);
      tma_prefetch_desc(&tmXA);
      tma_prefetch_desc(&tmXB);
      uint32_t it = 0;
      bool ok = true;
      for (int u = pair; u < num_tiles && ok; u += num_pairs) {
        int mb, nb;
        tile_coords(u, num_m2, num_n, p.group_m, mb, nb);
        const int ablk = 2 * mb + rank_i;  // this CTA's 128-row block of A
        for (int kb = 0; kb < KB; ++kb) {
          const int s = it % S;
          if (!wait_bounded(empty_bar(s), ((it / S) & 1u) ^ 1u, wctx, kRoleProducer)) {
            ok = false;
            break;
          }
          const uint32_t cfull = mapa_cluster(full_bar(s), 0);
          uint8_t* a_s = smem + s * Cfg::STAGE_BYTES;
          uint8_t* sf = sf_base + s * Cfg::SF_STAGE_BYTES;
          if (rank == 0) mbar_arrive_expect_tx(full_bar(s), 2 * Cfg::STAGE_BYTES);
          mbar_arrive_expect_tx(sf_full_bar(s), Cfg::SF_STAGE_BYTES);
          tma_load_2d_pair(smem_addr(a_s), &tmA, cfull, kb * Cfg::BK, ablk * Cfg::BM);
          if (NV)  // this CTA's 128 rows of B^T (K-major)
            tma_load_2d_pair(smem_addr(a_s + Cfg::A_BYTES), &tmB, cfull, kb * Cfg::BK,
                             nb * Cfg::BN + Cfg::B_HALF * rank_i);
          else
            tma_load_2d_pair(smem_addr(a_s + Cfg::A_BYTES), &tmB, cfull, nb * Cfg::BN + Cfg::B_HALF * rank_i,
                             kb * Cfg::BK);
          tma_load_2d(smem_addr(sf), &tmXA, sf_full_bar(s), 0, (ablk * KBw + Cfg::SETS * kb) * 2);
          tma_load_2d(smem_addr(sf + Cfg::SETS * Cfg::SF_BLOCK), &tmXB, sf_full_bar(s), 0,
                      (nb * KBw + Cfg::SETS * kb) * 4);
          ++it;
        }
      }
      if (!ok) {  // copies still in flight: the even CTA's full barriers see both CTAs' operands
        for (uint32_t j = (it > static_cast<uint32_t>(S) ? it - S : 0u); j < it; ++j) {
          if (rank == 0) wait_drain(full_bar(j % S), (j / S) & 1u, p.timeout_ns);
          wait_drain(sf_full_bar(j % S), (j / S) & 1u, p.timeout_ns);
        }
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer (even CTA)
    if (lane == 0 && rank == 0) {
      uint32_t it = 0, tiles = 0;
      bool ok = true;
      for (int u = pair; u < num_tiles && ok; u += num_pairs) {
        if (!wait_bounded(tempty_bar, (tiles & 1u) ^ 1u, wctx, kRoleMma)) break;
        tc_fence_after();
        for (int kb = 0; kb < KB; ++kb) {
          const int s = it % S;
          if (!wait_bounded(full_bar(s), (it / S) & 1u, wctx, kRoleMma) ||
              !wait_bounded_cluster(sf_ready_bar(s), (it / S) & 1u, wctx, kRoleMma)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sf_t = tmem_base + Cfg::SF_COL0 + s * Cfg::SF_COLS;
          const uint32_t a_base = smem_addr(smem + s * Cfg::STAGE_BYTES);
          const uint32_t b_base = a_base + Cfg::A_BYTES;
#pragma unroll
          for (int kk = 0; kk < Cfg::KSTEPS; ++kk) {
            const uint64_t adesc = smem_desc_sw128(a_base + kk * 32, 16, 1024);
            const uint64_t bdesc = NV ? smem_desc_sw128(b_base + kk * 32, 16, 1024)
                                      : smem_desc_sw128(b_base + kk * 32 * 128, Cfg::B_BYTES, 1024);
            const uint32_t acc = (kb > 0 || kk > 0) ? 1u : 0u;
            if (NV)
              mma_nvf4_pair(tmem_base, adesc, bdesc, IDESC, sf_t + 4 * kk, sf_t + Cfg::SFA_COLS + 8 * kk, acc);
            else
              mma_mxf8_pair(tmem_base, adesc, bdesc, mma_idesc<NV>(IDESC, kk), sf_t, sf_t + Cfg::SFA_COLS, acc);
          }
          mma_commit_pair_mc(empty_bar(s), 0x3);
          ++it;
        }
        if (!ok) break;
        mma_commit_pair_mc(tfull_bar, 0x3);
        ++tiles;
      }
      mma_commit_pair(drain_bar);
      wait_drain(drain_bar, 0u, p.timeout_ns);
    }
  }
  } else if (warp < Cfg::EPI_WARP0) {
    // ---------------------------------------------------------------- scale warps (each CTA)
    const int q = warp & 3;  // the TMEM lane quarter this warp may access
    const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
    const uint32_t ready0 = rank == 0 ? 0u : mapa_cluster(sf_ready_bar(0), 0);
    uint32_t it = 0;
    for (int u = pair; u < num_tiles; u += num_pairs) {
      bool ok = true;
      for (int kb = 0; kb < KB; ++kb) {
        const int s = it % S;
        bool w = wait_bounded(sf_full_bar(s), (it / S) & 1u, wctx, kRoleScales);
        if (!__all_sync(0xffffffffu, w)) {
          ok = false;
          break;
        }
        const uint8_t* sf = sf_base + s * Cfg::SF_STAGE_BYTES;
        const uint32_t col = tmem_base + lane_base + Cfg::SF_COL0 + s * Cfg::SF_COLS;
        // row `lane` of A's blocks (one per MMA set), then of B's (two per set)
        uint32_t a[4 * Cfg::SETS], b[8 * Cfg::SETS];
#pragma unroll
        for (int g = 0; g < 3 * Cfg::SETS; ++g) {
          const uint4 v = *reinterpret_cast<const uint4*>(sf + g * Cfg::SF_BLOCK + lane * 16);
          uint32_t* d = g < Cfg::SETS ? a + 4 * g : b + 4 * (g - Cfg::SETS);
          d[0] = v.x;
          d[1] = v.y;
          d[2] = v.z;
          d[3] = v.w;
        }
        if constexpr (NV) {
          tmem_st_x16(col, a);
          tmem_st_x32(col + Cfg::SFA_COLS, b);
        } else {
          tmem_st_x4(col, a);
          tmem_st_x8(col + Cfg::SFA_COLS, b);
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (rank == 0)
            mbar_arrive(sf_ready_bar(s));
          else
            mbar_arrive_cluster_relaxed(ready0 + 8u * static_cast<uint32_t>(s));
        }
        ++it;
      }
      if (!ok) break;
    }
  } else {
    // ---------------------------------------------------------------- epilogue (each CTA)
    const int ew = warp - Cfg::EPI_WARP0;
    const int q = warp & 3;
    const int h = ew >> 2;
    const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
    uint32_t tiles = 0;
    for (int u = pair; u < num_tiles; u += num_pairs) {
      int mb, nb;
      tile_coords(u, num_m2, num_n, p.group_m, mb, nb);
      const int m = mb * 2 * Cfg::BM + Cfg::BM * rank_i + q * 32 + lane;
      const int ncol0 = nb * Cfg::BN + h * (Cfg::BN / 2);
      bool w = wait_bounded(tfull_bar, tiles & 1u, wctx, kRoleEpilogue);
      w = __all_sync(0xffffffffu, w);
      if (!w) break;
      tc_fence_after();
      uint32_t v[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld_x32(tmem_base + lane_base + h * (Cfg::BN / 2) + c * 32, v[c]);
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld_wait(v[c]);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster_relaxed(mapa_cluster(tempty_bar, 0));
      float acc[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int j = 0; j < 32; ++j) acc[c][j] = __uint_as_float(v[c][j]);
      epilogue_rows<4>(p, m, ncol0, acc);
      ++tiles;
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

// Tensor maps of the operands and of the two scale-block arrays (16-byte rows).  MX: A M x K
// bytes, B K x N (N-major boxes of 128 columns).  NVFP4: A M x K/2 bytes, B given as B^T,
// N x K/2 bytes (K-major boxes of b_rows rows); pitches in bytes.
template <bool NV>
bool mx_maps(const GemmArgs& a, int b_box, CUtensorMap* tmA, CUtensorMap* tmB, CUtensorMap* tmXA,
             CUtensorMap* tmXB) {
  const int64_t kbytes = NV ? a.K / 2 : a.K;
  const int64_t KBw = mx_words(a.K, NV);
  const int sets = NV ? 4 : 1;
  // the blocks of a stage are contiguous: fetched as rows of 256 bytes (2 per 128-row block
  // of A, 4 per 256-column block of B), which keeps the number of TMA rows per stage small
  const int64_t xa_rows = ((a.M + 127) / 128) * KBw * 2;
  const int64_t xb_rows = ((a.N + 255) / 256) * KBw * 4;
  const CUtensorMapDataType u8 = CU_TENSOR_MAP_DATA_TYPE_UINT8;
  const bool b_ok = NV ? make_tensor_map_2d(tmB, a.B, u8, 1, a.N, kbytes, a.ldb, 128, b_box)
                       : make_tensor_map_2d(tmB, a.B, u8, 1, a.K, a.N, a.ldb, b_box, 128);
  return b_ok && make_tensor_map_2d(tmA, a.A, u8, 1, a.M, kbytes, a.lda, 128, 128) &&
         make_tensor_map_2d(tmXA, a.mx_sat, u8, 1, xa_rows, 256, 256, 256, 2 * sets, CU_TENSOR_MAP_SWIZZLE_NONE) &&
         make_tensor_map_2d(tmXB, a.mx_sbt, u8, 1, xb_rows, 256, 256, 256, 4 * sets, CU_TENSOR_MAP_SWIZZLE_NONE);
}

template <uint32_t F, bool NV>
ll_status run_mx(const GemmArgs& a, const LaunchCtx& ctx) {
  using Cfg = MxCfg<NV>;
  auto kern = gemm_mx_kernel<F, NV>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM) != cudaSuccess) {
    cudaGetLastError();
    return LL_ERR_CUDA;
  }
  CUtensorMap tmA, tmB, tmXA, tmXB;
  if (!mx_maps<NV>(a, Cfg::B_BOX_N, &tmA, &tmB, &tmXA, &tmXB)) return LL_ERR_CUDA;
  const GemmParams p = make_gemm_params(a, ctx);
  const int num_tiles = ((a.M + Cfg::BM - 1) / Cfg::BM) * ((a.N + Cfg::BN - 1) / Cfg::BN);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_tiles < ctx.num_sms ? num_tiles : ctx.num_sms);
  cfg.blockDim = dim3(Cfg::THREADS);
  cfg.dynamicSmemBytes = Cfg::SMEM;
  cfg.stream = ctx.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kern, tmA, tmB, tmXA, tmXB, p) != cudaSuccess) {
    cudaGetLastError();
    return LL_ERR_CUDA;
  }
  return LL_OK;
}

template <uint32_t F, bool NV>
ll_status run_mx2(const GemmArgs& a, const LaunchCtx& ctx) {
  using Cfg = Mx2Cfg<NV>;
  auto kern = gemm_mx2_kernel<F, NV>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM) != cudaSuccess) {
    cudaGetLastError();
    return LL_ERR_CUDA;
  }
  // the kernel's setmaxnreg split needs the block launched with LAUNCH_REGS registers a
  // thread (an increase beyond what the block holds would never be granted)
  static int launch_regs = 0;
  if (launch_regs == 0) {
    cudaFuncAttributes fa;
    if (cudaFuncGetAttributes(&fa, kern) != cudaSuccess) {
      cudaGetLastError();
      return LL_ERR_CUDA;
    }
    launch_regs = fa.numRegs;
  }
  if (launch_regs * Cfg::THREADS < 128 * Cfg::REGS_CTRL + 128 * Cfg::REGS_SF + 256 * Cfg::REGS_EPI)
    return LL_ERR_UNSUPPORTED;
  CUtensorMap tmA, tmB, tmXA, tmXB;
  if (!mx_maps<NV>(a, Cfg::B_HALF, &tmA, &tmB, &tmXA, &tmXB)) return LL_ERR_CUDA;
  const GemmParams p = make_gemm_params(a, ctx);
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
  static int max_pairs[2][64] = {};
  if (ctx.device < 0 || ctx.device >= 64) return LL_ERR_NO_DEVICE;
  int& mp = max_pairs[NV ? 1 : 0][ctx.device];
  if (mp == 0) {
    cfg.gridDim = dim3(2 * (ctx.num_sms / 2));
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n <= 0) {
      cudaGetLastError();
      n = ctx.num_sms / 2;
    }
    mp = n;
  }
  const int tiles = ((a.M + 2 * Cfg::BM - 1) / (2 * Cfg::BM)) * ((a.N + Cfg::BN - 1) / Cfg::BN);
  cfg.gridDim = dim3(2 * (tiles < mp ? tiles : mp));
  if (cudaLaunchKernelEx(&cfg, kern, tmA, tmB, tmXA, tmXB, p) != cudaSuccess) {
    cudaGetLastError();
    return LL_ERR_CUDA;
  }
  return LL_OK;
}

}  // namespace

size_t mx_scale_block_bytes(int M, int N, int K, bool nv, size_t* a_bytes) {
  const size_t KBw = static_cast<size_t>(mx_words(K, nv));
  const size_t xa = static_cast<size_t>((M + 127) / 128) * KBw * 512;
  const size_t xb = static_cast<size_t>((N + 255) / 256) * KBw * 1024;
  if (a_bytes) *a_bytes = xa;
  return xa + xb;
}

ll_status launch_mx_scale_tiles(const GemmArgs& a, uint8_t* xa, uint8_t* xb, const LaunchCtx& ctx) {
  const bool nv = a.nvf4 != 0;
  const int KBw = mx_words(a.K, nv);                         // 4-code words per row
  const int nkb = nv ? (a.K + 15) / 16 : (a.K + 31) / 32;    // codes per row
  const uint32_t neutral = nv ? 0x38u : 0x7Fu;               // 1.0 as UE4M3 / E8M0
  const int G = (KBw + 3) / 4;
  mx_scale_tile_kernel<<<dim3((a.M + 127) / 128, G), 128, 0, ctx.stream>>>(a.mx_sa, a.ld_mx_sa, a.M, nkb, KBw, 0,
                                                                          neutral, xa);
  if (cudaGetLastError() != cudaSuccess) return LL_ERR_CUDA;
  // B: every 128-column block of each 256-column tile (a block past N gets neutral codes)
  mx_scale_tile_kernel<<<dim3(2 * ((a.N + 255) / 256), G), 128, 0, ctx.stream>>>(a.mx_sb, a.ld_mx_sb, a.N, nkb, KBw,
                                                                                 1, neutral, xb);
  return cudaGetLastError() == cudaSuccess ? LL_OK : LL_ERR_CUDA;
}

ll_status launch_gemm_mx(const GemmArgs& a, const LaunchCtx& ctx) {
  // CTA pairs once there are enough 256 x 256 tiles to occupy a quarter of the SM pairs;
  // the one-CTA kernel below that
  const int pair_tiles = ((a.M + 255) / 256) * ((a.N + 255) / 256);
  const bool pair = pair_tiles >= ctx.num_sms / 4;
  if (a.nvf4) return pair ? run_mx2<fmt_pair(1, 1), true>(a, ctx) : run_mx<fmt_pair(1, 1), true>(a, ctx);
  const bool a5 = a.in_type == LL_IN_E5M2, b5 = a.b_type == LL_IN_E5M2;
  if (pair) {
    if (!a5 && !b5) return run_mx2<fmt_pair(0, 0), false>(a, ctx);
    if (a5 && b5) return run_mx2<fmt_pair(1, 1), false>(a, ctx);
    if (!a5) return run_mx2<fmt_pair(0, 1), false>(a, ctx);
    return run_mx2<fmt_pair(1, 0), false>(a, ctx);
  }
  if (!a5 && !b5) return run_mx<fmt_pair(0, 0), false>(a, ctx);
  if (a5 && b5) return run_mx<fmt_pair(1, 1), false>(a, ctx);
  if (!a5) return run_mx<fmt_pair(0, 1), false>(a, ctx);
  return run_mx<fmt_pair(1, 0), false>(a, ctx);
}

}  // namespace ll
