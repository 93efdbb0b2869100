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
// One persistent CTA per SM walks 128 x 256 output tiles in the grouped order.  Roles:
//   warp 0      operand producer: TMA copies of A (128 rows x 128 K, K-major) and B (128 K
//               x 256 columns, N-major), 128-byte swizzle, into a 4-stage ring.
//   warp 2      scale blocks: every four stages a TMA copy brings the next 16 K blocks of
//               scale codes of the tile's 128 rows of A and 256 columns of B (their own
//               K-block-contiguous layout; three group buffers, requested two groups
//               ahead); the 32 lanes reorder each stage's codes into three 32 x 16-byte
//               blocks (row r of a block holds at byte 4j + b the code of item 32j + r for
//               K block b) in the stage's slot and arrive on its full barrier.
//   warp 1      TMEM allocator and MMA issuer.  Per stage, three tcgen05.cp copies put the
//               scale blocks into TMEM (replicated over the four lane quarters), then four
//               K = 32 MMAs each select their K block's byte of the scale words through
//               the scale-factor IDs of the instruction descriptor.
//   warps 3-10  epilogue.  They drain the tile's 128 x 256 FP32 accumulator from TMEM into
//               registers (32 rows x 128 columns per warp), hand TMEM back at once so the
//               next tile's MMAs run, then apply alpha / beta and store D from registers.
// TMEM: the accumulator in columns 0-255; stage s's scales in columns 256 + 16 s: A's in
// the first 4 (row m at lane m, column m / 32), B's in the next 8 (column n at lanes
// 32 q + n % 32 of every quarter q, column 4 + n / 32).  Every wait is bounded; on expiry
// the CTA records LL_ERR_DEVICE_TIMEOUT, drains its copies and MMAs, frees TMEM and exits.
#include <cstring>

#include "gemm_common.cuh"

namespace ll {

namespace {

struct MxCfg {
  static constexpr int BM = 128, BN = 256;
  static constexpr int BK = 128;                 // K elements (bytes) per stage
  static constexpr int UMMA_K = 32, KSTEPS = 4;  // one E8M0 K block per MMA
  static constexpr int A_BYTES = BM * 128;
  static constexpr int B_BOX_N = 128, B_BOXES = BN / B_BOX_N, B_BOX_BYTES = BK * 128;
  static constexpr int STAGE_BYTES = A_BYTES + B_BOXES * B_BOX_BYTES;  // 48 KB
  static constexpr int SF_BLOCK = 512;                                 // 32 rows x 16 bytes
  static constexpr int SF_STAGE_BYTES = 3 * SF_BLOCK;                  // A, B columns 0-127, 128-255
  static constexpr int STAGES = 4;
  // scale codes arrive by TMA as boxes of 16 K blocks (four stages) x the tile's rows of A
  // (128) and columns of B (256), in their natural K-block-contiguous layout, into two
  // group buffers; the producer reorders each stage's words into the tcgen05.cp blocks
  static constexpr int SG_KB = 16;                    // K blocks per group
  static constexpr int SG_A = BM * SG_KB, SG_B = BN * SG_KB;
  static constexpr int SG_BYTES = SG_A + SG_B;        // 6 KB
  static constexpr int SG_BUFS = 3;                   // groups requested two ahead
  static constexpr int EPI_WARP0 = 3, EPI_WARPS = 8;
  static constexpr int EPI_THREADS = 32 * EPI_WARPS;
  static constexpr int THREADS = 32 * (EPI_WARP0 + EPI_WARPS);
  static constexpr int TMEM_COLS = 512;
  static constexpr int SF_COL0 = BN, SF_COLS = 16;
  static constexpr int NBARS = 2 * STAGES + 3 + SG_BUFS;  // full, empty, tfull, tempty, drain, sgfull
  static constexpr int SMEM = STAGES * (STAGE_BYTES + SF_STAGE_BYTES) + SG_BUFS * SG_BYTES + NBARS * 8 + 16 + 1024;
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

template <uint32_t AB_FMT>
__global__ void __launch_bounds__(MxCfg::THREADS, 1)
    gemm_mx_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmSA, const __grid_constant__ CUtensorMap tmSB,
                   const GemmParams p) {
  using Cfg = MxCfg;
  constexpr int S = Cfg::STAGES;
  constexpr uint32_t IDESC = make_idesc_mx(AB_FMT, Cfg::BN, Cfg::BM);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sf_base = smem + S * Cfg::STAGE_BYTES;
  uint8_t* sg_base = sf_base + S * Cfg::SF_STAGE_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sg_base + Cfg::SG_BUFS * Cfg::SG_BYTES);
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
  auto sgfull_bar = [&](int b) { return smem_addr(bars + 2 * S + 3 + b); };

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full_bar(s), 2);  // the operand copies (with their bytes) and the scale blocks
      mbar_init(empty_bar(s), 1);
    }
    mbar_init(tfull_bar, 1);
    mbar_init(tempty_bar, Cfg::EPI_THREADS);
    mbar_init(drain_bar, 1);
    for (int b = 0; b < Cfg::SG_BUFS; ++b) mbar_init(sgfull_bar(b), 1);
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
  const int KB = (p.K + Cfg::BK - 1) / Cfg::BK;  // stages per tile
  const int NG = (KB + 3) / 4;                   // scale groups per tile (16 K blocks each)

  // programmatic dependent launch: L2 prefetch of the first ring of operand tiles, then
  // the wait for the previous kernel of the stream (scales, C and D come after it)
  if (warp == 0 && lane == 0 && static_cast<int>(blockIdx.x) < num_tiles) {
    int mb, nb;
    tile_coords(blockIdx.x, num_m, num_n, p.group_m, mb, nb);
    const int pre = KB < S ? KB : S;
    for (int kb = 0; kb < pre; ++kb) {
      tma_prefetch_l2(&tmA, kb * Cfg::BK, mb * Cfg::BM);
      for (int j = 0; j < Cfg::B_BOXES; ++j) tma_prefetch_l2(&tmB, nb * Cfg::BN + j * Cfg::B_BOX_N, kb * Cfg::BK);
    }
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");

  if (warp == 0) {
    // ---------------------------------------------------------------- operand producer
    if (lane == 0) {
      tma_prefetch_desc(&tmA);
      tma_prefetch_desc(&tmB);
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
          mbar_arrive_expect_tx(full_bar(s), Cfg::STAGE_BYTES);
          tma_load_2d(smem_addr(a_s), &tmA, full_bar(s), kb * Cfg::BK, mb * Cfg::BM);
#pragma unroll
          for (int j = 0; j < Cfg::B_BOXES; ++j)
            tma_load_2d(smem_addr(b_s + j * Cfg::B_BOX_BYTES), &tmB, full_bar(s), nb * Cfg::BN + j * Cfg::B_BOX_N,
                        kb * Cfg::BK);
          ++it;
        }
      }
      if (!ok) {  // wait for the copies still in flight before the CTA can exit
        for (uint32_t j = (it > static_cast<uint32_t>(S) ? it - S : 0u); j < it; ++j)
          wait_drain(full_bar(j % S), (j / S) & 1u, p.timeout_ns);
      }
    }
  } else if (warp == 2) {
    // ---------------------------------------------------------------- scale blocks
    // This CTA's stages in order: stage i is K block i % KB of its (i / KB)-th tile.  Scale
    // group g (this CTA's g-th run of four stages of one tile) lands in buffer g % 3 and is
    // requested two groups ahead, so it is in place when its first stage comes.
    if (lane == 0) {
      tma_prefetch_desc(&tmSA);
      tma_prefetch_desc(&tmSB);
    }
    const int my_tiles = static_cast<int>(blockIdx.x) < num_tiles
                             ? (num_tiles - static_cast<int>(blockIdx.x) + static_cast<int>(gridDim.x) - 1) /
                                   static_cast<int>(gridDim.x)
                             : 0;
    const uint32_t total = static_cast<uint32_t>(my_tiles) * static_cast<uint32_t>(KB);
    const uint32_t groups = static_cast<uint32_t>(my_tiles) * static_cast<uint32_t>(NG);
    uint32_t g_requested = 0, g_waited = 0;  // scale groups requested / seen complete
    auto request_group = [&](uint32_t g) {  // lane 0
      if (g >= groups) return;
      g_requested = g + 1;
      int mb, nb;
      tile_coords(blockIdx.x + static_cast<int>(g / NG) * gridDim.x, num_m, num_n, p.group_m, mb, nb);
      const int x = static_cast<int>(g % NG) * Cfg::SG_KB;  // first K block (a multiple of 16 bytes)
      uint8_t* buf = sg_base + (g % Cfg::SG_BUFS) * Cfg::SG_BYTES;
      const uint32_t bar = sgfull_bar(g % Cfg::SG_BUFS);
      mbar_arrive_expect_tx(bar, Cfg::SG_BYTES);
      tma_load_2d(smem_addr(buf), &tmSA, bar, x, mb * Cfg::BM);
      tma_load_2d(smem_addr(buf + Cfg::SG_A), &tmSB, bar, x, nb * Cfg::BN);
    };
    if (lane == 0) {
      request_group(0);
      request_group(1);
    }
    bool ok = true;
    for (uint32_t i = 0; i < total && ok; ++i) {
      const int kb = static_cast<int>(i % KB);
      const uint32_t g = (i / KB) * NG + kb / 4;
      const int c = kb & 3;  // stage within the group
      const uint8_t* grp = sg_base + (g % Cfg::SG_BUFS) * Cfg::SG_BYTES;
      if (c == 0) {
        bool ok_g = wait_bounded(sgfull_bar(g % Cfg::SG_BUFS), (g / Cfg::SG_BUFS) & 1u, wctx, kRoleProducer);
        ok_g = __all_sync(0xffffffffu, ok_g);
        if (!ok_g) {
          ok = false;
          break;
        }
        g_waited = g + 1;
        fence_proxy_async_smem();  // every lane's reads of buffer (g + 2) % 3 (group g - 1) ...
        __syncwarp();
        if (lane == 0) request_group(g + 2);  // ... come before its refill
      }
      // this stage's words: K blocks 4c .. 4c + 3 of the group for row 32 j + lane of A and
      // column 32 j + lane of B (group rows are 16 bytes: K blocks 0-15 of the group)
      uint32_t w[12];
#pragma unroll
      for (int j = 0; j < 4; ++j) w[j] = *reinterpret_cast<const uint32_t*>(grp + (32 * j + lane) * 16 + 4 * c);
#pragma unroll
      for (int j = 0; j < 8; ++j)
        w[4 + j] = *reinterpret_cast<const uint32_t*>(grp + Cfg::SG_A + (32 * j + lane) * 16 + 4 * c);
      const int s = i % S;
      bool ok_w = wait_bounded(empty_bar(s), ((i / S) & 1u) ^ 1u, wctx, kRoleProducer);
      ok_w = __all_sync(0xffffffffu, ok_w);
      if (!ok_w) {
        ok = false;
        break;
      }
      uint8_t* sf = sf_base + s * Cfg::SF_STAGE_BYTES;
      *reinterpret_cast<uint4*>(sf + lane * 16) = make_uint4(w[0], w[1], w[2], w[3]);
      *reinterpret_cast<uint4*>(sf + Cfg::SF_BLOCK + lane * 16) = make_uint4(w[4], w[5], w[6], w[7]);
      *reinterpret_cast<uint4*>(sf + 2 * Cfg::SF_BLOCK + lane * 16) = make_uint4(w[8], w[9], w[10], w[11]);
      fence_proxy_async_smem();  // the generic-proxy writes, for tcgen05.cp's reads
      __syncwarp();
      if (lane == 0) mbar_arrive(full_bar(s));
    }
    if (!ok && lane == 0) {  // scale groups still in flight land before the CTA may exit
      for (uint32_t g = g_waited; g < g_requested; ++g)
        wait_drain(sgfull_bar(g % Cfg::SG_BUFS), (g / Cfg::SG_BUFS) & 1u, p.timeout_ns);
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
          tmem_cp_32x128b_x4(sf_t, smem_desc_plain16(sf_s));
          tmem_cp_32x128b_x4(sf_t + 4, smem_desc_plain16(sf_s + Cfg::SF_BLOCK));
          tmem_cp_32x128b_x4(sf_t + 8, smem_desc_plain16(sf_s + 2 * Cfg::SF_BLOCK));
          const uint32_t a_base = smem_addr(smem + s * Cfg::STAGE_BYTES);
          const uint32_t b_base = a_base + Cfg::A_BYTES;
#pragma unroll
          for (int kk = 0; kk < Cfg::KSTEPS; ++kk) {
            const uint64_t adesc = smem_desc_sw128(a_base + kk * 32, 16, 1024);
            const uint64_t bdesc = smem_desc_sw128(b_base + kk * Cfg::UMMA_K * 128, Cfg::B_BOX_BYTES, 1024);
            mma_mxf8(tmem_base, adesc, bdesc, IDESC | sf_ids(kk), sf_t, sf_t + 4, (kb > 0 || kk > 0) ? 1u : 0u);
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

template <uint32_t F>
ll_status run_mx(const GemmArgs& a, const LaunchCtx& ctx) {
  using Cfg = MxCfg;
  auto kern = gemm_mx_kernel<F>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM) != cudaSuccess) {
    cudaGetLastError();
    return LL_ERR_CUDA;
  }
  CUtensorMap tmA, tmB;
  if (!make_tensor_map_2d(&tmA, a.A, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, a.M, a.K, a.lda, Cfg::BK, Cfg::BM))
    return LL_ERR_CUDA;
  if (!make_tensor_map_2d(&tmB, a.B, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, a.K, a.N, a.ldb, Cfg::B_BOX_N, Cfg::BK))
    return LL_ERR_CUDA;
  // scale codes: K-block-contiguous rows with 16-byte-multiple pitches (repacked otherwise)
  const int64_t nkb = (a.K + 31) / 32;
  CUtensorMap tmSA, tmSB;
  if (!make_tensor_map_2d(&tmSA, a.mx_sa, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, a.M, nkb, a.ld_mx_sa, Cfg::SG_KB, Cfg::BM,
                          CU_TENSOR_MAP_SWIZZLE_NONE))
    return LL_ERR_CUDA;
  if (!make_tensor_map_2d(&tmSB, a.mx_sb, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, a.N, nkb, a.ld_mx_sb, Cfg::SG_KB, Cfg::BN,
                          CU_TENSOR_MAP_SWIZZLE_NONE))
    return LL_ERR_CUDA;
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
  if (cudaLaunchKernelEx(&cfg, kern, tmA, tmB, tmSA, tmSB, p) != cudaSuccess) {
    cudaGetLastError();
    return LL_ERR_CUDA;
  }
  return LL_OK;
}

}  // namespace

ll_status launch_gemm_mx(const GemmArgs& a, const LaunchCtx& ctx) {
  const bool a5 = a.in_type == LL_IN_E5M2, b5 = a.b_type == LL_IN_E5M2;
  if (!a5 && !b5) return run_mx<fmt_pair(0, 0)>(a, ctx);
  if (a5 && b5) return run_mx<fmt_pair(1, 1)>(a, ctx);
  if (!a5) return run_mx<fmt_pair(0, 1)>(a, ctx);
  return run_mx<fmt_pair(1, 0)>(a, ctx);
}

}  // namespace ll
