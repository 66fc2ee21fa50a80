// Persistent warp-specialised bf16 GEMM on the 5th-generation tensor cores.
//
//   C[M, N] = A[M, K] . W[N, K]^T, fp32 accumulation in tensor memory, then a
//   fused epilogue (bias, GELU, gated residual into the fp32 stream, or the
//   head-major Q/K/V scatter with rotary embedding).
//
// Roles (320 threads): warp 0 issues TMA loads of 128x64 A and BNx64 W tiles
// (128-byte swizzle) into a STAGES-deep shared-memory ring; warp 1 issues
// tcgen05.mma (M=128, N=BN, K=16) from one thread into one of two TMEM
// accumulators; warps 2-9 drain the other accumulator through tcgen05.ld
// (warp w reads TMEM lanes 32*(w%4)..+31 = its 32 rows, two warps per lane
// quadrant splitting the column chunks) and run the epilogue,
// so the epilogue of tile i overlaps the main loop of tile i+1.  One CTA per
// SM walks the tile list with stride gridDim.x; tiles are ordered N-fastest so
// CTAs running together share the same A rows through L2.
//
// Every mbarrier wait is bounded (common.cuh); on a timeout the CTA records
// the failure in *err, winds down, waits for its own copies and MMAs in
// flight, frees its TMEM and exits.
#include "epilogue.cuh"
#include "tmap.h"

namespace dit {

// Warps 2 .. 2+EPI_WARPS-1 drain the accumulator; two per TMEM lane quadrant,
// each taking every other 32-column chunk of the tile.
constexpr int EPI_WARPS = 8;
constexpr int GEMM_THREADS = 32 * (2 + EPI_WARPS);

template <int BN>
struct TcGemmCfg {
  static constexpr int BM = 128, BK = 64;
  static constexpr int A_BYTES = BM * BK * 2;
  static constexpr int B_BYTES = BN * BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int STAGES = (BN == 256) ? 4 : (BN == 128 ? 6 : 8);
  static constexpr int TMEM_COLS = (2 * BN < 32) ? 32 : 2 * BN;
  static constexpr int BAR_BYTES = 256;
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + BAR_BYTES + 1024;
  static constexpr uint32_t IDESC = umma_idesc_bf16(BM, BN, false);
};

template <int BN>
__global__ void __launch_bounds__(GEMM_THREADS, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, int64_t M,
                   int N, int K, EpiParams ep, int* err) {
  using C = TcGemmCfg<BN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::STAGES * C::STAGE_BYTES);
  uint64_t* empty = full + C::STAGES;
  uint64_t* tfull = empty + C::STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], EPI_WARPS);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) tmem_alloc(tmem_slot, C::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const int m_tiles = (int)((M + C::BM - 1) / C::BM);
  const int n_tiles = (N + BN - 1) / BN;
  const int k_blocks = (K + C::BK - 1) / C::BK;
  const int num_tiles = m_tiles * n_tiles;

  if (warp == 0) {
    // ------------------------------------------------ TMA producer (one thread)
    if (lane == 0) {
      uint32_t stage = 0, phase = 0;
      int issued[C::STAGES];
#pragma unroll
      for (int s = 0; s < C::STAGES; ++s) issued[s] = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
        const int mb = tile / n_tiles, nb = tile - mb * n_tiles;
        for (int kb = 0; kb < k_blocks; ++kb) {
          ok = mbar_wait(&empty[stage], phase ^ 1, abort_flag, err, 11);
          if (!ok) break;
          uint8_t* sa = smem + stage * C::STAGE_BYTES;
          mbar_arrive_expect_tx(&full[stage], C::STAGE_BYTES);
          tma_load_2d(sa, &tmA, &full[stage], kb * C::BK, mb * C::BM);
          tma_load_2d(sa + C::A_BYTES, &tmB, &full[stage], kb * C::BK, nb * BN);
          ++issued[stage];
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      if (!ok) {
        // wind down: let every copy this thread started land before the CTA exits
        volatile int no_abort = 0;
        for (int s = 0; s < C::STAGES; ++s)
          if (issued[s] > 0) mbar_wait(&full[s], (uint32_t)((issued[s] - 1) & 1), &no_abort, nullptr, 0);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer (one thread)
    // The whole role runs on lane 0: a warp that diverges and reconverges
    // around every MMA burst costs the tensor pipe a large share of its rate.
    if (lane == 0) {
      uint32_t stage = 0, phase = 0, local = 0;
      bool ok = true;
      const uint64_t a_desc = umma_desc_sw128(smem_u32(smem), 16, 1024);
      const uint64_t b_desc = umma_desc_sw128(smem_u32(smem) + C::A_BYTES, 16, 1024);
      for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x, ++local) {
        const uint32_t acc = local & 1, aphase = (local >> 1) & 1;
        ok = mbar_wait(&tempty[acc], aphase ^ 1, abort_flag, err, 12);
        if (!ok) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int kb = 0; kb < k_blocks; ++kb) {
          ok = mbar_wait(&full[stage], phase, abort_flag, err, 13);
          if (!ok) break;
          tc_fence_after();
          const uint64_t ad = umma_desc_add(a_desc, stage * C::STAGE_BYTES);
          const uint64_t bd = umma_desc_add(b_desc, stage * C::STAGE_BYTES);
#pragma unroll
          for (int k = 0; k < C::BK / 16; ++k)
            umma_ss(d_tmem, umma_desc_add(ad, k * 32), umma_desc_add(bd, k * 32), C::IDESC, (kb | k) != 0);
          umma_commit(&empty[stage]);
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        umma_commit(&tfull[acc]);
      }
      // all MMAs issued by this thread complete before TMEM is released
      umma_commit(drain);
      volatile int no_abort = 0;
      mbar_wait(drain, 0, &no_abort, nullptr, 0);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------ epilogue warps
    const int q = warp & 3;
    const int half = (warp - 2) / 4;
    const int row_in_tile = q * 32 + lane;
    uint32_t local = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x, ++local) {
      const uint32_t acc = local & 1, aphase = (local >> 1) & 1;
      ok = __all_sync(0xffffffffu, mbar_wait(&tfull[acc], aphase, abort_flag, err, 14));
      if (!ok) break;
      tc_fence_after();
      const int mb = tile / n_tiles, nb = tile - mb * n_tiles;
      const int64_t row = (int64_t)mb * C::BM + row_in_tile;
#pragma unroll 1
      for (int c = half; c < BN / 32; c += 2) {
        uint32_t r[32];
        tmem_ld32(tmem_base + acc * BN + c * 32 + ((uint32_t)(q * 32) << 16), r);
        tmem_ld_wait();
        const int col0 = nb * BN + c * 32;
        if (row < M && col0 < N) {
          float v[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
          epilogue_chunk<__nv_bfloat16, 32>(ep, row, col0, v);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[acc]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

template <int BN>
static cudaError_t launch_gemm_tc(const GemmArgs& g, int* err, int num_sms, cudaStream_t s) {
  using C = TcGemmCfg<BN>;
  CUtensorMap ta, tb;
  const uint64_t da[2] = {(uint64_t)g.K, (uint64_t)g.M}, sa[1] = {(uint64_t)g.lda * 2};
  const uint32_t ba[2] = {64, 128};
  const uint64_t db[2] = {(uint64_t)g.K, (uint64_t)g.N}, sb[1] = {(uint64_t)g.K * 2};
  const uint32_t bb[2] = {64, (uint32_t)BN};
  if (!make_tmap_bf16(&ta, g.A, 2, da, sa, ba) || !make_tmap_bf16(&tb, g.W, 2, db, sb, bb))
    return cudaErrorInvalidValue;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e =
        cudaFuncSetAttribute(gemm_tc_kernel<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const int64_t tiles = ((g.M + 127) / 128) * ((g.N + BN - 1) / BN);
  const int grid = (int)(tiles < num_sms ? tiles : num_sms);
  gemm_tc_kernel<BN><<<grid, GEMM_THREADS, C::SMEM_BYTES, s>>>(ta, tb, g.M, g.N, g.K, g.epi, err);
  return cudaGetLastError();
}

cudaError_t gemm_bf16_tc(const GemmArgs& g, int* err, int num_sms, cudaStream_t s) {
  if (g.M == 0 || g.N == 0) return cudaSuccess;
  // alignment rules of the tensor maps: 16-byte rows and bases
  if ((g.K % 8) || (g.lda % 8) || (reinterpret_cast<uintptr_t>(g.A) & 15) || (reinterpret_cast<uintptr_t>(g.W) & 15))
    return cudaErrorInvalidValue;
  if (g.N % 256 == 0) return launch_gemm_tc<256>(g, err, num_sms, s);
  if (g.N % 128 == 0) return launch_gemm_tc<128>(g, err, num_sms, s);
  return launch_gemm_tc<64>(g, err, num_sms, s);
}

}  // namespace dit
