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
// quadrant taking alternate column units) and run the epilogue, so the
// epilogue of tile i overlaps the main loop of tile i+1.  Each epilogue warp
// stages a finished 32-row x 128-byte unit in its own swizzled 4 KB shared
// buffer and hands it to the TMA unit: a tiled store for bf16/fp32 outputs,
// a reduce-add into the fp32 stream for the gated residual (the SM never
// reads x), a 3-D store into [batch*head, token, channel] for the Q/K/V
// scatter.  Full 128-byte lines leave the SM instead of 16-byte pieces of 32
// rows per instruction, which keeps the L2 free for the operand stream.  (A
// head-major unit whose 32 rows cross a batch boundary is stored directly.)
// One CTA per
// SM walks the tile list with stride gridDim.x; tiles are ordered N-fastest so
// CTAs running together share the same A rows through L2.
//
// Widths that are multiples of 256 with main loops of 16 K blocks or more
// run on CTA pairs (clusters of two): a
// 256 x 256 tile per pair, one tcgen05.mma.cta_group::2 (M = 256) per K step
// issued by the leader CTA, each CTA loading its own 128 rows of A and 128 of
// the tile's 256 W rows.  The L2 then serves 32 KB per CTA and K block
// instead of 48 KB; operand delivery from L2 is what limits the 128 x 256
// single-CTA main loop once the epilogue's stores compete with it.  The
// epilogue is unchanged: each CTA drains its own 128 x 256 accumulator.
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

// F8: e4m3 operands (kind::f8f6f4); a K block is then 128 elements, the same
// 128 bytes per tile row as 64 bf16 elements, so the tiles, swizzle and
// descriptors are the same and only the MMA kind and K per MMA change.
//
// PAIR: the tile is 256 x BN and runs on a cluster of two CTAs (one
// tcgen05.mma.cta_group::2 of M = 256 per K step, issued by the leader).  Each
// CTA loads its own 128 rows of A and half of the tile's BN rows of W, so a
// CTA reads 32 KB per K block instead of 48 KB, and holds its 128 x BN part
// of the accumulator.
template <int BN, bool F8 = false, bool PAIR = false>
struct TcGemmCfg {
  static constexpr int BM = 128, BK = F8 ? 128 : 64;
  static constexpr int ESZ = F8 ? 1 : 2;
  static constexpr int BN_CTA = PAIR ? BN / 2 : BN;  // W rows one CTA loads per tile
  static constexpr int A_BYTES = BM * BK * ESZ;
  static constexpr int B_BYTES = BN_CTA * BK * ESZ;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int STAGES = PAIR ? 6 : (BN == 256) ? 4 : (BN == 128 ? 6 : 8);
  static constexpr int TMEM_COLS = (2 * BN < 32) ? 32 : 2 * BN;
  static constexpr int BAR_BYTES = 256;
  static constexpr int STG_BYTES = 32 * 128;  // one epilogue warp's staging unit
  static constexpr int STG_OFF = STAGES * STAGE_BYTES;
  static constexpr int BAR_OFF = STG_OFF + EPI_WARPS * STG_BYTES;
  static constexpr int SMEM_BYTES = BAR_OFF + BAR_BYTES + 1024;
  static constexpr int MMA_M = PAIR ? 2 * BM : BM;
  static constexpr uint32_t IDESC = F8 ? umma_idesc_e4m3(MMA_M, BN) : umma_idesc_bf16(MMA_M, BN, false);
  static constexpr int K_PER_MMA = F8 ? 32 : 16;  // 32 bytes of each row per MMA either way
};

// Output tensor maps of the TMA epilogue: m[0] = output (x for EPI_RESID,
// with m[1] the same x in whole-tile boxes for the L2 prefetch);
// EPI_HEADS: m[s] = section s as [B*H][seq_total][hd].
struct EpiMaps {
  CUtensorMap m[3];
};

// The problems of one launch: NP GEMMs with the same N and K, each with its
// own operands, row count and epilogue.  Their tile lists run back to back
// (problem 0 first), so the tiles of a small problem fill the last wave of a
// large one instead of running as a short launch of their own (the two
// streams of a dual-stream block: 8192 image rows and 1024 condition rows).
template <int NP>
struct GemmBatch {
  CUtensorMap tmA[NP];
  CUtensorMap tmB[NP];
  EpiMaps maps[NP];
  EpiParams ep[NP];
  int64_t M[NP];
  int m_tiles[NP];
  int tile_end[NP];  // end (exclusive) of problem p's tiles in the launch's tile list
  int group_n;       // n-tiles per column group (see tile_coords)
};

// Tile t of a problem with m_tiles row tiles -> (mb, nb).  Tiles run in
// column groups of gn n-tiles (the last group narrower), N-fastest within a
// group: the CTAs of a wave then read one group's W columns, which stay in L2
// while the group streams A, instead of every W column of the layer (an image
// FFN1 layer's W is 75 MB; in plain N-fastest order its launch read 1.27 GB
// from DRAM for 0.21 GB of operands).  gn = n_tiles is plain N-fastest order.
DIT_DEV void tile_coords(int t, int m_tiles, int n_tiles, int gn, int* mb, int* nb) {
  const int per_group = m_tiles * gn;
  const int g = t / per_group;
  const int within = t - g * per_group;
  const int rest = n_tiles - g * gn;
  const int width = rest < gn ? rest : gn;
  *mb = within / width;
  *nb = g * gn + (within - *mb * width);
}

// Problem of a launch-wide tile index; *t = the tile's index within it.
template <int NP>
DIT_DEV int locate_tile(const GemmBatch<NP>& P, int tile, int* t) {
  int p = 0;
#pragma unroll
  for (int i = 0; i + 1 < NP; ++i) p += tile >= P.tile_end[i] ? 1 : 0;
  *t = p ? tile - P.tile_end[p - 1] : tile;
  return p;
}

// Drain one accumulator tile through shared memory and TMA.  UW = columns per
// 128-byte unit (64 bf16 or 32 fp32).  The warp owns rows row0..row0+31 and
// units u = half, half+2, ...; it releases the accumulator (lane 0 calls
// release(), an arrival on the accumulator's tempty barrier) as soon as its
// last tcgen05.ld has completed.
template <int BN, int UW, class Release>
DIT_DEV void drain_tile_tma(const EpiParams& ep, const EpiMaps& maps, uint32_t tacc, int64_t row0, int64_t M, int N,
                            int nb, int half, uint8_t* stg, Release release, int* err) {
  constexpr int NU = BN / UW;
  const int lane = threadIdx.x & 31;
  const int64_t row = row0 + lane;
  // rows past M are computed from row M-1 (never stored) so every table read stays in range
  const int64_t vrow = row < M ? row : M - 1;
  if (half >= NU) {
    __syncwarp();
    if (lane == 0) release();
    return;
  }
#pragma unroll 1
  for (int u = half; u < NU; u += 2) {
    float v[UW];
    {
      uint32_t r[UW];
      tmem_ld32(tacc + u * UW, *reinterpret_cast<uint32_t(*)[32]>(&r[0]));
      if constexpr (UW == 64) tmem_ld32(tacc + u * UW + 32, *reinterpret_cast<uint32_t(*)[32]>(&r[32]));
      // no memory clobber: the epilogue's bias and scale loads may issue
      // while the tensor-memory load is in flight
      tmem_ld_wait_regs(*reinterpret_cast<uint32_t(*)[32]>(&r[0]));
      if constexpr (UW == 64) tmem_ld_wait_regs(*reinterpret_cast<uint32_t(*)[32]>(&r[32]));
#pragma unroll
      for (int j = 0; j < UW; ++j) v[j] = __uint_as_float(r[j]);
    }
    if (u + 2 >= NU) {
      tc_fence_before();
      __syncwarp();
      if (lane == 0) release();
    }
    const int col0 = nb * BN + u * UW;
    if (col0 >= N || row0 >= M) continue;
    epilogue_values<__nv_bfloat16, UW>(ep, vrow, col0, v);
    int64_t b = 0;
    int t0 = 0;
    if (ep.kind == EPI_HEADS) {
      b = row0 / ep.rows_per_batch;
      t0 = (int)(row0 - b * ep.rows_per_batch);
      if (t0 + 32 > ep.rows_per_batch || row0 + 32 > M) {
        // the unit's rows cross a batch boundary: plain stores, one row per lane
        if (row < M) epilogue_store<__nv_bfloat16, UW>(ep, row, col0, v);
        continue;
      }
    }
    // the previous unit's TMA read of the staging buffer must be complete
    if (lane == 0) bulk_wait_read0();
    __syncwarp();
    uint8_t* rowp = stg + lane * 128;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      uint4 w;
      if constexpr (UW == 64) {
        w.x = pack_bf16x2(v[8 * j + 0], v[8 * j + 1]);
        w.y = pack_bf16x2(v[8 * j + 2], v[8 * j + 3]);
        w.z = pack_bf16x2(v[8 * j + 4], v[8 * j + 5]);
        w.w = pack_bf16x2(v[8 * j + 6], v[8 * j + 7]);
      } else {
        w = make_uint4(__float_as_uint(v[4 * j + 0]), __float_as_uint(v[4 * j + 1]), __float_as_uint(v[4 * j + 2]),
                       __float_as_uint(v[4 * j + 3]));
      }
      // 128-byte swizzle: 16-byte chunk j of row r sits at chunk j ^ (r % 8)
      *reinterpret_cast<uint4*>(rowp + ((j ^ (lane & 7)) << 4)) = w;
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      if (ep.kind == EPI_RESID) {
        tma_reduce_add_2d(&maps.m[0], stg, col0, (int)row0);
      } else if (ep.kind == EPI_HEADS) {
        const int sec = col0 / ep.D;
        const int cc = col0 - sec * ep.D;
        const int h = cc / ep.hd;
        if (DIT_BOUNDS(sec >= 0 && sec < 3 && ep.dst[sec] && cc - h * ep.hd + UW <= ep.hd && h < ep.H &&
                           ep.tok_off + t0 + 32 <= ep.seq_total && (b + 1) * ep.rows_per_batch <= M,
                       err, 61))
          tma_store_3d(&maps.m[sec], stg, cc - h * ep.hd, ep.tok_off + t0, (int)(b * ep.H + h));
      } else {
        tma_store_2d(&maps.m[0], stg, col0, (int)row0);
      }
      bulk_commit();
    }
  }
}

template <int BN, int NP, bool F8, bool PAIR>
__global__ void __launch_bounds__(GEMM_THREADS, 1)
    gemm_tc_kernel(const __grid_constant__ GemmBatch<NP> P, int N, int K, int* err) {
  using C = TcGemmCfg<BN, F8, PAIR>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
  uint64_t* empty = full + C::STAGES;
  uint64_t* tfull = empty + C::STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // CTA pair: rank 0 (the leader) issues the MMAs of both CTAs.  Its full[s]
  // counts the operand bytes of both CTAs (the peer's loads complete on it),
  // its tempty[a] the epilogue warps of both; the leader's commits arrive on
  // empty[s] and tfull[a] of both CTAs.  The peer's own full and tempty stay
  // unused.
  const uint32_t rank = PAIR ? cluster_ctarank() : 0;
  const bool leader = rank == 0;
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], PAIR ? 2 * EPI_WARPS : EPI_WARPS);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
#pragma unroll
    for (int p = 0; p < NP; ++p) {
      if (P.M[p] == 0) continue;  // no tiles, no tensor maps
      tma_prefetch_desc(&P.tmA[p]);
      tma_prefetch_desc(&P.tmB[p]);
    }
  }
  if (warp == 1) {
    if constexpr (PAIR)
      tmem_alloc_pair(tmem_slot, C::TMEM_COLS);
    else
      tmem_alloc(tmem_slot, C::TMEM_COLS);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // both CTAs' barriers are initialised before any remote arrival or copy
  if constexpr (PAIR) cluster_sync();
  const uint32_t tmem_base = *tmem_slot;
  // a role that gives up also stops the other CTA's waits
  auto abort_pair = [&]() {
    if constexpr (PAIR) st_cluster_u32(cluster_map((const void*)abort_flag, rank ^ 1u), 1u);
  };

  const int n_tiles = (N + BN - 1) / BN;
  const int k_blocks = (K + C::BK - 1) / C::BK;
  const int num_tiles = P.tile_end[NP - 1];
  // Both CTAs of a pair walk the same tile list; tile (mb, nb) of a pair
  // launch is 256 rows, of which CTA `rank` holds 128-row block 2 mb + rank.
  const int first = PAIR ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
  const int stride = PAIR ? (int)(gridDim.x >> 1) : (int)gridDim.x;

  if (warp == 0) {
    // ------------------------------------------------ TMA producer (one thread)
    if (lane == 0) {
      uint32_t stage = 0, phase = 0;
      int issued[C::STAGES];
#pragma unroll
      for (int s = 0; s < C::STAGES; ++s) issued[s] = 0;
      bool ok = true;
      // W tiles are reused by every row tile: keep them in L2 ahead of the
      // streamed A rows (FFN2, whose A is the 1.2 GB MLP hidden, 3 % faster)
      const uint64_t w_policy = l2_policy_evict_last();
      const uint32_t full_leader = PAIR ? cluster_map(full, 0) : 0;
      for (int tile = first; ok && tile < num_tiles; tile += stride) {
        int t, mb, nb;
        const int p = locate_tile(P, tile, &t);
        tile_coords(t, P.m_tiles[p], n_tiles, P.group_n, &mb, &nb);
        if (!DIT_BOUNDS(p >= 0 && p < NP && mb >= 0 && mb < P.m_tiles[p] && nb >= 0 && nb < n_tiles, err, 60)) {
          *abort_flag = 1;  // the other roles' waits return at once: the CTA winds down
          abort_pair();
          ok = false;
          break;
        }
        const CUtensorMap* tmA = &P.tmA[p];
        const CUtensorMap* tmB = &P.tmB[p];
        const int a_row = PAIR ? (2 * mb + (int)rank) * C::BM : mb * C::BM;
        const int b_row = nb * BN + (int)rank * C::BN_CTA;
        // Short main loops (K <= 2048): the residual rows this tile adds into
        // go to L2 now, so the epilogue's reduce-add a tile later does not
        // wait for DRAM (0.54 -> 0.51 ms for a video block's two
        // out-projections).  With long main loops the reduce has time to
        // spare and the prefetch only slowed the GEMM (FFN2 +3 %).
        if (P.ep[p].kind == EPI_RESID && P.ep[p].tma && k_blocks <= 32)
          tma_prefetch_l2_2d(&P.maps[p].m[1], nb * BN, a_row);
        for (int kb = 0; kb < k_blocks; ++kb) {
          ok = mbar_wait(&empty[stage], phase ^ 1, abort_flag, err, 11);
          if (!ok) break;
          uint8_t* sa = smem + stage * C::STAGE_BYTES;
          if constexpr (PAIR) {
            // the leader's arrival brings the bytes of both CTAs' loads
            if (leader) mbar_arrive_expect_tx(&full[stage], 2 * C::STAGE_BYTES);
            const uint32_t fb = full_leader + stage * (uint32_t)sizeof(uint64_t);
            tma_load_2d_pair(sa, tmA, fb, kb * C::BK, a_row);
            tma_load_2d_pair_hint(sa + C::A_BYTES, tmB, fb, kb * C::BK, b_row, w_policy);
          } else {
            mbar_arrive_expect_tx(&full[stage], C::STAGE_BYTES);
            tma_load_2d(sa, tmA, &full[stage], kb * C::BK, a_row);
            tma_load_2d_hint(sa + C::A_BYTES, tmB, &full[stage], kb * C::BK, b_row, w_policy);
          }
          ++issued[stage];
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) abort_pair();
      }
      if (!ok) {
        // wind down: let every copy this thread started land before the CTA exits
        volatile int no_abort = 0;
        if (leader) {
          for (int s = 0; s < C::STAGES; ++s)
            if (issued[s] > 0) mbar_wait(&full[s], (uint32_t)((issued[s] - 1) & 1), &no_abort, nullptr, 0);
        } else {
          // the peer's loads complete on the leader's barriers, whose phases
          // need the leader's arrivals as well: give them a fixed time to land
          const uint64_t t0 = globaltimer_ns();
          while (globaltimer_ns() - t0 < 200000ull) {
          }
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer (one thread)
    // The whole role runs on lane 0: a warp that diverges and reconverges
    // around every MMA burst costs the tensor pipe a large share of its rate.
    // In a pair only the leader's issues.
    if (lane == 0 && leader) {
      uint32_t stage = 0, phase = 0, local = 0;
      bool ok = true;
      const uint64_t a_desc = umma_desc_sw128(smem_u32(smem), 16, 1024);
      const uint64_t b_desc = umma_desc_sw128(smem_u32(smem) + C::A_BYTES, 16, 1024);
      for (int tile = first; ok && tile < num_tiles; tile += stride, ++local) {
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
          for (int k = 0; k < C::BK / C::K_PER_MMA; ++k) {
            const uint64_t ak = umma_desc_add(ad, k * 32), bk = umma_desc_add(bd, k * 32);
            const uint32_t accum = (kb | k) != 0;
            if constexpr (PAIR && F8)
              umma_ss_f8_pair(d_tmem, ak, bk, C::IDESC, accum);
            else if constexpr (PAIR)
              umma_ss_pair(d_tmem, ak, bk, C::IDESC, accum);
            else if constexpr (F8)
              umma_ss_f8(d_tmem, ak, bk, C::IDESC, accum);
            else
              umma_ss(d_tmem, ak, bk, C::IDESC, accum);
          }
          if constexpr (PAIR)
            umma_commit_pair(&empty[stage], 0x3);
          else
            umma_commit(&empty[stage]);
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        if constexpr (PAIR)
          umma_commit_pair(&tfull[acc], 0x3);
        else
          umma_commit(&tfull[acc]);
      }
      if (!ok) abort_pair();
      // all MMAs issued by this thread complete before TMEM is released
      if constexpr (PAIR)
        umma_commit_pair(drain, 0x1);
      else
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
    uint8_t* stg = smem + C::STG_OFF + (warp - 2) * C::STG_BYTES;
    const uint32_t tempty_leader = PAIR ? cluster_map(tempty, 0) : 0;
    uint32_t local = 0;
    bool ok = true;
    for (int tile = first; tile < num_tiles; tile += stride, ++local) {
      const uint32_t acc = local & 1, aphase = (local >> 1) & 1;
      ok = mbar_wait_warp(&tfull[acc], aphase, abort_flag, err, 14);
      if (!ok) break;
      tc_fence_after();
      int t, mb, nb;
      const int p = locate_tile(P, tile, &t);
      tile_coords(t, P.m_tiles[p], n_tiles, P.group_n, &mb, &nb);
      const EpiParams& ep = P.ep[p];
      const int64_t M = P.M[p];
      const int64_t tile_row0 = PAIR ? (int64_t)(2 * mb + (int)rank) * C::BM : (int64_t)mb * C::BM;
      const uint32_t tacc = tmem_base + acc * BN + ((uint32_t)(q * 32) << 16);
      // this warp is done with accumulator `acc` (tensor-memory reads complete)
      auto release = [&]() {
        if constexpr (PAIR)
          mbar_arrive_cluster(tempty_leader + acc * (uint32_t)sizeof(uint64_t));
        else
          mbar_arrive(&tempty[acc]);
      };
      if (ep.tma) {
        const int64_t row0 = tile_row0 + q * 32;
        if (ep.kind == EPI_F32 || ep.kind == EPI_RESID)
          drain_tile_tma<BN, 32>(ep, P.maps[p], tacc, row0, M, N, nb, half, stg, release, err);
        else
          drain_tile_tma<BN, 64>(ep, P.maps[p], tacc, row0, M, N, nb, half, stg, release, err);
        continue;
      }
      const int64_t row = tile_row0 + row_in_tile;
#pragma unroll 1
      for (int c = half; c < BN / 32; c += 2) {
        uint32_t r[32];
        tmem_ld32(tacc + c * 32, r);
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
      if (lane == 0) release();
    }
    if (!ok && lane == 0) abort_pair();
    // every TMA store of this warp has read its staging buffer and landed
    if (lane == 0) bulk_wait0();
    __syncwarp();
  }
  tc_fence_before();
  __syncthreads();
  // A pair frees its tensor memory together, once the leader's MMAs have all
  // completed (its MMA thread waited on `drain`) and neither CTA has remote
  // arrivals or copies left to make into the other.
  if constexpr (PAIR) cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    if constexpr (PAIR)
      tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
    else
      tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// Tensor maps for the TMA epilogue; false leaves the epilogue on plain stores
// (unaligned output, row stride not a multiple of 16 bytes, head_dim not a
// multiple of 64, or the driver rejecting a map).
static bool make_epi_maps(const EpiParams& e, int64_t M, int N, EpiMaps* maps) {
  switch (e.kind) {
    case EPI_F32: {
      if (!aligned16(e.out) || e.ldo % 4 || e.ldo < N) return false;
      const uint64_t d[2] = {(uint64_t)N, (uint64_t)M}, st[1] = {(uint64_t)e.ldo * 4};
      const uint32_t box[2] = {32, 32};
      return make_tmap(&maps->m[0], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, e.out, 2, d, st, box);
    }
    case EPI_ACT:
    case EPI_GELU: {
      if (!aligned16(e.out) || e.ldo % 8 || e.ldo < N) return false;
      const uint64_t d[2] = {(uint64_t)N, (uint64_t)M}, st[1] = {(uint64_t)e.ldo * 2};
      const uint32_t box[2] = {64, 32};
      return make_tmap_bf16(&maps->m[0], e.out, 2, d, st, box);
    }
    case EPI_RESID: {
      if (!aligned16(e.x) || N % 4) return false;
      const uint64_t d[2] = {(uint64_t)N, (uint64_t)M}, st[1] = {(uint64_t)N * 4};
      const uint32_t box[2] = {32, 32};
      // m[1]: the same tensor in boxes of a whole 128 x 256 output tile (L2 prefetch)
      const uint32_t pbox[2] = {256, 128};
      return make_tmap(&maps->m[0], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, e.x, 2, d, st, box) &&
             make_tmap(&maps->m[1], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, e.x, 2, d, st, pbox, CU_TENSOR_MAP_SWIZZLE_NONE);
    }
    case EPI_HEADS: {
      if (e.hd % 64 || e.rows_per_batch <= 0 || M % e.rows_per_batch) return false;
      const int64_t BH = (M / e.rows_per_batch) * e.H;
      const uint64_t d[3] = {(uint64_t)e.hd, (uint64_t)e.seq_total, (uint64_t)BH};
      const uint64_t st[2] = {(uint64_t)e.hd * 2, (uint64_t)e.seq_total * e.hd * 2};
      const uint32_t box[3] = {64, 32, 1};
      for (int sec = 0; sec < 3; ++sec) {
        if (!e.dst[sec]) continue;
        if (!aligned16(e.dst[sec]) || !make_tmap_bf16(&maps->m[sec], e.dst[sec], 3, d, st, box)) return false;
      }
      return true;
    }
  }
  return false;
}

// Clusters of two GEMM CTAs that fit on the device at once (per device,
// queried at the first pair launch).  A persistent pair launch never asks for
// more: a cluster that had to wait for a slot would run its whole tile list
// after the others.
static int pair_clusters(const void* kernel, cudaLaunchConfig_t cfg, int num_sms) {
  static int cached[kMaxDevices] = {};  // 0: not asked yet, -1: none fit
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  if (cached[dev] == 0) {
    int n = 0;
    cfg.gridDim = dim3(2 * (num_sms / 2));
    if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess) {
      (void)cudaGetLastError();  // the query's error is not the launch's
      n = 0;
    }
    cached[dev] = n <= 0 ? -1 : (n < num_sms / 2 ? n : num_sms / 2);
  }
  return cached[dev] > 0 ? cached[dev] : 0;
}

template <int BN, int NP, bool F8, bool PAIR>
static cudaError_t launch_gemm_tc(const GemmArgs* gs, int* err, int num_sms, cudaStream_t s) {
  using C = TcGemmCfg<BN, F8, PAIR>;
  constexpr int TILE_M = PAIR ? 2 * C::BM : C::BM;
  GemmBatch<NP> P{};
  const int n_tiles = (gs[0].N + BN - 1) / BN;
  int tiles = 0;
  for (int p = 0; p < NP; ++p) {
    const GemmArgs& g = gs[p];
    P.ep[p] = g.epi;
    P.M[p] = g.M;
    if (g.M > 0) {
      const uint64_t da[2] = {(uint64_t)g.K, (uint64_t)g.M}, sa[1] = {(uint64_t)g.lda * C::ESZ};
      const uint32_t ba[2] = {(uint32_t)C::BK, 128};
      const uint64_t db[2] = {(uint64_t)g.K, (uint64_t)g.N}, sb[1] = {(uint64_t)g.K * C::ESZ};
      const uint32_t bb[2] = {(uint32_t)C::BK, (uint32_t)C::BN_CTA};
      const CUtensorMapDataType dt = F8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
      if (!make_tmap(&P.tmA[p], dt, g.A, 2, da, sa, ba) || !make_tmap(&P.tmB[p], dt, g.W, 2, db, sb, bb))
        return cudaErrorInvalidValue;
      P.ep[p].tma = make_epi_maps(P.ep[p], g.M, g.N, &P.maps[p]) ? 1 : 0;
    }
    P.m_tiles[p] = (int)((g.M + TILE_M - 1) / TILE_M);
    tiles += P.m_tiles[p] * n_tiles;
    P.tile_end[p] = tiles;
  }
  // Column groups whose W slice is at most ~40 MB (every W of the video
  // layers fits whole: plain N-fastest order there).  Each group streams A
  // once more, so groups are used only while A is no larger than W: the
  // image FFN2 (A 226 MB, W 75 MB) read slightly more in two groups (887 MB)
  // than in one (853 MB).
  const int64_t w_tile_bytes = (int64_t)BN * gs[0].K * C::ESZ;
  const int64_t a_bytes = gs[0].M * gs[0].K * C::ESZ, w_bytes = (int64_t)gs[0].N * gs[0].K * C::ESZ;
  int64_t gn = ((int64_t)40 << 20) / w_tile_bytes;
  if (gn < 1) gn = 1;
  if (a_bytes > w_bytes) gn = n_tiles;
  P.group_n = (int)(gn < n_tiles ? gn : n_tiles);
  if (tiles == 0) return cudaSuccess;
  static SmemAttr attr;
  const void* kernel = reinterpret_cast<const void*>(gemm_tc_kernel<BN, NP, F8, PAIR>);
  cudaError_t e = ensure_smem_attr(kernel, C::SMEM_BYTES, attr);
  if (e != cudaSuccess) return e;
  if constexpr (PAIR) {
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 2;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg{};
    cfg.blockDim = dim3(GEMM_THREADS);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    cfg.stream = s;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    const int max_clusters = pair_clusters(kernel, cfg, num_sms);
    // no two-CTA cluster fits next to this kernel's resources: single CTAs
    if (max_clusters <= 0) return launch_gemm_tc<BN, NP, F8, false>(gs, err, num_sms, s);
    const int clusters = tiles < max_clusters ? tiles : max_clusters;
    cfg.gridDim = dim3(2 * clusters);
    e = cudaLaunchKernelEx(&cfg, gemm_tc_kernel<BN, NP, F8, true>, P, gs[0].N, gs[0].K, err);
    return e != cudaSuccess ? e : cudaGetLastError();
  } else {
    const int grid = tiles < num_sms ? tiles : num_sms;
    gemm_tc_kernel<BN, NP, F8, false><<<grid, GEMM_THREADS, C::SMEM_BYTES, s>>>(P, gs[0].N, gs[0].K, err);
    return cudaGetLastError();
  }
}

// alignment rules of the operand tensor maps: 16-byte rows and bases
static bool operands_ok(const GemmArgs& g, int esz) {
  const int per16 = 16 / esz;
  return !((g.K % per16) || (g.lda % per16) || (reinterpret_cast<uintptr_t>(g.A) & 15) ||
           (reinterpret_cast<uintptr_t>(g.W) & 15));
}

// Widths that are multiples of 256 run on CTA pairs (256 x 256 tiles) when a
// tile's main loop has at least kPairMinKBlocks K blocks; the others on single
// CTAs with 128 x 256, 128 x 128 or 128 x 64 tiles.  A pair's MMA waits until
// both CTAs' epilogues have drained the accumulator, so where the epilogue of
// a tile outlasts the main loop of the next the pair runs at the pace of the
// slower CTA: the video e4m3 projections (K = 1536: 12 K blocks) were 7-12 %
// slower on pairs, every GEMM with 24 K blocks or more (bf16 video and image,
// e4m3 image) 4-15 % faster.
constexpr int kPairMinKBlocks = 16;
static int g_cta_pairs = 1;  // 0 never, 1 by main-loop length, 2 always
void set_gemm_cta_pairs(int mode) { g_cta_pairs = mode < 0 ? 0 : (mode > 2 ? 2 : mode); }

template <int NP, bool F8>
static cudaError_t launch_by_width(const GemmArgs* gs, int* err, int num_sms, cudaStream_t s) {
  const int N = gs[0].N;
  if (N % 256 == 0) {
    const int k_blocks = (gs[0].K + TcGemmCfg<256, F8>::BK - 1) / TcGemmCfg<256, F8>::BK;
    const bool pair = g_cta_pairs == 2 || (g_cta_pairs == 1 && k_blocks >= kPairMinKBlocks);
    if (pair && num_sms >= 2) return launch_gemm_tc<256, NP, F8, true>(gs, err, num_sms, s);
    return launch_gemm_tc<256, NP, F8, false>(gs, err, num_sms, s);
  }
  if (N % 128 == 0) return launch_gemm_tc<128, NP, F8, false>(gs, err, num_sms, s);
  return launch_gemm_tc<64, NP, F8, false>(gs, err, num_sms, s);
}

template <bool F8>
static cudaError_t gemm_single(const GemmArgs& g, int* err, int num_sms, cudaStream_t s) {
  if (g.M == 0 || g.N == 0) return cudaSuccess;
  if (!operands_ok(g, F8 ? 1 : 2)) return cudaErrorInvalidValue;
  if (F8 && (!g.epi.a_scale || !g.epi.w_scale)) return cudaErrorInvalidValue;
  return launch_by_width<1, F8>(&g, err, num_sms, s);
}

template <bool F8>
static cudaError_t gemm_pair(const GemmArgs& g0, const GemmArgs& g1, int* err, int num_sms, cudaStream_t s) {
  if (g0.N != g1.N || g0.K != g1.K) return cudaErrorInvalidValue;
  if (g0.N == 0 || (g0.M == 0 && g1.M == 0)) return cudaSuccess;
  for (const GemmArgs* g : {&g0, &g1}) {
    if (g->M == 0) continue;
    if (!operands_ok(*g, F8 ? 1 : 2)) return cudaErrorInvalidValue;
    if (F8 && (!g->epi.a_scale || !g->epi.w_scale)) return cudaErrorInvalidValue;
  }
  const GemmArgs gs[2] = {g0, g1};
  return launch_by_width<2, F8>(gs, err, num_sms, s);
}

cudaError_t gemm_bf16_tc(const GemmArgs& g, int* err, int num_sms, cudaStream_t s) {
  return gemm_single<false>(g, err, num_sms, s);
}
cudaError_t gemm_bf16_tc_pair(const GemmArgs& g0, const GemmArgs& g1, int* err, int num_sms, cudaStream_t s) {
  return gemm_pair<false>(g0, g1, err, num_sms, s);
}
cudaError_t gemm_e4m3_tc(const GemmArgs& g, int* err, int num_sms, cudaStream_t s) {
  return gemm_single<true>(g, err, num_sms, s);
}
cudaError_t gemm_e4m3_tc_pair(const GemmArgs& g0, const GemmArgs& g1, int* err, int num_sms, cudaStream_t s) {
  return gemm_pair<true>(g0, g1, err, num_sms, s);
}

}  // namespace dit

static_assert(dit::TcGemmCfg<256>::SMEM_BYTES <= 232448 && dit::TcGemmCfg<128>::SMEM_BYTES <= 232448 &&
                  dit::TcGemmCfg<64>::SMEM_BYTES <= 232448 && dit::TcGemmCfg<256, false, true>::SMEM_BYTES <= 232448 &&
                  dit::TcGemmCfg<256, true, true>::SMEM_BYTES <= 232448,
              "GEMM tile set exceeds 227 KB of shared memory");
