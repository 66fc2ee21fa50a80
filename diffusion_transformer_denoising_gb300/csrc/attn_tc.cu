// Bidirectional multi-head attention (no mask), head_dim 128, bf16 in/out,
// fp32 softmax and accumulation, on the 5th-generation tensor cores.
//
// One CTA = 128 query rows of one (batch, head).  Each row's 128 key columns
// per step are split into two halves, each with its own online-softmax state
// (running max m_h, sum l_h) and its own output accumulator O_h; the halves
// are merged once at the end:
//     O = (2^(m_0-M) O_0 + 2^(m_1-M) O_1) / (2^(m_0-M) l_0 + 2^(m_1-M) l_1).
// Warps 0-3 run the softmax of key half 0 and warps 4-7 that of half 1 (warp
// w reads TMEM lane quadrant w%4, i.e. 32 query rows), so no warp ever waits
// for another inside the loop.  Warp 8 streams K and V tiles of 128 keys
// with TMA through two 3-stage rings; warp 9 issues the MMAs from one thread,
// one uninterrupted burst "PV_j, S_{j+2}" per key tile after two waits:
//     S_j = Q K_j^T                 (SS, K-major operands in shared memory)
//     O_h += P_j[:, half h] V_j[half h]   (TS: P from tensor memory, V N-major)
// Tensor memory (512 columns): S double buffer [0,128) [128,256); O_0 at
// [256,384); O_1 at [384,512).  P_j (packed bf16 pairs) overwrites the first
// 64 columns of its S slot once the softmax has read them.  tcgen05.mma
// operations of a CTA execute in issue order, so PV_j has read P_j before
// S_{j+2} overwrites the slot.
// Every tcgen05.commit costs the tensor pipe a few hundred cycles, so there
// is exactly one per key tile: after "PV_j, S_{j+2}" the MMA thread commits
// to done[(j+2) % 3].  Completion i of that ring (i = 0, 1 for S_0, S_1;
// i = j+2 for PV_j together with S_{j+2}) tells the softmax that S_i is in
// TMEM, the producer that K_{i} and V_{i-2} stages are free, and a lazy O
// rescale that PV_{i-2} has landed.  Each waiter takes the completions of a
// barrier in order, and completion i+3 cannot happen before K_{i+3} is
// loaded, so a parity wait never aliases.  O is rescaled lazily (only when a
// max grows by more than 2^8).
//
// All waits are bounded (common.cuh); on a timeout the CTA flags *err, waits
// for its own copies and MMAs, frees TMEM and exits.
#include "epilogue.cuh"
#include "tmap.h"

namespace dit {

namespace fa {
constexpr int BQ = 128, BKV = 128, HD = 128, KST = 3, VST = 3;
constexpr int TILE_BYTES = 128 * HD * 2;   // 32 KB: two 16 KB swizzle blocks of 64 channels
constexpr int Q_OFF = 0;
constexpr int K_OFF = Q_OFF + TILE_BYTES;
constexpr int V_OFF = K_OFF + KST * TILE_BYTES;
constexpr int BAR_OFF = V_OFF + VST * TILE_BYTES;
constexpr int XCH_OFF = BAR_OFF + 256;     // float[4][128]: m_0, m_1, l_0, l_1 per row
// The tiles need 1024-byte alignment.  The dynamic shared window of a kernel
// without static shared memory starts 1024-aligned (checked at entry), so no
// alignment slack is reserved and the total stays under 227 KB.
constexpr int SMEM_BYTES = XCH_OFF + 4 * BQ * 4;
constexpr int NUM_THREADS = 320;           // 8 softmax warps, TMA warp, MMA warp
constexpr int TMA_WARP = 8, MMA_WARP = 9;
constexpr uint32_t TM_S = 0, TM_O = 256;
constexpr uint32_t IDESC_S = umma_idesc_bf16(128, 128, false);
constexpr uint32_t IDESC_O = umma_idesc_bf16(128, 128, true);
constexpr float RESCALE_THRESHOLD = 8.0f;  // log2 units
}  // namespace fa

__global__ void __launch_bounds__(fa::NUM_THREADS, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, AttnArgs a, float scale_log2, int* err) {
  using namespace fa;
  extern __shared__ __align__(1024) uint8_t smem[];
  if (smem_u32(smem) & 1023) {  // uniform across the CTA: nothing has started yet
    if (threadIdx.x == 0) atomicCAS(err, 0, 20);
    return;
  }
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + BAR_OFF);
  uint64_t* q_full = bars;        // Q, K_0 and K_1
  uint64_t* xf = bars + 1;        // [3] tile pair j: V_j and K_{j+2} (see the producer)
  uint64_t* done = bars + 7;      // [3] MMA completion ring (see above)
  uint64_t* p_ready = bars + 10;  // [2] per S slot
  uint64_t* drain = bars + 12;
  uint64_t* fin = bars + 13;      // [4] per lane quadrant
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 17);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* xch = reinterpret_cast<float*>(smem + XCH_OFF);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bh = blockIdx.z * a.H + blockIdx.y;
  const int q0 = blockIdx.x * BQ;
  const int nkv = (a.Lk + BKV - 1) / BKV;
  // Each CTA walks the key tiles in a rotated order (the result does not
  // depend on the order), so CTAs running together read different K/V tiles.
  const int kv_rot = (int)(blockIdx.x % (unsigned)nkv);

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < 3; ++s) {
      mbar_init(&xf[s], 1);
      mbar_init(&done[s], 1);
    }
    for (int b = 0; b < 2; ++b) mbar_init(&p_ready[b], 8);
    mbar_init(drain, 1);
    for (int i = 0; i < 4; ++i) mbar_init(&fin[i], 2);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == TMA_WARP && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  if (warp == MMA_WARP) tmem_alloc(tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == TMA_WARP) {
    // ------------------------------------------------ TMA producer (one thread)
    // Loads are grouped so that the MMA thread waits once per key tile: barrier
    // xf[j % 3] covers V_j and K_{j+2}, exactly what "PV_j, S_{j+2}" reads.  Both
    // stages are free once completion j-1 (PV_{j-3}, S_{j-1}) has landed.
    if (lane == 0) {
      int issued[3] = {0, 0, 0};
      bool ok = true;
      auto load_tile = [&](const CUtensorMap* tm, uint8_t* dst, uint64_t* bar, int tile) {
        const int jt = (tile + kv_rot) % nkv;
        tma_load_3d(dst, tm, bar, 0, jt * BKV, bh);
        tma_load_3d(dst + TILE_BYTES / 2, tm, bar, 64, jt * BKV, bh);
      };
      mbar_arrive_expect_tx(q_full, (nkv > 1 ? 3 : 2) * TILE_BYTES);
      tma_load_3d(smem + Q_OFF, &tmQ, q_full, 0, q0, bh);
      tma_load_3d(smem + Q_OFF + TILE_BYTES / 2, &tmQ, q_full, 64, q0, bh);
      load_tile(&tmK, smem + K_OFF, q_full, 0);
      if (nkv > 1) load_tile(&tmK, smem + K_OFF + TILE_BYTES, q_full, 1);
      for (int j = 0; j < nkv; ++j) {
        if (j >= 1) ok = mbar_wait(&done[(j - 1) % 3], (uint32_t)(((j - 1) / 3) & 1), abort_flag, err, 21);
        if (!ok) break;
        const bool has_k = j + 2 < nkv;
        mbar_arrive_expect_tx(&xf[j % 3], (has_k ? 2 : 1) * TILE_BYTES);
        load_tile(&tmV, smem + V_OFF + (j % VST) * TILE_BYTES, &xf[j % 3], j);
        if (has_k) load_tile(&tmK, smem + K_OFF + ((j + 2) % KST) * TILE_BYTES, &xf[j % 3], j + 2);
        ++issued[j % 3];
      }
      if (!ok) {
        // wind down: every copy this thread started lands before the CTA exits
        volatile int no_abort = 0;
        mbar_wait(q_full, 0, &no_abort, nullptr, 0);
        for (int s = 0; s < 3; ++s)
          if (issued[s] > 0) mbar_wait(&xf[s], (uint32_t)((issued[s] - 1) & 1), &no_abort, nullptr, 0);
      }
    }
    __syncwarp();
  } else if (warp == MMA_WARP) {
    // ------------------------------------------------ MMA issuer (one thread)
    // The whole role runs on lane 0: a warp that diverges and reconverges
    // around every MMA burst costs the tensor pipe a large share of its rate.
    if (lane == 0) {
      auto wait1 = [&](uint64_t* bar, uint32_t parity, int site) -> bool {
        return mbar_wait(bar, parity, abort_flag, err, site);
      };
      // base descriptors, built once; per MMA only a constant is added
      const uint64_t q_desc = umma_desc_sw128(smem_u32(smem + Q_OFF), 16, 1024);
      const uint64_t k_desc = umma_desc_sw128(smem_u32(smem + K_OFF), 16, 1024);
      const uint64_t v_desc = umma_desc_sw128(smem_u32(smem + V_OFF), 16384, 1024);
      // S_j = Q K_j^T into S slot j % 2 (no commit here); K_j is resident
      auto issue_s = [&](int j) {
        const uint64_t kd = umma_desc_add(k_desc, (j % KST) * TILE_BYTES);
        const uint32_t d_tmem = tmem + TM_S + (j & 1) * 128;
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk) {
          const uint32_t off = (kk >> 2) * (TILE_BYTES / 2) + (kk & 3) * 32;
          umma_ss(d_tmem, umma_desc_add(q_desc, off), umma_desc_add(kd, off), IDESC_S, kk != 0);
        }
      };
      bool ok = wait1(q_full, 0, 24);
      if (ok) {
        tc_fence_after();
        issue_s(0);
        umma_commit(&done[0]);  // completion 0: S_0
        if (nkv > 1) {
          issue_s(1);
          umma_commit(&done[1]);  // completion 1: S_1
        }
      }
      // One uninterrupted burst per key tile: the issuing thread does nothing
      // between MMAs (any wait or detour there idles the tensor pipe).
      for (int j = 0; ok && j < nkv; ++j) {
        ok = wait1(&p_ready[j & 1], (uint32_t)((j >> 1) & 1), 25) &&
             wait1(&xf[j % 3], (uint32_t)((j / 3) & 1), 26);
        if (!ok) break;
        tc_fence_after();
        const uint64_t vd = umma_desc_add(v_desc, (j % VST) * TILE_BYTES);
        const uint32_t p_tmem = tmem + TM_S + (j & 1) * 128;
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            // keys 64h+16kk.. of V (8-row groups 1 KB apart; channel halves 16 KB apart)
            umma_ts(tmem + TM_O + h * 128, p_tmem + h * 32 + kk * 8, umma_desc_add(vd, (4 * h + kk) * 2048),
                    IDESC_O, (j | kk) != 0);
          }
        if (j + 2 < nkv) issue_s(j + 2);
        umma_commit(&done[(j + 2) % 3]);  // completion j+2: PV_j (+ S_{j+2})
      }
      umma_commit(drain);
      volatile int no_abort = 0;
      mbar_wait(drain, 0, &no_abort, nullptr, 0);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------ softmax warps 0-7
    const int q = warp & 3, h = warp >> 2;
    const uint32_t lane_off = (uint32_t)(q * 32) << 16;
    const uint32_t o_col = tmem + TM_O + h * 128 + lane_off;
    const int row = q * 32 + lane;
    float m_used = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < nkv; ++j) {
      ok = __all_sync(0xffffffffu, mbar_wait(&done[j % 3], (uint32_t)((j / 3) & 1), abort_flag, err, 31));
      if (!ok) break;
      tc_fence_after();
      const uint32_t s_col = tmem + TM_S + (j & 1) * 128 + lane_off;
      float s[64];
      {
        uint32_t r[64];
        tmem_ld32(s_col + h * 64, *reinterpret_cast<uint32_t(*)[32]>(&r[0]));
        tmem_ld32(s_col + h * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&r[32]));
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 64; ++i) s[i] = __uint_as_float(r[i]);
      }
      const int valid = a.Lk - ((j + kv_rot) % nkv) * BKV - h * 64;
      if (valid < 64) {
#pragma unroll
        for (int i = 0; i < 64; ++i)
          if (i >= valid) s[i] = -INFINITY;
      }
      // row max: four independent chains of three-input max over s[4..59], then s[60..63]
      float m4[4] = {s[0], s[1], s[2], s[3]};
#pragma unroll
      for (int i = 4; i + 8 <= 60; i += 8)
#pragma unroll
        for (int k = 0; k < 4; ++k) m4[k] = fmax3(m4[k], s[i + 2 * k], s[i + 2 * k + 1]);
#pragma unroll
      for (int k = 0; k < 4; ++k) m4[k] = fmaxf(m4[k], s[60 + k]);
      const float mx = fmaxf(fmax3(m4[0], m4[1], m4[2]), m4[3]);
      const float m_new = fmaxf(m_used, mx * scale_log2);
      float alpha = 1.f;
      if (j == 0) {
        m_used = m_new;
      } else {
        const bool need = m_new - m_used > RESCALE_THRESHOLD;
        if (__any_sync(0xffffffffu, need)) {
          // O_h must hold PV_{j-1} (completion j+1) before it is rescaled
          ok = __all_sync(0xffffffffu, mbar_wait(&done[(j + 1) % 3], (uint32_t)(((j + 1) / 3) & 1), abort_flag, err, 32));
          if (!ok) break;
          tc_fence_after();
          if (need) {
            alpha = ex2_approx(m_used - m_new);
            m_used = m_new;
          }
#pragma unroll 1
          for (int c = 0; c < HD / 32; ++c) {
            uint32_t r[32];
            tmem_ld32(o_col + c * 32, r);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
            tmem_st32(o_col + c * 32, r);
          }
        }
      }
      // a half that has seen no valid key yet keeps m = -inf and p = 0
      const float mref = (m_used == -INFINITY) ? 0.f : m_used;
      const float2 sc2 = make_float2(scale_log2, scale_log2), nm2 = make_float2(-mref, -mref);
      float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
      uint32_t pk[32];
#pragma unroll
      for (int i = 0; i < 64; i += 2) {
        const float2 x = ffma2(make_float2(s[i], s[i + 1]), sc2, nm2);
        const float2 p = make_float2(ex2_approx(x.x), ex2_approx(x.y));
        acc[(i >> 1) & 3] = fadd2(acc[(i >> 1) & 3], p);
        pk[i / 2] = pack_bf16x2(p.x, p.y);
      }
      const float2 a01 = fadd2(acc[0], acc[1]), a23 = fadd2(acc[2], acc[3]);
      l = l * alpha + ((a01.x + a01.y) + (a23.x + a23.y));
      tmem_st32(s_col + h * 32, pk);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_ready[j & 1]);
    }
    if (ok) {
      // PV_{nkv-1} is completion nkv+1
      ok = __all_sync(0xffffffffu, mbar_wait(&done[(nkv + 1) % 3], (uint32_t)(((nkv + 1) / 3) & 1), abort_flag, err, 33));
    }
    if (ok) {
      // merge the two halves: swap (m, l) with the partner warp of the quadrant
      xch[h * BQ + row] = m_used;
      xch[(2 + h) * BQ + row] = l;
      __syncwarp();
      if (lane == 0) mbar_arrive(&fin[q]);
      ok = __all_sync(0xffffffffu, mbar_wait(&fin[q], 0, abort_flag, err, 34));
    }
    if (ok) {
      tc_fence_after();
      const float m_o = xch[(1 - h) * BQ + row], l_o = xch[(3 - h) * BQ + row];
      const float M = fmaxf(m_used, m_o);
      const float a_s = (m_used == -INFINITY) ? 0.f : ex2_approx(m_used - M);
      const float a_o = (m_o == -INFINITY) ? 0.f : ex2_approx(m_o - M);
      const float inv = 1.f / (l * a_s + l_o * a_o);
      const int tok = q0 + row;
      const int D = a.H * HD;
      __nv_bfloat16* out = nullptr;
      if (tok < a.Lq) {
        out = (tok < a.split)
                  ? static_cast<__nv_bfloat16*>(a.o1) + ((int64_t)blockIdx.z * a.split + tok) * D
                  : static_cast<__nv_bfloat16*>(a.o2) +
                        ((int64_t)blockIdx.z * (a.Lq - a.split) + (tok - a.split)) * D;
        out += blockIdx.y * HD + h * 64;
      }
      // this warp writes channels [64h, 64h+64) from both accumulators
      const uint32_t self_col = tmem + TM_O + h * 128 + h * 64 + lane_off;
      const uint32_t oth_col = tmem + TM_O + (1 - h) * 128 + h * 64 + lane_off;
#pragma unroll 1
      for (int c = 0; c < 2; ++c) {
        uint32_t r1[32], r2[32];
        tmem_ld32(self_col + c * 32, r1);
        tmem_ld32(oth_col + c * 32, r2);
        tmem_ld_wait();
        if (out) {
          float v[32];
#pragma unroll
          for (int i = 0; i < 32; ++i)
            v[i] = (__uint_as_float(r1[i]) * a_s + __uint_as_float(r2[i]) * a_o) * inv;
          store_chunk<__nv_bfloat16, 32>(out + c * 32, v);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == MMA_WARP) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

cudaError_t attention_bf16_tc(const AttnArgs& a, int* err, cudaStream_t s) {
  using namespace fa;
  if (a.Lq == 0 || a.B == 0) return cudaSuccess;
  if (a.hd != HD || a.Lk <= 0) return cudaErrorInvalidValue;
  CUtensorMap tq, tk, tv;
  const uint32_t box[3] = {64, 128, 1};
  const uint64_t dq[3] = {(uint64_t)HD, (uint64_t)a.Lq, (uint64_t)a.B * a.H};
  const uint64_t sq[2] = {(uint64_t)HD * 2, (uint64_t)a.Lq * HD * 2};
  const uint64_t dk[3] = {(uint64_t)HD, (uint64_t)a.Lk, (uint64_t)a.B * a.H};
  const uint64_t sk[2] = {(uint64_t)HD * 2, (uint64_t)a.Lk * HD * 2};
  if (!make_tmap_bf16(&tq, a.q, 3, dq, sq, box) || !make_tmap_bf16(&tk, a.k, 3, dk, sk, box) ||
      !make_tmap_bf16(&tv, a.v, 3, dk, sk, box))
    return cudaErrorInvalidValue;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  dim3 grid((a.Lq + BQ - 1) / BQ, a.H, a.B);
  const float scale_log2 = 1.4426950408889634f / sqrtf((float)HD);
  attn_tc_kernel<<<grid, NUM_THREADS, SMEM_BYTES, s>>>(tq, tk, tv, a, scale_log2, err);
  return cudaGetLastError();
}

}  // namespace dit

static_assert(dit::fa::SMEM_BYTES <= 232448, "attention tile set exceeds 227 KB of shared memory");
