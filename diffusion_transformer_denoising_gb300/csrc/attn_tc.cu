// Bidirectional multi-head attention (no mask), head_dim 128, bf16 in/out,
// fp32 softmax and accumulation, on the 5th-generation tensor cores.
//
// One CTA = 128 query rows of one (batch, head).  Warps 0-3 run the online
// softmax (thread = query row = TMEM lane), warp 4 streams K/V tiles of 128
// keys with TMA through a 3-stage ring, warp 5 issues the MMAs:
//     S_j = Q K_j^T          (SS: both operands in shared memory, K-major)
//     O  += P_j V_j          (TS: P from tensor memory, V N-major in smem)
// Tensor memory (512 columns): S double buffer [0,128) [128,256), O [256,384),
// P double buffer [384,448) [448,512) as packed bf16 pairs.  S_{j+1} is
// computed while the softmax works on S_j.  The running max is updated
// lazily: O is rescaled only when a row's max grows by more than 2^8, so most
// steps never touch O from the CUDA cores.
//
// All waits are bounded (common.cuh); on a timeout the CTA flags *err, waits
// for its own copies and MMAs, frees TMEM and exits.
#include "epilogue.cuh"
#include "tmap.h"

namespace dit {

namespace fa {
constexpr int BQ = 128, BKV = 128, HD = 128, STAGES = 3;
constexpr int TILE_BYTES = BKV * HD * 2;   // 32 KB: two 16 KB swizzle blocks of 64 channels
constexpr int Q_OFF = 0;
constexpr int KV_OFF = TILE_BYTES;
constexpr int STAGE_BYTES = 2 * TILE_BYTES;  // K then V
constexpr int BAR_OFF = KV_OFF + STAGES * STAGE_BYTES;
constexpr int SMEM_BYTES = BAR_OFF + 256 + 1024;
constexpr uint32_t TM_S = 0, TM_O = 256, TM_P = 384;
constexpr uint32_t IDESC_S = umma_idesc_bf16(128, 128, false);
constexpr uint32_t IDESC_O = umma_idesc_bf16(128, 128, true);
constexpr float RESCALE_THRESHOLD = 8.0f;  // log2 units
}  // namespace fa

__global__ void __launch_bounds__(192, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, AttnArgs a, float scale_log2, int* err) {
  using namespace fa;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + BAR_OFF);
  uint64_t* q_full = bars;
  uint64_t* k_full = bars + 1;        // [3]
  uint64_t* v_full = bars + 4;        // [3]
  uint64_t* kv_empty = bars + 7;      // [3]
  uint64_t* s_full = bars + 10;       // [2]
  uint64_t* p_ready = bars + 12;      // [2]
  uint64_t* o_done = bars + 14;
  uint64_t* drain = bars + 15;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 16);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bh = blockIdx.z * a.H + blockIdx.y;
  const int q0 = blockIdx.x * BQ;
  const int nkv = (a.Lk + BKV - 1) / BKV;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&s_full[b], 1);
      mbar_init(&p_ready[b], 4);
    }
    mbar_init(o_done, 1);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 4 && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  if (warp == 5) tmem_alloc(tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 4) {
    // ------------------------------------------------ TMA producer
    int issued[STAGES] = {0, 0, 0};
    bool q_issued = false, ok = true;
    if (lane == 0) {
      mbar_arrive_expect_tx(q_full, TILE_BYTES);
      tma_load_3d(smem + Q_OFF, &tmQ, q_full, 0, q0, bh);
      tma_load_3d(smem + Q_OFF + TILE_BYTES / 2, &tmQ, q_full, 64, q0, bh);
      q_issued = true;
    }
    for (int j = 0; j < nkv; ++j) {
      const int st = j % STAGES;
      const uint32_t ph = (uint32_t)((j / STAGES) & 1);
      if (lane == 0) ok = mbar_wait(&kv_empty[st], ph ^ 1, abort_flag, err, 21);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      if (lane == 0) {
        uint8_t* kb = smem + KV_OFF + st * STAGE_BYTES;
        mbar_arrive_expect_tx(&k_full[st], TILE_BYTES);
        tma_load_3d(kb, &tmK, &k_full[st], 0, j * BKV, bh);
        tma_load_3d(kb + TILE_BYTES / 2, &tmK, &k_full[st], 64, j * BKV, bh);
        mbar_arrive_expect_tx(&v_full[st], TILE_BYTES);
        tma_load_3d(kb + TILE_BYTES, &tmV, &v_full[st], 0, j * BKV, bh);
        tma_load_3d(kb + TILE_BYTES + TILE_BYTES / 2, &tmV, &v_full[st], 64, j * BKV, bh);
      }
      ++issued[st];
    }
    if (!ok && lane == 0) {
      volatile int no_abort = 0;
      if (q_issued) mbar_wait(q_full, 0, &no_abort, nullptr, 0);
      for (int s = 0; s < STAGES; ++s)
        if (issued[s] > 0) {
          mbar_wait(&k_full[s], (uint32_t)((issued[s] - 1) & 1), &no_abort, nullptr, 0);
          mbar_wait(&v_full[s], (uint32_t)((issued[s] - 1) & 1), &no_abort, nullptr, 0);
        }
    }
  } else if (warp == 5) {
    // ------------------------------------------------ MMA issuer
    const uint32_t qa = smem_u32(smem + Q_OFF);
    bool ok = true;
    if (lane == 0) ok = mbar_wait(q_full, 0, abort_flag, err, 22);
    ok = __shfl_sync(0xffffffffu, ok, 0);
    auto issue_s = [&](int j) -> bool {
      const int st = j % STAGES;
      bool r = true;
      if (lane == 0) r = mbar_wait(&k_full[st], (uint32_t)((j / STAGES) & 1), abort_flag, err, 23);
      r = __shfl_sync(0xffffffffu, r, 0);
      if (!r) return false;
      tc_fence_after();
      if (lane == 0) {
        const uint32_t ka = smem_u32(smem + KV_OFF + st * STAGE_BYTES);
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk) {
          const uint32_t off = (kk >> 2) * (TILE_BYTES / 2) + (kk & 3) * 32;
          umma_ss(tmem + TM_S + (j & 1) * 128, umma_desc_sw128(qa + off, 16, 1024),
                  umma_desc_sw128(ka + off, 16, 1024), IDESC_S, kk != 0);
        }
        umma_commit(&s_full[j & 1]);
      }
      __syncwarp();
      return true;
    };
    if (ok) ok = issue_s(0);
    for (int j = 0; ok && j < nkv; ++j) {
      if (j + 1 < nkv) {
        ok = issue_s(j + 1);
        if (!ok) break;
      }
      const int st = j % STAGES;
      if (lane == 0) {
        ok = mbar_wait(&p_ready[j & 1], (uint32_t)((j >> 1) & 1), abort_flag, err, 24) &&
             mbar_wait(&v_full[st], (uint32_t)((j / STAGES) & 1), abort_flag, err, 25);
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      if (lane == 0) {
        const uint32_t va = smem_u32(smem + KV_OFF + st * STAGE_BYTES + TILE_BYTES);
#pragma unroll
        for (int kk = 0; kk < BKV / 16; ++kk) {
          // V tile [128 keys][128 ch]: keys are the K dimension (8-row groups
          // 1 KB apart), channels the N dimension (64-wide halves 16 KB apart).
          umma_ts(tmem + TM_O, tmem + TM_P + (j & 1) * 64 + kk * 8, umma_desc_sw128(va + kk * 2048, 16384, 1024),
                  IDESC_O, (j | kk) != 0);
        }
        umma_commit(&kv_empty[st]);
        umma_commit(o_done);
      }
      __syncwarp();
    }
    if (lane == 0) {
      umma_commit(drain);
      volatile int no_abort = 0;
      mbar_wait(drain, 0, &no_abort, nullptr, 0);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------ softmax warps 0-3
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    float m_used = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < nkv; ++j) {
      if (lane == 0) ok = mbar_wait(&s_full[j & 1], (uint32_t)((j >> 1) & 1), abort_flag, err, 26);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      float s[BKV];
#pragma unroll
      for (int c = 0; c < BKV / 32; ++c) {
        uint32_t r[32];
        tmem_ld32(tmem + TM_S + (j & 1) * 128 + c * 32 + lane_off, r);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) s[c * 32 + i] = __uint_as_float(r[i]);
      }
      const int valid = a.Lk - j * BKV;
      if (valid < BKV) {
#pragma unroll
        for (int i = 0; i < BKV; ++i)
          if (i >= valid) s[i] = -INFINITY;
      }
      float mx = s[0];
#pragma unroll
      for (int i = 1; i < BKV; ++i) mx = fmaxf(mx, s[i]);
      const float m_new = fmaxf(m_used, mx * scale_log2);
      bool need;
      float alpha;
      if (j == 0) {
        need = false;
        alpha = 0.f;
        m_used = m_new;
      } else {
        need = m_new - m_used > RESCALE_THRESHOLD;
        alpha = need ? ex2_approx(m_used - m_new) : 1.f;
        if (need) m_used = m_new;
      }
      float rs = 0.f;
      uint32_t pk[BKV / 2];
#pragma unroll
      for (int i = 0; i < BKV; i += 2) {
        const float p0 = ex2_approx(fmaf(s[i], scale_log2, -m_used));
        const float p1 = ex2_approx(fmaf(s[i + 1], scale_log2, -m_used));
        rs += p0 + p1;
        pk[i / 2] = pack_bf16x2(p0, p1);
      }
      l = l * alpha + rs;
      {
        uint32_t r[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) r[i] = pk[i];
        tmem_st32(tmem + TM_P + (j & 1) * 64 + lane_off, r);
#pragma unroll
        for (int i = 0; i < 32; ++i) r[i] = pk[32 + i];
        tmem_st32(tmem + TM_P + (j & 1) * 64 + 32 + lane_off, r);
      }
      tmem_st_wait();
      if (j > 0) {
        // P_j may only be consumed after O holds P_{j-1} V_{j-1}; rescale then
        if (lane == 0) ok = mbar_wait(o_done, (uint32_t)((j - 1) & 1), abort_flag, err, 27);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        tc_fence_after();
        if (__any_sync(0xffffffffu, need)) {
#pragma unroll 1
          for (int c = 0; c < HD / 32; ++c) {
            uint32_t r[32];
            tmem_ld32(tmem + TM_O + c * 32 + lane_off, r);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
            tmem_st32(tmem + TM_O + c * 32 + lane_off, r);
          }
          tmem_st_wait();
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_ready[j & 1]);
    }
    if (ok) {
      if (lane == 0) ok = mbar_wait(o_done, (uint32_t)((nkv - 1) & 1), abort_flag, err, 28);
      ok = __shfl_sync(0xffffffffu, ok, 0);
    }
    if (ok) {
      tc_fence_after();
      const int t = q0 + warp * 32 + lane;
      const int D = a.H * HD;
      __nv_bfloat16* out = nullptr;
      if (t < a.Lq) {
        out = (t < a.split)
                  ? static_cast<__nv_bfloat16*>(a.o1) + ((int64_t)blockIdx.z * a.split + t) * D
                  : static_cast<__nv_bfloat16*>(a.o2) + ((int64_t)blockIdx.z * (a.Lq - a.split) + (t - a.split)) * D;
        out += blockIdx.y * HD;
      }
      const float inv = 1.f / l;
#pragma unroll 1
      for (int c = 0; c < HD / 32; ++c) {
        uint32_t r[32];
        tmem_ld32(tmem + TM_O + c * 32 + lane_off, r);
        tmem_ld_wait();
        if (out) {
          float v[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]) * inv;
          store_chunk<__nv_bfloat16, 32>(out + c * 32, v);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
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
  attn_tc_kernel<<<grid, 192, SMEM_BYTES, s>>>(tq, tk, tv, a, scale_log2, err);
  return cudaGetLastError();
}

}  // namespace dit
