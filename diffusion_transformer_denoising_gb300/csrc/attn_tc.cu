// Bidirectional multi-head attention (no mask), head_dim 128, bf16 in/out,
// fp32 softmax and accumulation, on the 5th-generation tensor cores.
//
// Two kernels share the method -- per key tile j
//     S_j = Q K_j^T            (tcgen05.mma, A and B from shared memory)
//     P_j = 2^(S_j*c - m)      (softmax warps, bf16, written to tensor memory)
//     O  += P_j V_j            (tcgen05.mma, A = P_j from tensor memory)
// with the online-softmax running row max m and row sum l (c = log2(e)/sqrt(d))
// -- and differ in how a CTA is laid out:
//   attn_tc_kernel    short key ranges (cross-attention over the text tokens,
//                     the joint image attention): 128-key tiles, persistent
//                     CTAs that each walk many (query tile, batch*head) items;
//   attn_wide_kernel  long key ranges (video self-attention): 192-key tiles,
//                     one CTA per item (further down).
//
// attn_tc_kernel: one item = 128 query rows of one (batch, head).
//
// The tensor pipe idles whenever its issuing thread stops issuing (a wait, a
// fence, a commit all leave a gap), and a single chain of MMAs into one
// accumulator does not keep it full.  So two threads issue: one warp the S
// products, another the PV products.  Each waits only for its own inputs, and
// while one waits the other's MMAs keep the pipe busy.  This needs S_{j+2}
// and PV_j to be independent, so P has its own tensor-memory slots:
//     S slots [0,128) [128,256)   P slots [256,320) [320,384)   O [384,512)
// S_{j+2} is issued into slot j%2 as soon as the softmax has copied S_j into
// registers; P_j goes to P slot j%2 once PV_{j-2} has consumed P_{j-2}.
//
// Softmax: 8 warps.  Warp w reads TMEM lane quadrant q = w%4 (query rows
// 32q..32q+31) and key columns [64h, 64h+64) of every tile, h = w/4.  The two
// warps of a quadrant share one O, so they share each row's reference max m.
// Per tile each warp first evaluates 2^(s*c - m) against the current m
// without computing a row max, and raises a flag when a row's tile sum
// exceeds SUM_LIMIT (only then can a p be large).  One 64-thread barrier
// reduction (bar.red.or) tells both warps whether any flag is up; if so (and
// on the first tile) they compute the tile's row max, exchange it in shared
// memory (rounded to bf16: any common reference is exact), move the rows
// whose max grew by more than 2^8 to it (O and l rescaled) and redo those
// rows.  Both warps get the same reduction, so they always take the same
// path and their barriers stay matched.
//
// Two loader warps stream K and V with TMA through rings of KST and VST
// stages (K_j is loaded once S_{j-KST} has completed, V_j once PV_{j-VST}
// has).  Completions are signalled by tcgen05.commit to rings s_done[SR]
// (loader of K), pv_done[PR] (loader of V, O rescale, end) and tile_ready[SR],
// which takes two commits per tile -- S_j from the S thread and PV_{j-2} from
// the PV thread -- so the softmax of tile j makes a single wait for "S_j is
// in tensor memory and P slot j%2 is free".  Every waiter's next completion
// on a barrier needs an action of its own first, so a parity wait never
// aliases.
//
// Persistence: a CTA per item would spend more on start-up (barrier set-up,
// tensor memory, the first Q and K loads) than on the item's few tiles, so
// one CTA per SM walks every gridDim-th item.  Tiles are counted over all of
// a CTA's items, so every ring runs on across item boundaries; the K loader
// refills the Q buffer once the previous item's last S product has
// completed, and the first PV product of an item (which overwrites O) waits
// until the softmax warps have read out the previous item's O (o_free).  The
// output goes through shared memory and TMA tensor stores (three V stages
// make the room).
//
// Per-tile integer work on the softmax path is kept to compares and adds
// (the ring slots and the rotated key tile advance incrementally): a
// division or modulo by a runtime value there costs several percent.
//
// All waits are bounded (common.cuh); on a timeout the CTA flags *err, keeps
// the softmax warps' named barriers matched, waits for its own copies and
// MMAs, frees tensor memory and exits.
#include "epilogue.cuh"
#include "tmap.h"

namespace dit {

namespace fa {
constexpr int BQ = 128, BKV = 128, HD = 128;
// K stages, V stages, and the completion rings of S_j and PV_j.  S runs about
// two tiles ahead of PV, so K needs less lead than V.  A ring must be at least
// as long as the stage count its loader waits on (SR >= KST, PR >= VST) so that
// no parity wait can alias.
constexpr int KST = 2, VST = 3, SR = 3, PR = 4;
constexpr int TILE_BYTES = 128 * HD * 2;   // 32 KB: two 16 KB swizzle blocks of 64 channels
constexpr int Q_OFF = 0;
constexpr int K_OFF = Q_OFF + TILE_BYTES;

// Exchange areas (after the barriers, see Layout): bf16 row maxima
// [2 parities][NQ][128] and, apart from them, the float row sums [NQ][128] an
// item's epilogue combines (a partner warp that has moved on to the next
// item's first tile may already be writing maxima).
// The tiles need 1024-byte alignment.  The dynamic shared window of a kernel
// without static shared memory starts 1024-aligned (checked at entry), so no
// alignment slack is reserved and the total stays under 227 KB.
constexpr int SM_WARPS = 8;                       // softmax warps
constexpr int NQ = SM_WARPS / 4;                  // warps per TMEM lane quadrant
constexpr int KPW = BKV / NQ;                     // key columns per softmax warp
// Each item's output goes through shared memory and TMA: every softmax warp
// stages its 32 rows x 64 channels (4 KB, 128-byte swizzle) and issues one
// tensor store.  (Per-lane 16-byte stores of 32 different rows cost ~3700
// cycles per item, half the time of a 4-tile item.)
struct Layout {
  static constexpr int V_OFF = K_OFF + KST * TILE_BYTES;
  static constexpr int STG_OFF = V_OFF + VST * TILE_BYTES;  // [SM_WARPS][32 rows][128 B]
  static constexpr int STG_BYTES = SM_WARPS * 32 * 128;
  static constexpr int BAR_OFF = STG_OFF + STG_BYTES;
  static constexpr int XCH_OFF = BAR_OFF + 256;
  static constexpr int XSUM_OFF = XCH_OFF + 2 * NQ * BQ * 2;
  static constexpr int SMEM_BYTES = XSUM_OFF + NQ * BQ * 4;
};
static_assert(SR >= KST && PR >= VST && VST <= 4, "completion rings shorter than the stage rings");
constexpr int NUM_THREADS = 32 * (SM_WARPS + 4);  // + K/Q loader, S-MMA, PV-MMA, V loader warps
constexpr int TMA_WARP = SM_WARPS, S_WARP = SM_WARPS + 1, PV_WARP = SM_WARPS + 2, VTMA_WARP = SM_WARPS + 3;
constexpr uint32_t TM_S = 0, TM_P = 256, TM_O = 384;
constexpr uint32_t IDESC_S = umma_idesc_bf16(128, 128, false);
constexpr uint32_t IDESC_O = umma_idesc_bf16(128, 128, true);
// A row moves to a new reference max only when its max grew by more than 2^8.
constexpr float RESCALE_THRESHOLD = 8.0f;  // log2 units
// A tile's exponentials are kept against the running reference max while
// the row's tile sum stays below this (each p <= 2^14, far from overflow:
// bf16 and fp32 keep their relative precision at any such magnitude).
constexpr float SUM_LIMIT = 16384.0f;
// Key ranges of at most this many 128-key tiles run on attn_tc_kernel's
// persistent CTAs (one per SM, each walking several items so that one item's
// start overlaps the previous one's end); longer ones on attn_wide_kernel,
// one CTA per item, whose fixed cost is small next to the item.
constexpr int PERSIST_MAX_KV_TILES = 64;

// tcgen05.ld of 64 columns (one instruction) straight into float registers
DIT_DEV void tmem_ld64f(uint32_t taddr, float (&r)[64]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,"
      "%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,"
      "%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];"
      : "=f"(r[0]), "=f"(r[1]), "=f"(r[2]), "=f"(r[3]), "=f"(r[4]), "=f"(r[5]), "=f"(r[6]), "=f"(r[7]),
        "=f"(r[8]), "=f"(r[9]), "=f"(r[10]), "=f"(r[11]), "=f"(r[12]), "=f"(r[13]), "=f"(r[14]), "=f"(r[15]),
        "=f"(r[16]), "=f"(r[17]), "=f"(r[18]), "=f"(r[19]), "=f"(r[20]), "=f"(r[21]), "=f"(r[22]), "=f"(r[23]),
        "=f"(r[24]), "=f"(r[25]), "=f"(r[26]), "=f"(r[27]), "=f"(r[28]), "=f"(r[29]), "=f"(r[30]), "=f"(r[31]),
        "=f"(r[32]), "=f"(r[33]), "=f"(r[34]), "=f"(r[35]), "=f"(r[36]), "=f"(r[37]), "=f"(r[38]), "=f"(r[39]),
        "=f"(r[40]), "=f"(r[41]), "=f"(r[42]), "=f"(r[43]), "=f"(r[44]), "=f"(r[45]), "=f"(r[46]), "=f"(r[47]),
        "=f"(r[48]), "=f"(r[49]), "=f"(r[50]), "=f"(r[51]), "=f"(r[52]), "=f"(r[53]), "=f"(r[54]), "=f"(r[55]),
        "=f"(r[56]), "=f"(r[57]), "=f"(r[58]), "=f"(r[59]), "=f"(r[60]), "=f"(r[61]), "=f"(r[62]), "=f"(r[63])
      : "r"(taddr));
}

// p = 2^(s*c - m) for the KPW scores of one row, packed to bf16 pairs; returns
// the row sum of the (unrounded) p.  Masked keys (s = -inf) give exactly 0.
template <int NV>
DIT_DEV float exp_tile(const float (&s)[NV], uint32_t (&pk)[NV / 2], float scale_log2, float m) {
  const float2 sc2 = make_float2(scale_log2, scale_log2), nm2 = make_float2(-m, -m);
  float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
  for (int i = 0; i < NV; i += 2) {
    const float2 x = ffma2(make_float2(s[i], s[i + 1]), sc2, nm2);
    const float2 p = make_float2(ex2_approx(x.x), ex2_approx(x.y));
    acc[(i >> 1) & 3] = fadd2(acc[(i >> 1) & 3], p);
    pk[i / 2] = pack_bf16x2(p.x, p.y);
  }
  const float2 a01 = fadd2(acc[0], acc[1]), a23 = fadd2(acc[2], acc[3]);
  return (a01.x + a01.y) + (a23.x + a23.y);
}
}  // namespace fa

// tmO[0] / tmO[1]: the outputs o1 / o2 as [B][rows][H*128] in boxes of
// 64 channels x 32 rows, used when bit 0 / bit 1 of o_tma is set.
struct AttnOutMaps {
  CUtensorMap m[2];
};

__global__ void __launch_bounds__(fa::NUM_THREADS, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const __grid_constant__ AttnOutMaps tmO, int o_tma,
                   AttnArgs a, float scale_log2, int* err) {
  using namespace fa;
  using Lay = Layout;
  extern __shared__ __align__(1024) uint8_t smem[];
  if (smem_u32(smem) & 1023) {  // uniform across the CTA: nothing has started yet
    if (threadIdx.x == 0) atomicCAS(err, 0, 20);
    return;
  }
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Lay::BAR_OFF);
  uint64_t* q_full = bars;         // Q tile
  uint64_t* kf = bars + 1;              // [KST] K stage loaded
  uint64_t* vf = kf + KST;              // [VST] V stage loaded
  uint64_t* s_done = vf + VST;          // [SR] S_j complete (ring by j % SR)
  uint64_t* pv_done = s_done + SR;      // [PR] PV_j complete (ring by j % PR)
  uint64_t* s_free = pv_done + PR;      // [2] softmax has copied S slot j % 2 (one arrival per softmax warp)
  uint64_t* p_ready = s_free + 2;       // [2] P slot j % 2 written (one arrival per softmax warp)
  uint64_t* drain = p_ready + 2;        // [2] final commit of each MMA thread
  uint64_t* tile_ready = drain + 2;     // [SR] S_G and PV_{G-2} complete (two commits)
  uint64_t* o_free = tile_ready + SR;   // O of an item read out (one arrival per softmax warp)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(o_free + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  __nv_bfloat16* xmax = reinterpret_cast<__nv_bfloat16*>(smem + Lay::XCH_OFF);
  float* xsum = reinterpret_cast<float*>(smem + Lay::XSUM_OFF);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nq = (a.Lq + BQ - 1) / BQ;
  const int nkv = (a.Lk + BKV - 1) / BKV;
  // the key tile that has fewer than BKV keys, if any (its masked columns
  // read -inf)
  const int partial_jt = (a.Lk % BKV) ? nkv - 1 : -1;
  // An item is one (query tile, batch*head).  The CTA takes items
  // blockIdx.x, + gridDim.x, ... (the grid never exceeds the item count).
  // Key tiles are counted over all items of the CTA (G), so every ring runs
  // on across item boundaries.
  const int n_items = a.B * a.H * nq;
  const int my_items = (n_items - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x;
  auto item_bh = [&](int k) -> int { return ((int)blockIdx.x + k * (int)gridDim.x) / nq; };
  auto item_qt = [&](int k) -> int { return ((int)blockIdx.x + k * (int)gridDim.x) % nq; };
  // Each item walks the key tiles in a rotated order (the result does not
  // depend on the order), so items running together read different K/V tiles.
  auto item_rot = [&](int k) -> int { return item_qt(k) % nkv; };

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int i = 0; i < KST; ++i) mbar_init(&kf[i], 1);
    for (int i = 0; i < VST; ++i) mbar_init(&vf[i], 1);
    for (int i = 0; i < SR; ++i) mbar_init(&s_done[i], 1);
    for (int i = 0; i < PR; ++i) mbar_init(&pv_done[i], 1);
    for (int i = 0; i < SR; ++i) mbar_init(&tile_ready[i], 2);
    // tiles 0 and 1 have no PV_{j-2}: its arrival is made up front
    mbar_arrive(&tile_ready[0]);
    mbar_arrive(&tile_ready[1 % SR]);
    mbar_init(o_free, SM_WARPS);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&s_free[b], SM_WARPS);
      mbar_init(&p_ready[b], SM_WARPS);
      mbar_init(&drain[b], 1);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == TMA_WARP && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  if (warp == S_WARP) tmem_alloc(tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == TMA_WARP || warp == VTMA_WARP) {
    // ------------------------------------------------ TMA producers (one thread each)
    // K and V run on separate threads: S runs about two tiles ahead of PV,
    // so a K load must not queue behind the wait for a V stage.  The K
    // thread also loads each item's Q tile, once the previous item's last
    // S product has read the buffer.
    if (lane == 0) {
      const bool is_k = warp == TMA_WARP;
      const CUtensorMap* tm = is_k ? &tmK : &tmV;
      uint64_t* full = is_k ? kf : vf;
      uint64_t* consumed = is_k ? s_done : pv_done;
      const int nst = is_k ? KST : VST, ring = is_k ? SR : PR;
      uint8_t* stages = smem + (is_k ? K_OFF : Lay::V_OFF);
      int issued[4] = {0, 0, 0, 0};
      int q_issued = 0;
      bool ok = true;
      int G = 0;
      for (int k = 0; ok && k < my_items; ++k) {
        const int bh = item_bh(k), qt = item_qt(k), kv_rot = item_rot(k);
        if (is_k) {
          if (k > 0) {
            const int c = G - 1;  // the previous item's last S product
            ok = mbar_wait(&s_done[c % SR], (uint32_t)((c / SR) & 1), abort_flag, err, 21);
            if (!ok) break;
          }
          mbar_arrive_expect_tx(q_full, TILE_BYTES);
          tma_load_3d(smem + Q_OFF, &tmQ, q_full, 0, qt * BQ, bh);
          tma_load_3d(smem + Q_OFF + TILE_BYTES / 2, &tmQ, q_full, 64, qt * BQ, bh);
          ++q_issued;
        }
        if (!DIT_BOUNDS(bh >= 0 && bh < a.B * a.H && qt >= 0 && qt < nq && kv_rot >= 0 && kv_rot < nkv, err, 62)) {
          *abort_flag = 1;  // every other wait of the CTA returns at once
          ok = false;
          break;
        }
        for (int j = 0; j < nkv; ++j, ++G) {
          // stage G % nst was last read by S_{G-nst} (K) or PV_{G-nst} (V)
          if (G >= nst) {
            const int c = G - nst;
            ok = mbar_wait(&consumed[c % ring], (uint32_t)((c / ring) & 1), abort_flag, err, is_k ? 21 : 22);
            if (!ok) break;
          }
          const int jt = j + kv_rot < nkv ? j + kv_rot : j + kv_rot - nkv;
          uint8_t* dst = stages + (G % nst) * TILE_BYTES;
          mbar_arrive_expect_tx(&full[G % nst], TILE_BYTES);
          tma_load_3d(dst, tm, &full[G % nst], 0, jt * BKV, bh);
          tma_load_3d(dst + TILE_BYTES / 2, tm, &full[G % nst], 64, jt * BKV, bh);
          ++issued[G % nst];
        }
      }
      if (!ok) {
        // wind down: every copy this thread started lands before the CTA exits
        volatile int no_abort = 0;
        if (q_issued > 0) mbar_wait(q_full, (uint32_t)((q_issued - 1) & 1), &no_abort, nullptr, 0);
        for (int st = 0; st < nst; ++st)
          if (issued[st] > 0) mbar_wait(&full[st], (uint32_t)((issued[st] - 1) & 1), &no_abort, nullptr, 0);
      }
    }
    __syncwarp();
  } else if (warp == S_WARP) {
    // ------------------------------------------------ S = Q K^T issuer (one thread)
    if (lane == 0) {
      const uint64_t q_desc = umma_desc_sw128(smem_u32(smem + Q_OFF), 16, 1024);
      const uint64_t k_desc = umma_desc_sw128(smem_u32(smem + K_OFF), 16, 1024);
      bool ok = true;
      int G = 0;
      for (int k = 0; ok && k < my_items; ++k) {
        // Q of item k
        ok = mbar_wait(q_full, (uint32_t)(k & 1), abort_flag, err, 23);
        for (int j = 0; ok && j < nkv; ++j, ++G) {
          // slot G%2 is free once the softmax has copied S_{G-2}
          if (G >= 2) ok = mbar_wait(&s_free[G & 1], (uint32_t)(((G - 2) >> 1) & 1), abort_flag, err, 24);
          ok = ok && mbar_wait(&kf[G % KST], (uint32_t)((G / KST) & 1), abort_flag, err, 25);
          if (!ok) break;
          tc_fence_after();
          const uint64_t kd = umma_desc_add(k_desc, (G % KST) * TILE_BYTES);
          const uint32_t d_tmem = tmem + TM_S + (G & 1) * 128;
#pragma unroll
          for (int kk = 0; kk < HD / 16; ++kk) {
            const uint32_t off = (kk >> 2) * (TILE_BYTES / 2) + (kk & 3) * 32;
            umma_ss(d_tmem, umma_desc_add(q_desc, off), umma_desc_add(kd, off), IDESC_S, kk != 0);
          }
          umma_commit(&s_done[G % SR]);
          umma_commit(&tile_ready[G % SR]);
        }
      }
      // all MMAs issued by this thread complete before tensor memory is released
      umma_commit(&drain[0]);
      volatile int no_abort = 0;
      mbar_wait(&drain[0], 0, &no_abort, nullptr, 0);
    }
    __syncwarp();
  } else if (warp == PV_WARP) {
    // ------------------------------------------------ O += P V issuer (one thread)
    if (lane == 0) {
      const uint64_t v_desc = umma_desc_sw128(smem_u32(smem + Lay::V_OFF), 16384, 1024);
      bool ok = true;
      int G = 0;
      for (int k = 0; ok && k < my_items; ++k) {
        for (int j = 0; ok && j < nkv; ++j, ++G) {
          ok = mbar_wait(&p_ready[G & 1], (uint32_t)((G >> 1) & 1), abort_flag, err, 26) &&
               mbar_wait(&vf[G % VST], (uint32_t)((G / VST) & 1), abort_flag, err, 27);
          // the first product of an item overwrites O: the previous item's O
          // must have been read out
          if (j == 0 && k > 0) ok = ok && mbar_wait(o_free, (uint32_t)((k - 1) & 1), abort_flag, err, 28);
          if (!ok) break;
          tc_fence_after();
          const uint64_t vd = umma_desc_add(v_desc, (G % VST) * TILE_BYTES);
          const uint32_t p_tmem = tmem + TM_P + (G & 1) * 64;
#pragma unroll
          for (int kk = 0; kk < BKV / 16; ++kk) {
            // keys 16kk..16kk+15: P columns 8kk.. (bf16 pairs), V rows 16kk.. (8-row groups 1 KB apart)
            umma_ts(tmem + TM_O, p_tmem + kk * 8, umma_desc_add(vd, kk * 2048), IDESC_O, (j | kk) != 0);
          }
          umma_commit(&pv_done[G % PR]);
          umma_commit(&tile_ready[(G + 2) % SR]);
        }
      }
      umma_commit(&drain[1]);
      volatile int no_abort = 0;
      mbar_wait(&drain[1], 0, &no_abort, nullptr, 0);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------ softmax warps
    const int q = warp & 3, h = warp >> 2;
    const uint32_t lane_off = (uint32_t)(q * 32) << 16;
    const uint32_t o_col = tmem + TM_O + h * KPW + lane_off;  // this warp's O (and output) channels
    const int row = q * 32 + lane;
    bool ok = true;
    int G = 0;
    int tr_slot = 0;
    uint32_t tr_phase = 0;  // tile_ready slot G % SR and its parity
    for (int k = 0; k < my_items; ++k) {
    const int kv_rot = item_rot(k);
    int jt = kv_rot;  // key tile of the item's tile j
    float m_used = -INFINITY, l = 0.f;
    // The loop never breaks: after a failed wait the warp skips the work but
    // still meets its quadrant partners at every named barrier.
    for (int j = 0; j < nkv; ++j, ++G, jt = (jt + 1 == nkv) ? 0 : jt + 1) {
      float s[KPW];
      uint32_t pk[KPW / 2];
      float tsum = 0.f;
      bool big = true;  // a warp that skipped its work asks for the slow path
      bool p_stored = false;
      const uint32_t p_col = tmem + TM_P + (G & 1) * 64 + h * (KPW / 2) + lane_off;
      ok = ok && mbar_wait_warp(&tile_ready[tr_slot], tr_phase, abort_flag, err, 31);
      if (++tr_slot == SR) {
        tr_slot = 0;
        tr_phase ^= 1u;
      }
      if (ok) {
        tc_fence_after();
        {
          static_assert(KPW == 64, "one 64-column load per tile");
          tmem_ld64f(tmem + TM_S + (G & 1) * 128 + h * KPW + lane_off, s);
          tmem_ld_wait();
        }
        // S slot j%2 may now take S_{j+2}
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&s_free[G & 1]);
        // only the last key tile can be partial
        if (jt == partial_jt) {
          const int valid = a.Lk - jt * BKV - h * KPW;
#pragma unroll
          for (int i = 0; i < KPW; ++i)
            if (i >= valid) s[i] = -INFINITY;
        }
        // Fast path: the exponentials against the current reference max, no
        // row max.  A row whose tile sum exceeds SUM_LIMIT (so some p may be
        // large) is flagged and redone below against the tile's row max.
        if (j > 0) {
          tsum = exp_tile(s, pk, scale_log2, m_used);
          big = !(tsum <= SUM_LIMIT);
          // P_j goes to tensor memory now, while the quadrant agrees on the
          // path below (the store's latency overlaps the barrier); a slow
          // path stores it again before P_j is signalled
          if constexpr (KPW == 64)
            tmem_st32(p_col, *reinterpret_cast<const uint32_t(*)[32]>(pk));
          else
            tmem_st16(p_col, *reinterpret_cast<const uint32_t(*)[16]>(pk));
          p_stored = true;
        }
      }
      // one barrier of the quadrant's warps that ORs their flags: all of them
      // get the same answer, take the same path and keep the barriers matched
      if (named_bar_or(1 + q, 32 * NQ, big)) {
        // slow path: the row max of the tile over the quadrant's warps
        if (ok) {
          float m4[4] = {s[0], s[1], s[2], s[3]};
#pragma unroll
          for (int i = 4; i + 8 <= KPW - 4; i += 8)
#pragma unroll
            for (int k = 0; k < 4; ++k) m4[k] = fmax3(m4[k], s[i + 2 * k], s[i + 2 * k + 1]);
#pragma unroll
          for (int k = 0; k < 4; ++k) m4[k] = fmaxf(m4[k], s[KPW - 4 + k]);
          xmax[((j & 1) * NQ + h) * BQ + row] =
              __float2bfloat16_rn(fmaxf(fmax3(m4[0], m4[1], m4[2]), m4[3]) * scale_log2);
        }
        named_bar_sync(1 + q, 32 * NQ);
        if (!ok) continue;
        const __nv_bfloat16* xm = xmax + (j & 1) * NQ * BQ + row;
        float m_tile = __bfloat162float(xm[0]);
#pragma unroll
        for (int w = 1; w < NQ; ++w) m_tile = fmaxf(m_tile, __bfloat162float(xm[w * BQ]));
        // rows whose max grew by more than 2^8 (every row of the first tile)
        // move to the tile max; the others keep their fast-path exponentials
        const bool row_big = m_tile - m_used > RESCALE_THRESHOLD;
        const float m_new = row_big ? m_tile : m_used;
        if (j > 0) {
          // O (and l) move to the new reference; O must hold PV_{j-1} first
          ok = mbar_wait_warp(&pv_done[(G - 1) % PR], (uint32_t)(((G - 1) / PR) & 1), abort_flag, err, 32);
          if (!ok) continue;
          tc_fence_after();
          const float alpha = ex2_approx(m_used - m_new);  // 1 for rows kept
          l *= alpha;
#pragma unroll 1
          for (int c = 0; c < KPW / 32; ++c) {
            uint32_t r[32];
            tmem_ld32(o_col + c * 32, r);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
            tmem_st32(o_col + c * 32, r);
          }
        }
        if (row_big) {
          m_used = m_new;
          tsum = exp_tile(s, pk, scale_log2, m_used);
        }
        if (p_stored) tmem_st_wait();  // the early store lands before it is replaced
        p_stored = false;
      }
      if (!ok) continue;
      l += tsum;
      if (!p_stored) {
        if constexpr (KPW == 64)
          tmem_st32(p_col, *reinterpret_cast<const uint32_t(*)[32]>(pk));
        else
          tmem_st16(p_col, *reinterpret_cast<const uint32_t(*)[16]>(pk));
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_ready[G & 1]);
    }
    tmem_st_wait();  // a P store left in flight by a failed wait lands before tensor memory is reused
    // O is final once PV_{nkv-1} has completed
    ok = ok && mbar_wait_warp(&pv_done[(G - 1) % PR], (uint32_t)(((G - 1) / PR) & 1), abort_flag, err, 34);
    // the quadrant's partial row sums (same reference max) go through the
    // row-sum area once every warp of the quadrant has read the previous
    // item's sums from it
    named_bar_sync(1 + q, 32 * NQ);
    xsum[h * BQ + row] = l;
    named_bar_sync(1 + q, 32 * NQ);
    if (ok) {
      tc_fence_after();
      float lt = 0.f;
#pragma unroll
      for (int w = 0; w < NQ; ++w) lt += xsum[w * BQ + row];
      const float inv = 1.f / lt;
      const int tok0 = item_qt(k) * BQ + q * 32;  // the warp's first row
      const int tok = tok0 + lane;
      const int bh = item_bh(k), b = bh / a.H, head = bh - b * a.H;
      const int D = a.H * HD;
      // TMA path: the warp's 32 rows lie in one output (units across the
      // split between o1 and o2 take the per-lane stores; rows past the last
      // token are clipped by the tensor map)
      int map = -1;
      if (tok0 + 32 <= a.split || a.split == a.Lq)
        map = (o_tma & 1) ? 0 : -1;
      else if (tok0 >= a.split)
        map = (o_tma & 2) ? 1 : -1;
      if (map >= 0) {
        if (tok0 < a.Lq && DIT_BOUNDS(bh < a.B * a.H && tok0 >= 0, err, 63)) {
          uint8_t* stg = smem + Lay::STG_OFF + warp * (32 * 128);
          // the staging buffer's previous tensor store has read it
          if (lane == 0) bulk_wait_read0();
          __syncwarp();
          uint8_t* rowp = stg + lane * 128;
#pragma unroll 1
          for (int c = 0; c < KPW / 32; ++c) {
            uint32_t r[32];
            tmem_ld32(o_col + c * 32, r);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              uint4 w;
              w.x = pack_bf16x2(__uint_as_float(r[8 * j + 0]) * inv, __uint_as_float(r[8 * j + 1]) * inv);
              w.y = pack_bf16x2(__uint_as_float(r[8 * j + 2]) * inv, __uint_as_float(r[8 * j + 3]) * inv);
              w.z = pack_bf16x2(__uint_as_float(r[8 * j + 4]) * inv, __uint_as_float(r[8 * j + 5]) * inv);
              w.w = pack_bf16x2(__uint_as_float(r[8 * j + 6]) * inv, __uint_as_float(r[8 * j + 7]) * inv);
              // 128-byte swizzle: 16-byte chunk n of row r sits at chunk n ^ (r % 8)
              *reinterpret_cast<uint4*>(rowp + (((c * 4 + j) ^ (lane & 7)) << 4)) = w;
            }
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            // rows past the end of the output are clipped by the tensor map
            tma_store_3d(&tmO.m[map], stg, head * HD + h * KPW, map == 0 ? tok0 : tok0 - a.split, b);
            bulk_commit();
          }
        }
      } else {
        __nv_bfloat16* out = nullptr;
        if (tok < a.Lq && DIT_BOUNDS(bh < a.B * a.H && tok >= 0, err, 63)) {
          out = (tok < a.split)
                    ? static_cast<__nv_bfloat16*>(a.o1) + ((int64_t)b * a.split + tok) * D
                    : static_cast<__nv_bfloat16*>(a.o2) + ((int64_t)b * (a.Lq - a.split) + (tok - a.split)) * D;
          out += head * HD + h * KPW;
        }
#pragma unroll 1
        for (int c = 0; c < KPW / 32; ++c) {
          uint32_t r[32];
          tmem_ld32(o_col + c * 32, r);
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
    // O may now take the next item's products
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(o_free);
    }
    // every tensor store of this warp has landed before the CTA exits
    if (lane == 0) bulk_wait0();
    __syncwarp();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == S_WARP) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ---------------------------------------------------------------------------
// Long key ranges (self-attention over thousands of tokens): key tiles of 192.
//
// With 128-key tiles (the kernel above, once also used here) a long key range
// is bound by the softmax: each tile costs its eight softmax warps a fixed
// ~600 cycles (the wait for S, the tensor-memory load, the quadrant's barrier,
// the P store) on top of the exponentials, ~1450 cycles in all, while the
// tile's 16 MMAs take ~1070.  Here a tile holds 192 keys and twelve softmax
// warps (three per lane quadrant, 64 keys each) share it: the fixed cost is
// paid once per 192 keys.  Measured on the video self-attention (32760
// tokens, batch 2): ~1900 cycles per 192-key tile, 7.96 ms per launch
// against 8.42 ms with 128-key tiles.
// Tensor memory then holds one S tile, two P slots and O:
//     S [0,192)   P slots [192,288) [288,384)   O [384,512)
// S_{j+1} is issued into the single S tile once every softmax warp has copied
// S_j into registers; P_j goes to slot j%2 once PV_{j-2} has read it.  As in
// the kernel above, two threads issue: one the S products (one chain of
// M128 x N192 MMAs per tile), one the PV products (twelve M128 x N128 MMAs
// into O).  A single thread issuing both was measured at ~2400 cycles per
// tile against ~1600 of MMA work: each MMA it issues holds it for about the
// MMA's duration, so PV_{j-1} and S_{j+1} could never overlap.  With two
// threads the two products interleave in the pipe and both run at its full
// rate.  (Holding PV_{j-1} back until S_{j+1} was issued, so that S_{j+1}
// completes sooner, made the kernel 10 % slower: PV then runs as a lone
// chain of dependent MMAs.)  The softmax of tile j makes one wait, on
// tile_ready (two commits: S_j from the S thread, PV_{j-2} from the PV
// thread).
//
// One loader thread streams Q, then K and V in two stages each (48 KB per
// 192-key tile), in the order their stages free up: K_{t+1} once S_{t-1} has
// completed, V_t once PV_{t-2} has.
//
// The softmax itself is the one above (fast path against the running
// reference max, one bar.red.or per quadrant per tile, row max and rescale
// only when a row's tile sum exceeds SUM_LIMIT), with NQ = 3.  O's 128
// channels are read out (rescale, epilogue) in 32-column chunks, chunk c by
// warp c % 3 of the quadrant.
namespace fw {
constexpr int BQ = 128, BKV = 192, HD = 128;
constexpr int SM_WARPS = 12;
constexpr int NQ = SM_WARPS / 4;   // softmax warps per lane quadrant
constexpr int KPW = BKV / NQ;      // key columns per softmax warp
static_assert(KPW == 64, "one 64-column tensor-memory load per warp and tile");
constexpr int NUM_THREADS = 32 * (SM_WARPS + 3);
constexpr int LOAD_WARP = SM_WARPS, S_WARP = SM_WARPS + 1, PV_WARP = SM_WARPS + 2;
constexpr int Q_BYTES = BQ * HD * 2;         // 32 KB: two 16 KB boxes of 64 channels
constexpr int KV_BOX = BKV * 64 * 2;         // 24 KB: 192 rows x 64 channels
constexpr int KV_BYTES = 2 * KV_BOX;         // one K or V tile
constexpr int STAGES = 2;
constexpr int Q_OFF = 0;
constexpr int K_OFF = Q_OFF + Q_BYTES;
constexpr int V_OFF = K_OFF + STAGES * KV_BYTES;
constexpr int BAR_OFF = V_OFF + STAGES * KV_BYTES;
// bf16 row maxima [2 parities][NQ][BQ]; once the last tile is done the same
// bytes take the float row sums [NQ][BQ] (one item per CTA)
constexpr int XCH_OFF = BAR_OFF + 256;
constexpr int SMEM_BYTES = XCH_OFF + 2 * NQ * BQ * 2;
static_assert(NQ * BQ * 4 <= 2 * NQ * BQ * 2, "row-sum area larger than the row-max area it reuses");
constexpr int SR = 4, PR = 4;  // completion rings of S_j and PV_j (powers of two)
constexpr uint32_t TM_S = 0, TM_P = 192, TM_O = 384;
constexpr uint32_t IDESC_S = umma_idesc_bf16(128, BKV, false);
constexpr uint32_t IDESC_O = umma_idesc_bf16(128, 128, true);
}  // namespace fw

__global__ void __launch_bounds__(fw::NUM_THREADS, 1)
    attn_wide_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV, AttnArgs a, float scale_log2, int* err) {
  using namespace fw;
  using fa::exp_tile;
  using fa::tmem_ld64f;
  extern __shared__ __align__(1024) uint8_t smem[];
  if (smem_u32(smem) & 1023) {  // uniform across the CTA: nothing has started yet
    if (threadIdx.x == 0) atomicCAS(err, 0, 20);
    return;
  }
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + BAR_OFF);
  uint64_t* q_full = bars;              // Q tile
  uint64_t* kf = bars + 1;              // [STAGES] K stage loaded
  uint64_t* vf = kf + STAGES;           // [STAGES] V stage loaded
  uint64_t* s_done = vf + STAGES;       // [SR] S_j complete
  uint64_t* pv_done = s_done + SR;      // [PR] PV_j complete
  uint64_t* tile_ready = pv_done + PR;  // [SR] S_j and PV_{j-2} complete (two commits)
  uint64_t* s_free = tile_ready + SR;   // softmax has copied S_j (one arrival per softmax warp)
  uint64_t* p_ready = s_free + 1;       // [2] P slot j % 2 written (one arrival per softmax warp)
  uint64_t* drain = p_ready + 2;        // [2] final commit of each MMA thread
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  __nv_bfloat16* xmax = reinterpret_cast<__nv_bfloat16*>(smem + XCH_OFF);
  float* xsum = reinterpret_cast<float*>(smem + XCH_OFF);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nkv = (a.Lk + BKV - 1) / BKV;
  const int partial_jt = (a.Lk % BKV) ? nkv - 1 : -1;
  const int qt = (int)blockIdx.x, bh = (int)(blockIdx.z * a.H + blockIdx.y);
  // Key tiles in a rotated order (the result does not depend on it), so the
  // CTAs running together read different K/V tiles.
  const int kv_rot = (int)(blockIdx.x % (unsigned)nkv);

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(&kf[i], 1);
      mbar_init(&vf[i], 1);
    }
    for (int i = 0; i < SR; ++i) mbar_init(&s_done[i], 1);
    for (int i = 0; i < PR; ++i) mbar_init(&pv_done[i], 1);
    for (int i = 0; i < SR; ++i) mbar_init(&tile_ready[i], 2);
    // tiles 0 and 1 have no PV_{j-2}: its arrival is made up front
    mbar_arrive(&tile_ready[0]);
    mbar_arrive(&tile_ready[1]);
    mbar_init(s_free, SM_WARPS);
    mbar_init(&p_ready[0], SM_WARPS);
    mbar_init(&p_ready[1], SM_WARPS);
    mbar_init(&drain[0], 1);
    mbar_init(&drain[1], 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == LOAD_WARP && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  if (warp == S_WARP) tmem_alloc(tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == LOAD_WARP) {
    // ------------------------------------------------ TMA producer (one thread)
    if (lane == 0) {
      int k_issued[STAGES] = {0, 0}, v_issued[STAGES] = {0, 0};
      bool ok = DIT_BOUNDS(bh >= 0 && bh < a.B * a.H && qt >= 0 && qt * BQ < a.Lq && kv_rot < nkv, err, 62);
      if (!ok) *abort_flag = 1;  // every other wait of the CTA returns at once
      auto load_kv = [&](const CUtensorMap* tm, uint64_t* full, uint8_t* dst, int t) {
        const int jt = t + kv_rot < nkv ? t + kv_rot : t + kv_rot - nkv;
        mbar_arrive_expect_tx(full, KV_BYTES);
        tma_load_3d(dst, tm, full, 0, jt * BKV, bh);
        tma_load_3d(dst + KV_BOX, tm, full, 64, jt * BKV, bh);
      };
      if (ok) {
        mbar_arrive_expect_tx(q_full, Q_BYTES);
        tma_load_3d(smem + Q_OFF, &tmQ, q_full, 0, qt * BQ, bh);
        tma_load_3d(smem + Q_OFF + Q_BYTES / 2, &tmQ, q_full, 64, qt * BQ, bh);
        load_kv(&tmK, &kf[0], smem + K_OFF, 0);
        ++k_issued[0];
      }
      for (int t = 0; ok && t < nkv; ++t) {
        if (t + 1 < nkv) {
          // K stage (t+1) % 2 was last read by S_{t-1}
          if (t >= 1) {
            ok = mbar_wait(&s_done[(t - 1) & (SR - 1)], (uint32_t)(((t - 1) / SR) & 1), abort_flag, err, 50);
            if (!ok) break;
          }
          load_kv(&tmK, &kf[(t + 1) & 1], smem + K_OFF + ((t + 1) & 1) * KV_BYTES, t + 1);
          ++k_issued[(t + 1) & 1];
        }
        // V stage t % 2 was last read by PV_{t-2}
        if (t >= 2) {
          ok = mbar_wait(&pv_done[(t - 2) & (PR - 1)], (uint32_t)(((t - 2) / PR) & 1), abort_flag, err, 51);
          if (!ok) break;
        }
        load_kv(&tmV, &vf[t & 1], smem + V_OFF + (t & 1) * KV_BYTES, t);
        ++v_issued[t & 1];
      }
      if (!ok) {
        // wind down: every copy this thread started lands before the CTA exits
        volatile int no_abort = 0;
        if (k_issued[0] > 0) mbar_wait(q_full, 0, &no_abort, nullptr, 0);
        for (int st = 0; st < STAGES; ++st) {
          if (k_issued[st] > 0) mbar_wait(&kf[st], (uint32_t)((k_issued[st] - 1) & 1), &no_abort, nullptr, 0);
          if (v_issued[st] > 0) mbar_wait(&vf[st], (uint32_t)((v_issued[st] - 1) & 1), &no_abort, nullptr, 0);
        }
      }
    }
    __syncwarp();
  } else if (warp == S_WARP) {
    // ------------------------------------------------ S = Q K^T issuer (one thread)
    if (lane == 0) {
      const uint64_t q_desc = umma_desc_sw128(smem_u32(smem + Q_OFF), 16, 1024);
      const uint64_t k_desc = umma_desc_sw128(smem_u32(smem + K_OFF), 16, 1024);
      bool ok = mbar_wait(q_full, 0, abort_flag, err, 52);
      for (int t = 0; ok && t < nkv; ++t) {
        // the S tile is free once every softmax warp has copied S_{t-1}
        if (t >= 1) ok = mbar_wait(s_free, (uint32_t)((t - 1) & 1), abort_flag, err, 56);
        ok = ok && mbar_wait(&kf[t & 1], (uint32_t)((t >> 1) & 1), abort_flag, err, 53);
        if (!ok) break;
        tc_fence_after();
        const uint64_t kd = umma_desc_add(k_desc, (t & 1) * KV_BYTES);
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk) {
          // channels 16kk..16kk+15: 32-byte steps inside a 128-byte swizzled row, boxes of 64 channels
          umma_ss(tmem + TM_S, umma_desc_add(q_desc, (kk >> 2) * (Q_BYTES / 2) + (kk & 3) * 32),
                  umma_desc_add(kd, (kk >> 2) * KV_BOX + (kk & 3) * 32), IDESC_S, kk != 0);
        }
        umma_commit(&s_done[t & (SR - 1)]);
        umma_commit(&tile_ready[t & (SR - 1)]);
      }
      // all MMAs issued by this thread complete before tensor memory is released
      umma_commit(&drain[0]);
      volatile int no_abort = 0;
      mbar_wait(&drain[0], 0, &no_abort, nullptr, 0);
    }
    __syncwarp();
  } else if (warp == PV_WARP) {
    // ------------------------------------------------ O += P V issuer (one thread)
    if (lane == 0) {
      const uint64_t v_desc = umma_desc_sw128(smem_u32(smem + V_OFF), KV_BOX, 1024);
      bool ok = true;
      for (int t = 0; ok && t < nkv; ++t) {
        ok = mbar_wait(&p_ready[t & 1], (uint32_t)((t >> 1) & 1), abort_flag, err, 54) &&
             mbar_wait(&vf[t & 1], (uint32_t)((t >> 1) & 1), abort_flag, err, 55);
        if (!ok) break;
        tc_fence_after();
        const uint64_t vd = umma_desc_add(v_desc, (t & 1) * KV_BYTES);
        const uint32_t p_tmem = tmem + TM_P + (t & 1) * (BKV / 2);
#pragma unroll
        for (int kk = 0; kk < BKV / 16; ++kk)
          // keys 16kk..16kk+15: P columns 8kk.. (bf16 pairs), V rows 16kk.. (8-row groups 1 KB apart)
          umma_ts(tmem + TM_O, p_tmem + kk * 8, umma_desc_add(vd, kk * 2048), IDESC_O, (t | kk) != 0);
        umma_commit(&pv_done[t & (PR - 1)]);
        umma_commit(&tile_ready[(t + 2) & (SR - 1)]);
      }
      umma_commit(&drain[1]);
      volatile int no_abort = 0;
      mbar_wait(&drain[1], 0, &no_abort, nullptr, 0);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------ softmax warps
    const int q = warp & 3, h = warp >> 2;
    const uint32_t lane_off = (uint32_t)(q * 32) << 16;
    const int row = q * 32 + lane;
    bool ok = true;
    float m_used = -INFINITY, l = 0.f;
    int jt = kv_rot;  // key tile of tile j
    // The loop never breaks: after a failed wait the warp skips the work but
    // still meets its quadrant partners at every named barrier.
    for (int j = 0; j < nkv; ++j, jt = (jt + 1 == nkv) ? 0 : jt + 1) {
      float s[KPW];
      uint32_t pk[KPW / 2];
      float tsum = 0.f;
      bool big = true;  // a warp that skipped its work asks for the slow path
      bool p_stored = false;
      const uint32_t p_col = tmem + TM_P + (j & 1) * (BKV / 2) + h * (KPW / 2) + lane_off;
      // S_j complete, and PV_{j-2}: P slot j%2 is free
      ok = ok && mbar_wait_warp(&tile_ready[j & (SR - 1)], (uint32_t)((j / SR) & 1), abort_flag, err, 57);
      if (ok) {
        tc_fence_after();
        tmem_ld64f(tmem + TM_S + h * KPW + lane_off, s);
        tmem_ld_wait();
        // the S tile may now take S_{j+1}
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(s_free);
        if (jt == partial_jt) {
          const int valid = a.Lk - jt * BKV - h * KPW;
#pragma unroll
          for (int i = 0; i < KPW; ++i)
            if (i >= valid) s[i] = -INFINITY;
        }
        if (j > 0) {
          tsum = exp_tile(s, pk, scale_log2, m_used);
          big = !(tsum <= fa::SUM_LIMIT);
          tmem_st32(p_col, *reinterpret_cast<const uint32_t(*)[32]>(pk));
          p_stored = true;
        }
      }
      if (named_bar_or(1 + q, 32 * NQ, big)) {
        // slow path: the row max of the tile over the quadrant's warps
        if (ok) {
          float m4[4] = {s[0], s[1], s[2], s[3]};
#pragma unroll
          for (int i = 4; i + 8 <= KPW - 4; i += 8)
#pragma unroll
            for (int k = 0; k < 4; ++k) m4[k] = fmax3(m4[k], s[i + 2 * k], s[i + 2 * k + 1]);
#pragma unroll
          for (int k = 0; k < 4; ++k) m4[k] = fmaxf(m4[k], s[KPW - 4 + k]);
          xmax[((j & 1) * NQ + h) * BQ + row] =
              __float2bfloat16_rn(fmaxf(fmax3(m4[0], m4[1], m4[2]), m4[3]) * scale_log2);
        }
        named_bar_sync(1 + q, 32 * NQ);
        if (!ok) continue;
        const __nv_bfloat16* xm = xmax + (j & 1) * NQ * BQ + row;
        float m_tile = __bfloat162float(xm[0]);
#pragma unroll
        for (int w = 1; w < NQ; ++w) m_tile = fmaxf(m_tile, __bfloat162float(xm[w * BQ]));
        // rows whose max grew by more than 2^8 (every row of the first tile)
        // move to the tile max; the others keep their fast-path exponentials
        const bool row_big = m_tile - m_used > fa::RESCALE_THRESHOLD;
        const float alpha = row_big ? ex2_approx(m_used - m_tile) : 1.f;  // O's factor: 1 for rows kept
        const bool any_big = __any_sync(0xffffffffu, row_big);
        if (any_big || !p_stored) {
          // P_j again, every lane of the warp (a row that keeps its reference
          // recomputes the same values), from the scores still in registers:
          // the S tile may already hold S_{j+1}
          if (row_big) m_used = m_tile;
          tsum = exp_tile(s, pk, scale_log2, m_used);
          if (p_stored) tmem_st_wait();  // the early store lands before it is replaced
          tmem_st32(p_col, *reinterpret_cast<const uint32_t(*)[32]>(pk));
          p_stored = true;
        }
        if (j > 0 && any_big) {
          // O (and l) move to the new reference; O must hold PV_{j-1} first.
          // (PV_j reads P_j only after p_ready, below.)
          ok = mbar_wait_warp(&pv_done[(j - 1) & (PR - 1)], (uint32_t)(((j - 1) / PR) & 1), abort_flag, err, 57);
          if (!ok) continue;
          tc_fence_after();
          l *= alpha;
#pragma unroll 1
          for (int c = h; c < HD / 32; c += NQ) {
            uint32_t r[32];
            tmem_ld32(tmem + TM_O + c * 32 + lane_off, r);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
            tmem_st32(tmem + TM_O + c * 32 + lane_off, r);
          }
        }
      }
      if (!ok) continue;
      l += tsum;
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_ready[j & 1]);
    }
    tmem_st_wait();  // a P store left in flight by a failed wait lands before tensor memory is reused
    // O is final once PV_{nkv-1} has completed
    ok = ok && mbar_wait_warp(&pv_done[(nkv - 1) & (PR - 1)], (uint32_t)(((nkv - 1) / PR) & 1), abort_flag, err, 57);
    // the quadrant's partial row sums (same reference max) meet in the
    // exchange area once every warp of the quadrant is past its last tile
    named_bar_sync(1 + q, 32 * NQ);
    xsum[h * BQ + row] = l;
    named_bar_sync(1 + q, 32 * NQ);
    if (ok) {
      tc_fence_after();
      float lt = 0.f;
#pragma unroll
      for (int w = 0; w < NQ; ++w) lt += xsum[w * BQ + row];
      const float inv = 1.f / lt;
      const int tok = qt * BQ + row;
      const int b = bh / a.H, head = bh - b * a.H;
      const int D = a.H * HD;
      __nv_bfloat16* out = nullptr;
      if (tok < a.Lq && DIT_BOUNDS(bh < a.B * a.H && tok >= 0, err, 63)) {
        out = (tok < a.split)
                  ? static_cast<__nv_bfloat16*>(a.o1) + ((int64_t)b * a.split + tok) * D
                  : static_cast<__nv_bfloat16*>(a.o2) + ((int64_t)b * (a.Lq - a.split) + (tok - a.split)) * D;
        out += head * HD;
      }
#pragma unroll 1
      for (int c = h; c < HD / 32; c += NQ) {
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
  if (warp == S_WARP) {
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
  static SmemAttr attr_persist;
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(attn_tc_kernel), Layout::SMEM_BYTES, attr_persist);
  static int sms_of[kMaxDevices] = {};
  int dev = 0;
  if (e == cudaSuccess) e = cudaGetDevice(&dev);
  if (e == cudaSuccess && !sms_of[dev]) e = cudaDeviceGetAttribute(&sms_of[dev], cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const int num_sms = sms_of[dev];
  const int nq = (a.Lq + BQ - 1) / BQ, nkv = (a.Lk + BKV - 1) / BKV;
  const float scale_log2 = 1.4426950408889634f / sqrtf((float)HD);
  if (nkv <= PERSIST_MAX_KV_TILES) {
    // short key ranges: one CTA per SM walking every gridDim-th item, so each
    // item's start overlaps the previous one's end
    const int64_t items = (int64_t)a.B * a.H * nq;
    if (items > INT32_MAX) return cudaErrorInvalidValue;
    const int grid = (int)(items < num_sms ? items : num_sms);
    // output tensor maps [B][rows][H*128]: o1 holds tokens [0, split), o2 the rest
    AttnOutMaps om{};
    int o_tma = 0;
    const uint32_t obox[3] = {64, 32, 1};
    auto omap = [&](CUtensorMap* t, void* base, int rows) -> bool {
      if (!base || rows <= 0 || (reinterpret_cast<uintptr_t>(base) & 15)) return false;
      const uint64_t d[3] = {(uint64_t)a.H * HD, (uint64_t)rows, (uint64_t)a.B};
      const uint64_t st[2] = {(uint64_t)a.H * HD * 2, (uint64_t)rows * a.H * HD * 2};
      return make_tmap_bf16(t, base, 3, d, st, obox);
    };
    if (omap(&om.m[0], a.o1, a.split)) o_tma |= 1;
    if (omap(&om.m[1], a.o2, a.Lq - a.split)) o_tma |= 2;
    attn_tc_kernel<<<grid, NUM_THREADS, Layout::SMEM_BYTES, s>>>(tq, tk, tv, om, o_tma, a, scale_log2, err);
  } else {
    // long key ranges: one CTA per (query tile, batch*head), 192-key tiles
    CUtensorMap tk_w, tv_w;
    const uint32_t box_w[3] = {64, (uint32_t)fw::BKV, 1};
    if (!make_tmap_bf16(&tk_w, a.k, 3, dk, sk, box_w) || !make_tmap_bf16(&tv_w, a.v, 3, dk, sk, box_w))
      return cudaErrorInvalidValue;
    static SmemAttr attr_wide;
    e = ensure_smem_attr(reinterpret_cast<const void*>(attn_wide_kernel), fw::SMEM_BYTES, attr_wide);
    if (e != cudaSuccess) return e;
    dim3 grid(nq, a.H, a.B);
    attn_wide_kernel<<<grid, fw::NUM_THREADS, fw::SMEM_BYTES, s>>>(tq, tk_w, tv_w, a, scale_log2, err);
  }
  return cudaGetLastError();
}

}  // namespace dit

static_assert(dit::fa::Layout::SMEM_BYTES <= 232448 && dit::fw::SMEM_BYTES <= 232448,
              "attention tile set exceeds 227 KB of shared memory");
static_assert(dit::fa::Layout::STG_OFF % 1024 == 0, "swizzled staging buffers need 1024-byte alignment");
