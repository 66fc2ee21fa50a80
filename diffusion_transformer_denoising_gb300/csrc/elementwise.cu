// Memory-bound kernels of the denoiser step: modulated LayerNorm, timestep
// embedding MLP, modulation tables, latent packing, guidance + Euler.
// All use coalesced 128-bit accesses where the layout allows and one warp
// per row for row reductions.
#include <math.h>
#include "common.cuh"
#include "kernels.h"
#include "tmap.h"

namespace dit {

DIT_DEV float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

DIT_DEV float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Quantize a warp's row held as y[NCH] float4 (lane owns float4 c = lane + 32 i
// while c < n4) to e4m3 bytes at dst (row of n4 * 4 bytes) with its scale
// max|row| / 448 written by lane 0 to *row_scale.
template <int NCH>
DIT_DEV void store_row_e4m3(const float4 (&y)[NCH], int n4, uint8_t* dst, float* row_scale) {
  const int lane = threadIdx.x & 31;
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < NCH; ++i)
    if (lane + 32 * i < n4)
      amax = fmaxf(amax, fmaxf(fmaxf(fabsf(y[i].x), fabsf(y[i].y)), fmaxf(fabsf(y[i].z), fabsf(y[i].w))));
  amax = warp_max(amax);
  const float sc = amax > 0.f ? amax / kE4M3Max : 1.f;
  const float inv = amax > 0.f ? kE4M3Max / amax : 1.f;
#pragma unroll
  for (int i = 0; i < NCH; ++i) {
    const int c = lane + 32 * i;
    if (c < n4) reinterpret_cast<uint32_t*>(dst)[c] = pack_e4m3x4(y[i].x * inv, y[i].y * inv, y[i].z * inv, y[i].w * inv);
  }
  if (lane == 0) *row_scale = sc;
}

static inline unsigned blocks_for(int64_t n, int per_block, int cap = 152 * 32) {
  int64_t b = (n + per_block - 1) / per_block;
  if (b < 1) b = 1;
  return (unsigned)(b > cap ? cap : b);
}

// ---------------------------------------------------------------- LayerNorm + adaLN
// One warp per row; the row stays in registers (NCH float4 per lane) so x is
// read once.  Statistics in fp32: mean, then the centred second moment.
template <int NCH, int OUT>
__global__ void __launch_bounds__(256) ln_mod_kernel(const float* __restrict__ x, int64_t rows, int D, int rpb,
                                                     const float* __restrict__ shift,
                                                     const float* __restrict__ scale, int64_t mbs, float eps,
                                                     void* __restrict__ out, float* __restrict__ row_scale) {
  const int lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (row >= rows) return;
  const int n4 = D >> 2;
  const float4* xr = reinterpret_cast<const float4*>(x + row * D);
  float4 v[NCH];
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < NCH; ++i) {
    const int c = lane + 32 * i;
    if (c < n4) {
      v[i] = __ldg(xr + c);
      s += (v[i].x + v[i].y) + (v[i].z + v[i].w);
    } else {
      v[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
  const float mean = warp_sum(s) / (float)D;
  float q = 0.f;
#pragma unroll
  for (int i = 0; i < NCH; ++i) {
    const int c = lane + 32 * i;
    if (c < n4) {
      const float a = v[i].x - mean, b = v[i].y - mean, cc = v[i].z - mean, d = v[i].w - mean;
      q += (a * a + b * b) + (cc * cc + d * d);
    }
  }
  const float rstd = 1.0f / sqrtf(warp_sum(q) / (float)D + eps);
  const int64_t bi = row / rpb;
  const float4* sh4 = shift ? reinterpret_cast<const float4*>(shift + bi * mbs) : nullptr;
  const float4* sc4 = scale ? reinterpret_cast<const float4*>(scale + bi * mbs) : nullptr;
#pragma unroll
  for (int i = 0; i < NCH; ++i) {
    const int c = lane + 32 * i;
    if (c >= n4) continue;
    float4 y = make_float4((v[i].x - mean) * rstd, (v[i].y - mean) * rstd, (v[i].z - mean) * rstd,
                           (v[i].w - mean) * rstd);
    if (sc4) {
      const float4 a = __ldg(sc4 + c), b = __ldg(sh4 + c);
      y.x = fmaf(y.x, 1.f + a.x, b.x);
      y.y = fmaf(y.y, 1.f + a.y, b.y);
      y.z = fmaf(y.z, 1.f + a.z, b.z);
      y.w = fmaf(y.w, 1.f + a.w, b.w);
    }
    if constexpr (OUT == LN_BF16) {
      uint2 u;
      u.x = pack_bf16x2(y.x, y.y);
      u.y = pack_bf16x2(y.z, y.w);
      reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(out) + row * D)[c] = u;
    } else if constexpr (OUT == LN_F32) {
      reinterpret_cast<float4*>(static_cast<float*>(out) + row * D)[c] = y;
    } else {
      v[i] = y;  // quantized below, once the row's max is known
    }
  }
  if constexpr (OUT == LN_E4M3) store_row_e4m3<NCH>(v, n4, static_cast<uint8_t*>(out) + row * D, row_scale + row);
}

// bf16-output variant with the rows staged in shared memory by bulk copies.
// One CTA per SM walks rows blockIdx.x, blockIdx.x + gridDim.x, ...; lane 0
// of warp 0 keeps up to `stages` rows in flight (bulk copies into a ring of
// row slots), and each of the LN_CONSUMERS other warps takes every
// LN_CONSUMERS-th row of the CTA: it moves the row from its slot into
// registers (the slot goes back to the copier at once), forms the mean and
// the centred variance with warp shuffles and writes the modulated bf16 row.
// The modulation of every batch element (shift and 1 + scale) is copied to
// shared memory once per CTA.  Against the register-resident kernel above,
// which issues a warp's loads only when the warp starts and re-reads 2 D
// floats of modulation per row through L1, each SM keeps ~100-150 KB of reads
// in flight while its warps compute.  One launch may normalise two row sets
// of the same width (the image and condition streams of a dual-stream
// block): their rows are numbered back to back.
constexpr int LN_CONSUMERS = 8;
constexpr int LN_STAGED_THREADS = 32 * (1 + LN_CONSUMERS);
constexpr int LN_MOD_SMEM = 96 * 1024;   // modulation of all batch elements, at most
constexpr int LN_RING_SMEM = 200 * 1024; // ring + modulation

struct LnSeg {
  const float* x = nullptr;        // [rows, D]
  void* out = nullptr;             // [rows, D] bf16, or e4m3 bytes with row_scale[rows]
  float* row_scale = nullptr;
  const float* shift = nullptr;    // [batch] rows of stride mbs; NULL in both segments = plain LN
  const float* scale = nullptr;
  int64_t mbs = 0;
  int rows = 0, rpb = 1;
  int mod0 = 0;                    // first modulation entry of this segment in shared memory
};
struct LnSegs {
  LnSeg s[2];
  int nmod = 0;                    // modulation entries (batch elements of both segments)
};

template <int NCH, bool F8>
__global__ void __launch_bounds__(LN_STAGED_THREADS, 1)
    ln_mod_staged_kernel(const __grid_constant__ LnSegs P, int D, float eps, int stages, int* err) {
  extern __shared__ __align__(16) uint8_t ln_smem[];
  const bool modulate = P.s[0].shift != nullptr;
  float* ring = reinterpret_cast<float*>(ln_smem);
  float4* smod = reinterpret_cast<float4*>(ln_smem + (size_t)stages * D * 4);  // [nmod][2][D/4]
  const int n4 = D >> 2;
  const size_t mod_f4 = modulate ? (size_t)P.nmod * 2 * n4 : 0;
  uint64_t* full = reinterpret_cast<uint64_t*>(smod + mod_f4);
  uint64_t* empty = full + stages;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + stages);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rows0 = P.s[0].rows, rows = rows0 + P.s[1].rows;
  if (threadIdx.x == 0) {
    for (int i = 0; i < stages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (modulate) {
    for (int i = threadIdx.x; i < P.nmod * n4; i += blockDim.x) {
      const int e = i / n4, c = i - e * n4;
      const int sg = e >= P.s[1].mod0 && P.s[1].rows > 0 ? 1 : 0;
      const LnSeg& g = P.s[sg];
      const int64_t b = e - g.mod0;
      const float4 a = __ldg(reinterpret_cast<const float4*>(g.scale + b * g.mbs) + c);
      smod[(size_t)(2 * e) * n4 + c] = __ldg(reinterpret_cast<const float4*>(g.shift + b * g.mbs) + c);
      smod[(size_t)(2 * e + 1) * n4 + c] = make_float4(1.f + a.x, 1.f + a.y, 1.f + a.z, 1.f + a.w);
    }
  }
  __syncthreads();
  const int nloc = rows > (int)blockIdx.x ? (rows - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
  if (warp == 0) {
    // ------------------------------------------------ copier (one thread)
    if (lane == 0) {
      const uint32_t row_bytes = (uint32_t)D * 4u;
      int issued = 0, slot = 0;
      uint32_t use = 0;
      bool ok = true;
      for (int k = 0; k < nloc; ++k) {
        if (use > 0) {
          ok = mbar_wait(&empty[slot], (use - 1) & 1, abort_flag, err, 41);
          if (!ok) break;
        }
        const int row = (int)blockIdx.x + k * (int)gridDim.x;
        if (!DIT_BOUNDS(row >= 0 && row < rows && slot >= 0 && slot < stages, err, 64)) {
          *abort_flag = 1;
          ok = false;
          break;
        }
        const float* src = row < rows0 ? P.s[0].x + (int64_t)row * D : P.s[1].x + (int64_t)(row - rows0) * D;
        mbar_arrive_expect_tx(&full[slot], row_bytes);
        bulk_load(ring + (size_t)slot * D, src, row_bytes, &full[slot]);
        ++issued;
        if (++slot == stages) {
          slot = 0;
          ++use;
        }
      }
      if (!ok) {
        // wind down: the last copy into each slot lands before the CTA exits
        volatile int no_abort = 0;
        for (int sl = 0; sl < stages && sl < issued; ++sl)
          mbar_wait(&full[sl], (uint32_t)((issued - 1 - sl) / stages) & 1, &no_abort, nullptr, 0);
      }
    }
    return;
  }
  // -------------------------------------------------- consumer warps
  const float inv_d = 1.0f / (float)D;
  for (int k = warp - 1; k < nloc; k += LN_CONSUMERS) {
    const int slot = k % stages;
    if (!mbar_wait_warp(&full[slot], (uint32_t)(k / stages) & 1, abort_flag, err, 42)) break;
    const float4* src = reinterpret_cast<const float4*>(ring + (size_t)slot * D);
    float4 v[NCH];
    float sum = 0.f;
#pragma unroll
    for (int i = 0; i < NCH; ++i) {
      const int c = lane + 32 * i;
      if (c < n4) {
        v[i] = src[c];
        sum += (v[i].x + v[i].y) + (v[i].z + v[i].w);
      } else {
        v[i] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[slot]);
    const float mean = warp_sum(sum) * inv_d;
    float q = 0.f;
#pragma unroll
    for (int i = 0; i < NCH; ++i) {
      const int c = lane + 32 * i;
      if (c < n4) {
        const float a = v[i].x - mean, b = v[i].y - mean, cc = v[i].z - mean, d = v[i].w - mean;
        q += (a * a + b * b) + (cc * cc + d * d);
      }
    }
    const float rstd = 1.0f / sqrtf(warp_sum(q) * inv_d + eps);
    const int row = (int)blockIdx.x + k * (int)gridDim.x;
    const int sg = row < rows0 ? 0 : 1;
    const int lr = row - sg * rows0;
    const LnSeg& g = P.s[sg];
    const int e = g.mod0 + lr / g.rpb;
    if (!DIT_BOUNDS(lr >= 0 && lr < g.rows && (!modulate || (e >= 0 && e < P.nmod)), err, 65)) break;
    const float4* sh4 = smod + (size_t)(2 * e) * n4;
    const float4* sc4 = sh4 + n4;
    uint2* dst = reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(g.out) + (int64_t)lr * D);
#pragma unroll
    for (int i = 0; i < NCH; ++i) {
      const int c = lane + 32 * i;
      if (c >= n4) continue;
      float4 y = make_float4((v[i].x - mean) * rstd, (v[i].y - mean) * rstd, (v[i].z - mean) * rstd,
                             (v[i].w - mean) * rstd);
      if (modulate) {
        const float4 a = sc4[c], b = sh4[c];
        y.x = fmaf(y.x, a.x, b.x);
        y.y = fmaf(y.y, a.y, b.y);
        y.z = fmaf(y.z, a.z, b.z);
        y.w = fmaf(y.w, a.w, b.w);
      }
      if constexpr (F8) {
        v[i] = y;  // quantized below, once the row's max is known
      } else {
        uint2 u;
        u.x = pack_bf16x2(y.x, y.y);
        u.y = pack_bf16x2(y.z, y.w);
        dst[c] = u;
      }
    }
    if constexpr (F8) store_row_e4m3<NCH>(v, n4, static_cast<uint8_t*>(g.out) + (int64_t)lr * D, g.row_scale + lr);
  }
}

// Staged launch over one or two segments; false (nothing launched) when the
// modulation of all batch elements does not fit its shared-memory budget.
// Ring: what is left of ~200 KB, at most 24 rows (144 KB of 1536-wide rows,
// more than one SM needs in flight to cover DRAM latency at its share of the
// bandwidth), a multiple of LN_CONSUMERS; one CTA per SM (fewer when there
// are fewer rows).
template <int NCH, bool F8>
static bool ln_staged_launch(LnSegs P, int D, float eps, int* err, int num_sms, cudaStream_t s, cudaError_t* status) {
  const int row_bytes = D * 4;
  int nmod = 0;
  for (int i = 0; i < 2; ++i) {
    P.s[i].mod0 = nmod;
    if (P.s[i].rows > 0) nmod += (P.s[i].rows + P.s[i].rpb - 1) / P.s[i].rpb;
  }
  P.nmod = nmod;
  const size_t mod_bytes = P.s[0].shift ? (size_t)nmod * 2 * D * 4 : 0;
  if (mod_bytes > (size_t)LN_MOD_SMEM) return false;
  // The ring holds a multiple of LN_CONSUMERS rows, so slot s only ever
  // holds rows of consumer warp s % LN_CONSUMERS, which takes its rows in
  // order: a warp then never waits on a slot whose previous fill it has not
  // consumed itself, and the one-bit phase parity of the slot barriers cannot
  // alias (a warp running two fills ahead of the copier would otherwise pass
  // a stale phase and arrive on the slot twice).
  int stages = (int)((LN_RING_SMEM - mod_bytes) / row_bytes);
  if (stages > 24) stages = 24;
  stages -= stages % LN_CONSUMERS;
  if (stages < LN_CONSUMERS) return false;
  const size_t smem = (size_t)stages * row_bytes + mod_bytes + 2 * sizeof(uint64_t) * stages + 16;
  static SmemAttr attr;
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(ln_mod_staged_kernel<NCH, F8>), (int)smem, attr);
  if (e != cudaSuccess) {
    *status = e;
    return true;
  }
  const int rows = P.s[0].rows + P.s[1].rows;
  const int grid = rows < num_sms ? rows : num_sms;
  ln_mod_staged_kernel<NCH, F8><<<grid, LN_STAGED_THREADS, smem, s>>>(P, D, eps, stages, err);
  *status = cudaGetLastError();
  return true;
}

// The staged kernel takes a segment whose x is 16-byte and out 8-byte aligned.
static bool staged_ok(const LnArgs& a) {
  return (reinterpret_cast<uintptr_t>(a.x) & 15) == 0 && (reinterpret_cast<uintptr_t>(a.out) & 7) == 0;
}

static bool ln_staged(const LnArgs* a, int nseg, int D, float eps, int* err, int num_sms, cudaStream_t s,
                      cudaError_t* status, bool f8) {
  LnSegs P;
  int64_t rows = 0;
  for (int i = 0; i < nseg; ++i) {
    if (!staged_ok(a[i]) || a[i].rpb <= 0) return false;
    if (i > 0 && (a[i].shift == nullptr) != (a[0].shift == nullptr)) return false;
    if (f8 && !a[i].row_scale) return false;
    P.s[i].x = a[i].x;
    P.s[i].out = a[i].out;
    P.s[i].row_scale = a[i].row_scale;
    P.s[i].shift = a[i].shift;
    P.s[i].scale = a[i].scale;
    P.s[i].mbs = a[i].mbs;
    P.s[i].rows = (int)a[i].rows;
    P.s[i].rpb = a[i].rpb;
    rows += a[i].rows;
  }
  if (rows >= (int64_t)1 << 31) return false;
  const int nch = (D / 4 + 31) / 32;
  if (f8) {
    if (nch <= 4) return ln_staged_launch<4, true>(P, D, eps, err, num_sms, s, status);
    if (nch <= 12) return ln_staged_launch<12, true>(P, D, eps, err, num_sms, s, status);
    if (nch <= 24) return ln_staged_launch<24, true>(P, D, eps, err, num_sms, s, status);
    return false;
  }
  if (nch <= 4) return ln_staged_launch<4, false>(P, D, eps, err, num_sms, s, status);
  if (nch <= 12) return ln_staged_launch<12, false>(P, D, eps, err, num_sms, s, status);
  if (nch <= 24) return ln_staged_launch<24, false>(P, D, eps, err, num_sms, s, status);
  return false;
}

template <int NCH>
static cudaError_t ln_launch(const float* x, int64_t rows, int D, int rpb, const float* sh, const float* sc,
                             int64_t mbs, float eps, void* out, int out_kind, float* row_scale, cudaStream_t s) {
  const unsigned grid = (unsigned)((rows + 7) / 8);
  if (out_kind == LN_BF16)
    ln_mod_kernel<NCH, LN_BF16><<<grid, 256, 0, s>>>(x, rows, D, rpb, sh, sc, mbs, eps, out, row_scale);
  else if (out_kind == LN_E4M3)
    ln_mod_kernel<NCH, LN_E4M3><<<grid, 256, 0, s>>>(x, rows, D, rpb, sh, sc, mbs, eps, out, row_scale);
  else
    ln_mod_kernel<NCH, LN_F32><<<grid, 256, 0, s>>>(x, rows, D, rpb, sh, sc, mbs, eps, out, row_scale);
  return cudaGetLastError();
}

cudaError_t ln_modulate(const float* x, int64_t rows, int D, int rpb, const float* shift, const float* scale,
                        int64_t mbs, float eps, void* out, int out_kind, int* err, int num_sms, cudaStream_t s,
                        float* row_scale) {
  if (rows == 0) return cudaSuccess;
  if (D % 4) return cudaErrorInvalidValue;
  if (out_kind == LN_E4M3 && (!row_scale || (reinterpret_cast<uintptr_t>(out) & 3))) return cudaErrorInvalidValue;
  if (out_kind != LN_F32) {
    LnArgs a{x, rows, rpb, shift, scale, mbs, out};
    a.row_scale = row_scale;
    cudaError_t st = cudaSuccess;
    if (ln_staged(&a, 1, D, eps, err, num_sms, s, &st, out_kind == LN_E4M3)) return st;
  }
  const int nch = (D / 4 + 31) / 32;
#define DIT_LN_CASE(n) \
  if (nch <= n) return ln_launch<n>(x, rows, D, rpb, shift, scale, mbs, eps, out, out_kind, row_scale, s);
  DIT_LN_CASE(1)
  DIT_LN_CASE(2)
  DIT_LN_CASE(4)
  DIT_LN_CASE(8)
  DIT_LN_CASE(12)
  DIT_LN_CASE(16)
  DIT_LN_CASE(24)
  DIT_LN_CASE(32)
#undef DIT_LN_CASE
  return cudaErrorInvalidValue;
}

cudaError_t ln_modulate_pair(const LnArgs& a, const LnArgs& b, int D, float eps, int out_kind, int* err,
                             int num_sms, cudaStream_t s, int* launches) {
  if (D % 4) return cudaErrorInvalidValue;
  *launches = 1;
  if (out_kind != LN_F32 && a.rows > 0 && b.rows > 0) {
    const LnArgs ab[2] = {a, b};
    cudaError_t st = cudaSuccess;
    if (ln_staged(ab, 2, D, eps, err, num_sms, s, &st, out_kind == LN_E4M3)) return st;
  }
  *launches = (a.rows > 0) + (b.rows > 0);
  cudaError_t e = ln_modulate(a.x, a.rows, D, a.rpb, a.shift, a.scale, a.mbs, eps, a.out, out_kind, err, num_sms, s,
                              a.row_scale);
  if (e != cudaSuccess) return e;
  return ln_modulate(b.x, b.rows, D, b.rpb, b.shift, b.scale, b.mbs, eps, b.out, out_kind, err, num_sms, s,
                     b.row_scale);
}

// ---------------------------------------------------------------- weight quantization
// One warp per row: max |w| over the row, then w * 448 / max to e4m3.
template <typename T>
__global__ void __launch_bounds__(256) quantize_rows_kernel(const T* __restrict__ src, int64_t rows, int K,
                                                            uint8_t* __restrict__ dst, float* __restrict__ scale) {
  const int lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (row >= rows) return;
  const T* r = src + row * K;
  auto ld = [&](int k) -> float {
    if constexpr (sizeof(T) == 2) return __bfloat162float(r[k]);
    else return r[k];
  };
  float amax = 0.f;
  for (int k = lane; k < K; k += 32) amax = fmaxf(amax, fabsf(ld(k)));
  amax = warp_max(amax);
  const float inv = amax > 0.f ? kE4M3Max / amax : 1.f;
  for (int k = 4 * lane; k < K; k += 128)  // K is a multiple of 16
    *reinterpret_cast<uint32_t*>(dst + row * K + k) =
        pack_e4m3x4(ld(k) * inv, ld(k + 1) * inv, ld(k + 2) * inv, ld(k + 3) * inv);
  if (lane == 0) scale[row] = amax > 0.f ? amax / kE4M3Max : 1.f;
}

cudaError_t quantize_rows_e4m3(const void* src, bool src_bf16, int64_t rows, int K, uint8_t* dst, float* scale,
                               cudaStream_t s) {
  if (rows == 0) return cudaSuccess;
  if (K % 16) return cudaErrorInvalidValue;
  const unsigned grid = (unsigned)((rows + 7) / 8);
  if (src_bf16)
    quantize_rows_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(src), rows, K, dst, scale);
  else
    quantize_rows_kernel<float><<<grid, 256, 0, s>>>(static_cast<const float*>(src), rows, K, dst, scale);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- timestep MLP
template <typename WT>
DIT_DEV float wload(const WT* w, int64_t i);
template <>
DIT_DEV float wload<float>(const float* w, int64_t i) { return __ldg(w + i); }
template <>
DIT_DEV float wload<__nv_bfloat16>(const __nv_bfloat16* w, int64_t i) { return __bfloat162float(w[i]); }

// hidden[b, j] = SiLU(W1[j, :] . e(t_b) + b1[j]); one warp per output.
// The sinusoid's arguments reach 1000 rad, so they are formed in double.
template <typename WT>
__global__ void __launch_bounds__(256) temb_fc1_kernel(const float* t_dev, double t0, const float* sig,
                                                       const int* step, int fq, int D,
                                                       const WT* __restrict__ w1, const float* __restrict__ b1,
                                                       float* hidden) {
  extern __shared__ float e[];
  const int b = blockIdx.y;
  // t per batch element from t_dev, or t0 * sig[*step] (t0 = the timestep
  // scale) from the loop's device schedule, or t0 itself
  const double t = t_dev ? (double)t_dev[b] : (sig ? t0 * (double)sig[*step] : t0);
  const int half = fq / 2;
  for (int k = threadIdx.x; k < half; k += blockDim.x) {
    const double a = t * pow(10000.0, -(double)k / (double)half);
    double sv, cv;
    sincos(a, &sv, &cv);
    e[k] = (float)cv;
    e[half + k] = (float)sv;
  }
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const int j = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (j >= D) return;
  float acc = 0.f;
  for (int k = lane; k < fq; k += 32) acc = fmaf(wload(w1, (int64_t)j * fq + k), e[k], acc);
  acc = warp_sum(acc) + b1[j];
  if (lane == 0) hidden[(int64_t)b * D + j] = acc / (1.f + expf(-acc));
}

// mod[b, i] = W2[i, :] . hidden[b] + b2[i]; one warp per output.
template <typename WT>
__global__ void __launch_bounds__(256) temb_fc2_kernel(int D, const WT* __restrict__ w2,
                                                       const float* __restrict__ b2, const float* hidden,
                                                       float* mod) {
  extern __shared__ float h[];
  const int b = blockIdx.y;
  for (int k = threadIdx.x; k < D; k += blockDim.x) h[k] = hidden[(int64_t)b * D + k];
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const int i = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (i >= 6 * D) return;
  float acc = 0.f;
  for (int k = lane; k < D; k += 32) acc = fmaf(wload(w2, (int64_t)i * D + k), h[k], acc);
  acc = warp_sum(acc);
  if (lane == 0) mod[(int64_t)b * 6 * D + i] = acc + b2[i];
}

static cudaError_t timestep_mlp_any(const float* t_dev, double t0, const float* sig, const int* step, int batch,
                                    int fq, int D, const void* w1, const float* b1, const void* w2, const float* b2,
                                    bool w_bf16, float* hidden, float* mod, cudaStream_t s) {
  dim3 g1((D + 7) / 8, batch), g2((6 * D + 7) / 8, batch);
  if (w_bf16) {
    temb_fc1_kernel<__nv_bfloat16><<<g1, 256, fq * sizeof(float), s>>>(
        t_dev, t0, sig, step, fq, D, static_cast<const __nv_bfloat16*>(w1), b1, hidden);
    temb_fc2_kernel<__nv_bfloat16><<<g2, 256, D * sizeof(float), s>>>(
        D, static_cast<const __nv_bfloat16*>(w2), b2, hidden, mod);
  } else {
    temb_fc1_kernel<float><<<g1, 256, fq * sizeof(float), s>>>(t_dev, t0, sig, step, fq, D,
                                                               static_cast<const float*>(w1), b1, hidden);
    temb_fc2_kernel<float><<<g2, 256, D * sizeof(float), s>>>(D, static_cast<const float*>(w2), b2, hidden,
                                                              mod);
  }
  return cudaGetLastError();
}

cudaError_t timestep_mlp(const float* t_dev, double t0, int batch, int fq, int D, const void* w1, const float* b1,
                         const void* w2, const float* b2, bool w_bf16, float* hidden, float* mod, cudaStream_t s) {
  return timestep_mlp_any(t_dev, t0, nullptr, nullptr, batch, fq, D, w1, b1, w2, b2, w_bf16, hidden, mod, s);
}

cudaError_t timestep_mlp_sched(const float* sig, const int* step, double scale, int fq, int D, const void* w1,
                               const float* b1, const void* w2, const float* b2, bool w_bf16, float* hidden,
                               float* mod, cudaStream_t s) {
  return timestep_mlp_any(nullptr, scale, sig, step, 1, fq, D, w1, b1, w2, b2, w_bf16, hidden, mod, s);
}

__global__ void step_advance_kernel(int* step) {
  if (threadIdx.x == 0 && blockIdx.x == 0) *step += 1;
}

cudaError_t step_advance(int* step, cudaStream_t s) {
  step_advance_kernel<<<1, 32, 0, s>>>(step);
  return cudaGetLastError();
}

cudaError_t timestep_mlp_preload(bool w_bf16) {
  cudaFuncAttributes a;
  cudaError_t e = w_bf16 ? cudaFuncGetAttributes(&a, temb_fc1_kernel<__nv_bfloat16>)
                         : cudaFuncGetAttributes(&a, temb_fc1_kernel<float>);
  if (e == cudaSuccess)
    e = w_bf16 ? cudaFuncGetAttributes(&a, temb_fc2_kernel<__nv_bfloat16>)
               : cudaFuncGetAttributes(&a, temb_fc2_kernel<float>);
  return e;
}

// ---------------------------------------------------------------- modulation tables
__global__ void add_tables_kernel(const float* __restrict__ mod, int batch, int D, int rows,
                                  const float* __restrict__ tab, int ntab, float* __restrict__ out) {
  const int64_t per = (int64_t)rows * D;
  const int64_t n = (int64_t)ntab * batch * per;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t k = i / (batch * per);
    const int64_t r = i - k * batch * per;
    const int64_t b = r / per;
    const int64_t jc = r - b * per;
    out[i] = mod[b * 6 * D + jc] + tab[k * per + jc];
  }
}

cudaError_t add_tables(const float* mod, int batch, int D, int rows, const float* tables, int ntab, float* out,
                       cudaStream_t s) {
  const int64_t n = (int64_t)ntab * batch * rows * D;
  if (n == 0) return cudaSuccess;
  add_tables_kernel<<<blocks_for(n, 256), 256, 0, s>>>(mod, batch, D, rows, tables, ntab, out);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- latent packing
struct PatchGeom {
  int C, T, H, W, pt, ph, pw, gt, gh, gw, P;
  int64_t N;
};
static PatchGeom geom(int C, int T, int H, int W, int pt, int ph, int pw) {
  PatchGeom g{C, T, H, W, pt, ph, pw, T / pt, H / ph, W / pw, C * pt * ph * pw, 0};
  g.N = (int64_t)g.gt * g.gh * g.gw;
  return g;
}
// latent element (c, t, h, w) -> (token n, patch index j)
DIT_DEV void latent_to_token(const PatchGeom& g, int c, int t, int h, int w, int64_t& n, int& j) {
  n = ((int64_t)(t / g.pt) * g.gh + h / g.ph) * g.gw + w / g.pw;
  j = ((c * g.pt + t % g.pt) * g.ph + h % g.ph) * g.pw + w % g.pw;
}

template <bool kBf16>
__global__ void patchify_kernel(const float* __restrict__ lat, int Bl, int copies, PatchGeom g, void* tokens) {
  const int64_t per = (int64_t)g.C * g.T * g.H * g.W;
  const int64_t n = (int64_t)Bl * per;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t b = i / per;
    int64_t r = i - b * per;
    const int w = (int)(r % g.W); r /= g.W;
    const int h = (int)(r % g.H); r /= g.H;
    const int t = (int)(r % g.T);
    const int c = (int)(r / g.T);
    int64_t tok; int j;
    latent_to_token(g, c, t, h, w, tok, j);
    const float v = lat[i];
    for (int cp = 0; cp < copies; ++cp) {
      const int64_t o = (((int64_t)cp * Bl + b) * g.N + tok) * g.P + j;
      if constexpr (kBf16) static_cast<__nv_bfloat16*>(tokens)[o] = __float2bfloat16_rn(v);
      else static_cast<float*>(tokens)[o] = v;
    }
  }
}

cudaError_t patchify(const float* lat, int Bl, int copies, int C, int T, int H, int W, int pt, int ph, int pw,
                     void* tokens, bool out_bf16, cudaStream_t s) {
  const PatchGeom g = geom(C, T, H, W, pt, ph, pw);
  const int64_t n = (int64_t)Bl * C * T * H * W;
  if (n == 0) return cudaSuccess;
  if (out_bf16) patchify_kernel<true><<<blocks_for(n, 256), 256, 0, s>>>(lat, Bl, copies, g, tokens);
  else patchify_kernel<false><<<blocks_for(n, 256), 256, 0, s>>>(lat, Bl, copies, g, tokens);
  return cudaGetLastError();
}

__global__ void unpatchify_kernel(const float* __restrict__ tok, int B, PatchGeom g, float* __restrict__ lat) {
  const int64_t per = (int64_t)g.C * g.T * g.H * g.W;
  const int64_t n = (int64_t)B * per;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t b = i / per;
    int64_t r = i - b * per;
    const int w = (int)(r % g.W); r /= g.W;
    const int h = (int)(r % g.H); r /= g.H;
    const int t = (int)(r % g.T);
    const int c = (int)(r / g.T);
    int64_t tk; int j;
    latent_to_token(g, c, t, h, w, tk, j);
    lat[i] = tok[(b * g.N + tk) * g.P + j];
  }
}

cudaError_t unpatchify(const float* tok, int B, int C, int T, int H, int W, int pt, int ph, int pw, float* lat,
                       cudaStream_t s) {
  const PatchGeom g = geom(C, T, H, W, pt, ph, pw);
  const int64_t n = (int64_t)B * C * T * H * W;
  if (n == 0) return cudaSuccess;
  unpatchify_kernel<<<blocks_for(n, 256), 256, 0, s>>>(tok, B, g, lat);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- guidance + Euler
// Euler increment of the loop's current step: sigma[i+1] - sigma[i] of the
// device schedule, rounded once to fp32 (the host-side flow_euler_step rounds
// the same difference of the same values).
DIT_DEV float sched_dsig(const float* sig, const int* step) {
  const int i = *step;
  return (float)((double)sig[i + 1] - (double)sig[i]);
}

__global__ void cfg_euler_tokens_kernel(const float* __restrict__ vt, int Bl, int cfg, float gs, const float* sig,
                                        const int* step, PatchGeom g, float* __restrict__ lat) {
  const float dsig = sched_dsig(sig, step);
  const int64_t per = (int64_t)g.C * g.T * g.H * g.W;
  const int64_t n = (int64_t)Bl * per;
  const int64_t half = (int64_t)Bl * g.N * g.P;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t b = i / per;
    int64_t r = i - b * per;
    const int w = (int)(r % g.W); r /= g.W;
    const int h = (int)(r % g.H); r /= g.H;
    const int t = (int)(r % g.T);
    const int c = (int)(r / g.T);
    int64_t tk; int j;
    latent_to_token(g, c, t, h, w, tk, j);
    const int64_t o = (b * g.N + tk) * g.P + j;
    const float vc = vt[o];
    const float v = cfg ? fmaf(gs, vc - vt[half + o], vt[half + o]) : vc;
    lat[i] = fmaf(dsig, v, lat[i]);
  }
}

// Coalesced form: one CTA per grid row of tokens (batch b, grid t index it,
// grid h index ih; its gw tokens are gw*P contiguous floats in token layout).
// One thread copies the row of both passes' velocities into shared memory
// with bulk copies while every thread loads the latent float4s it will
// update (the C*pt*ph latent rows the tokens cover), so all of a CTA's loads
// are in flight together; then guidance + Euler and 128-bit stores.  Needs
// W % 4 == 0, P % 4 == 0 and 16-byte aligned buffers.
constexpr int CE_PER_THREAD = 4;  // latent float4s a thread keeps in flight
__global__ void __launch_bounds__(128, 8) cfg_euler_rows_kernel(const float* __restrict__ vt, int Bl, int cfg, float gs,
                                                            const float* sig, const int* step, PatchGeom g,
                                                            float* __restrict__ lat, int* err) {
  extern __shared__ __align__(16) uint8_t ce_smem[];
  __shared__ int ce_abort;
  const int row_floats = g.gw * g.P;
  float* vcs = reinterpret_cast<float*>(ce_smem);
  float* vus = vcs + row_floats;
  uint64_t* bar = reinterpret_cast<uint64_t*>(vus + row_floats);
  const int ih = blockIdx.x % g.gh;
  const int it = (blockIdx.x / g.gh) % g.gt;
  const int b = blockIdx.x / (g.gh * g.gt);
  const int64_t tok0 = ((int64_t)b * g.N + ((int64_t)it * g.gh + ih) * g.gw) * g.P;  // first float of the row
  const int64_t half = (int64_t)Bl * g.N * g.P;
  if (threadIdx.x == 0) {
    ce_abort = 0;
    mbar_init(bar, 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const uint32_t bytes = (uint32_t)row_floats * 4u;
    mbar_arrive_expect_tx(bar, cfg ? 2 * bytes : bytes);
    bulk_load(vcs, vt + tok0, bytes, bar);
    if (cfg) bulk_load(vus, vt + half + tok0, bytes, bar);
  }
  const float dsig = sched_dsig(sig, step);
  const int wq = g.W / 4;
  const int n4 = g.C * g.pt * g.ph * wq;
  // latent float4 k of the CTA: latent row (c, a, e) = k / wq, columns w0..w0+3
  auto lat_index = [&](int k, int* jrow, int* w0) -> int64_t {
    const int row = k / wq;
    *w0 = (k - row * wq) * 4;
    const int e = row % g.ph, a = (row / g.ph) % g.pt, c = row / (g.ph * g.pt);
    *jrow = ((c * g.pt + a) * g.ph + e) * g.pw;  // patch index of (c, a, e, 0)
    return ((((int64_t)b * g.C + c) * g.T + it * g.pt + a) * g.H + ih * g.ph + e) * g.W + *w0;
  };
  bool waited = false, ok = true;
  for (int base = threadIdx.x; base < n4; base += blockDim.x * CE_PER_THREAD) {
    float4 x[CE_PER_THREAD];
#pragma unroll
    for (int q = 0; q < CE_PER_THREAD; ++q) {
      const int k = base + q * (int)blockDim.x;
      if (k >= n4) break;
      int jrow, w0;
      x[q] = *reinterpret_cast<const float4*>(lat + lat_index(k, &jrow, &w0));
    }
    if (!waited) {
      ok = mbar_wait(bar, 0, &ce_abort, err, 43);
      waited = true;
    }
    if (!ok) break;
#pragma unroll
    for (int q = 0; q < CE_PER_THREAD; ++q) {
      const int k = base + q * (int)blockDim.x;
      if (k >= n4) break;
      int jrow, w0;
      const int64_t li = lat_index(k, &jrow, &w0);
      float xv[4] = {x[q].x, x[q].y, x[q].z, x[q].w};
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int w = w0 + r, iw = w / g.pw;
        const int idx = iw * g.P + jrow + (w - iw * g.pw);
        const float vc = vcs[idx];
        const float v = cfg ? fmaf(gs, vc - vus[idx], vus[idx]) : vc;
        xv[r] = fmaf(dsig, v, xv[r]);
      }
      *reinterpret_cast<float4*>(lat + li) = make_float4(xv[0], xv[1], xv[2], xv[3]);
    }
  }
  // the copies land before the CTA exits, whichever threads had work
  if (!waited && threadIdx.x == 0) mbar_wait(bar, 0, &ce_abort, err, 43);
}

cudaError_t cfg_euler_tokens(const float* vt, int Bl, bool cfg, float gs, const float* sig, const int* step, int C,
                             int T, int H, int W, int pt, int ph, int pw, float* lat, int* err, cudaStream_t s) {
  const PatchGeom g = geom(C, T, H, W, pt, ph, pw);
  const int64_t n = (int64_t)Bl * C * T * H * W;
  if (n == 0) return cudaSuccess;
  const size_t row_bytes = (size_t)g.gw * g.P * sizeof(float);
  const bool aligned = ((reinterpret_cast<uintptr_t>(vt) | reinterpret_cast<uintptr_t>(lat)) & 15) == 0;
  const int64_t nrows = (int64_t)Bl * g.gt * g.gh;
  const size_t smem = 2 * row_bytes + 16;
  if (aligned && W % 4 == 0 && g.P % 4 == 0 && smem <= 48 * 1024 && nrows <= INT32_MAX) {
    cfg_euler_rows_kernel<<<(int)nrows, 128, smem, s>>>(vt, Bl, cfg ? 1 : 0, gs, sig, step, g, lat, err);
  } else {
    cfg_euler_tokens_kernel<<<blocks_for(n, 256), 256, 0, s>>>(vt, Bl, cfg ? 1 : 0, gs, sig, step, g, lat);
  }
  return cudaGetLastError();
}

__global__ void cfg_kernel(const float* __restrict__ vc, const float* __restrict__ vu, float gs, float* v,
                           int64_t n) {
  const int64_t n4 = n / 4;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const int64_t i0 = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  const bool vec = ((reinterpret_cast<uintptr_t>(vc) | reinterpret_cast<uintptr_t>(vu) |
                     reinterpret_cast<uintptr_t>(v)) & 15) == 0;
  int64_t done = 0;
  if (vec) {
    for (int64_t i = i0; i < n4; i += stride) {
      const float4 a = reinterpret_cast<const float4*>(vc)[i], b = reinterpret_cast<const float4*>(vu)[i];
      reinterpret_cast<float4*>(v)[i] =
          make_float4(fmaf(gs, a.x - b.x, b.x), fmaf(gs, a.y - b.y, b.y), fmaf(gs, a.z - b.z, b.z),
                      fmaf(gs, a.w - b.w, b.w));
    }
    done = n4 * 4;
  }
  for (int64_t i = done + i0; i < n; i += stride) v[i] = fmaf(gs, vc[i] - vu[i], vu[i]);
}

__global__ void euler_kernel_(float* x, const float* __restrict__ v, float dsig, int64_t n) {
  const int64_t n4 = n / 4;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const int64_t i0 = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  const bool vec = ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(v)) & 15) == 0;
  int64_t done = 0;
  if (vec) {
    for (int64_t i = i0; i < n4; i += stride) {
      float4 a = reinterpret_cast<float4*>(x)[i];
      const float4 b = reinterpret_cast<const float4*>(v)[i];
      a.x = fmaf(dsig, b.x, a.x); a.y = fmaf(dsig, b.y, a.y);
      a.z = fmaf(dsig, b.z, a.z); a.w = fmaf(dsig, b.w, a.w);
      reinterpret_cast<float4*>(x)[i] = a;
    }
    done = n4 * 4;
  }
  for (int64_t i = done + i0; i < n; i += stride) x[i] = fmaf(dsig, v[i], x[i]);
}

cudaError_t cfg_combine_kernel(const float* vc, const float* vu, float g, float* v, int64_t n, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  cfg_kernel<<<blocks_for(n / 4 + 1, 256), 256, 0, s>>>(vc, vu, g, v, n);
  return cudaGetLastError();
}

cudaError_t euler_kernel(float* x, const float* v, float dsig, int64_t n, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  euler_kernel_<<<blocks_for(n / 4 + 1, 256), 256, 0, s>>>(x, v, dsig, n);
  return cudaGetLastError();
}

__global__ void f32_to_bf16_kernel(const float* __restrict__ in, __nv_bfloat16* __restrict__ out, int64_t n) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
    out[i] = __float2bfloat16_rn(in[i]);
}

cudaError_t f32_to_bf16(const float* in, void* out, int64_t n, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  f32_to_bf16_kernel<<<blocks_for(n, 256), 256, 0, s>>>(in, static_cast<__nv_bfloat16*>(out), n);
  return cudaGetLastError();
}

__global__ void bf16_to_f32_kernel(const __nv_bfloat16* __restrict__ in, float* __restrict__ out, int64_t n) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
    out[i] = __bfloat162float(in[i]);
}

cudaError_t bf16_to_f32(const void* in, float* out, int64_t n, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  bf16_to_f32_kernel<<<blocks_for(n, 256), 256, 0, s>>>(static_cast<const __nv_bfloat16*>(in), out, n);
  return cudaGetLastError();
}

// Test hook for the bounded-wait failure path: one warp waits on an mbarrier
// that nothing ever arrives on.  The wait gives up after DIT_WAIT_LIMIT_NS,
// records `site` in *err and the kernel returns; the context stays usable.
__global__ void debug_stall_kernel(int* err, int site) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait(&bar, 0, &abort_flag, err, site);
}

cudaError_t debug_stall(int* err, int site, cudaStream_t s) {
  debug_stall_kernel<<<1, 32, 0, s>>>(err, site);
  return cudaGetLastError();
}

}  // namespace dit
