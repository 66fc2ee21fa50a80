// GEMM epilogues applied to a chunk of NV consecutive columns of one output
// row while the accumulators are still in registers: bias, GELU (tanh form),
// gated residual update of the fp32 stream, or the head-major Q/K/V scatter
// with rotary embedding of interleaved channel pairs.
#pragma once
#include <type_traits>
#include "common.cuh"
#include "kernels.h"

namespace dit {

template <typename T>
DIT_DEV T to_act(float v);
template <>
DIT_DEV float to_act<float>(float v) { return v; }
template <>
DIT_DEV __nv_bfloat16 to_act<__nv_bfloat16>(float v) { return __float2bfloat16_rn(v); }

// Store NV values to dst (16-byte aligned when NV * sizeof(T) >= 16 and the
// caller passes an aligned address).
template <typename T, int NV>
DIT_DEV void store_chunk(T* dst, const float (&v)[NV]) {
  if constexpr (std::is_same<T, float>::value) {
    if constexpr (NV % 4 == 0) {
#pragma unroll
      for (int j = 0; j < NV; j += 4)
        *reinterpret_cast<float4*>(dst + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
    } else {
#pragma unroll
      for (int j = 0; j < NV; ++j) dst[j] = v[j];
    }
  } else {
    if constexpr (NV % 8 == 0) {
#pragma unroll
      for (int j = 0; j < NV; j += 8) {
        uint4 u;
        u.x = pack_bf16x2(v[j + 0], v[j + 1]);
        u.y = pack_bf16x2(v[j + 2], v[j + 3]);
        u.z = pack_bf16x2(v[j + 4], v[j + 5]);
        u.w = pack_bf16x2(v[j + 6], v[j + 7]);
        *reinterpret_cast<uint4*>(dst + j) = u;
      }
    } else if constexpr (NV % 2 == 0) {
#pragma unroll
      for (int j = 0; j < NV; j += 2) *reinterpret_cast<uint32_t*>(dst + j) = pack_bf16x2(v[j], v[j + 1]);
    } else {
#pragma unroll
      for (int j = 0; j < NV; ++j) dst[j] = __float2bfloat16_rn(v[j]);
    }
  }
}

template <bool kFast>
DIT_DEV float gelu_tanh(float x) {
  const float k0 = 0.7978845608028654f;  // sqrt(2/pi)
  const float u = k0 * (x + 0.044715f * x * x * x);
  const float t = kFast ? tanh_approx(u) : tanhf(u);
  return 0.5f * x * (1.0f + t);
}

// Element-wise part of the epilogue for columns [col0, col0 + NV) of row
// `row` (row < M): bias, then GELU (EPI_GELU), the gate factor (EPI_RESID:
// v becomes gate * v, the increment of x) or the rotary embedding of
// interleaved channel pairs (EPI_HEADS).  col0 is a multiple of NV; for
// EPI_HEADS NV divides hd and D and is a multiple of 4.
//
// The tensor-core path (bf16 activations) works on pairs of columns with the
// packed f32x2 instructions (fma / mul / add .rn.f32x2: the same IEEE
// rounding per element, half the instructions).  The instruction count
// matters beyond the epilogue itself: the epilogue warps share the SM's
// schedulers with the thread that issues the MMAs, and measured per 256 x 256
// tile of the video FFN1 GEMM the main loop took 16,250 cycles with the
// scalar bias + GELU, 14,520 with the packed form and ~13,000 with no
// epilogue arithmetic at all.
template <typename ActT, int NV>
DIT_DEV void epilogue_values(const EpiParams& p, int64_t row, int col0, float (&v)[NV]) {
  constexpr bool kFast = std::is_same<ActT, __nv_bfloat16>::value;
  constexpr bool kPair = kFast && NV % 4 == 0;  // packed pairs (v[2i], v[2i+1])
  auto pr = [&](int j) { return make_float2(v[j], v[j + 1]); };
  auto put = [&](int j, float2 x) {
    v[j] = x.x;
    v[j + 1] = x.y;
  };
  const bool full = col0 + NV <= p.N;
  // 8-bit operands: the row scale of A and the column scale of W are undone
  // together with the bias add (v = v * sa * w_scale + bias); whole chunks
  // read bias and scales as float4 (both are 256-byte aligned arrays and col0
  // is a multiple of NV)
  const float sa = p.a_scale ? __ldg(p.a_scale + row) : 1.f;
  const bool vec = full && NV % 4 == 0 &&
                   ((reinterpret_cast<uintptr_t>(p.bias) | reinterpret_cast<uintptr_t>(p.w_scale)) & 15) == 0;
  if (vec) {
#pragma unroll
    for (int j = 0; j < NV; j += 4) {
      const float4 b = p.bias ? __ldg(reinterpret_cast<const float4*>(p.bias + col0 + j)) : make_float4(0.f, 0.f, 0.f, 0.f);
      if (p.a_scale) {
        const float4 w = __ldg(reinterpret_cast<const float4*>(p.w_scale + col0 + j));
        if constexpr (kPair) {
          const float2 sa2 = make_float2(sa, sa);
          put(j, ffma2(pr(j), fmul2(sa2, make_float2(w.x, w.y)), make_float2(b.x, b.y)));
          put(j + 2, ffma2(pr(j + 2), fmul2(sa2, make_float2(w.z, w.w)), make_float2(b.z, b.w)));
        } else {
          v[j + 0] = fmaf(v[j + 0], sa * w.x, b.x);
          v[j + 1] = fmaf(v[j + 1], sa * w.y, b.y);
          v[j + 2] = fmaf(v[j + 2], sa * w.z, b.z);
          v[j + 3] = fmaf(v[j + 3], sa * w.w, b.w);
        }
      } else if constexpr (kPair) {
        put(j, fadd2(pr(j), make_float2(b.x, b.y)));
        put(j + 2, fadd2(pr(j + 2), make_float2(b.z, b.w)));
      } else {
        v[j + 0] += b.x;
        v[j + 1] += b.y;
        v[j + 2] += b.z;
        v[j + 3] += b.w;
      }
    }
  } else {
#pragma unroll
    for (int j = 0; j < NV; ++j) {
      if (!full && col0 + j >= p.N) continue;
      if (p.a_scale) v[j] *= sa * __ldg(p.w_scale + col0 + j);
      if (p.bias) v[j] += __ldg(p.bias + col0 + j);
    }
  }
  if (p.kind == EPI_GELU) {
    if constexpr (kPair) {
      // 0.5 x (1 + tanh(u)), u = x (k0 + k0 c x^2) = k0 (x + c x^3)
      const float2 k0 = make_float2(0.7978845608028654f, 0.7978845608028654f);
      const float2 k0c = make_float2(0.7978845608028654f * 0.044715f, 0.7978845608028654f * 0.044715f);
      const float2 half = make_float2(0.5f, 0.5f);
#pragma unroll
      for (int j = 0; j < NV; j += 2) {
        const float2 x = pr(j);
        const float2 u = fmul2(x, ffma2(fmul2(x, x), k0c, k0));
        const float2 hx = fmul2(x, half);
        put(j, ffma2(hx, make_float2(tanh_approx(u.x), tanh_approx(u.y)), hx));
      }
    } else {
#pragma unroll
      for (int j = 0; j < NV; ++j) v[j] = gelu_tanh<kFast>(v[j]);
    }
  } else if (p.kind == EPI_RESID) {
    if (p.gate) {
      const float* g = p.gate + (row / p.rows_per_batch) * p.gate_bstride + col0;
      if (full && (p.gate_bstride % 4 == 0) && (NV % 4 == 0)) {
#pragma unroll
        for (int j = 0; j < NV; j += 4) {
          const float4 gv = __ldg(reinterpret_cast<const float4*>(g + j));
          if constexpr (kPair) {
            put(j, fmul2(pr(j), make_float2(gv.x, gv.y)));
            put(j + 2, fmul2(pr(j + 2), make_float2(gv.z, gv.w)));
          } else {
            v[j + 0] *= gv.x;
            v[j + 1] *= gv.y;
            v[j + 2] *= gv.z;
            v[j + 3] *= gv.w;
          }
        }
      } else {
#pragma unroll
        for (int j = 0; j < NV; ++j)
          if (col0 + j < p.N) v[j] *= __ldg(g + j);
      }
    }
  } else if (p.kind == EPI_HEADS) {
    const int sec = col0 / p.D;
    const int c = (col0 - sec * p.D) % p.hd;
    const int t = (int)(row % p.rows_per_batch);
    if (p.rope && ((p.rope_mask >> sec) & 1)) {
      if constexpr (kFast && NV % 8 == 0) {
        // The angle pos * inv_freq is formed here instead of read from the
        // (cos, sin) table: one lane per row would fetch 16 bytes from a
        // different table row per load, a scattered stream that costs the
        // epilogue more than the main loop.  The angle (at most a few
        // hundred radians) is reduced to [-pi, pi] with a two-constant
        // Cody-Waite step (2 pi = 6.28125 + 1.9353...e-3, the first part
        // exact for small multiples), then passed to the fast sincos.  Two
        // channel pairs at a time in packed f32x2 form.
        const int iw = t % p.rope_g2, th = t / p.rope_g2;
        const float pos_t = (float)(th / p.rope_g1), pos_h = (float)(th % p.rope_g1), pos_w = (float)iw;
        const float4* inv4 = reinterpret_cast<const float4*>(p.rope_inv + c / 2);
        const float2 inv2pi = make_float2(0.159154943091895336f, 0.159154943091895336f);
        const float2 c1 = make_float2(6.28125f, 6.28125f), c2 = make_float2(1.93530717958647692e-3f, 1.93530717958647692e-3f);
#pragma unroll
        for (int j = 0; j < NV; j += 8) {
          const float4 f4 = __ldg(inv4 + j / 8);
#pragma unroll
          for (int k = 0; k < 4; k += 2) {
            const int pp = c / 2 + j / 2 + k;
            const float pos0 = pp < p.rope_b0 ? pos_t : (pp < p.rope_b1 ? pos_h : pos_w);
            const float pos1 = pp + 1 < p.rope_b0 ? pos_t : (pp + 1 < p.rope_b1 ? pos_h : pos_w);
            const float2 ang = fmul2(make_float2(pos0, pos1), k ? make_float2(f4.z, f4.w) : make_float2(f4.x, f4.y));
            const float2 tn = fmul2(ang, inv2pi);
            const float2 nn = make_float2(-rintf(tn.x), -rintf(tn.y));
            const float2 r = ffma2(nn, c2, ffma2(nn, c1, ang));
            float sn0, cs0, sn1, cs1;
            __sincosf(r.x, &sn0, &cs0);
            __sincosf(r.y, &sn1, &cs1);
            // (a, b) -> (a cos - b sin, a sin + b cos) for both pairs
            const float a0 = v[j + 2 * k], b0 = v[j + 2 * k + 1], a1 = v[j + 2 * k + 2], b1 = v[j + 2 * k + 3];
            put(j + 2 * k, ffma2(make_float2(a0, a0), make_float2(cs0, sn0), fmul2(make_float2(-b0, b0), make_float2(sn0, cs0))));
            put(j + 2 * k + 2, ffma2(make_float2(a1, a1), make_float2(cs1, sn1), fmul2(make_float2(-b1, b1), make_float2(sn1, cs1))));
          }
        }
      } else {
        // two (cos, sin) pairs per 16-byte load: c is a multiple of 4 channels
        const float4* cs = reinterpret_cast<const float4*>(p.rope + (int64_t)t * (p.hd / 2) + c / 2);
#pragma unroll
        for (int j = 0; j < NV; j += 4) {
          const float4 r = __ldg(cs + j / 4);
          const float a0 = v[j], b0 = v[j + 1], a1 = v[j + 2], b1 = v[j + 3];
          v[j] = a0 * r.x - b0 * r.y;
          v[j + 1] = a0 * r.y + b0 * r.x;
          v[j + 2] = a1 * r.z - b1 * r.w;
          v[j + 3] = a1 * r.w + b1 * r.z;
        }
      }
    }
  }
}

// Write the values produced by epilogue_values with plain per-thread stores
// (EPI_RESID adds them into the fp32 stream x).
template <typename ActT, int NV>
DIT_DEV void epilogue_store(const EpiParams& p, int64_t row, int col0, const float (&v)[NV]) {
  const bool full = col0 + NV <= p.N;
  switch (p.kind) {
    case EPI_F32: {
      float* o = static_cast<float*>(p.out) + row * p.ldo + col0;
      if (full && (p.ldo % 4 == 0)) {
        store_chunk<float, NV>(o, v);
      } else {
        for (int j = 0; j < NV; ++j)
          if (col0 + j < p.N) o[j] = v[j];
      }
      break;
    }
    case EPI_GELU:
    case EPI_ACT: {
      ActT* o = static_cast<ActT*>(p.out) + row * p.ldo + col0;
      if (full && (p.ldo % 8 == 0)) {
        store_chunk<ActT, NV>(o, v);
      } else {
        for (int j = 0; j < NV; ++j)
          if (col0 + j < p.N) o[j] = to_act<ActT>(v[j]);
      }
      break;
    }
    case EPI_RESID: {
      float* xr = p.x + row * (int64_t)p.N + col0;
      if (full && (p.N % 4 == 0) && (NV % 4 == 0)) {
#pragma unroll
        for (int j = 0; j < NV; j += 4) {
          float4 xv = *reinterpret_cast<float4*>(xr + j);
          xv.x += v[j + 0];
          xv.y += v[j + 1];
          xv.z += v[j + 2];
          xv.w += v[j + 3];
          *reinterpret_cast<float4*>(xr + j) = xv;
        }
      } else {
        for (int j = 0; j < NV; ++j)
          if (col0 + j < p.N) xr[j] += v[j];
      }
      break;
    }
    case EPI_HEADS: {
      const int sec = col0 / p.D;
      const int cc = col0 - sec * p.D;
      const int h = cc / p.hd;
      const int c = cc - h * p.hd;
      const int64_t b = row / p.rows_per_batch;
      const int t = (int)(row - b * p.rows_per_batch);
      ActT* o = static_cast<ActT*>(p.dst[sec]) + ((b * p.H + h) * (int64_t)p.seq_total + p.tok_off + t) * p.hd + c;
      store_chunk<ActT, NV>(o, v);
      break;
    }
  }
}

// The whole epilogue of NV columns of one row (row < M).
template <typename ActT, int NV>
DIT_DEV void epilogue_chunk(const EpiParams& p, int64_t row, int col0, float (&v)[NV]) {
  epilogue_values<ActT, NV>(p, row, col0, v);
  epilogue_store<ActT, NV>(p, row, col0, v);
}

}  // namespace dit
