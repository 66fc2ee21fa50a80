// fp32 CUDA-core kernels of the test precision: a tiled GEMM with the shared
// epilogues, and a flash-style attention with an online softmax.  They give
// the fp32-accumulate reference mode of the GPU path (all activations fp32).
#include "epilogue.cuh"

namespace dit {

// ---------------------------------------------------------------- GEMM
// 64 x 64 output tile, K step 16, 256 threads, 4 x 4 outputs per thread.
constexpr int SG_BM = 64, SG_BN = 64, SG_BK = 16;

__global__ void __launch_bounds__(256) gemm_f32_kernel(const float* __restrict__ A, int64_t lda,
                                                       const float* __restrict__ W, int64_t M, int N, int K,
                                                       EpiParams ep) {
  __shared__ float As[SG_BK][SG_BM + 4];
  __shared__ float Ws[SG_BK][SG_BN + 4];
  const int tid = threadIdx.x;
  const int tx = tid & 15, ty = tid >> 4;
  const int64_t m0 = (int64_t)blockIdx.y * SG_BM;
  const int n0 = blockIdx.x * SG_BN;
  float acc[4][4] = {};
  // each thread stages 4 elements of each operand tile: row lr, k lk..lk+3
  const int lr = tid >> 2, lk = (tid & 3) * 4;
  for (int k0 = 0; k0 < K; k0 += SG_BK) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int k = k0 + lk + j;
      const int64_t am = m0 + lr;
      As[lk + j][lr] = (am < M && k < K) ? A[am * lda + k] : 0.f;
      const int wn = n0 + lr;
      Ws[lk + j][lr] = (wn < N && k < K) ? W[(int64_t)wn * K + k] : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < SG_BK; ++k) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[k][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = Ws[k][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
  const int col0 = n0 + tx * 4;
  if (col0 >= N) return;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int64_t row = m0 + ty * 4 + i;
    if (row < M) epilogue_chunk<float, 4>(ep, row, col0, acc[i]);
  }
}

cudaError_t gemm_f32(const GemmArgs& g, cudaStream_t s) {
  if (g.M == 0 || g.N == 0) return cudaSuccess;
  dim3 grid((g.N + SG_BN - 1) / SG_BN, (unsigned)((g.M + SG_BM - 1) / SG_BM));
  gemm_f32_kernel<<<grid, 256, 0, s>>>(static_cast<const float*>(g.A), g.lda, static_cast<const float*>(g.W),
                                        g.M, g.N, g.K, g.epi);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- attention
// One CTA = 32 query rows of one (batch, head); 128 threads, 4 per row.
// Keys/values stream through shared memory 64 at a time.
constexpr int SA_BQ = 32, SA_BK = 64;

template <int HD>
__global__ void __launch_bounds__(128) attn_f32_kernel(AttnArgs a, float scale_log2) {
  extern __shared__ float sm[];
  float* Qs = sm;                          // [32][HD+1]
  float* Ks = Qs + SA_BQ * (HD + 1);       // [64][HD+1]
  float* Vs = Ks + SA_BK * (HD + 1);       // [64][HD]
  float* Ps = Vs + SA_BK * HD;             // [32][65]
  const int tid = threadIdx.x, r = tid >> 2, sub = tid & 3;
  const int b = blockIdx.z, h = blockIdx.y;
  const int q0 = blockIdx.x * SA_BQ;
  const float* Q = static_cast<const float*>(a.q) + ((int64_t)b * a.H + h) * a.Lq * HD;
  const float* Kp = static_cast<const float*>(a.k) + ((int64_t)b * a.H + h) * a.Lk * HD;
  const float* Vp = static_cast<const float*>(a.v) + ((int64_t)b * a.H + h) * a.Lk * HD;
  for (int i = tid; i < SA_BQ * HD; i += 128) {
    const int rr = i / HD, c = i - rr * HD;
    Qs[rr * (HD + 1) + c] = (q0 + rr < a.Lq) ? Q[(int64_t)(q0 + rr) * HD + c] : 0.f;
  }
  constexpr int NO = HD / 4;
  float o[NO];
#pragma unroll
  for (int i = 0; i < NO; ++i) o[i] = 0.f;
  float m = -INFINITY, l = 0.f;
  for (int k0 = 0; k0 < a.Lk; k0 += SA_BK) {
    __syncthreads();
    for (int i = tid; i < SA_BK * HD; i += 128) {
      const int kk = i / HD, c = i - kk * HD;
      const bool ok = k0 + kk < a.Lk;
      Ks[kk * (HD + 1) + c] = ok ? Kp[(int64_t)(k0 + kk) * HD + c] : 0.f;
      Vs[kk * HD + c] = ok ? Vp[(int64_t)(k0 + kk) * HD + c] : 0.f;
    }
    __syncthreads();
    float s[16];
    float mx = -INFINITY;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const int kk = sub + 4 * j;
      float acc = 0.f;
#pragma unroll 8
      for (int c = 0; c < HD; ++c) acc = fmaf(Qs[r * (HD + 1) + c], Ks[kk * (HD + 1) + c], acc);
      s[j] = (k0 + kk < a.Lk) ? acc * scale_log2 : -INFINITY;
      mx = fmaxf(mx, s[j]);
    }
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    const float m_new = fmaxf(m, mx);
    const float alpha = exp2f(m - m_new);
    float ps = 0.f;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const float p = exp2f(s[j] - m_new);
      ps += p;
      Ps[r * 65 + sub + 4 * j] = p;
    }
    l = l * alpha + ps;
    m = m_new;
    __syncwarp();
#pragma unroll
    for (int i = 0; i < NO; ++i) o[i] *= alpha;
    for (int kk = 0; kk < SA_BK; ++kk) {
      const float p = Ps[r * 65 + kk];
#pragma unroll
      for (int i = 0; i < NO; ++i) o[i] = fmaf(p, Vs[kk * HD + sub + 4 * i], o[i]);
    }
  }
  l += __shfl_xor_sync(0xffffffffu, l, 1);
  l += __shfl_xor_sync(0xffffffffu, l, 2);
  const int t = q0 + r;
  if (t >= a.Lq) return;
  const int D = a.H * HD;
  float* out = (t < a.split) ? static_cast<float*>(a.o1) + ((int64_t)b * a.split + t) * D
                             : static_cast<float*>(a.o2) + ((int64_t)b * (a.Lq - a.split) + (t - a.split)) * D;
  out += h * HD;
  const float inv = 1.f / l;
#pragma unroll
  for (int i = 0; i < NO; ++i) out[sub + 4 * i] = o[i] * inv;
}

template <int HD>
static cudaError_t launch_attn_f32(const AttnArgs& a, cudaStream_t s) {
  const size_t smem = sizeof(float) * (SA_BQ * (HD + 1) + SA_BK * (HD + 1) + SA_BK * HD + SA_BQ * 65);
  cudaError_t e = cudaFuncSetAttribute(attn_f32_kernel<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid((a.Lq + SA_BQ - 1) / SA_BQ, a.H, a.B);
  const float scale_log2 = 1.4426950408889634f / sqrtf((float)HD);
  attn_f32_kernel<HD><<<grid, 128, smem, s>>>(a, scale_log2);
  return cudaGetLastError();
}

cudaError_t attention_f32(const AttnArgs& a, cudaStream_t s) {
  if (a.Lq == 0 || a.B == 0) return cudaSuccess;
  switch (a.hd) {
    case 32: return launch_attn_f32<32>(a, s);
    case 64: return launch_attn_f32<64>(a, s);
    case 128: return launch_attn_f32<128>(a, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace dit
