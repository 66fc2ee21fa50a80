// Internal launch interface between the C ABI layer (dit_api.cu) and the
// kernel translation units.  Nothing here is exported from libdit.so.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

namespace dit {

// Error-word sites: bounded waits that gave up use 1..59 (and the stall test
// hook its own site); the checks of the debug bounds build
// (-DDIT_DEBUG_BOUNDS) use DIT_BOUNDS_SITE_MIN..DIT_BOUNDS_SITE_MAX.
constexpr int DIT_BOUNDS_SITE_MIN = 60;
constexpr int DIT_BOUNDS_SITE_MAX = 79;

// ------------------------------------------------------------------ GEMM
// C[M, N] = A[M, K] . W[N, K]^T (+ bias), followed by one fused epilogue.
enum EpiKind : int {
  EPI_F32 = 0,    // out_f32[row * ldo + col] = acc + bias
  EPI_ACT = 1,    // out_act[row * ldo + col] = acc + bias       (activation dtype)
  EPI_GELU = 2,   // out_act[row * ldo + col] = gelu_tanh(acc + bias)
  EPI_RESID = 3,  // x[row * N + col] += gate[b, col] * (acc + bias)   (gate NULL = 1)
  EPI_HEADS = 4   // scatter sections of D columns into head-major [B, H, S, hd] (+ RoPE)
};

struct EpiParams {
  int kind = EPI_F32;
  int M = 0, N = 0;
  const float* bias = nullptr;
  void* out = nullptr;
  int64_t ldo = 0;
  // residual update
  float* x = nullptr;
  const float* gate = nullptr;
  int64_t gate_bstride = 0;
  int rows_per_batch = 1;  // also used by EPI_HEADS
  // head-major scatter: column n -> section n / D, head (n % D) / hd, channel n % hd;
  // row r -> batch r / rows_per_batch, token tok_off + r % rows_per_batch of seq_total
  void* dst[3] = {nullptr, nullptr, nullptr};
  int D = 0, hd = 0, H = 0, seq_total = 0, tok_off = 0, rope_mask = 0;
  const float2* rope = nullptr;  // [rows_per_batch][hd / 2] (cos, sin)
  // the same rotation evaluated in the kernel (bf16 tensor-core path): token
  // t = (it * rope_g1 + ih) * rope_g2 + iw; channel pair p turns by
  // pos * rope_inv[p], pos = it for p < rope_b0, ih for p < rope_b1, else iw
  const float* rope_inv = nullptr;  // [hd / 2]
  int rope_g1 = 0, rope_g2 = 0, rope_b0 = 0, rope_b1 = 0;
  // set by the tensor-core GEMM launcher when its output tensor maps are valid
  // (the epilogue then stores through shared memory with TMA)
  int tma = 0;
  // 8-bit GEMM: the accumulator of row r, column n is multiplied by
  // a_scale[r] * w_scale[n] (the scales the two operands were quantized with)
  // before the bias and the rest of the epilogue
  const float* a_scale = nullptr;
  const float* w_scale = nullptr;
};

struct GemmArgs {
  const void* A = nullptr;  // [M, K] row-major, row stride lda elements
  int64_t M = 0;
  int K = 0;
  int64_t lda = 0;
  const void* W = nullptr;  // [N, K] row-major (row stride K)
  int N = 0;
  EpiParams epi;
};

// fp32 CUDA-core GEMM (test precision).
cudaError_t gemm_f32(const GemmArgs& g, cudaStream_t s);
// bf16 tcgen05 GEMM (production precision); err = device error word for
// bounded waits; num_sms = persistent grid size.
cudaError_t gemm_bf16_tc(const GemmArgs& g, int* err, int num_sms, cudaStream_t s);
// Two bf16 GEMMs with the same N and K in one persistent launch (g0's tiles
// first, then g1's); either may have M = 0.
cudaError_t gemm_bf16_tc_pair(const GemmArgs& g0, const GemmArgs& g1, int* err, int num_sms, cudaStream_t s);
// e4m3 tcgen05 GEMM (kind::f8f6f4): A [M, K] and W [N, K] bytes (row strides
// lda and K bytes, multiples of 16), fp32 accumulation; the epilogue applies
// epi.a_scale / epi.w_scale.  Single and paired forms as above.
cudaError_t gemm_e4m3_tc(const GemmArgs& g, int* err, int num_sms, cudaStream_t s);
cudaError_t gemm_e4m3_tc_pair(const GemmArgs& g0, const GemmArgs& g1, int* err, int num_sms, cudaStream_t s);
// GEMMs whose N is a multiple of 256 on clusters of two CTAs sharing
// cta_group::2 MMAs of 256 x 256 tiles: 0 never (single CTAs, 128 x 256),
// 1 (default) when the main loop has at least 16 K blocks, 2 always.
void set_gemm_cta_pairs(int mode);
// Row-wise e4m3 quantization of a weight matrix: src [rows, K] (fp32 or bf16)
// -> dst [rows, K] e4m3 bytes and scale[rows] = max|row| / 448 (1 for a zero
// row), dst = src / scale rounded to nearest.
cudaError_t quantize_rows_e4m3(const void* src, bool src_bf16, int64_t rows, int K, uint8_t* dst, float* scale,
                               cudaStream_t s);

// ------------------------------------------------------------------ attention
// Q [B, H, Lq, hd], K/V [B, H, Lk, hd] head-major; output token-major rows of
// width D = H * hd: token t < split goes to o1[b, t], else o2[b, t - split].
struct AttnArgs {
  const void* q = nullptr;
  const void* k = nullptr;
  const void* v = nullptr;
  int B = 0, H = 0, Lq = 0, Lk = 0, hd = 0;
  void* o1 = nullptr;
  void* o2 = nullptr;
  int split = 0;
};
cudaError_t attention_f32(const AttnArgs& a, cudaStream_t s);
cudaError_t attention_bf16_tc(const AttnArgs& a, int* err, cudaStream_t s);

// ------------------------------------------------------------------ elementwise
// h[r, :] = LN(x[r, :]) * (1 + scale[b]) + shift[b], b = r / rows_per_batch;
// shift/scale NULL = plain LN.  Output bf16 (out_bf16) or fp32.  The bf16
// path stages rows through shared memory on a grid of at most num_sms CTAs;
// err = device error word for its bounded waits.
// Output kinds: LN_F32, LN_BF16, or LN_E4M3 (e4m3 bytes, each row divided by
// its scale max|row| / 448, written to row_scale[row]).
enum LnOut : int { LN_F32 = 0, LN_BF16 = 1, LN_E4M3 = 2 };
cudaError_t ln_modulate(const float* x, int64_t rows, int D, int rows_per_batch, const float* shift,
                        const float* scale, int64_t mod_bstride, float eps, void* out, int out_kind, int* err,
                        int num_sms, cudaStream_t s, float* row_scale = nullptr);
// One LayerNorm of a pair: x [rows, D] -> out, modulation of batch element
// r / rpb at shift/scale + (r / rpb) * mbs (both NULL = plain LN).
struct LnArgs {
  const float* x;
  int64_t rows;
  int rpb;
  const float* shift;
  const float* scale;
  int64_t mbs;
  void* out;
  float* row_scale = nullptr;  // LN_E4M3 output: per-row scale
};
// Two LayerNorms of the same width in one launch where the staged bf16 path
// takes them (both modulated or both plain), else one launch each;
// *launches = the number of kernels launched.
cudaError_t ln_modulate_pair(const LnArgs& a, const LnArgs& b, int D, float eps, int out_kind, int* err,
                             int num_sms, cudaStream_t s, int* launches);
// Sinusoidal timestep embedding + 2-layer MLP: mod[b, 6D] for each t[b].
// hidden_scratch: float[batch * D].
// t_dev NULL: every batch element uses t0.
cudaError_t timestep_mlp(const float* t_dev, double t0, int batch, int freq_dim, int D, const void* w1, const float* b1,
                         const void* w2, const float* b2, bool w_bf16, float* hidden_scratch, float* mod,
                         cudaStream_t s);
// Loads the timestep MLP's kernels for the current device (under lazy module
// loading a kernel's code is otherwise loaded, and its device memory taken,
// at its first launch).
cudaError_t timestep_mlp_preload(bool w_bf16);
// The loop's timestep MLP: t = scale * sig[*step] from the device schedule
// and step counter (batch 1).
cudaError_t timestep_mlp_sched(const float* sig, const int* step, double scale, int freq_dim, int D, const void* w1,
                               const float* b1, const void* w2, const float* b2, bool w_bf16, float* hidden,
                               float* mod, cudaStream_t s);
// *step += 1 (one thread), enqueued at the end of every loop step.
cudaError_t step_advance(int* step, cudaStream_t s);
// Largest hidden width whose activation vector the second MLP kernel keeps
// in shared memory without an opt-in (48 KB).
constexpr int kTimestepMlpMaxHidden = 12288;
// out[k, b, j, c] = mod[b, j*D + c] + tables[k, j, c] for k < ntab, j < rows
// (tables contiguous [ntab, rows, D]).
cudaError_t add_tables(const float* mod, int batch, int D, int rows, const float* tables, int ntab, float* out,
                       cudaStream_t s);
// latents [Bl, C, T, H, W] -> tokens [copies * Bl, N, C*pt*ph*pw] (copies of the batch back to back)
cudaError_t patchify(const float* lat, int Bl, int copies, int C, int T, int H, int W, int pt, int ph, int pw,
                     void* tokens, bool out_bf16, cudaStream_t s);
// tokens [B, N, P] -> latents [B, C, T, H, W]
cudaError_t unpatchify(const float* tok, int B, int C, int T, int H, int W, int pt, int ph, int pw, float* lat,
                       cudaStream_t s);
// Fused guidance + Euler + unpatchify over velocity tokens vt [2*Bl or Bl, N, P]:
// lat += dsig * (vu + g (vc - vu)) (or vc alone when !cfg).
// Guidance + Euler update of the loop, reading velocity tokens; the Euler
// increment of the current step comes from the device schedule sig and the
// device step counter.
cudaError_t cfg_euler_tokens(const float* vt, int Bl, bool cfg, float g, const float* sig, const int* step, int C,
                             int T, int H, int W, int pt, int ph, int pw, float* lat, int* err, cudaStream_t s);
cudaError_t cfg_combine_kernel(const float* vc, const float* vu, float g, float* v, int64_t n, cudaStream_t s);
cudaError_t euler_kernel(float* x, const float* v, float dsig, int64_t n, cudaStream_t s);
cudaError_t f32_to_bf16(const float* in, void* out, int64_t n, cudaStream_t s);
cudaError_t bf16_to_f32(const void* in, float* out, int64_t n, cudaStream_t s);

// Test hook: a kernel whose bounded wait runs out and records `site` in *err.
cudaError_t debug_stall(int* err, int site, cudaStream_t s);

}  // namespace dit
