/*
 * dit.h -- C ABI of the GB300 denoiser stage (libdit.so).
 *
 * The denoiser stage runs the network's forward passes over the whole step
 * schedule, with the sampler advancing the latent after each of them
 * (SGLang-Diffusion "Disaggregated Diffusion Pipeline", Quick Start, role
 * table: "denoiser").  Its inputs are the latents, the
 * timestep / sigma schedule in the exact order used, the positive prompt
 * embeddings and, when classifier-free guidance is on, the negative ones
 * (SGLang-Diffusion "Support New Diffusion Models", section 4, table of the
 * fields DenoisingStage requires).  The network is called with
 * hidden_states / encoder_hidden_states / timestep, once with the positive
 * and once with the negative condition (same page, section 2 "Pipeline
 * Config").  Velocities are flow predictions integrated with a flow-matching
 * Euler step on a shifted sigma schedule (stable-diffusion.cpp "Model
 * Configuration Conventions", "Sampling And Geometry").
 *
 * Conventions for every call:
 *   - Every pointer documented "device" is a CUDA device pointer owned by the
 *     caller; the library never frees it.  Host pointers are read before the
 *     call returns.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Work is enqueued asynchronously on it; results are ready once
 *     the stream is synchronised (dit_synchronize does that and also reports
 *     a device-side timeout).
 *   - Argument errors are detected on the host before anything is launched;
 *     outputs are then left untouched.  Nothing aborts the process: every
 *     failure is a status code, with a message from dit_last_error().
 *   - There is no CPU fallback and no silent precision change: a call the
 *     GPU path cannot serve returns an error.
 *   - One model owns one device workspace that every forward call of that
 *     model reuses (block scratch, loop state, the timestep MLP's hidden
 *     activations).  Calls on the same model must therefore be ordered on
 *     the GPU: issue them on one stream, or order the streams with events.
 *     Calls of one model on two unordered streams race on the workspace.
 *     Separate models share nothing and may run concurrently.
 *   - Floating-point tensors crossing the ABI are float32, row-major, densely
 *     packed, in the layouts given per call.  B is the batch of network
 *     passes; in the loop B = 2 x requests with CFG (conditional passes
 *     first, then unconditional ones).
 */
#ifndef DIT_H
#define DIT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  DIT_OK = 0,
  DIT_ERR_INVALID_ARG = 1, /* bad pointer, value, schedule or flag          */
  DIT_ERR_SHAPE = 2,       /* inconsistent or unsupported tensor shape      */
  DIT_ERR_NOT_LOADED = 3,  /* forward called before a complete weight load  */
  DIT_ERR_OOM = 4,         /* device allocation failed                      */
  DIT_ERR_CUDA = 5,        /* a CUDA runtime/driver call failed             */
  DIT_ERR_TIMEOUT = 6      /* a kernel gave up a bounded wait (see dit_synchronize) */
} dit_status;

enum { DIT_PREC_BF16 = 0, DIT_PREC_F32 = 1, DIT_PREC_FP8 = 2 };
enum { DIT_COND_CROSS = 0, DIT_COND_JOINT = 1 };
enum { DIT_DTYPE_F32 = 0, DIT_DTYPE_BF16 = 1 };
/* dit_denoise_loop flags */
enum {
  DIT_LOOP_PARTIAL_SCHEDULE = 1, /* allow sigmas[0] != 1 or sigmas[n] != 0                     */
  DIT_LOOP_CUDA_GRAPH = 2        /* replay one captured step as a CUDA graph (see the loop call) */
};

/*
 * Model configuration, copied by dit_create.  Mirrors the C++ "*Config"
 * convention of stable-diffusion.cpp "Model Configuration Conventions"
 * (Config Types / Runner And Model Responsibilities): derived once, passed to
 * the model, never re-scanned.
 *   in_channels   latent channels C (stable-diffusion.cpp ModelGeometry latent_channels)
 *   patch[3]      patch size (pt, ph, pw) over (T, H, W) of the latent
 *   hidden        D = heads * head_dim
 *   mlp           F, width of the GELU MLP
 *   cond_dim      Dc, width of a condition token (must equal hidden in joint mode)
 *   freq_dim      width of the sinusoidal timestep embedding (even)
 *   rope_axes[3]  rotary channels per axis (t, h, w), each even, summing to
 *                 head_dim, or all zero for no rotation
 *   cond_mode     DIT_COND_CROSS: cross-attention to condition tokens;
 *                 DIT_COND_JOINT: dual-stream joint attention with them
 *   precision     DIT_PREC_BF16: bf16 weights/activations, fp32 accumulate
 *                 (tcgen05 tensor cores; requires head_dim == 128);
 *                 DIT_PREC_FP8: as bf16, except that the GEMMs fed by a
 *                 LayerNorm (self-attention Q/K/V, cross-attention Q, MLP
 *                 up-projection) take e4m3 operands: weights quantized at
 *                 load with one scale per output row, the LayerNorm output
 *                 with one scale per token row (requires hidden % 16 == 0);
 *                 DIT_PREC_F32: fp32 everywhere (test mode, CUDA cores)
 *   ln_eps, rope_theta, timestep_scale (t = timestep_scale * sigma)
 */
typedef struct {
  int32_t in_channels;
  int32_t patch[3];
  int32_t hidden;
  int32_t heads;
  int32_t head_dim;
  int32_t mlp;
  int32_t depth;
  int32_t cond_dim;
  int32_t freq_dim;
  int32_t rope_axes[3];
  int32_t cond_mode;
  int32_t precision;
  float ln_eps;
  float rope_theta;
  float timestep_scale;
} dit_config;

/* One named parameter for dit_load_weights.  `data` may be a host or a
 * device pointer (unified addressing decides); dtype is DIT_DTYPE_F32 or
 * DIT_DTYPE_BF16; shape[0..ndim) must equal the expected shape. */
typedef struct {
  const char* name;
  int32_t ndim;
  int64_t shape[4];
  int32_t dtype;
  const void* data;
} dit_tensor;

typedef struct dit_model dit_model;

/* Create a model on CUDA device `device`.  Validates the configuration
 * (DIT_ERR_INVALID_ARG / DIT_ERR_SHAPE) before touching the GPU. */
dit_status dit_create(const dit_config* cfg, int device, dit_model** out);

/* Copy parameters into the model's own device arena (converted to the
 * model's storage precision).  Strict: every name must be a known parameter,
 * appear once across all calls, and have the expected shape; otherwise
 * DIT_ERR_SHAPE and nothing of this call is kept (SGLang-Diffusion "Support
 * New Diffusion Models", "Reuse component loaders": strict key and shape
 * checks, fail instead of falling back).  The forward calls return
 * DIT_ERR_NOT_LOADED until every parameter has been loaded.  Synchronous.
 * With DIT_PREC_FP8 the weights of the self-attention Q/K/V, cross-attention
 * Q and MLP up-projection are quantized here on the device to e4m3 with one
 * scale per output row (max |row| / 448); the others are stored as bf16. */
dit_status dit_load_weights(dit_model* m, const dit_tensor* tensors, int n);

/* Host-only queries on a configuration (no GPU needed): the number of
 * parameters a model of this configuration expects, and the name (copied into
 * name_buf, NUL-terminated) and shape of the i-th, in load order.  Linear
 * weights are [out_features, in_features]; each block carries a learned
 * [6, hidden] modulation table (shift1, scale1, gate1, shift2, scale2,
 * gate2) added to the shared timestep modulation. */
int dit_num_params(const dit_config* cfg);
dit_status dit_param_info(const dit_config* cfg, int i, char* name_buf, int buf_len, int32_t* ndim,
                          int64_t shape[4]);

/* a1: timestep embedding -> MLP -> shared modulation.
 *   t_host  host float[batch], the network timestep per batch element
 *   mod     device float[batch, 6*hidden] output */
dit_status dit_timestep_modulation(dit_model* m, const float* t_host, int batch, float* mod, void* stream);

/* The same computation as dit_timestep_modulation, for callers that must
 * not allocate device memory during the call: for example a serving thread
 * that may not trigger the implicit device synchronisation a cudaMalloc or
 * cudaFree can cause, or a host whose device memory is entirely handed to
 * its own pool allocator, so any allocation by this library would fail or
 * stall.  (The pages have no counterpart; this is an interface addition.)
 * The call allocates nothing: it never calls cudaMalloc, cudaFree or any
 * allocating library routine, and it loads no module.  Its scratch (the
 * timesteps and the MLP's hidden activations) lives in one fixed array of
 * this library's device memory (about 1 MiB), which every GPU that loads the
 * library holds until the process exits.
 *   batch <= DIT_NOALLOC_MAX_BATCH, batch * hidden <= DIT_NOALLOC_MAX_HIDDEN,
 *   and hidden, freq_dim <= 12288 (one activation vector held in 48 KB of
 *   shared memory); otherwise DIT_ERR_INVALID_ARG (nothing is launched).
 * Set-up happens in dit_create, with the model's device current: it looks up
 * the array's device address on that device and loads the kernels this call
 * launches.  So create the model before any stream capture.  All calls share
 * the one array: calls whose work overlaps on the GPU (for example on two
 * streams without ordering between them) race with each other.  Every byte
 * of scratch a call reads it has written itself first. */
enum { DIT_NOALLOC_MAX_BATCH = 64, DIT_NOALLOC_MAX_HIDDEN = 262144 };
dit_status dit_timestep_modulation_noalloc(dit_model* m, const float* t_host, int batch, float* mod, void* stream);

/* a2: patchify + patch embedding.
 *   latents device float[batch, C, T, H, W]; latent_thw = {T, H, W}, each
 *           divisible by the patch size (else DIT_ERR_SHAPE)
 *   x       device float[batch, N, hidden] output, N = (T/pt)(H/ph)(W/pw),
 *           tokens in row-major (t, h, w) grid order */
dit_status dit_patch_embed(dit_model* m, const float* latents, int batch, const int32_t latent_thw[3],
                           float* x, void* stream);

/* a3-a9: one DiT block, in place on the residual stream(s).  The network
 * call of the pages (hidden_states = x, encoder_hidden_states = cond or xc,
 * the timestep through `mod`: SGLang-Diffusion "Support New Diffusion
 * Models", section 2 "Pipeline Config"), restricted to one block; rotary
 * positions follow the token grid ("Verify the Port": rotary shape and style
 * must match).
 *   block   0 .. depth-1
 *   x       device float[batch, N, hidden], image/video token stream, in/out
 *   xc      joint mode: device float[batch, cond_len, hidden], condition-token
 *           stream, in/out; cross mode: must be NULL
 *   mod     device float[batch, 6*hidden], the shared timestep modulation from
 *           dit_timestep_modulation (the block adds its own table)
 *   cond    cross mode: device float[batch, cond_len, cond_dim] condition
 *           tokens; joint mode: must be NULL
 *   grid    token grid {T/pt, H/ph, W/pw} (N = product), sets RoPE positions */
dit_status dit_block_forward(dit_model* m, int block, float* x, float* xc, const float* mod,
                             const float* cond, int batch, const int32_t grid[3], int cond_len,
                             void* stream);

/* a10: final layer (LN + head modulation + linear) and unpatchify.
 *   x  device float[batch, N, hidden];  mod as above
 *   v  device float[batch, C, T, H, W] output velocity */
dit_status dit_final_layer(dit_model* m, const float* x, const float* mod, int batch,
                           const int32_t latent_thw[3], float* v, void* stream);

/* a11 (first half): classifier-free guidance v = vu + g (vc - vu) over n
 * floats (device pointers; v may alias vc or vu).  The positive and negative
 * passes and the guidance scale: SGLang-Diffusion "Support New Diffusion
 * Models", section 1 "Sampling Params" (guidance_scale) and section 2
 * "Pipeline Config" (pos/neg kwargs).  n < 0, a NULL pointer with n > 0 or a
 * non-finite g: DIT_ERR_INVALID_ARG. */
dit_status cfg_combine(const float* vc, const float* vu, float g, float* v, int64_t n, void* stream);

/* a11 (second half): flow-matching Euler update x += (sigma_next - sigma) v
 * over n floats, in place on device x.  Flow prediction integrated on the
 * shifted sigma schedule: stable-diffusion.cpp "Model Configuration
 * Conventions", "Sampling And Geometry" (flow prediction, default flow
 * shift, flow denoisers).  n < 0, a NULL pointer with n > 0 or a non-finite
 * sigma: DIT_ERR_INVALID_ARG. */
dit_status flow_euler_step(float* x, const float* v, float sigma, float sigma_next, int64_t n,
                           void* stream);

/* The whole denoiser stage for `batch` requests: the denoiser role of
 * SGLang-Diffusion "Disaggregated Diffusion Pipeline" (Quick Start, role
 * table), with the inputs that "Support New Diffusion Models" section 4 lists
 * for the denoising stage (latents, the sigma schedule in the order used,
 * positive and negative condition embeddings, number of steps); the error
 * cases follow that page's "Verify the Port" failure points (reversed
 * timesteps, missing negative embeddings with CFG on, latent shape).
 *   latents  device float[batch, C, T, H, W], initial noise in, denoised out
 *   cond     device float[batch, cond_len, cond_dim] positive condition
 *   uncond   device float[batch, cond_len, cond_dim] negative condition, or
 *            NULL for no guidance (then `guidance` must be 1)
 *   sigmas   host float[n_steps + 1], already shifted, strictly decreasing,
 *            sigmas[0] == 1 and sigmas[n_steps] == 0 unless
 *            DIT_LOOP_PARTIAL_SCHEDULE is set (resuming part of a schedule)
 *   Per step i: t = timestep_scale * sigmas[i]; v from the network on the
 *   2*batch conditional+unconditional passes; v = vu + g (vc - vu);
 *   latents += (sigmas[i+1] - sigmas[i]) v.  Condition-token keys/values of
 *   cross-attention are computed once per call (they do not depend on the
 *   step). */
/*   With DIT_LOOP_CUDA_GRAPH the launches of one step are captured once (on
 *   a stream the model owns; nothing runs during the capture) into a CUDA
 *   graph that is then launched n_steps times on `stream`.  Every step reads
 *   its timestep and Euler increment from a device copy of `sigmas` through a
 *   device step counter, so the same graph serves every step; the result is
 *   bitwise the same as without the flag.  The graph is kept in the model and
 *   reused by later calls whose pointers, shapes, guidance and n_steps are
 *   the same; otherwise it is captured again.  Cannot be combined with
 *   per-launch timing (dit_profile_start with timing on): DIT_ERR_INVALID_ARG. */
dit_status dit_denoise_loop(dit_model* m, float* latents, int batch, const int32_t latent_thw[3],
                            const float* cond, const float* uncond, int cond_len,
                            const float* sigmas, int n_steps, float guidance, uint32_t flags,
                            void* stream);

/* Synchronise `stream` and report DIT_ERR_TIMEOUT if a kernel of this model
 * abandoned a bounded wait since the last check (its outputs are then
 * invalid; the flag is cleared). */
dit_status dit_synchronize(dit_model* m, void* stream);

/* Per-kernel accounting of this model's launches, for measurement.
 * dit_profile_start resets the counters and, when `timing` is non-zero,
 * records a CUDA event pair on the launching stream around every launch.
 * dit_profile_stop synchronises the device and returns, per kernel kind,
 * the number of kernel launches and (with timing) their summed device time
 * in milliseconds.  counts/ms: host arrays of DIT_KERNEL_KINDS entries. */
enum {
  DIT_KERNEL_GEMM_QKV = 0,    /* self-attention Q/K/V projection (+RoPE scatter)  */
  DIT_KERNEL_GEMM_OUT = 1,    /* attention output projections (gated residual)   */
  DIT_KERNEL_GEMM_CROSS_Q = 2,
  DIT_KERNEL_GEMM_CROSS_KV = 3,
  DIT_KERNEL_GEMM_FFN1 = 4,   /* MLP up-projection + GELU                         */
  DIT_KERNEL_GEMM_FFN2 = 5,   /* MLP down-projection (gated residual)             */
  DIT_KERNEL_GEMM_EMBED = 6,  /* patch embedding and final linear                 */
  DIT_KERNEL_ATTN_SELF = 7,
  DIT_KERNEL_ATTN_CROSS = 8,
  DIT_KERNEL_LN = 9,          /* LayerNorm + adaLN modulation                     */
  DIT_KERNEL_SMALL = 10,      /* timestep MLP, tables, packing, casts             */
  DIT_KERNEL_CFG_EULER = 11,  /* guidance + Euler update of the loop              */
  DIT_KERNEL_KINDS = 12
};
dit_status dit_profile_start(dit_model* m, int timing);
dit_status dit_profile_stop(dit_model* m, int64_t* counts, double* ms);

/* Bytes of device memory held by the model (weights + workspace). */
int64_t dit_device_bytes(const dit_model* m);

void dit_destroy(dit_model* m);
const char* dit_status_string(dit_status s);
/* Message of the last failing call on this thread ("" if none). */
const char* dit_last_error(void);

/* Test hook: make the next `n`-th device allocation of any model fail with
 * DIT_ERR_OOM (0 disables).  Host-side only; used to test failure paths. */
void dit_debug_fail_alloc_after(int n);

/* Test hook: where GEMMs whose output width is a multiple of 256 run on
 * clusters of two CTAs that share one tcgen05.mma of 256 x 256
 * (cta_group::2) instead of single CTAs with 128 x 256 tiles.  mode 1 (the
 * default): when the GEMM's main loop has at least 16 K blocks (K >= 1024 in
 * bf16, K >= 2048 in e4m3); 0: never; 2: always.  Other values are clamped
 * to 0..2.  Process-wide; takes effect at the next launch (a CUDA graph
 * captured before keeps the kernels it captured).  Both paths give the same
 * bits; the hook exists to compare them. */
void dit_debug_gemm_cta_pairs(int mode);

/* Test hook for the device-side failure path.  Enqueues on `stream` a kernel
 * whose bounded wait on a barrier that nothing ever arrives on gives up after
 * the library's wait limit (1.5 s) and records DIT_DEBUG_STALL_SITE in the
 * model's error word; the next dit_synchronize then returns DIT_ERR_TIMEOUT
 * (and clears the word).  Nothing faults or hangs, and the model stays
 * usable.  Returns DIT_ERR_INVALID_ARG for a NULL model, DIT_ERR_CUDA if the
 * launch fails. */
enum { DIT_DEBUG_STALL_SITE = 99 };
dit_status dit_debug_stall(dit_model* m, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* DIT_H */
