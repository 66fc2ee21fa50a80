// C ABI of the denoiser stage: model object, weight arena, workspace and the
// per-block / per-step launch schedule.  All arithmetic runs in the kernels
// of this library; this file validates arguments, lays out device memory and
// enqueues launches on the caller's stream.
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <string>
#include <unordered_map>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "../../include/dit.h"
#include "kernels.h"

using namespace dit;

// ============================================================== error state
static thread_local char g_last_error[512] = "";
static int g_fail_alloc_after = 0;  // test hook: fail the n-th next allocation

static dit_status fail(dit_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return s;
}

#define CU_TRY(expr)                                                                                    \
  do {                                                                                                  \
    cudaError_t e_ = (expr);                                                                            \
    if (e_ != cudaSuccess) return fail(DIT_ERR_CUDA, "%s failed: %s", #expr, cudaGetErrorString(e_)); \
  } while (0)
#define DIT_TRY(expr)                 \
  do {                                \
    dit_status s_ = (expr);           \
    if (s_ != DIT_OK) return s_;      \
  } while (0)

static dit_status dev_alloc(void** p, size_t bytes) {
  *p = nullptr;
  if (bytes == 0) return DIT_OK;
  if (g_fail_alloc_after > 0 && --g_fail_alloc_after == 0)
    return fail(DIT_ERR_OOM, "device allocation of %zu bytes failed (injected)", bytes);
  cudaError_t e = cudaMalloc(p, bytes);
  if (e != cudaSuccess) {
    cudaGetLastError();
    *p = nullptr;
    return fail(e == cudaErrorMemoryAllocation ? DIT_ERR_OOM : DIT_ERR_CUDA, "cudaMalloc(%zu) failed: %s", bytes,
                cudaGetErrorString(e));
  }
  return DIT_OK;
}

// ============================================================== parameters
struct ParamSpec {
  std::string name;
  std::vector<int64_t> shape;
};

static std::vector<ParamSpec> param_specs(const dit_config& c) {
  const int64_t D = c.hidden, F = c.mlp, Dc = c.cond_dim, fq = c.freq_dim;
  const int64_t P = (int64_t)c.in_channels * c.patch[0] * c.patch[1] * c.patch[2];
  std::vector<ParamSpec> s = {{"patch_embed.weight", {D, P}},      {"patch_embed.bias", {D}},
                              {"time_mlp.fc1.weight", {D, fq}},    {"time_mlp.fc1.bias", {D}},
                              {"time_mlp.fc2.weight", {6 * D, D}}, {"time_mlp.fc2.bias", {6 * D}}};
  for (int b = 0; b < c.depth; ++b) {
    const std::string p = "blocks." + std::to_string(b) + ".";
    const int nstreams = c.cond_mode == DIT_COND_CROSS ? 1 : 2;
    for (int st = 0; st < nstreams; ++st) {
      const std::string q = p + (st ? "ctx." : "");
      s.push_back({q + "mod_table", {6, D}});
      s.push_back({q + "attn.qkv.weight", {3 * D, D}});
      s.push_back({q + "attn.qkv.bias", {3 * D}});
      s.push_back({q + "attn.out.weight", {D, D}});
      s.push_back({q + "attn.out.bias", {D}});
      if (st == 0 && c.cond_mode == DIT_COND_CROSS) {
        s.push_back({p + "cross.q.weight", {D, D}});
        s.push_back({p + "cross.q.bias", {D}});
        s.push_back({p + "cross.kv.weight", {2 * D, Dc}});
        s.push_back({p + "cross.kv.bias", {2 * D}});
        s.push_back({p + "cross.out.weight", {D, D}});
        s.push_back({p + "cross.out.bias", {D}});
      }
      s.push_back({q + "mlp.fc1.weight", {F, D}});
      s.push_back({q + "mlp.fc1.bias", {F}});
      s.push_back({q + "mlp.fc2.weight", {D, F}});
      s.push_back({q + "mlp.fc2.bias", {D}});
    }
  }
  s.push_back({"head.mod_table", {2, D}});
  s.push_back({"head.weight", {P, D}});
  s.push_back({"head.bias", {P}});
  return s;
}

static dit_status validate_config(const dit_config* c) {
  if (!c) return fail(DIT_ERR_INVALID_ARG, "config is NULL");
  if (c->in_channels <= 0 || c->patch[0] <= 0 || c->patch[1] <= 0 || c->patch[2] <= 0 || c->hidden <= 0 ||
      c->heads <= 0 || c->head_dim <= 0 || c->mlp <= 0 || c->depth <= 0 || c->cond_dim <= 0 || c->freq_dim <= 0)
    return fail(DIT_ERR_INVALID_ARG, "config sizes must be positive");
  if (c->heads * c->head_dim != c->hidden)
    return fail(DIT_ERR_SHAPE, "hidden (%d) != heads (%d) * head_dim (%d)", c->hidden, c->heads, c->head_dim);
  if (c->freq_dim % 2) return fail(DIT_ERR_INVALID_ARG, "freq_dim must be even");
  if (c->cond_mode != DIT_COND_CROSS && c->cond_mode != DIT_COND_JOINT)
    return fail(DIT_ERR_INVALID_ARG, "unknown cond_mode %d", c->cond_mode);
  if (c->precision != DIT_PREC_BF16 && c->precision != DIT_PREC_F32 && c->precision != DIT_PREC_FP8)
    return fail(DIT_ERR_INVALID_ARG, "unknown precision %d", c->precision);
  const int ra = c->rope_axes[0] + c->rope_axes[1] + c->rope_axes[2];
  for (int i = 0; i < 3; ++i)
    if (c->rope_axes[i] < 0 || c->rope_axes[i] % 2)
      return fail(DIT_ERR_INVALID_ARG, "rope_axes must be even and non-negative");
  if (ra != 0 && ra != c->head_dim)
    return fail(DIT_ERR_INVALID_ARG, "rope_axes sum %d must equal head_dim %d (or 0 for no rotation)", ra,
                c->head_dim);
  if (c->cond_mode == DIT_COND_JOINT && c->cond_dim != c->hidden)
    return fail(DIT_ERR_SHAPE, "joint mode needs cond_dim == hidden");
  if (!(c->ln_eps >= 0.f) || !(c->rope_theta > 0.f) || !(c->timestep_scale > 0.f))
    return fail(DIT_ERR_INVALID_ARG, "ln_eps >= 0, rope_theta > 0 and timestep_scale > 0 required");
  if (c->hidden % 4) return fail(DIT_ERR_SHAPE, "hidden must be a multiple of 4");
  if (c->precision == DIT_PREC_FP8 && c->hidden % 16)
    return fail(DIT_ERR_SHAPE, "fp8 precision requires hidden to be a multiple of 16");
  if (c->precision == DIT_PREC_BF16 || c->precision == DIT_PREC_FP8) {
    if (c->head_dim != 128) return fail(DIT_ERR_SHAPE, "bf16 precision requires head_dim 128");
    if (c->mlp % 8 || c->cond_dim % 8)
      return fail(DIT_ERR_SHAPE, "bf16 precision requires mlp and cond_dim multiples of 8");
    const int P = c->in_channels * c->patch[0] * c->patch[1] * c->patch[2];
    if (P % 8) return fail(DIT_ERR_SHAPE, "bf16 precision requires C*pt*ph*pw to be a multiple of 8");
  } else {
    if (c->head_dim != 32 && c->head_dim != 64 && c->head_dim != 128)
      return fail(DIT_ERR_SHAPE, "fp32 precision supports head_dim 32, 64 or 128");
  }
  return DIT_OK;
}

// ============================================================== model
// Scratch of dit_timestep_modulation_noalloc: DIT_NOALLOC_MAX_BATCH timesteps
// followed by DIT_NOALLOC_MAX_HIDDEN hidden activations, in module memory
// that no call allocates or frees.  In host code the symbol is a host-side
// stand-in; dit_create looks up its device address with the model's device
// current (which also loads this file's module there) and keeps it in the
// model, so the no-allocation call itself never triggers a module load.
static __device__ __align__(256) float g_noalloc_scratch[DIT_NOALLOC_MAX_BATCH + DIT_NOALLOC_MAX_HIDDEN];

struct Param {
  ParamSpec spec;
  bool matrix;  // linear weight: stored in the activation dtype
  bool fp8;     // stored as e4m3 bytes with one fp32 scale per output row (fp8 precision)
  size_t offset;
  size_t scale_offset;
  int64_t numel;
  bool loaded;
};

// In fp8 precision the weights of the GEMMs whose input comes from a
// LayerNorm (self-attention Q/K/V of both streams, cross-attention Q, MLP
// up-projection of both streams) are kept in e4m3; the LayerNorm writes their
// input in e4m3 with one scale per row.
static bool fp8_weight(const std::string& n) {
  auto ends = [&](const char* suf) {
    const size_t l = strlen(suf);
    return n.size() >= l && n.compare(n.size() - l, l, suf) == 0;
  };
  return n.rfind("blocks.", 0) == 0 &&
         (ends(".attn.qkv.weight") || ends(".cross.q.weight") || ends(".mlp.fc1.weight"));
}

struct Workspace {
  void* base = nullptr;
  size_t bytes = 0;
  size_t used = 0;
  void* take(size_t n) {
    n = (n + 255) & ~size_t(255);
    void* p = static_cast<char*>(base) + used;
    used += n;
    return p;
  }
};

struct dit_model {
  dit_config cfg;
  int device = 0;
  int num_sms = 0;
  bool bf16 = true;
  bool fp8 = false;  // e4m3 GEMMs after the LayerNorms (DIT_PREC_FP8)
  size_t act = 2;  // bytes per activation element
  std::vector<Param> params;
  std::unordered_map<std::string, int> index;
  char* arena = nullptr;
  size_t arena_bytes = 0;
  size_t tables_off = 0, ctx_tables_off = 0;  // contiguous [depth][6][D] fp32
  int n_loaded = 0;
  int* d_err = nullptr;
  float* d_t = nullptr;
  int d_t_cap = 0;
  void* ws = nullptr;
  size_t ws_bytes = 0;
  float2* rope = nullptr;
  float* noalloc_scratch = nullptr;  // device address of g_noalloc_scratch on this device
  // dit_denoise_loop with DIT_LOOP_CUDA_GRAPH: one captured step, replayed
  struct LoopGraph {
    cudaGraphExec_t exec = nullptr;
    std::vector<uint64_t> key;                // every pointer and scalar the captured step holds
    int64_t counts[DIT_KERNEL_KINDS] = {};  // kernel launches of one step, by kind
  } graph;
  cudaStream_t capture_stream = nullptr;
  bool capturing = false;
  int rope_grid[3] = {0, 0, 0};
  size_t rope_bytes = 0;
  // launch accounting (dit_profile_start / dit_profile_stop)
  bool prof_timing = false;
  int64_t prof_counts[DIT_KERNEL_KINDS] = {};
  struct Rec {
    int kind;
    cudaEvent_t a, b;
  };
  std::vector<Rec> prof_rec;
  std::vector<cudaEvent_t> prof_pool;
  size_t prof_next = 0;

  const void* W(const std::string& n) const { return arena + params[index.at(n)].offset; }
  // per-output-row scales of an e4m3 weight (nullptr for the others)
  const float* S(const std::string& n) const {
    const Param& p = params[index.at(n)];
    return p.fp8 ? reinterpret_cast<const float*>(arena + p.scale_offset) : nullptr;
  }
  const float* V(const std::string& n) const {
    return reinterpret_cast<const float*>(arena + params[index.at(n)].offset);
  }
  std::string blk(int b, const char* suffix) const { return "blocks." + std::to_string(b) + "." + suffix; }
};

static bool is_matrix(const std::string& n) {
  return n.size() > 7 && n.compare(n.size() - 7, 7, ".weight") == 0;
}

extern "C" int dit_num_params(const dit_config* cfg) {
  if (validate_config(cfg) != DIT_OK) return -1;
  return (int)param_specs(*cfg).size();
}

extern "C" dit_status dit_param_info(const dit_config* cfg, int i, char* name_buf, int buf_len, int32_t* ndim,
                                     int64_t shape[4]) {
  DIT_TRY(validate_config(cfg));
  const auto s = param_specs(*cfg);
  if (i < 0 || i >= (int)s.size()) return fail(DIT_ERR_INVALID_ARG, "parameter index %d out of range", i);
  if (!name_buf || buf_len <= (int)s[i].name.size() || !ndim || !shape)
    return fail(DIT_ERR_INVALID_ARG, "output buffers missing or too small");
  memcpy(name_buf, s[i].name.c_str(), s[i].name.size() + 1);
  *ndim = (int32_t)s[i].shape.size();
  for (int d = 0; d < 4; ++d) shape[d] = d < *ndim ? s[i].shape[d] : 1;
  return DIT_OK;
}

extern "C" void dit_debug_fail_alloc_after(int n) { g_fail_alloc_after = n; }
extern "C" void dit_debug_gemm_cta_pairs(int mode) { dit::set_gemm_cta_pairs(mode); }

extern "C" const char* dit_status_string(dit_status s) {
  switch (s) {
    case DIT_OK: return "ok";
    case DIT_ERR_INVALID_ARG: return "invalid argument";
    case DIT_ERR_SHAPE: return "shape error";
    case DIT_ERR_NOT_LOADED: return "weights not loaded";
    case DIT_ERR_OOM: return "out of device memory";
    case DIT_ERR_CUDA: return "CUDA error";
    case DIT_ERR_TIMEOUT: return "device wait timed out";
  }
  return "unknown status";
}

extern "C" const char* dit_last_error(void) { return g_last_error; }

extern "C" void dit_destroy(dit_model* m) {
  if (!m) return;
  int prev = 0;
  if (cudaGetDevice(&prev) == cudaSuccess) cudaSetDevice(m->device);
  cudaFree(m->arena);
  cudaFree(m->d_err);
  cudaFree(m->d_t);
  cudaFree(m->ws);
  cudaFree(m->rope);
  for (auto e : m->prof_pool) cudaEventDestroy(e);
  if (m->graph.exec) cudaGraphExecDestroy(m->graph.exec);
  if (m->capture_stream) cudaStreamDestroy(m->capture_stream);
  cudaSetDevice(prev);
  delete m;
}

extern "C" dit_status dit_create(const dit_config* cfg, int device, dit_model** out) {
  g_last_error[0] = 0;
  if (!out) return fail(DIT_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  DIT_TRY(validate_config(cfg));
  dit_model* m = new dit_model();
  m->cfg = *cfg;
  m->device = device;
  m->bf16 = cfg->precision != DIT_PREC_F32;
  m->fp8 = cfg->precision == DIT_PREC_FP8;
  m->act = m->bf16 ? 2 : 4;
  // arena layout: block modulation tables first, contiguous per stream
  const int64_t D = cfg->hidden;
  const size_t tab_bytes = (size_t)cfg->depth * 6 * D * sizeof(float);
  size_t off = 0;
  m->tables_off = off;
  off += (tab_bytes + 255) & ~size_t(255);
  if (cfg->cond_mode == DIT_COND_JOINT) {
    m->ctx_tables_off = off;
    off += (tab_bytes + 255) & ~size_t(255);
  }
  for (auto& sp : param_specs(*cfg)) {
    Param p;
    p.spec = sp;
    p.matrix = is_matrix(sp.name);
    p.fp8 = m->fp8 && p.matrix && fp8_weight(sp.name);
    p.scale_offset = 0;
    p.numel = 1;
    for (auto d : sp.shape) p.numel *= d;
    p.loaded = false;
    const std::string& n = sp.name;
    const bool table = n.size() > 9 && n.compare(n.size() - 9, 9, "mod_table") == 0 && n.rfind("blocks.", 0) == 0;
    if (table) {
      const int b = atoi(n.c_str() + 7);
      const bool ctx = n.find(".ctx.") != std::string::npos;
      p.offset = (ctx ? m->ctx_tables_off : m->tables_off) + (size_t)b * 6 * D * sizeof(float);
    } else {
      p.offset = off;
      const size_t bytes = (size_t)p.numel * (p.fp8 ? 1 : (p.matrix ? m->act : sizeof(float)));
      off += (bytes + 255) & ~size_t(255);
      if (p.fp8) {
        p.scale_offset = off;
        off += ((size_t)sp.shape[0] * sizeof(float) + 255) & ~size_t(255);
      }
    }
    m->index[n] = (int)m->params.size();
    m->params.push_back(p);
  }
  m->arena_bytes = off;
  cudaError_t e = cudaSetDevice(device);
  if (e != cudaSuccess) {
    delete m;
    return fail(DIT_ERR_CUDA, "cudaSetDevice(%d) failed: %s", device, cudaGetErrorString(e));
  }
  e = cudaDeviceGetAttribute(&m->num_sms, cudaDevAttrMultiProcessorCount, device);
  int major = 0, minor = 0;
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, device);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, device);
  if (e != cudaSuccess) {
    delete m;
    return fail(DIT_ERR_CUDA, "device query failed: %s", cudaGetErrorString(e));
  }
  if (major * 10 + minor != 103) {
    delete m;
    return fail(DIT_ERR_CUDA, "libdit.so is built for sm_103a; device %d is sm_%d%d", device, major, minor);
  }
  dit_status st = dev_alloc(reinterpret_cast<void**>(&m->arena), m->arena_bytes);
  if (st == DIT_OK) st = dev_alloc(reinterpret_cast<void**>(&m->d_err), sizeof(int));
  if (st != DIT_OK) {
    dit_destroy(m);
    return st;
  }
  if (cudaMemset(m->d_err, 0, sizeof(int)) != cudaSuccess) {
    dit_destroy(m);
    return fail(DIT_ERR_CUDA, "cudaMemset failed");
  }
  {
    // set-up of the no-allocation entry point, done here so that its calls
    // never load a module: the fixed scratch's device address, and the
    // timestep MLP kernels it launches
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e == cudaSuccess && !p) e = cudaErrorInvalidSymbol;
    if (e == cudaSuccess) e = timestep_mlp_preload(m->bf16);
    if (e != cudaSuccess) {
      dit_destroy(m);
      return fail(DIT_ERR_CUDA, "set-up of the fixed scratch failed: %s", cudaGetErrorString(e));
    }
    m->noalloc_scratch = static_cast<float*>(p);
  }
  if (getenv("DIT_VERBOSE"))
    fprintf(stderr,
            "dit: hidden=%d heads=%d head_dim=%d mlp=%d depth=%d cond=%s precision=%s params=%zu arena=%.1f MB\n",
            cfg->hidden, cfg->heads, cfg->head_dim, cfg->mlp, cfg->depth,
            cfg->cond_mode == DIT_COND_CROSS ? "cross" : "joint", m->bf16 ? "bf16" : "fp32", m->params.size(),
            m->arena_bytes / 1e6);
  *out = m;
  return DIT_OK;
}

extern "C" int64_t dit_device_bytes(const dit_model* m) {
  if (!m) return 0;
  return (int64_t)(m->arena_bytes + m->ws_bytes + m->rope_bytes + sizeof(int) + m->d_t_cap * sizeof(float));
}

extern "C" dit_status dit_load_weights(dit_model* m, const dit_tensor* t, int n) {
  g_last_error[0] = 0;
  if (!m || (n > 0 && !t) || n < 0) return fail(DIT_ERR_INVALID_ARG, "NULL model or tensor list");
  // validate the whole call first: nothing is kept if any entry is wrong
  std::vector<int> idx(n);
  std::unordered_map<std::string, int> seen;
  for (int i = 0; i < n; ++i) {
    if (!t[i].name) return fail(DIT_ERR_SHAPE, "tensor %d has no name", i);
    auto it = m->index.find(t[i].name);
    if (it == m->index.end()) return fail(DIT_ERR_SHAPE, "unknown parameter '%s'", t[i].name);
    if (seen.count(t[i].name) || m->params[it->second].loaded)
      return fail(DIT_ERR_SHAPE, "parameter '%s' given twice", t[i].name);
    seen[t[i].name] = i;
    const Param& p = m->params[it->second];
    bool shape_ok = t[i].ndim == (int)p.spec.shape.size();
    for (int d = 0; shape_ok && d < t[i].ndim; ++d) shape_ok = t[i].shape[d] == p.spec.shape[d];
    if (!shape_ok) return fail(DIT_ERR_SHAPE, "parameter '%s' has the wrong shape", t[i].name);
    if (t[i].dtype != DIT_DTYPE_F32 && t[i].dtype != DIT_DTYPE_BF16)
      return fail(DIT_ERR_INVALID_ARG, "parameter '%s' has an unknown dtype", t[i].name);
    if (!t[i].data) return fail(DIT_ERR_INVALID_ARG, "parameter '%s' has no data", t[i].name);
    idx[i] = it->second;
  }
  CU_TRY(cudaSetDevice(m->device));
  // staging buffer for dtype conversion (largest tensor needing it)
  size_t stage_bytes = 0;
  for (int i = 0; i < n; ++i) {
    const Param& p = m->params[idx[i]];
    const bool want_bf16 = p.matrix && m->bf16;
    const bool have_bf16 = t[i].dtype == DIT_DTYPE_BF16;
    if (want_bf16 != have_bf16 || p.fp8) stage_bytes = std::max(stage_bytes, (size_t)p.numel * (have_bf16 ? 2 : 4));
  }
  void* stage = nullptr;
  DIT_TRY(dev_alloc(&stage, stage_bytes));
  dit_status st = DIT_OK;
  for (int i = 0; i < n && st == DIT_OK; ++i) {
    Param& p = m->params[idx[i]];
    char* dst = m->arena + p.offset;
    const bool want_bf16 = p.matrix && m->bf16;
    const bool have_bf16 = t[i].dtype == DIT_DTYPE_BF16;
    const size_t src_bytes = (size_t)p.numel * (have_bf16 ? 2 : 4);
    cudaError_t e;
    if (p.fp8) {
      // e4m3 with one scale per output row, quantized on the device
      e = cudaMemcpy(stage, t[i].data, src_bytes, cudaMemcpyDefault);
      if (e == cudaSuccess)
        e = quantize_rows_e4m3(stage, have_bf16, p.spec.shape[0], (int)p.spec.shape[1], reinterpret_cast<uint8_t*>(dst),
                               reinterpret_cast<float*>(m->arena + p.scale_offset), 0);
      if (e == cudaSuccess) e = cudaDeviceSynchronize();
    } else if (want_bf16 == have_bf16) {
      e = cudaMemcpy(dst, t[i].data, src_bytes, cudaMemcpyDefault);
    } else {
      e = cudaMemcpy(stage, t[i].data, src_bytes, cudaMemcpyDefault);
      if (e == cudaSuccess)
        e = want_bf16 ? f32_to_bf16(static_cast<const float*>(stage), dst, p.numel, 0)
                      : bf16_to_f32(stage, reinterpret_cast<float*>(dst), p.numel, 0);
      if (e == cudaSuccess) e = cudaDeviceSynchronize();
    }
    if (e != cudaSuccess) st = fail(DIT_ERR_CUDA, "copying '%s' failed: %s", t[i].name, cudaGetErrorString(e));
  }
  cudaFree(stage);
  if (st != DIT_OK) return st;
  for (int i = 0; i < n; ++i) {
    m->params[idx[i]].loaded = true;
    ++m->n_loaded;
  }
  return DIT_OK;
}

// ============================================================== helpers
static dit_status require_loaded(const dit_model* m) {
  if (!m) return fail(DIT_ERR_INVALID_ARG, "model is NULL");
  if (m->n_loaded != (int)m->params.size())
    return fail(DIT_ERR_NOT_LOADED, "%d of %zu parameters loaded", m->n_loaded, m->params.size());
  return DIT_OK;
}

// NVTX range names of the kernel kinds (host-side annotations for a profiler
// timeline; without an attached tool each push/pop is a no-op call).
static const char* const kKindNames[DIT_KERNEL_KINDS] = {
    "gemm_qkv", "gemm_out", "gemm_cross_q", "gemm_cross_kv", "gemm_ffn1", "gemm_ffn2",
    "gemm_embed", "attn_self", "attn_cross", "ln", "small", "cfg_euler"};

// A named NVTX range for the lifetime of the object.
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  NvtxRange(const char* fmt, int i) {
    char buf[48];
    snprintf(buf, sizeof(buf), fmt, i);
    nvtxRangePushA(buf);
  }
  ~NvtxRange() { nvtxRangePop(); }
};

// Counts the kernels a launcher enqueues, names them with an NVTX range and,
// while timing is on, brackets them with an event pair on the launching stream.
struct Launch {
  dit_model* m;
  int kind, n;
  cudaStream_t s;
  cudaEvent_t a = nullptr;
  static cudaEvent_t event(dit_model* m) {
    if (m->prof_next == m->prof_pool.size()) {
      cudaEvent_t e = nullptr;
      if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
      m->prof_pool.push_back(e);
    }
    return m->prof_pool[m->prof_next++];
  }
  Launch(dit_model* m_, int kind_, int n_, cudaStream_t s_) : m(m_), kind(kind_), n(n_), s(s_) {
    nvtxRangePushA(kKindNames[kind]);
    if (m->prof_timing && !m->capturing && (a = event(m))) cudaEventRecord(a, s);
  }
  ~Launch() {
    nvtxRangePop();
    m->prof_counts[kind] += n;
    if (a) {
      cudaEvent_t b = event(m);
      if (b) {
        cudaEventRecord(b, s);
        m->prof_rec.push_back({kind, a, b});
      }
    }
  }
};
#define LAUNCH(kind, n, expr)             \
  do {                                    \
    Launch l_(m, kind, n, s);             \
    cudaError_t e_ = (expr);              \
    if (e_ != cudaSuccess) return fail(DIT_ERR_CUDA, "%s failed: %s", #expr, cudaGetErrorString(e_)); \
  } while (0)

static dit_status ensure_ws(dit_model* m, size_t bytes) {
  if (bytes <= m->ws_bytes) return DIT_OK;
  if (m->ws) {
    CU_TRY(cudaDeviceSynchronize());
    cudaFree(m->ws);
    m->ws = nullptr;
    m->ws_bytes = 0;
  }
  DIT_TRY(dev_alloc(&m->ws, bytes));
  m->ws_bytes = bytes;
  return DIT_OK;
}

// rotary table [N][hd/2] of (cos, sin) for a token grid, built in double on
// the host once per grid shape
static dit_status ensure_rope(dit_model* m, const int32_t g[3]) {
  const dit_config& c = m->cfg;
  if (c.rope_axes[0] + c.rope_axes[1] + c.rope_axes[2] == 0) return DIT_OK;
  if (m->rope && g[0] == m->rope_grid[0] && g[1] == m->rope_grid[1] && g[2] == m->rope_grid[2]) return DIT_OK;
  const int64_t N = (int64_t)g[0] * g[1] * g[2];
  const int half = c.head_dim / 2;
  std::vector<float2> tab((size_t)N * half);
  int64_t n = 0;
  for (int it = 0; it < g[0]; ++it)
    for (int ih = 0; ih < g[1]; ++ih)
      for (int iw = 0; iw < g[2]; ++iw, ++n) {
        const int pos[3] = {it, ih, iw};
        int p = 0;
        for (int a = 0; a < 3; ++a)
          for (int j = 0; j < c.rope_axes[a] / 2; ++j, ++p) {
            const double ang = pos[a] * pow((double)c.rope_theta, -2.0 * j / c.rope_axes[a]);
            tab[(size_t)n * half + p] = make_float2((float)cos(ang), (float)sin(ang));
          }
      }
  if (m->rope) {
    CU_TRY(cudaDeviceSynchronize());
    cudaFree(m->rope);
    m->rope = nullptr;
  }
  // followed by the inverse frequency of each pair, for kernels that form
  // the angles themselves
  std::vector<float> inv(half);
  for (int a = 0, p = 0; a < 3; ++a)
    for (int j = 0; j < c.rope_axes[a] / 2; ++j, ++p)
      inv[p] = (float)pow((double)c.rope_theta, -2.0 * j / c.rope_axes[a]);
  const size_t tab_bytes = tab.size() * sizeof(float2);
  const size_t bytes = tab_bytes + half * sizeof(float);
  DIT_TRY(dev_alloc(reinterpret_cast<void**>(&m->rope), bytes));
  m->rope_bytes = bytes;
  CU_TRY(cudaMemcpy(m->rope, tab.data(), tab_bytes, cudaMemcpyHostToDevice));
  CU_TRY(cudaMemcpy(reinterpret_cast<uint8_t*>(m->rope) + tab_bytes, inv.data(), half * sizeof(float),
                    cudaMemcpyHostToDevice));
  memcpy(m->rope_grid, g, sizeof(m->rope_grid));
  return DIT_OK;
}

static dit_status do_gemm(dit_model* m, int kind, const void* A, int64_t M, int K, int64_t lda, const void* W, int N,
                          const EpiParams& ep, cudaStream_t s) {
  GemmArgs g;
  g.A = A;
  g.M = M;
  g.K = K;
  g.lda = lda;
  g.W = W;
  g.N = N;
  g.epi = ep;
  g.epi.M = (int)M;
  g.epi.N = N;
  Launch l_(m, kind, 1, s);
  cudaError_t e = ep.a_scale ? gemm_e4m3_tc(g, m->d_err, m->num_sms, s)
                  : m->bf16  ? gemm_bf16_tc(g, m->d_err, m->num_sms, s)
                             : gemm_f32(g, s);
  if (e != cudaSuccess) return fail(DIT_ERR_CUDA, "GEMM launch (M=%lld N=%d K=%d) failed: %s", (long long)M, N, K,
                                    cudaGetErrorString(e));
  return DIT_OK;
}

// Two GEMMs with the same N and K (the image and condition streams of a
// dual-stream block): one launch on the tensor-core path, two on the fp32 path.
static dit_status do_gemm_pair(dit_model* m, int kind, const void* A0, int64_t M0, const void* W0, const EpiParams& ep0,
                               const void* A1, int64_t M1, const void* W1, const EpiParams& ep1, int K, int N,
                               cudaStream_t s) {
  GemmArgs g[2];
  const void* A[2] = {A0, A1};
  const void* W[2] = {W0, W1};
  const int64_t M[2] = {M0, M1};
  const EpiParams* ep[2] = {&ep0, &ep1};
  for (int i = 0; i < 2; ++i) {
    g[i].A = A[i];
    g[i].M = M[i];
    g[i].K = K;
    g[i].lda = K;
    g[i].W = W[i];
    g[i].N = N;
    g[i].epi = *ep[i];
    g[i].epi.M = (int)M[i];
    g[i].epi.N = N;
  }
  cudaError_t e = cudaSuccess;
  if (m->bf16) {
    Launch l_(m, kind, 1, s);
    e = ep0.a_scale ? gemm_e4m3_tc_pair(g[0], g[1], m->d_err, m->num_sms, s)
                    : gemm_bf16_tc_pair(g[0], g[1], m->d_err, m->num_sms, s);
  } else {
    Launch l_(m, kind, 2, s);
    e = gemm_f32(g[0], s);
    if (e == cudaSuccess) e = gemm_f32(g[1], s);
  }
  if (e != cudaSuccess)
    return fail(DIT_ERR_CUDA, "GEMM pair launch (M=%lld+%lld N=%d K=%d) failed: %s", (long long)M0, (long long)M1, N, K,
                cudaGetErrorString(e));
  return DIT_OK;
}

// The two streams' LayerNorms of a dual-stream block (one launch on the
// staged bf16 path).
static dit_status ln_pair(dit_model* m, const LnArgs& a, const LnArgs& b, cudaStream_t s) {
  Launch l_(m, DIT_KERNEL_LN, 0, s);
  int n = 0;
  const int kind = a.row_scale ? LN_E4M3 : (m->bf16 ? LN_BF16 : LN_F32);
  cudaError_t e = ln_modulate_pair(a, b, m->cfg.hidden, m->cfg.ln_eps, kind, m->d_err, m->num_sms, s, &n);
  l_.n = n;
  if (e != cudaSuccess) return fail(DIT_ERR_CUDA, "LayerNorm pair launch failed: %s", cudaGetErrorString(e));
  return DIT_OK;
}

static dit_status do_attn(dit_model* m, int kind, const void* q, const void* k, const void* v, int B, int Lq, int Lk,
                          void* o1, void* o2, int split, cudaStream_t s) {
  AttnArgs a;
  a.q = q;
  a.k = k;
  a.v = v;
  a.B = B;
  a.H = m->cfg.heads;
  a.Lq = Lq;
  a.Lk = Lk;
  a.hd = m->cfg.head_dim;
  a.o1 = o1;
  a.o2 = o2;
  a.split = split;
  Launch l_(m, kind, 1, s);
  cudaError_t e = m->bf16 ? attention_bf16_tc(a, m->d_err, s) : attention_f32(a, s);
  if (e != cudaSuccess)
    return fail(DIT_ERR_CUDA, "attention launch (Lq=%d Lk=%d) failed: %s", Lq, Lk, cudaGetErrorString(e));
  return DIT_OK;
}

#define K_TRY(expr)                                                                                       \
  do {                                                                                                    \
    cudaError_t e_ = (expr);                                                                              \
    if (e_ != cudaSuccess) return fail(DIT_ERR_CUDA, "%s failed: %s", #expr, cudaGetErrorString(e_));   \
  } while (0)

static EpiParams epi_heads(const dit_model* m, const float* bias, void* d0, void* d1, void* d2, int rpb, int seq_total,
                           int tok_off, int rope_mask) {
  EpiParams e;
  e.kind = EPI_HEADS;
  e.bias = bias;
  e.dst[0] = d0;
  e.dst[1] = d1;
  e.dst[2] = d2;
  e.D = m->cfg.hidden;
  e.hd = m->cfg.head_dim;
  e.H = m->cfg.heads;
  e.rows_per_batch = rpb;
  e.seq_total = seq_total;
  e.tok_off = tok_off;
  e.rope_mask = m->rope ? rope_mask : 0;
  e.rope = m->rope;
  if (m->rope) {
    const int64_t n = (int64_t)m->rope_grid[0] * m->rope_grid[1] * m->rope_grid[2];
    e.rope_inv = reinterpret_cast<const float*>(m->rope + n * (m->cfg.head_dim / 2));
    e.rope_g1 = m->rope_grid[1];
    e.rope_g2 = m->rope_grid[2];
    e.rope_b0 = m->cfg.rope_axes[0] / 2;
    e.rope_b1 = (m->cfg.rope_axes[0] + m->cfg.rope_axes[1]) / 2;
  }
  return e;
}
static EpiParams epi_resid(const float* bias, float* x, const float* gate, int64_t gate_bstride, int rpb) {
  EpiParams e;
  e.kind = EPI_RESID;
  e.bias = bias;
  e.x = x;
  e.gate = gate;
  e.gate_bstride = gate_bstride;
  e.rows_per_batch = rpb;
  return e;
}
static EpiParams epi_store(int kind, const float* bias, void* out, int64_t ldo) {
  EpiParams e;
  e.kind = kind;
  e.bias = bias;
  e.out = out;
  e.ldo = ldo;
  return e;
}

// Scratch buffers of one block evaluation.
struct BlockBufs {
  void* h;         // [B, max(N, L), D] act (LN output)
  void* q;         // [B, H, S, hd] act, S = N (cross) or L + N (joint)
  void* k;
  void* v;
  void* a;         // [B, N, D] act attention output (image stream)
  void* ac;        // [B, L, D] act (joint: condition stream)
  void* g;         // [B, max(N, L), F] act MLP hidden
  void* cond_act;  // [B, L, Dc] act (cross mode, bf16 copy of the condition)
  void* kc;        // [B, H, L, hd] act (cross mode, this block's keys)
  void* vc;
  void* hc;        // [B, L, D] act (joint: condition-stream LN output)
  void* gc;        // [B, L, F] act (joint: condition-stream MLP hidden)
  float* hs;       // [B, max(N, L)] row scales of h when it holds e4m3 (fp8 precision)
  float* hcs;      // [B, L] row scales of hc (joint, fp8 precision)
};

static size_t block_ws_bytes(const dit_model* m, int B, int N, int L) {
  const dit_config& c = m->cfg;
  const size_t a = m->act;
  const int64_t NL = std::max(N, L);
  const int64_t S = c.cond_mode == DIT_COND_JOINT ? (int64_t)N + L : N;
  size_t t = 0;
  auto add = [&](int64_t elems, size_t es) { t += ((size_t)elems * es + 255) & ~size_t(255); };
  add((int64_t)B * NL * c.hidden, a);      // h
  for (int i = 0; i < 3; ++i) add((int64_t)B * S * c.hidden, a);  // q k v
  add((int64_t)B * N * c.hidden, a);       // a
  add((int64_t)B * L * c.hidden, a);       // ac
  add((int64_t)B * NL * c.mlp, a);         // g
  add((int64_t)B * L * c.cond_dim, a);     // cond_act
  add((int64_t)B * L * c.hidden, a);       // kc
  add((int64_t)B * L * c.hidden, a);       // vc
  if (c.cond_mode == DIT_COND_JOINT) {
    add((int64_t)B * L * c.hidden, a);     // hc
    add((int64_t)B * L * c.mlp, a);        // gc
  }
  if (m->fp8) {
    add((int64_t)B * NL, 4);               // hs
    add((int64_t)B * L, 4);                // hcs
  }
  return t;
}

static BlockBufs carve_block(const dit_model* m, Workspace& w, int B, int N, int L) {
  const dit_config& c = m->cfg;
  const size_t a = m->act;
  const int64_t NL = std::max(N, L);
  const int64_t S = c.cond_mode == DIT_COND_JOINT ? (int64_t)N + L : N;
  BlockBufs b;
  b.h = w.take((size_t)B * NL * c.hidden * a);
  b.q = w.take((size_t)B * S * c.hidden * a);
  b.k = w.take((size_t)B * S * c.hidden * a);
  b.v = w.take((size_t)B * S * c.hidden * a);
  b.a = w.take((size_t)B * N * c.hidden * a);
  b.ac = w.take((size_t)B * L * c.hidden * a);
  b.g = w.take((size_t)B * NL * c.mlp * a);
  b.cond_act = w.take((size_t)B * L * c.cond_dim * a);
  b.kc = w.take((size_t)B * L * c.hidden * a);
  b.vc = w.take((size_t)B * L * c.hidden * a);
  b.hc = b.gc = nullptr;
  if (c.cond_mode == DIT_COND_JOINT) {
    b.hc = w.take((size_t)B * L * c.hidden * a);
    b.gc = w.take((size_t)B * L * c.mlp * a);
  }
  b.hs = b.hcs = nullptr;
  if (m->fp8) {
    b.hs = static_cast<float*>(w.take((size_t)B * NL * 4));
    b.hcs = static_cast<float*>(w.take((size_t)B * L * 4));
  }
  return b;
}

// LayerNorm feeding a GEMM: e4m3 + row scales in fp8 precision, else the
// activation dtype.
static int ln_out_kind(const dit_model* m) { return m->fp8 ? LN_E4M3 : (m->bf16 ? LN_BF16 : LN_F32); }
// The same epilogue with the operand scales of an e4m3 GEMM (no change when
// the weight is not e4m3).
static EpiParams scaled(EpiParams e, const float* a_scale, const float* w_scale) {
  if (w_scale) {
    e.a_scale = a_scale;
    e.w_scale = w_scale;
  }
  return e;
}

// Cross-attention keys/values of the condition tokens for one block:
// [B*L, Dc] x W_kv^T -> head-major kc, vc.
static dit_status cross_kv(dit_model* m, int blk, const void* cond_act, int B, int L, void* kc, void* vc,
                           cudaStream_t s) {
  const dit_config& c = m->cfg;
  EpiParams ep = epi_heads(m, m->V(m->blk(blk, "cross.kv.bias")), kc, vc, nullptr, L, L, 0, 0);
  return do_gemm(m, DIT_KERNEL_GEMM_CROSS_KV, cond_act, (int64_t)B * L, c.cond_dim, c.cond_dim, m->W(m->blk(blk, "cross.kv.weight")),
                 2 * c.hidden, ep, s);
}

// One DiT block on the residual stream(s).  mod/modc point at this block's
// [6][D] modulation (plus b * mod_bstride per batch element).
static dit_status run_block(dit_model* m, int blk, float* x, float* xc, const float* mod, const float* modc,
                            int64_t mod_bstride, const void* kc, const void* vc, int B, int N, int L,
                            bool ctx_out_needed, const BlockBufs& bb, cudaStream_t s) {
  NvtxRange range("dit.block %d", blk);
  const dit_config& c = m->cfg;
  const int D = c.hidden, F = c.mlp;
  const float eps = c.ln_eps;
  const int lk = ln_out_kind(m);  // LayerNorm outputs that feed a GEMM directly
  float* hs = bb.hs;              // their row scales (fp8 precision), else unused
  auto Wt = [&](const char* n) { return m->W(m->blk(blk, n)); };
  auto Sc = [&](const char* n) { return m->S(m->blk(blk, n)); };
  if (c.cond_mode == DIT_COND_CROSS) {
    const int64_t R = (int64_t)B * N;
    // self-attention half
    LAUNCH(DIT_KERNEL_LN, 1, ln_modulate(x, R, D, N, mod + 0 * D, mod + 1 * D, mod_bstride, eps, bb.h, lk, m->d_err, m->num_sms, s, hs));
    DIT_TRY(do_gemm(m, DIT_KERNEL_GEMM_QKV, bb.h, R, D, D, Wt("attn.qkv.weight"), 3 * D,
                    scaled(epi_heads(m, m->V(m->blk(blk, "attn.qkv.bias")), bb.q, bb.k, bb.v, N, N, 0, 0x3), hs,
                           Sc("attn.qkv.weight")), s));
    DIT_TRY(do_attn(m, DIT_KERNEL_ATTN_SELF, bb.q, bb.k, bb.v, B, N, N, bb.a, nullptr, N, s));
    DIT_TRY(do_gemm(m, DIT_KERNEL_GEMM_OUT, bb.a, R, D, D, Wt("attn.out.weight"), D,
                    epi_resid(m->V(m->blk(blk, "attn.out.bias")), x, mod + 2 * D, mod_bstride, N), s));
    // cross-attention half: plain LN, no rotation, ungated residual
    LAUNCH(DIT_KERNEL_LN, 1, ln_modulate(x, R, D, N, nullptr, nullptr, 0, eps, bb.h, lk, m->d_err, m->num_sms, s, hs));
    DIT_TRY(do_gemm(m, DIT_KERNEL_GEMM_CROSS_Q, bb.h, R, D, D, Wt("cross.q.weight"), D,
                    scaled(epi_heads(m, m->V(m->blk(blk, "cross.q.bias")), bb.q, nullptr, nullptr, N, N, 0, 0), hs,
                           Sc("cross.q.weight")), s));
    DIT_TRY(do_attn(m, DIT_KERNEL_ATTN_CROSS, bb.q, kc, vc, B, N, L, bb.a, nullptr, N, s));
    DIT_TRY(do_gemm(m, DIT_KERNEL_GEMM_OUT, bb.a, R, D, D, Wt("cross.out.weight"), D,
                    epi_resid(m->V(m->blk(blk, "cross.out.bias")), x, nullptr, 0, N), s));
    // MLP half
    LAUNCH(DIT_KERNEL_LN, 1, ln_modulate(x, R, D, N, mod + 3 * D, mod + 4 * D, mod_bstride, eps, bb.h, lk, m->d_err, m->num_sms, s, hs));
    DIT_TRY(do_gemm(m, DIT_KERNEL_GEMM_FFN1, bb.h, R, D, D, Wt("mlp.fc1.weight"), F,
                    scaled(epi_store(EPI_GELU, m->V(m->blk(blk, "mlp.fc1.bias")), bb.g, F), hs, Sc("mlp.fc1.weight")),
                    s));
    DIT_TRY(do_gemm(m, DIT_KERNEL_GEMM_FFN2, bb.g, R, F, F, Wt("mlp.fc2.weight"), D,
                    epi_resid(m->V(m->blk(blk, "mlp.fc2.bias")), x, mod + 5 * D, mod_bstride, N), s));
    return DIT_OK;
  }
  // joint (dual-stream) block: sequence [condition; image].  The two streams'
  // GEMMs of equal shape run as one launch (image rows first, condition rows
  // after), so the condition stream's 1024 rows fill the image GEMM's last wave.
  const int S = L + N;
  const int64_t R = (int64_t)B * N, Rc = (int64_t)B * L;
  float* hcs = bb.hcs;
  auto ln_args = [&](const float* xx, int64_t rows, int rpb, const float* sh, const float* sc, void* out,
                     float* rs) {
    LnArgs a{xx, rows, rpb, sh, sc, mod_bstride, out};
    a.row_scale = m->fp8 ? rs : nullptr;
    return a;
  };
  DIT_TRY(ln_pair(m, ln_args(x, R, N, mod + 0 * D, mod + 1 * D, bb.h, hs),
                  ln_args(xc, Rc, L, modc + 0 * D, modc + 1 * D, bb.hc, hcs), s));
  DIT_TRY(do_gemm_pair(m, DIT_KERNEL_GEMM_QKV,
                       bb.h, R, Wt("attn.qkv.weight"),
                       scaled(epi_heads(m, m->V(m->blk(blk, "attn.qkv.bias")), bb.q, bb.k, bb.v, N, S, L, 0x3), hs,
                              Sc("attn.qkv.weight")),
                       bb.hc, Rc, Wt("ctx.attn.qkv.weight"),
                       scaled(epi_heads(m, m->V(m->blk(blk, "ctx.attn.qkv.bias")), bb.q, bb.k, bb.v, L, S, 0, 0), hcs,
                              Sc("ctx.attn.qkv.weight")),
                       D, 3 * D, s));
  DIT_TRY(do_attn(m, DIT_KERNEL_ATTN_SELF, bb.q, bb.k, bb.v, B, S, S, bb.ac, bb.a, L, s));
  if (!ctx_out_needed) {
    // last block: the condition stream's output is never read
    DIT_TRY(do_gemm(m, DIT_KERNEL_GEMM_OUT, bb.a, R, D, D, Wt("attn.out.weight"), D,
                    epi_resid(m->V(m->blk(blk, "attn.out.bias")), x, mod + 2 * D, mod_bstride, N), s));
    LAUNCH(DIT_KERNEL_LN, 1, ln_modulate(x, R, D, N, mod + 3 * D, mod + 4 * D, mod_bstride, eps, bb.h, lk, m->d_err, m->num_sms, s, hs));
    DIT_TRY(do_gemm(m, DIT_KERNEL_GEMM_FFN1, bb.h, R, D, D, Wt("mlp.fc1.weight"), F,
                    scaled(epi_store(EPI_GELU, m->V(m->blk(blk, "mlp.fc1.bias")), bb.g, F), hs, Sc("mlp.fc1.weight")),
                    s));
    DIT_TRY(do_gemm(m, DIT_KERNEL_GEMM_FFN2, bb.g, R, F, F, Wt("mlp.fc2.weight"), D,
                    epi_resid(m->V(m->blk(blk, "mlp.fc2.bias")), x, mod + 5 * D, mod_bstride, N), s));
    return DIT_OK;
  }
  DIT_TRY(do_gemm_pair(m, DIT_KERNEL_GEMM_OUT,
                       bb.a, R, Wt("attn.out.weight"),
                       epi_resid(m->V(m->blk(blk, "attn.out.bias")), x, mod + 2 * D, mod_bstride, N),
                       bb.ac, Rc, Wt("ctx.attn.out.weight"),
                       epi_resid(m->V(m->blk(blk, "ctx.attn.out.bias")), xc, modc + 2 * D, mod_bstride, L),
                       D, D, s));
  DIT_TRY(ln_pair(m, ln_args(x, R, N, mod + 3 * D, mod + 4 * D, bb.h, hs),
                  ln_args(xc, Rc, L, modc + 3 * D, modc + 4 * D, bb.hc, hcs), s));
  DIT_TRY(do_gemm_pair(m, DIT_KERNEL_GEMM_FFN1,
                       bb.h, R, Wt("mlp.fc1.weight"),
                       scaled(epi_store(EPI_GELU, m->V(m->blk(blk, "mlp.fc1.bias")), bb.g, F), hs, Sc("mlp.fc1.weight")),
                       bb.hc, Rc, Wt("ctx.mlp.fc1.weight"),
                       scaled(epi_store(EPI_GELU, m->V(m->blk(blk, "ctx.mlp.fc1.bias")), bb.gc, F), hcs,
                              Sc("ctx.mlp.fc1.weight")),
                       D, F, s));
  DIT_TRY(do_gemm_pair(m, DIT_KERNEL_GEMM_FFN2,
                       bb.g, R, Wt("mlp.fc2.weight"),
                       epi_resid(m->V(m->blk(blk, "mlp.fc2.bias")), x, mod + 5 * D, mod_bstride, N),
                       bb.gc, Rc, Wt("ctx.mlp.fc2.weight"),
                       epi_resid(m->V(m->blk(blk, "ctx.mlp.fc2.bias")), xc, modc + 5 * D, mod_bstride, L),
                       F, D, s));
  return DIT_OK;
}

static dit_status check_latent(const dit_model* m, int batch, const int32_t thw[3]) {
  if (batch <= 0) return fail(DIT_ERR_INVALID_ARG, "batch must be positive");
  if (!thw) return fail(DIT_ERR_INVALID_ARG, "latent shape is NULL");
  for (int i = 0; i < 3; ++i) {
    if (thw[i] <= 0) return fail(DIT_ERR_SHAPE, "latent dims must be positive");
    if (thw[i] % m->cfg.patch[i])
      return fail(DIT_ERR_SHAPE, "latent dim %d (%d) not divisible by patch %d", i, thw[i], m->cfg.patch[i]);
  }
  return DIT_OK;
}

// ============================================================== ABI: pieces
extern "C" dit_status dit_timestep_modulation(dit_model* m, const float* t_host, int batch, float* mod,
                                              void* stream) {
  g_last_error[0] = 0;
  DIT_TRY(require_loaded(m));
  if (!t_host || !mod || batch <= 0) return fail(DIT_ERR_INVALID_ARG, "bad timestep arguments");
  for (int b = 0; b < batch; ++b)
    if (!isfinite(t_host[b])) return fail(DIT_ERR_INVALID_ARG, "timestep %d is not finite", b);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  CU_TRY(cudaSetDevice(m->device));
  if (m->d_t_cap < batch) {
    CU_TRY(cudaDeviceSynchronize());
    cudaFree(m->d_t);
    m->d_t = nullptr;
    m->d_t_cap = 0;
    DIT_TRY(dev_alloc(reinterpret_cast<void**>(&m->d_t), batch * sizeof(float)));
    m->d_t_cap = batch;
  }
  const size_t need = (size_t)batch * m->cfg.hidden * sizeof(float) + 256;
  DIT_TRY(ensure_ws(m, need));
  CU_TRY(cudaMemcpyAsync(m->d_t, t_host, batch * sizeof(float), cudaMemcpyHostToDevice, s));
  LAUNCH(DIT_KERNEL_SMALL, 2, timestep_mlp(m->d_t, 0.0, batch, m->cfg.freq_dim, m->cfg.hidden, m->W("time_mlp.fc1.weight"),
                     m->V("time_mlp.fc1.bias"), m->W("time_mlp.fc2.weight"), m->V("time_mlp.fc2.bias"), m->bf16,
                     static_cast<float*>(m->ws), mod, s));
  return DIT_OK;
}

extern "C" dit_status dit_timestep_modulation_noalloc(dit_model* m, const float* t_host, int batch, float* mod,
                                                      void* stream) {
  g_last_error[0] = 0;
  DIT_TRY(require_loaded(m));
  if (!t_host || !mod || batch <= 0) return fail(DIT_ERR_INVALID_ARG, "bad timestep arguments");
  if (batch > DIT_NOALLOC_MAX_BATCH)
    return fail(DIT_ERR_INVALID_ARG, "batch %d exceeds the fixed scratch limit of %d", batch,
                (int)DIT_NOALLOC_MAX_BATCH);
  if ((int64_t)batch * m->cfg.hidden > DIT_NOALLOC_MAX_HIDDEN)
    return fail(DIT_ERR_INVALID_ARG, "batch * hidden = %lld exceeds the fixed scratch limit of %d floats",
                (long long)batch * m->cfg.hidden, (int)DIT_NOALLOC_MAX_HIDDEN);
  if (m->cfg.hidden > kTimestepMlpMaxHidden || m->cfg.freq_dim > kTimestepMlpMaxHidden)
    return fail(DIT_ERR_INVALID_ARG, "hidden %d / freq_dim %d exceed the timestep MLP limit of %d", m->cfg.hidden,
                m->cfg.freq_dim, kTimestepMlpMaxHidden);
  for (int b = 0; b < batch; ++b)
    if (!isfinite(t_host[b])) return fail(DIT_ERR_INVALID_ARG, "timestep %d is not finite", b);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  CU_TRY(cudaSetDevice(m->device));
  float* scratch = m->noalloc_scratch;
  float* t_dev = scratch;                          // [batch] timesteps
  float* hidden = scratch + DIT_NOALLOC_MAX_BATCH;  // [batch, hidden], fully written by fc1 before fc2 reads it
  CU_TRY(cudaMemcpyAsync(t_dev, t_host, batch * sizeof(float), cudaMemcpyHostToDevice, s));
  LAUNCH(DIT_KERNEL_SMALL, 2, timestep_mlp(t_dev, 0.0, batch, m->cfg.freq_dim, m->cfg.hidden, m->W("time_mlp.fc1.weight"),
                                            m->V("time_mlp.fc1.bias"), m->W("time_mlp.fc2.weight"),
                                            m->V("time_mlp.fc2.bias"), m->bf16, hidden, mod, s));
  return DIT_OK;
}

extern "C" dit_status dit_patch_embed(dit_model* m, const float* lat, int batch, const int32_t thw[3], float* x,
                                      void* stream) {
  g_last_error[0] = 0;
  DIT_TRY(require_loaded(m));
  DIT_TRY(check_latent(m, batch, thw));
  if (!lat || !x) return fail(DIT_ERR_INVALID_ARG, "NULL tensor");
  const dit_config& c = m->cfg;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  CU_TRY(cudaSetDevice(m->device));
  const int64_t N = (int64_t)(thw[0] / c.patch[0]) * (thw[1] / c.patch[1]) * (thw[2] / c.patch[2]);
  const int P = c.in_channels * c.patch[0] * c.patch[1] * c.patch[2];
  DIT_TRY(ensure_ws(m, (size_t)batch * N * P * m->act + 256));
  LAUNCH(DIT_KERNEL_SMALL, 1, patchify(lat, batch, 1, c.in_channels, thw[0], thw[1], thw[2], c.patch[0], c.patch[1], c.patch[2], m->ws,
                 m->bf16, s));
  return do_gemm(m, DIT_KERNEL_GEMM_EMBED, m->ws, (int64_t)batch * N, P, P, m->W("patch_embed.weight"), c.hidden,
                 epi_store(EPI_F32, m->V("patch_embed.bias"), x, c.hidden), s);
}

extern "C" dit_status dit_block_forward(dit_model* m, int block, float* x, float* xc, const float* mod,
                                        const float* cond, int batch, const int32_t grid[3], int cond_len,
                                        void* stream) {
  g_last_error[0] = 0;
  DIT_TRY(require_loaded(m));
  const dit_config& c = m->cfg;
  if (block < 0 || block >= c.depth) return fail(DIT_ERR_INVALID_ARG, "block %d out of range", block);
  if (!x || !mod || batch <= 0 || !grid) return fail(DIT_ERR_INVALID_ARG, "NULL tensor or bad batch");
  if (grid[0] <= 0 || grid[1] <= 0 || grid[2] <= 0) return fail(DIT_ERR_SHAPE, "grid dims must be positive");
  if (cond_len <= 0) return fail(DIT_ERR_SHAPE, "cond_len must be positive");
  if (c.cond_mode == DIT_COND_CROSS && (!cond || xc))
    return fail(DIT_ERR_INVALID_ARG, "cross mode takes cond and no xc");
  if (c.cond_mode == DIT_COND_JOINT && (cond || !xc))
    return fail(DIT_ERR_INVALID_ARG, "joint mode takes xc and no cond");
  const int64_t N64 = (int64_t)grid[0] * grid[1] * grid[2];
  if (N64 > (1 << 24)) return fail(DIT_ERR_SHAPE, "too many tokens");
  const int N = (int)N64, L = cond_len, D = c.hidden;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  CU_TRY(cudaSetDevice(m->device));
  const size_t modtab_bytes = (size_t)2 * batch * 6 * D * sizeof(float);
  DIT_TRY(ensure_rope(m, grid));
  DIT_TRY(ensure_ws(m, block_ws_bytes(m, batch, N, L) + modtab_bytes + 4096));
  Workspace w{m->ws, m->ws_bytes, 0};
  BlockBufs bb = carve_block(m, w, batch, N, L);
  float* modtab = static_cast<float*>(w.take((size_t)batch * 6 * D * sizeof(float)));
  float* modtab_c = static_cast<float*>(w.take((size_t)batch * 6 * D * sizeof(float)));
  LAUNCH(DIT_KERNEL_SMALL, 1, add_tables(mod, batch, D, 6, m->V(m->blk(block, "mod_table")), 1, modtab, s));
  if (c.cond_mode == DIT_COND_JOINT)
    LAUNCH(DIT_KERNEL_SMALL, 1, add_tables(mod, batch, D, 6, m->V(m->blk(block, "ctx.mod_table")), 1, modtab_c, s));
  const void* kc = nullptr;
  const void* vc = nullptr;
  if (c.cond_mode == DIT_COND_CROSS) {
    const void* ca = cond;
    if (m->bf16) {
      LAUNCH(DIT_KERNEL_SMALL, 1, f32_to_bf16(cond, bb.cond_act, (int64_t)batch * L * c.cond_dim, s));
      ca = bb.cond_act;
    }
    DIT_TRY(cross_kv(m, block, ca, batch, L, bb.kc, bb.vc, s));
    kc = bb.kc;
    vc = bb.vc;
  }
  return run_block(m, block, x, xc, modtab, modtab_c, 6 * D, kc, vc, batch, N, L, true, bb, s);
}

extern "C" dit_status dit_final_layer(dit_model* m, const float* x, const float* mod, int batch,
                                      const int32_t thw[3], float* v, void* stream) {
  g_last_error[0] = 0;
  DIT_TRY(require_loaded(m));
  DIT_TRY(check_latent(m, batch, thw));
  if (!x || !mod || !v) return fail(DIT_ERR_INVALID_ARG, "NULL tensor");
  const dit_config& c = m->cfg;
  const int D = c.hidden;
  const int64_t N = (int64_t)(thw[0] / c.patch[0]) * (thw[1] / c.patch[1]) * (thw[2] / c.patch[2]);
  const int P = c.in_channels * c.patch[0] * c.patch[1] * c.patch[2];
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  CU_TRY(cudaSetDevice(m->device));
  Workspace w{nullptr, 0, 0};
  const size_t need = (size_t)batch * 2 * D * 4 + (size_t)batch * N * D * m->act + (size_t)batch * N * P * 4 + 1024;
  DIT_TRY(ensure_ws(m, need));
  w.base = m->ws;
  w.bytes = m->ws_bytes;
  float* headtab = static_cast<float*>(w.take((size_t)batch * 2 * D * 4));
  void* h = w.take((size_t)batch * N * D * m->act);
  float* vt = static_cast<float*>(w.take((size_t)batch * N * P * 4));
  LAUNCH(DIT_KERNEL_SMALL, 1, add_tables(mod, batch, D, 2, m->V("head.mod_table"), 1, headtab, s));
  LAUNCH(DIT_KERNEL_LN, 1, ln_modulate(x, batch * N, D, (int)N, headtab, headtab + D, 2 * D, c.ln_eps, h, m->bf16 ? LN_BF16 : LN_F32, m->d_err, m->num_sms, s));
  DIT_TRY(do_gemm(m, DIT_KERNEL_GEMM_EMBED, h, batch * N, D, D, m->W("head.weight"), P, epi_store(EPI_F32, m->V("head.bias"), vt, P), s));
  LAUNCH(DIT_KERNEL_SMALL, 1, unpatchify(vt, batch, c.in_channels, thw[0], thw[1], thw[2], c.patch[0], c.patch[1], c.patch[2], v, s));
  return DIT_OK;
}

extern "C" dit_status cfg_combine(const float* vc, const float* vu, float g, float* v, int64_t n, void* stream) {
  g_last_error[0] = 0;
  if (n < 0 || (n > 0 && (!vc || !vu || !v))) return fail(DIT_ERR_INVALID_ARG, "bad cfg_combine arguments");
  if (!isfinite(g)) return fail(DIT_ERR_INVALID_ARG, "guidance scale is not finite");
  K_TRY(cfg_combine_kernel(vc, vu, g, v, n, static_cast<cudaStream_t>(stream)));
  return DIT_OK;
}

extern "C" dit_status flow_euler_step(float* x, const float* v, float sigma, float sigma_next, int64_t n,
                                      void* stream) {
  g_last_error[0] = 0;
  if (n < 0 || (n > 0 && (!x || !v))) return fail(DIT_ERR_INVALID_ARG, "bad flow_euler_step arguments");
  if (!isfinite(sigma) || !isfinite(sigma_next)) return fail(DIT_ERR_INVALID_ARG, "sigma is not finite");
  const float dsig = (float)((double)sigma_next - (double)sigma);
  K_TRY(euler_kernel(x, v, dsig, n, static_cast<cudaStream_t>(stream)));
  return DIT_OK;
}

// ============================================================== ABI: loop
extern "C" dit_status dit_denoise_loop(dit_model* m, float* latents, int batch, const int32_t thw[3],
                                       const float* cond, const float* uncond, int cond_len, const float* sigmas,
                                       int n_steps, float guidance, uint32_t flags, void* stream) {
  g_last_error[0] = 0;
  DIT_TRY(require_loaded(m));
  DIT_TRY(check_latent(m, batch, thw));
  const dit_config& c = m->cfg;
  if (!latents || !cond) return fail(DIT_ERR_INVALID_ARG, "NULL latents or cond");
  if (cond_len <= 0) return fail(DIT_ERR_SHAPE, "cond_len must be positive");
  if (n_steps <= 0 || !sigmas) return fail(DIT_ERR_INVALID_ARG, "need n_steps > 0 and n_steps + 1 sigmas");
  if (flags & ~(uint32_t)(DIT_LOOP_PARTIAL_SCHEDULE | DIT_LOOP_CUDA_GRAPH))
    return fail(DIT_ERR_INVALID_ARG, "unknown flags");
  if ((flags & DIT_LOOP_CUDA_GRAPH) && m->prof_timing)
    return fail(DIT_ERR_INVALID_ARG, "DIT_LOOP_CUDA_GRAPH cannot be combined with per-launch timing (dit_profile_start)");
  if (!isfinite(guidance)) return fail(DIT_ERR_INVALID_ARG, "guidance is not finite");
  if (!uncond && guidance != 1.0f)
    return fail(DIT_ERR_INVALID_ARG, "guidance %g needs negative condition tokens (uncond is NULL)", guidance);
  for (int i = 0; i <= n_steps; ++i)
    if (!isfinite(sigmas[i])) return fail(DIT_ERR_INVALID_ARG, "sigma %d is not finite", i);
  for (int i = 0; i < n_steps; ++i)
    if (!(sigmas[i + 1] < sigmas[i]))
      return fail(DIT_ERR_INVALID_ARG, "sigmas must be strictly decreasing (reversed schedule?) at step %d", i);
  if (!(flags & DIT_LOOP_PARTIAL_SCHEDULE) && (sigmas[0] != 1.0f || sigmas[n_steps] != 0.0f))
    return fail(DIT_ERR_INVALID_ARG, "schedule must run from sigma 1 to 0 (set DIT_LOOP_PARTIAL_SCHEDULE to resume)");
  const bool cfg = uncond != nullptr;
  const int Bq = batch, B = cfg ? 2 * batch : batch;
  const int32_t grid[3] = {thw[0] / c.patch[0], thw[1] / c.patch[1], thw[2] / c.patch[2]};
  const int64_t N64 = (int64_t)grid[0] * grid[1] * grid[2];
  if (N64 > (1 << 24)) return fail(DIT_ERR_SHAPE, "too many tokens");
  const int N = (int)N64, L = cond_len, D = c.hidden, P = c.in_channels * c.patch[0] * c.patch[1] * c.patch[2];
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  CU_TRY(cudaSetDevice(m->device));
  DIT_TRY(ensure_rope(m, grid));

  // workspace: block scratch + loop state
  const size_t a = m->act;
  const int nst = c.cond_mode == DIT_COND_JOINT ? 2 : 1;
  size_t need = block_ws_bytes(m, B, N, L);
  need += (size_t)c.depth * nst * 6 * D * 4 + 2 * D * 4 + 6 * D * 4 + D * 4;  // tables, m, temb hidden
  need += (size_t)B * N * D * 4;                                                // x
  need += (size_t)B * L * D * 4;                                                // xc
  need += (size_t)B * N * P * a + (size_t)B * N * P * 4;                        // tokens, vt
  if (c.cond_mode == DIT_COND_CROSS) need += (size_t)c.depth * 2 * B * L * D * a;  // K/V cache
  need += (size_t)(n_steps + 1) * sizeof(float) + sizeof(int);                  // schedule, step counter
  need += 64 * 256;
  DIT_TRY(ensure_ws(m, need));
  Workspace w{m->ws, m->ws_bytes, 0};
  BlockBufs bb = carve_block(m, w, B, N, L);
  float* tabs = static_cast<float*>(w.take((size_t)c.depth * 6 * D * 4));
  float* tabs_c = nst == 2 ? static_cast<float*>(w.take((size_t)c.depth * 6 * D * 4)) : nullptr;
  float* headtab = static_cast<float*>(w.take((size_t)2 * D * 4));
  float* mvec = static_cast<float*>(w.take((size_t)6 * D * 4));
  float* thid = static_cast<float*>(w.take((size_t)D * 4));
  float* x = static_cast<float*>(w.take((size_t)B * N * D * 4));
  float* xc = static_cast<float*>(w.take((size_t)B * L * D * 4));
  void* tokens = w.take((size_t)B * N * P * a);
  float* vt = static_cast<float*>(w.take((size_t)B * N * P * 4));
  void* kvcache = c.cond_mode == DIT_COND_CROSS ? w.take((size_t)c.depth * 2 * B * L * D * a) : nullptr;
  int* step_dev = static_cast<int*>(w.take(sizeof(int)));
  float* sig_dev = static_cast<float*>(w.take((size_t)(n_steps + 1) * sizeof(float)));

  // condition rows: [cond (Bq); uncond (Bq)]
  const size_t cond_bytes = (size_t)Bq * L * c.cond_dim * 4;
  if (c.cond_mode == DIT_COND_CROSS) {
    // keys/values of the condition tokens do not depend on the step: once per call
    float* cf = xc;  // xc is unused in cross mode; borrow it to stage fp32 rows
    if ((size_t)B * L * c.cond_dim > (size_t)B * L * D) {
      // cond_dim > hidden: stage through the MLP scratch instead
      cf = static_cast<float*>(bb.g);
    }
    CU_TRY(cudaMemcpyAsync(cf, cond, cond_bytes, cudaMemcpyDeviceToDevice, s));
    if (cfg) CU_TRY(cudaMemcpyAsync(cf + (size_t)Bq * L * c.cond_dim, uncond, cond_bytes, cudaMemcpyDeviceToDevice, s));
    const void* ca = cf;
    if (m->bf16) {
      LAUNCH(DIT_KERNEL_SMALL, 1, f32_to_bf16(cf, bb.cond_act, (int64_t)B * L * c.cond_dim, s));
      ca = bb.cond_act;
    }
    const size_t per = (size_t)B * L * D * a;
    for (int blk = 0; blk < c.depth; ++blk) {
      char* kb = static_cast<char*>(kvcache) + (size_t)blk * 2 * per;
      DIT_TRY(cross_kv(m, blk, ca, B, L, kb, kb + per, s));
    }
  }
  // Device copy of the schedule and a step counter: every step reads its
  // timestep and Euler increment from them, so the launches of a step are
  // the same for every step (and can be captured once and replayed).
  CU_TRY(cudaMemcpyAsync(sig_dev, sigmas, (size_t)(n_steps + 1) * sizeof(float), cudaMemcpyHostToDevice, s));
  CU_TRY(cudaMemsetAsync(step_dev, 0, sizeof(int), s));
  const size_t per = (size_t)B * L * D * a;
  auto enqueue_step = [&](cudaStream_t s) -> dit_status {
    NvtxRange range("dit.step");
    LAUNCH(DIT_KERNEL_SMALL, 2, timestep_mlp_sched(sig_dev, step_dev, (double)c.timestep_scale, c.freq_dim, D,
                                                   m->W("time_mlp.fc1.weight"), m->V("time_mlp.fc1.bias"),
                                                   m->W("time_mlp.fc2.weight"), m->V("time_mlp.fc2.bias"), m->bf16,
                                                   thid, mvec, s));
    LAUNCH(DIT_KERNEL_SMALL, 1, add_tables(mvec, 1, D, 6, m->V("blocks.0.mod_table"), c.depth, tabs, s));
    if (tabs_c) LAUNCH(DIT_KERNEL_SMALL, 1, add_tables(mvec, 1, D, 6, m->V("blocks.0.ctx.mod_table"), c.depth, tabs_c, s));
    LAUNCH(DIT_KERNEL_SMALL, 1, add_tables(mvec, 1, D, 2, m->V("head.mod_table"), 1, headtab, s));
    LAUNCH(DIT_KERNEL_SMALL, 1, patchify(latents, Bq, cfg ? 2 : 1, c.in_channels, thw[0], thw[1], thw[2], c.patch[0], c.patch[1],
                   c.patch[2], tokens, m->bf16, s));
    DIT_TRY(do_gemm(m, DIT_KERNEL_GEMM_EMBED, tokens, (int64_t)B * N, P, P, m->W("patch_embed.weight"), D,
                    epi_store(EPI_F32, m->V("patch_embed.bias"), x, D), s));
    if (c.cond_mode == DIT_COND_JOINT) {
      CU_TRY(cudaMemcpyAsync(xc, cond, cond_bytes, cudaMemcpyDeviceToDevice, s));
      if (cfg) CU_TRY(cudaMemcpyAsync(xc + (size_t)Bq * L * D, uncond, cond_bytes, cudaMemcpyDeviceToDevice, s));
    }
    for (int blk = 0; blk < c.depth; ++blk) {
      const void* kc = nullptr;
      const void* vc = nullptr;
      if (kvcache) {
        kc = static_cast<char*>(kvcache) + (size_t)blk * 2 * per;
        vc = static_cast<const char*>(kc) + per;
      }
      DIT_TRY(run_block(m, blk, x, c.cond_mode == DIT_COND_JOINT ? xc : nullptr, tabs + (size_t)blk * 6 * D,
                        tabs_c ? tabs_c + (size_t)blk * 6 * D : nullptr, 0, kc, vc, B, N, L, blk + 1 < c.depth, bb,
                        s));
    }
    LAUNCH(DIT_KERNEL_LN, 1, ln_modulate(x, (int64_t)B * N, D, N, headtab, headtab + D, 0, c.ln_eps, bb.h, m->bf16 ? LN_BF16 : LN_F32, m->d_err, m->num_sms, s));
    DIT_TRY(do_gemm(m, DIT_KERNEL_GEMM_EMBED, bb.h, (int64_t)B * N, D, D, m->W("head.weight"), P,
                    epi_store(EPI_F32, m->V("head.bias"), vt, P), s));
    LAUNCH(DIT_KERNEL_CFG_EULER, 1, cfg_euler_tokens(vt, Bq, cfg, guidance, sig_dev, step_dev, c.in_channels, thw[0], thw[1],
                                                     thw[2], c.patch[0], c.patch[1], c.patch[2], latents, m->d_err, s));
    LAUNCH(DIT_KERNEL_SMALL, 1, step_advance(step_dev, s));
    return DIT_OK;
  };
  if (!(flags & DIT_LOOP_CUDA_GRAPH)) {
    for (int i = 0; i < n_steps; ++i) DIT_TRY(enqueue_step(s));
    return DIT_OK;
  }
  // Graph path: the step is captured once on the model's own stream (nothing
  // runs during capture) and replayed n_steps times on the caller's stream.
  // The capture is reused while every pointer and scalar it holds is the same.
  float gbits = guidance;
  uint32_t gu = 0;
  memcpy(&gu, &gbits, sizeof(gu));
  const std::vector<uint64_t> key = {
      (uint64_t)(uintptr_t)latents, (uint64_t)(uintptr_t)cond,  (uint64_t)(uintptr_t)uncond,
      (uint64_t)(uintptr_t)m->ws,   (uint64_t)m->ws_bytes,      (uint64_t)(uintptr_t)m->rope,
      (uint64_t)Bq,                 (uint64_t)thw[0],           (uint64_t)thw[1],
      (uint64_t)thw[2],             (uint64_t)L,                (uint64_t)gu,
      (uint64_t)(uintptr_t)sig_dev, (uint64_t)(uintptr_t)step_dev};
  if (!m->graph.exec || m->graph.key != key) {
    if (m->graph.exec) {
      cudaGraphExecDestroy(m->graph.exec);
      m->graph.exec = nullptr;
    }
    if (!m->capture_stream) CU_TRY(cudaStreamCreateWithFlags(&m->capture_stream, cudaStreamNonBlocking));
    // the capture stream starts after the schedule upload and counter reset above
    cudaEvent_t ready = nullptr;
    CU_TRY(cudaEventCreateWithFlags(&ready, cudaEventDisableTiming));
    cudaError_t e = cudaEventRecord(ready, s);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(m->capture_stream, ready, 0);
    cudaEventDestroy(ready);
    if (e != cudaSuccess) return fail(DIT_ERR_CUDA, "ordering the capture stream failed: %s", cudaGetErrorString(e));
    int64_t before[DIT_KERNEL_KINDS];
    memcpy(before, m->prof_counts, sizeof(before));
    CU_TRY(cudaStreamBeginCapture(m->capture_stream, cudaStreamCaptureModeRelaxed));
    m->capturing = true;
    const dit_status st = enqueue_step(m->capture_stream);
    m->capturing = false;
    cudaGraph_t graph = nullptr;
    e = cudaStreamEndCapture(m->capture_stream, &graph);
    if (st != DIT_OK) {
      if (graph) cudaGraphDestroy(graph);
      return st;
    }
    if (e != cudaSuccess) return fail(DIT_ERR_CUDA, "capturing the loop step failed: %s", cudaGetErrorString(e));
    e = cudaGraphInstantiate(&m->graph.exec, graph, 0);
    cudaGraphDestroy(graph);
    if (e != cudaSuccess) {
      m->graph.exec = nullptr;
      return fail(DIT_ERR_CUDA, "instantiating the loop step graph failed: %s", cudaGetErrorString(e));
    }
    // the capture launched nothing: its launches are counted when replayed
    for (int k = 0; k < DIT_KERNEL_KINDS; ++k) {
      m->graph.counts[k] = m->prof_counts[k] - before[k];
      m->prof_counts[k] = before[k];
    }
    m->graph.key = key;
  }
  for (int i = 0; i < n_steps; ++i) {
    CU_TRY(cudaGraphLaunch(m->graph.exec, s));
    for (int k = 0; k < DIT_KERNEL_KINDS; ++k) m->prof_counts[k] += m->graph.counts[k];
  }
  return DIT_OK;
}

extern "C" dit_status dit_synchronize(dit_model* m, void* stream) {
  g_last_error[0] = 0;
  if (!m) return fail(DIT_ERR_INVALID_ARG, "model is NULL");
  CU_TRY(cudaSetDevice(m->device));
  CU_TRY(cudaStreamSynchronize(static_cast<cudaStream_t>(stream)));
  int h = 0;
  CU_TRY(cudaMemcpy(&h, m->d_err, sizeof(int), cudaMemcpyDeviceToHost));
  if (h) {
    CU_TRY(cudaMemset(m->d_err, 0, sizeof(int)));
    if (h >= DIT_BOUNDS_SITE_MIN && h <= DIT_BOUNDS_SITE_MAX)
      return fail(DIT_ERR_CUDA, "device bounds check failed (site %d, debug build); outputs are invalid", h);
    return fail(DIT_ERR_TIMEOUT, "a kernel abandoned a bounded wait (site %d); outputs are invalid", h);
  }
  return DIT_OK;
}

extern "C" dit_status dit_debug_stall(dit_model* m, void* stream) {
  g_last_error[0] = 0;
  if (!m) return fail(DIT_ERR_INVALID_ARG, "model is NULL");
  CU_TRY(cudaSetDevice(m->device));
  K_TRY(debug_stall(m->d_err, DIT_DEBUG_STALL_SITE, static_cast<cudaStream_t>(stream)));
  return DIT_OK;
}

extern "C" dit_status dit_profile_start(dit_model* m, int timing) {
  g_last_error[0] = 0;
  if (!m) return fail(DIT_ERR_INVALID_ARG, "model is NULL");
  for (int k = 0; k < DIT_KERNEL_KINDS; ++k) m->prof_counts[k] = 0;
  m->prof_rec.clear();
  m->prof_next = 0;
  m->prof_timing = timing != 0;
  return DIT_OK;
}

extern "C" dit_status dit_profile_stop(dit_model* m, int64_t* counts, double* ms) {
  g_last_error[0] = 0;
  if (!m) return fail(DIT_ERR_INVALID_ARG, "model is NULL");
  CU_TRY(cudaSetDevice(m->device));
  CU_TRY(cudaDeviceSynchronize());
  double acc[DIT_KERNEL_KINDS] = {};
  for (const auto& r : m->prof_rec) {
    float t = 0.f;
    CU_TRY(cudaEventElapsedTime(&t, r.a, r.b));
    acc[r.kind] += t;
  }
  for (int k = 0; k < DIT_KERNEL_KINDS; ++k) {
    if (counts) counts[k] = m->prof_counts[k];
    if (ms) ms[k] = acc[k];
  }
  m->prof_timing = false;
  m->prof_rec.clear();
  m->prof_next = 0;
  return DIT_OK;
}
