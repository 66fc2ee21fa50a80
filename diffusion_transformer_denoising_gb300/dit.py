"""ctypes binding of libdit.so: the same entry points as include/dit.h, with
argument marshalling only (every step of the denoiser runs in the library's
CUDA kernels).  Tensors are passed by pointer: torch CUDA tensors (or any
object with data_ptr()) for device buffers, numpy arrays for host buffers.

The library is loaded on first use.  If it has not been built the binding
raises instead of falling back to anything else.
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
# DIT_LIB selects another build of the same library (the debug build with
# device-side bounds checks, libdit_debug.so); default: the release build.
LIB_PATH = os.environ.get("DIT_LIB") or os.path.join(_PKG, "libdit.so")

DIT_OK, DIT_ERR_INVALID_ARG, DIT_ERR_SHAPE, DIT_ERR_NOT_LOADED, DIT_ERR_OOM, DIT_ERR_CUDA, DIT_ERR_TIMEOUT = range(7)
PREC_BF16, PREC_F32, PREC_FP8 = 0, 1, 2
COND_CROSS, COND_JOINT = 0, 1
DTYPE_F32, DTYPE_BF16 = 0, 1
LOOP_PARTIAL_SCHEDULE = 1
LOOP_CUDA_GRAPH = 2

# every symbol include/dit.h declares
EXPORTS = ["dit_create", "dit_load_weights", "dit_num_params", "dit_param_info", "dit_timestep_modulation",
           "dit_patch_embed", "dit_block_forward", "dit_final_layer", "cfg_combine", "flow_euler_step",
           "dit_denoise_loop", "dit_synchronize", "dit_device_bytes", "dit_destroy", "dit_status_string",
           "dit_last_error", "dit_debug_fail_alloc_after", "dit_debug_gemm_cta_pairs", "dit_debug_stall", "dit_profile_start", "dit_profile_stop",
           "dit_timestep_modulation_noalloc"]
NOALLOC_MAX_BATCH, NOALLOC_MAX_HIDDEN = 64, 262144

KERNEL_KINDS = ["gemm_qkv", "gemm_out", "gemm_cross_q", "gemm_cross_kv", "gemm_ffn1", "gemm_ffn2", "gemm_embed",
                "attn_self", "attn_cross", "ln", "small", "cfg_euler"]


class DitConfig(C.Structure):
    _fields_ = [("in_channels", C.c_int32), ("patch", C.c_int32 * 3), ("hidden", C.c_int32),
                ("heads", C.c_int32), ("head_dim", C.c_int32), ("mlp", C.c_int32), ("depth", C.c_int32),
                ("cond_dim", C.c_int32), ("freq_dim", C.c_int32), ("rope_axes", C.c_int32 * 3),
                ("cond_mode", C.c_int32), ("precision", C.c_int32), ("ln_eps", C.c_float),
                ("rope_theta", C.c_float), ("timestep_scale", C.c_float)]


class DitTensor(C.Structure):
    _fields_ = [("name", C.c_char_p), ("ndim", C.c_int32), ("shape", C.c_int64 * 4), ("dtype", C.c_int32),
                ("data", C.c_void_p)]


class DitError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"[{status}] {msg}")
        self.status = status


_lib = None


def lib():
    """The loaded library (raises if libdit.so has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it first (python -m "
                           "diffusion_transformer_denoising_gb300.build or __graft_entry__.build())")
    L = C.CDLL(LIB_PATH)
    vp, i32, i64, f32 = C.c_void_p, C.c_int32, C.c_int64, C.c_float
    sig = {
        "dit_create": ([C.POINTER(DitConfig), C.c_int, C.POINTER(vp)], C.c_int),
        "dit_load_weights": ([vp, C.POINTER(DitTensor), C.c_int], C.c_int),
        "dit_num_params": ([C.POINTER(DitConfig)], C.c_int),
        "dit_param_info": ([C.POINTER(DitConfig), C.c_int, C.c_char_p, C.c_int, C.POINTER(i32),
                            C.POINTER(i64)], C.c_int),
        "dit_timestep_modulation": ([vp, C.POINTER(f32), C.c_int, vp, vp], C.c_int),
        "dit_timestep_modulation_noalloc": ([vp, C.POINTER(f32), C.c_int, vp, vp], C.c_int),
        "dit_patch_embed": ([vp, vp, C.c_int, C.POINTER(i32), vp, vp], C.c_int),
        "dit_block_forward": ([vp, C.c_int, vp, vp, vp, vp, C.c_int, C.POINTER(i32), C.c_int, vp], C.c_int),
        "dit_final_layer": ([vp, vp, vp, C.c_int, C.POINTER(i32), vp, vp], C.c_int),
        "cfg_combine": ([vp, vp, f32, vp, i64, vp], C.c_int),
        "flow_euler_step": ([vp, vp, f32, f32, i64, vp], C.c_int),
        "dit_denoise_loop": ([vp, vp, C.c_int, C.POINTER(i32), vp, vp, C.c_int, C.POINTER(f32), C.c_int, f32,
                              C.c_uint32, vp], C.c_int),
        "dit_synchronize": ([vp, vp], C.c_int),
        "dit_device_bytes": ([vp], i64),
        "dit_destroy": ([vp], None),
        "dit_status_string": ([C.c_int], C.c_char_p),
        "dit_last_error": ([], C.c_char_p),
        "dit_debug_fail_alloc_after": ([C.c_int], None),
        "dit_debug_gemm_cta_pairs": ([C.c_int], None),
        "dit_debug_stall": ([vp, vp], C.c_int),
        "dit_profile_start": ([vp, C.c_int], C.c_int),
        "dit_profile_stop": ([vp, C.POINTER(i64), C.POINTER(C.c_double)], C.c_int),
    }
    for name, (args, res) in sig.items():
        f = getattr(L, name)
        f.argtypes = args
        f.restype = res
    _lib = L
    return L


def _check(status: int):
    if status != DIT_OK:
        raise DitError(status, lib().dit_last_error().decode())


def _ptr(t):
    if t is None:
        return None
    if hasattr(t, "data_ptr"):
        return C.c_void_p(t.data_ptr())
    if isinstance(t, np.ndarray):
        return C.c_void_p(t.ctypes.data)
    if isinstance(t, int):
        return C.c_void_p(t)
    raise TypeError(f"cannot take a pointer of {type(t)}")


def _stream(stream):
    if stream is None:
        try:
            import torch
            if torch.cuda.is_available():
                return C.c_void_p(torch.cuda.current_stream().cuda_stream)
        except Exception:
            pass
        return None
    if hasattr(stream, "cuda_stream"):
        return C.c_void_p(stream.cuda_stream)
    return C.c_void_p(int(stream))


def make_config(cfg: dict) -> DitConfig:
    c = DitConfig()
    c.in_channels = cfg["in_channels"]
    c.patch[:] = list(cfg["patch"])
    for k in ("hidden", "heads", "head_dim", "mlp", "depth", "cond_dim", "freq_dim", "cond_mode", "precision"):
        setattr(c, k, int(cfg[k]))
    c.rope_axes[:] = list(cfg["rope_axes"])
    c.ln_eps, c.rope_theta, c.timestep_scale = cfg["ln_eps"], cfg["rope_theta"], cfg["timestep_scale"]
    return c


def dit_num_params(cfg: dict) -> int:
    return lib().dit_num_params(C.byref(make_config(cfg)))


def dit_param_info(cfg: dict, i: int):
    buf = C.create_string_buffer(256)
    nd = C.c_int32()
    shape = (C.c_int64 * 4)()
    _check(lib().dit_param_info(C.byref(make_config(cfg)), i, buf, 256, C.byref(nd), shape))
    return buf.value.decode(), tuple(shape[: nd.value])


def cfg_combine(vc, vu, g: float, v, n: int, stream=None):
    _check(lib().cfg_combine(_ptr(vc), _ptr(vu), g, _ptr(v), n, _stream(stream)))


def flow_euler_step(x, v, sigma: float, sigma_next: float, n: int, stream=None):
    _check(lib().flow_euler_step(_ptr(x), _ptr(v), sigma, sigma_next, n, _stream(stream)))


def dit_debug_fail_alloc_after(n: int):
    lib().dit_debug_fail_alloc_after(n)


def dit_debug_gemm_cta_pairs(mode: int):
    """0: GEMMs never on CTA pairs, 1 (default): when the main loop has >= 16
    K blocks, 2: always (widths that are multiples of 256)."""
    lib().dit_debug_gemm_cta_pairs(int(mode))


class DiT:
    """One dit_model: create, load weights, run pieces or the whole loop."""

    def __init__(self, cfg: dict, device: int = 0):
        self.cfg = dict(cfg)
        self._cfg = make_config(cfg)
        h = C.c_void_p()
        _check(lib().dit_create(C.byref(self._cfg), device, C.byref(h)))
        self.h = h

    def close(self):
        if getattr(self, "h", None):
            lib().dit_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def device_bytes(self) -> int:
        return lib().dit_device_bytes(self.h)

    def load_weights(self, weights: dict, chunk: int = 64):
        """weights: name -> numpy float32 array, or torch tensor (float32 or
        bfloat16, host or device)."""
        keep, items = [], list(weights.items())
        for s in range(0, len(items), chunk):
            arr = (DitTensor * len(items[s:s + chunk]))()
            for j, (name, w) in enumerate(items[s:s + chunk]):
                t = arr[j]
                t.name = name.encode()
                keep.append(t.name)
                if isinstance(w, np.ndarray):
                    w = np.ascontiguousarray(w, dtype=np.float32)
                    keep.append(w)
                    t.dtype = DTYPE_F32
                else:
                    import torch
                    w = w.contiguous()
                    keep.append(w)
                    if w.dtype == torch.bfloat16:
                        t.dtype = DTYPE_BF16
                    elif w.dtype == torch.float32:
                        t.dtype = DTYPE_F32
                    else:
                        raise TypeError(f"{name}: unsupported dtype {w.dtype}")
                t.ndim = len(w.shape)
                for d in range(4):
                    t.shape[d] = w.shape[d] if d < len(w.shape) else 1
                t.data = _ptr(w).value
            _check(lib().dit_load_weights(self.h, arr, len(arr)))

    def dit_timestep_modulation(self, t_host, mod, stream=None):
        t = np.ascontiguousarray(t_host, dtype=np.float32)
        _check(lib().dit_timestep_modulation(self.h, t.ctypes.data_as(C.POINTER(C.c_float)), len(t), _ptr(mod),
                                             _stream(stream)))

    def dit_timestep_modulation_noalloc(self, t_host, mod, stream=None):
        """dit_timestep_modulation without any device allocation (fixed
        library scratch; see include/dit.h for the limits)."""
        t = np.ascontiguousarray(t_host, dtype=np.float32)
        _check(lib().dit_timestep_modulation_noalloc(self.h, t.ctypes.data_as(C.POINTER(C.c_float)), len(t),
                                                     _ptr(mod), _stream(stream)))

    def dit_patch_embed(self, latents, batch: int, thw, x, stream=None):
        a = (C.c_int32 * 3)(*thw)
        _check(lib().dit_patch_embed(self.h, _ptr(latents), batch, a, _ptr(x), _stream(stream)))

    def dit_block_forward(self, block: int, x, xc, mod, cond, batch: int, grid, cond_len: int, stream=None):
        g = (C.c_int32 * 3)(*grid)
        _check(lib().dit_block_forward(self.h, block, _ptr(x), _ptr(xc), _ptr(mod), _ptr(cond), batch, g,
                                       cond_len, _stream(stream)))

    def dit_final_layer(self, x, mod, batch: int, thw, v, stream=None):
        a = (C.c_int32 * 3)(*thw)
        _check(lib().dit_final_layer(self.h, _ptr(x), _ptr(mod), batch, a, _ptr(v), _stream(stream)))

    def dit_denoise_loop(self, latents, batch: int, thw, cond, uncond, cond_len: int, sigmas, guidance: float,
                         flags: int = 0, stream=None):
        a = (C.c_int32 * 3)(*thw)
        sg = np.ascontiguousarray(sigmas, dtype=np.float32)
        _check(lib().dit_denoise_loop(self.h, _ptr(latents), batch, a, _ptr(cond), _ptr(uncond), cond_len,
                                      sg.ctypes.data_as(C.POINTER(C.c_float)), len(sg) - 1, guidance, flags,
                                      _stream(stream)))

    def dit_profile_start(self, timing: bool = True):
        _check(lib().dit_profile_start(self.h, 1 if timing else 0))

    def dit_profile_stop(self):
        """{kind: (launches, total device ms)} since dit_profile_start."""
        n = len(KERNEL_KINDS)
        counts, ms = (C.c_int64 * n)(), (C.c_double * n)()
        _check(lib().dit_profile_stop(self.h, counts, ms))
        return {k: (counts[i], ms[i]) for i, k in enumerate(KERNEL_KINDS)}

    def dit_synchronize(self, stream=None):
        _check(lib().dit_synchronize(self.h, _stream(stream)))

    def dit_debug_stall(self, stream=None):
        """Test hook: a device wait that runs out (see include/dit.h)."""
        _check(lib().dit_debug_stall(self.h, _stream(stream)))
