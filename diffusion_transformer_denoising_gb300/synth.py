"""Seeded synthetic inputs for the denoiser stage: model configurations, the
parameter list and the random tensors fed to both the CUDA path and the CPU
oracle.

This module holds no arithmetic of the method itself: it only names shapes,
draws random numbers and rounds them to bf16 where a configuration asks for
bf16 weights.  Both sides receive the very same arrays from here.

Workload shapes follow the pages' workloads:
  * video: Wan2.1-T2V-1.3B-shaped DiT on an 81-frame 480x832 request, i.e. a
    16-channel latent of 21 x 60 x 104 cut into (1,2,2) patches = 32760
    tokens (SGLang-Diffusion "Disaggregated Diffusion Pipeline",
    Single-Machine Example);
  * image: the 7B DiT of GLM-Image denoising a 1024x1024 image in 30-50 steps
    (LMSYS blog "SGL-Diffusion full-stack optimisation of AR+DiT"), 16 x 128 x
    128 latent, 2x2 patches = 4096 tokens plus 512 condition tokens;
  * tiny: a 2-block model small enough for the plain oracle to run the whole
    loop in well under a second.
"""
from __future__ import annotations

import copy
import numpy as np

PREC_BF16 = 0
PREC_F32 = 1
PREC_FP8 = 2   # bf16 activations; the LayerNorm-fed GEMMs in e4m3
COND_CROSS = 0
COND_JOINT = 1

_BASE = dict(in_channels=16, patch=(1, 2, 2), freq_dim=256, ln_eps=1e-6,
             rope_theta=1e4, timestep_scale=1000.0, precision=PREC_BF16)

CONFIGS = {
    # 4 x 16 x 16 latent, 2x2 patches -> 64 tokens, hidden 128, 4 heads of 32.
    "tiny": dict(_BASE, in_channels=4, hidden=128, heads=4, head_dim=32,
                 mlp=512, depth=2, cond_dim=128, rope_axes=(0, 16, 16),
                 cond_mode=COND_CROSS, precision=PREC_F32,
                 latent=(1, 16, 16), cond_len=16, steps=4, shift=3.0,
                 guidance=5.0),
    # Wan2.1-1.3B-shaped video DiT.
    "video": dict(_BASE, hidden=1536, heads=12, head_dim=128, mlp=8960,
                  depth=30, cond_dim=1536, rope_axes=(44, 42, 42),
                  cond_mode=COND_CROSS, latent=(21, 60, 104), cond_len=512,
                  steps=50, shift=5.0, guidance=5.0),
    # 7B-class dual-stream image DiT, condition tokens attend jointly.
    "image": dict(_BASE, hidden=3072, heads=24, head_dim=128, mlp=12288,
                  depth=30, cond_dim=3072, rope_axes=(0, 64, 64),
                  cond_mode=COND_JOINT, latent=(1, 128, 128), cond_len=512,
                  steps=30, shift=3.0, guidance=4.0),
}


def config(name: str, **overrides) -> dict:
    """A copy of a named configuration with fields overridden."""
    c = copy.deepcopy(CONFIGS[name])
    c.update(overrides)
    c["patch"] = tuple(c["patch"])
    c["rope_axes"] = tuple(c["rope_axes"])
    c["latent"] = tuple(c["latent"])
    return c


def patch_dim(cfg: dict) -> int:
    pt, ph, pw = cfg["patch"]
    return cfg["in_channels"] * pt * ph * pw


def grid(cfg: dict, latent=None) -> tuple:
    """Token grid (T', H', W') of a latent of spatial shape (T, H, W)."""
    T, H, W = latent if latent is not None else cfg["latent"]
    pt, ph, pw = cfg["patch"]
    return (T // pt, H // ph, W // pw)


def param_specs(cfg: dict) -> list:
    """Ordered (name, shape) list of every parameter of the model.

    Linear weights are stored [out_features, in_features].  Each block holds a
    learned 6 x D table added to the shared timestep modulation (shift1,
    scale1, gate1, shift2, scale2, gate2).  Joint-mode blocks carry a second
    set of weights for the condition-token stream under the prefix "ctx.".
    """
    D, F, Dc, P = cfg["hidden"], cfg["mlp"], cfg["cond_dim"], patch_dim(cfg)
    fq = cfg["freq_dim"]
    s = [("patch_embed.weight", (D, P)), ("patch_embed.bias", (D,)),
         ("time_mlp.fc1.weight", (D, fq)), ("time_mlp.fc1.bias", (D,)),
         ("time_mlp.fc2.weight", (6 * D, D)), ("time_mlp.fc2.bias", (6 * D,))]
    for b in range(cfg["depth"]):
        p = f"blocks.{b}."
        streams = [""] if cfg["cond_mode"] == COND_CROSS else ["", "ctx."]
        for st in streams:
            s += [(p + st + "mod_table", (6, D)),
                  (p + st + "attn.qkv.weight", (3 * D, D)),
                  (p + st + "attn.qkv.bias", (3 * D,)),
                  (p + st + "attn.out.weight", (D, D)),
                  (p + st + "attn.out.bias", (D,))]
            if st == "" and cfg["cond_mode"] == COND_CROSS:
                s += [(p + "cross.q.weight", (D, D)), (p + "cross.q.bias", (D,)),
                      (p + "cross.kv.weight", (2 * D, Dc)),
                      (p + "cross.kv.bias", (2 * D,)),
                      (p + "cross.out.weight", (D, D)),
                      (p + "cross.out.bias", (D,))]
            s += [(p + st + "mlp.fc1.weight", (F, D)), (p + st + "mlp.fc1.bias", (F,)),
                  (p + st + "mlp.fc2.weight", (D, F)), (p + st + "mlp.fc2.bias", (D,))]
    s += [("head.mod_table", (2, D)), ("head.weight", (P, D)), ("head.bias", (P,))]
    return s


def round_bf16(a: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bf16 (ties to even); returns float32
    arrays whose values are exactly representable in bf16."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32)


def _rng(seed: int, index: int) -> np.random.Generator:
    return np.random.default_rng([int(seed), int(index)])


def make_weights(cfg: dict, seed: int = 0, std: float = 0.02,
                 blocks=None) -> dict:
    """Every parameter ~ N(0, std^2), float32, one generator per tensor
    (seed, index in the parameter list), so a subset can be drawn alone.

    blocks: optional iterable of block indices to draw (others are skipped;
    non-block tensors are always drawn).  With precision bf16 the values are
    rounded to bf16 (also for fp8 precision, whose weights are quantized
    from these values on the device), the precision both sides then read.
    """
    keep = None if blocks is None else {f"blocks.{b}." for b in blocks}
    out = {}
    for i, (name, shape) in enumerate(param_specs(cfg)):
        if keep is not None and name.startswith("blocks.") and \
                not any(name.startswith(k) for k in keep):
            continue
        w = _rng(seed, i).standard_normal(shape, dtype=np.float32) * np.float32(std)
        if cfg["precision"] in (PREC_BF16, PREC_FP8):
            w = round_bf16(w)
        out[name] = w
    return out


def make_latent(cfg: dict, batch: int = 1, seed: int = 1, latent=None) -> np.ndarray:
    """Initial noise latent [batch, C, T, H, W] ~ N(0, 1), float32."""
    T, H, W = latent if latent is not None else cfg["latent"]
    x = _rng(seed, 10**6).standard_normal((batch, cfg["in_channels"], T, H, W),
                                          dtype=np.float32)
    return x


def make_cond(cfg: dict, batch: int = 1, seed: int = 2, length=None) -> np.ndarray:
    """Condition tokens [batch, L, Dc] ~ N(0, 1), float32 (bf16-rounded when the
    configuration is bf16, since the GPU path reads them as bf16)."""
    L = length if length is not None else cfg["cond_len"]
    c = _rng(seed, 10**6 + 1).standard_normal((batch, L, cfg["cond_dim"]),
                                              dtype=np.float32)
    if cfg["precision"] in (PREC_BF16, PREC_FP8):
        c = round_bf16(c)
    return c


def make_normal(shape, seed: int, index: int = 0, std: float = 1.0) -> np.ndarray:
    """A generic N(0, std^2) float32 array for kernel-level tests."""
    return _rng(seed, 2 * 10**6 + index).standard_normal(shape, dtype=np.float32) * np.float32(std)


def make_weights_torch(cfg: dict, seed: int = 0, std: float = 0.02, device="cuda"):
    """Device-side generation of the same parameter list for throughput runs
    where drawing billions of values on the host would dominate set-up time.
    Values come from torch's generator of that device (not identical to
    make_weights), bf16 unless the configuration is fp32."""
    import torch
    dt = torch.float32 if cfg["precision"] == PREC_F32 else torch.bfloat16
    g = torch.Generator(device=device)
    out = {}
    for i, (name, shape) in enumerate(param_specs(cfg)):
        g.manual_seed(seed * 1000003 + i)
        t = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
        out[name] = (t * std).to(dt)
    return out
