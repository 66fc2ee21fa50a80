"""CPU oracle for the denoiser stage: a plain, slow, float64 restatement of
what one denoising loop computes.  TEST INFRASTRUCTURE ONLY: the product
path never imports it.

Only tests/, __graft_entry__.smoke() and bench.py's cpu_baseline leg may use
this module.  It shares no code with the CUDA path and imports nothing from
it: every function takes plain numpy arrays and returns numpy arrays.

What the pages fix, and where:
  * the denoiser role: the network's forward passes repeated over the step
    loop, with the sampler advancing the latent between them
    (SGLang-Diffusion "Disaggregated Diffusion Pipeline", Quick Start, role
    table);
  * its inputs: latents, timesteps in the exact order, sigmas, positive and
    (with CFG) negative prompt embeddings, number of steps, raw latent shape
    (SGLang-Diffusion "Support New Diffusion Models", section 4 "Last-Resort
    Before-Denoising Stage", table of fields required by DenoisingStage);
  * the DiT forward kwargs hidden_states / encoder_hidden_states / timestep,
    run once with the positive and once with the negative embeddings for
    classifier-free guidance (same page, section 2 "Pipeline Config");
  * flow prediction with a flow shift and a flow denoiser (stable-diffusion.cpp
    "Model Configuration Conventions", "Sampling And Geometry");
  * rotary position embeddings and latent packing as things a port must match
    (SGLang-Diffusion "Support New Diffusion Models", "Verify the Port").
The block equations themselves are not on the pages; each reading taken where
they are silent is marked [R1]..[R14] at the function that applies it.

Arrays are float64 unless a caller passes another dtype.  Shapes: a token
sequence is [N, D] for one batch element; batch loops are explicit.
"""
from __future__ import annotations

import math
import numpy as np

F64 = np.float64


# --------------------------------------------------------------------------
# schedule (stable-diffusion.cpp "Sampling And Geometry": flow prediction with
# a default flow shift; SGLang-Diffusion "Verify the Port": timestep order and
# sigma values must match)
# --------------------------------------------------------------------------
def sigma_schedule(n_steps: int) -> np.ndarray:
    """[R1] n+1 sigmas going linearly from 1 to exactly 0."""
    return np.array([1.0 - i / n_steps for i in range(n_steps + 1)], dtype=F64)


def shift_sigma(sigma, shift: float):
    """[R1] flow shift: sigma' = s*sigma / (1 + (s-1)*sigma)."""
    sigma = np.asarray(sigma, dtype=F64)
    return shift * sigma / (1.0 + (shift - 1.0) * sigma)


def timesteps_from_sigmas(sigmas, scale: float = 1000.0) -> np.ndarray:
    """[R2] the network's timestep is t = 1000 * sigma'."""
    return np.asarray(sigmas, dtype=F64) * scale


# --------------------------------------------------------------------------
# timestep embedding -> adaLN modulation
# --------------------------------------------------------------------------
def timestep_embedding(t: float, dim: int = 256, base: float = 10000.0) -> np.ndarray:
    """[R3] sinusoid: [cos(t f_k) for k<dim/2] ++ [sin(t f_k)], f_k = base^(-k/(dim/2))."""
    half = dim // 2
    f = np.array([base ** (-k / half) for k in range(half)], dtype=F64)
    a = float(t) * f
    return np.concatenate([np.cos(a), np.sin(a)])


def silu(x):
    return x / (1.0 + np.exp(-x))


def linear(x, w, b=None):
    """y = x W^T + b with W stored [out, in]."""
    y = np.asarray(x, F64) @ np.asarray(w, F64).T
    if b is not None:
        y = y + np.asarray(b, F64)
    return y


def timestep_modulation(t: float, W: dict, cfg: dict) -> np.ndarray:
    """[R4] m = fc2(SiLU(fc1(e(t)))) in R^{6D}, shared by every block."""
    e = timestep_embedding(t, cfg["freq_dim"])
    h = silu(linear(e, W["time_mlp.fc1.weight"], W["time_mlp.fc1.bias"]))
    return linear(h, W["time_mlp.fc2.weight"], W["time_mlp.fc2.bias"])


def block_modulation(m: np.ndarray, table: np.ndarray, D: int):
    """[R4] (shift1, scale1, gate1, shift2, scale2, gate2) = m + table, each D wide."""
    mm = np.asarray(m, F64).reshape(6, D) + np.asarray(table, F64)
    return [mm[i] for i in range(6)]


# --------------------------------------------------------------------------
# elementary layers
# --------------------------------------------------------------------------
def layer_norm(x, eps: float):
    """[R6] LayerNorm over the last axis, no affine, population variance."""
    x = np.asarray(x, F64)
    mu = x.mean(axis=-1, keepdims=True)
    var = ((x - mu) ** 2).mean(axis=-1, keepdims=True)
    return (x - mu) / np.sqrt(var + eps)


def modulate(h, shift, scale):
    """adaLN: h * (1 + scale) + shift."""
    return h * (1.0 + np.asarray(scale, F64)) + np.asarray(shift, F64)


def gelu_tanh(x):
    """[R10] GELU in its tanh form: 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3)))."""
    x = np.asarray(x, F64)
    return 0.5 * x * (1.0 + np.tanh(math.sqrt(2.0 / math.pi) * (x + 0.044715 * x ** 3)))


def softmax_rows(s):
    s = np.asarray(s, F64)
    s = s - s.max(axis=-1, keepdims=True)
    p = np.exp(s)
    return p / p.sum(axis=-1, keepdims=True)


def attention(q, k, v):
    """Bidirectional scaled dot-product attention for one head, no mask:
    softmax(q k^T / sqrt(d)) v.  q [Nq, d], k [Nk, d], v [Nk, d]."""
    d = q.shape[-1]
    return softmax_rows(np.asarray(q, F64) @ np.asarray(k, F64).T / math.sqrt(d)) @ np.asarray(v, F64)


def multihead_attention(q, k, v, heads: int):
    """q [Nq, H*d], k/v [Nk, H*d] -> [Nq, H*d], head h on columns h*d..h*d+d-1."""
    d = q.shape[-1] // heads
    out = np.empty((q.shape[0], heads * d), dtype=F64)
    for h in range(heads):
        sl = slice(h * d, (h + 1) * d)
        out[:, sl] = attention(q[:, sl], k[:, sl], v[:, sl])
    return out


# --------------------------------------------------------------------------
# rotary position embedding (SGLang-Diffusion "Verify the Port": rotary shape
# and style must match)
# --------------------------------------------------------------------------
def token_positions(grid) -> np.ndarray:
    """[R5] integer (t, h, w) grid index of every token, tokens in row-major
    (t, h, w) order.  Returns [N, 3]."""
    gt, gh, gw = grid
    pos = np.zeros((gt * gh * gw, 3), dtype=np.int64)
    n = 0
    for it in range(gt):
        for ih in range(gh):
            for iw in range(gw):
                pos[n] = (it, ih, iw)
                n += 1
    return pos


def rope_angles(pos: np.ndarray, axes, theta: float) -> np.ndarray:
    """[R7][R8] angle of every rotary pair: the head dimension is split into
    per-axis sections of axes[a] channels (t, then h, then w); pair j of axis a
    turns by pos_a * theta^(-2j / axes[a]).  Returns [N, sum(axes)/2]."""
    cols = []
    for a, da in enumerate(axes):
        for j in range(da // 2):
            cols.append(pos[:, a].astype(F64) * theta ** (-2.0 * j / da))
    if not cols:
        return np.zeros((pos.shape[0], 0), dtype=F64)
    return np.stack(cols, axis=1)


def apply_rope(x, angles):
    """[R7] rotate interleaved pairs (x[2p], x[2p+1]) of every head by angle p:
    (a, b) -> (a cos - b sin, a sin + b cos).  x [N, H*d], angles [N, d/2]."""
    x = np.asarray(x, F64)
    N, HD = x.shape
    npair = angles.shape[1]
    d = 2 * npair
    out = x.copy()
    c, s = np.cos(angles), np.sin(angles)
    for h in range(HD // d):
        a = x[:, h * d + 0: h * d + d: 2]
        b = x[:, h * d + 1: h * d + d: 2]
        out[:, h * d + 0: h * d + d: 2] = a * c - b * s
        out[:, h * d + 1: h * d + d: 2] = a * s + b * c
    return out


# --------------------------------------------------------------------------
# latent packing (SGLang-Diffusion "Support New Diffusion Models": latent
# packing and raw_latent_shape)
# --------------------------------------------------------------------------
def patchify(latent, patch):
    """[R5] latent [C, T, H, W] -> tokens [N, C*pt*ph*pw]; tokens in row-major
    (t, h, w) grid order, each patch vector ordered (c, pt, ph, pw)."""
    C, T, H, W = latent.shape
    pt, ph, pw = patch
    gt, gh, gw = T // pt, H // ph, W // pw
    x = np.asarray(latent, F64).reshape(C, gt, pt, gh, ph, gw, pw)
    x = x.transpose(1, 3, 5, 0, 2, 4, 6)  # gt gh gw C pt ph pw
    return x.reshape(gt * gh * gw, C * pt * ph * pw)


def unpatchify(tokens, patch, shape):
    """Inverse of patchify: tokens [N, C*pt*ph*pw] -> [C, T, H, W]."""
    C, T, H, W = shape
    pt, ph, pw = patch
    gt, gh, gw = T // pt, H // ph, W // pw
    x = np.asarray(tokens, F64).reshape(gt, gh, gw, C, pt, ph, pw)
    x = x.transpose(3, 0, 4, 1, 5, 2, 6)  # C gt pt gh ph gw pw
    return x.reshape(C, T, H, W)


def patch_embed(latent, W, cfg):
    return linear(patchify(latent, cfg["patch"]), W["patch_embed.weight"], W["patch_embed.bias"])


# --------------------------------------------------------------------------
# DiT blocks
# --------------------------------------------------------------------------
def _rope_for(cfg, grid):
    if sum(cfg["rope_axes"]) == 0:
        return None
    return rope_angles(token_positions(grid), cfg["rope_axes"], cfg["rope_theta"])


def block_cross(x, m, ctx, W, b: int, cfg: dict, grid, rows=None, angles=None):
    """One cross-attention DiT block for one batch element [R6]-[R9].

    x [N, D] residual stream, m [6D] timestep modulation, ctx [L, Dc]
    condition tokens.  rows: optional index array; when given, only those
    output rows are computed (keys and values still use every token) and the
    result is [len(rows), D].
    """
    D, H, eps = cfg["hidden"], cfg["heads"], cfg["ln_eps"]
    p = f"blocks.{b}."
    sh1, sc1, g1, sh2, sc2, g2 = block_modulation(m, W[p + "mod_table"], D)
    x = np.asarray(x, F64)
    if angles is None:
        angles = _rope_for(cfg, grid)
    sel = np.arange(x.shape[0]) if rows is None else np.asarray(rows)
    # self-attention half
    h = modulate(layer_norm(x, eps), sh1, sc1)
    wqkv, bqkv = W[p + "attn.qkv.weight"], W[p + "attn.qkv.bias"]
    k = linear(h, wqkv[D:2 * D], bqkv[D:2 * D])
    v = linear(h, wqkv[2 * D:], bqkv[2 * D:])
    q = linear(h[sel], wqkv[:D], bqkv[:D])
    if angles is not None:
        q = apply_rope(q, angles[sel])
        k = apply_rope(k, angles)
    a = multihead_attention(q, k, v, H)
    xs = x[sel] + g1 * linear(a, W[p + "attn.out.weight"], W[p + "attn.out.bias"])
    # cross-attention half [R9]: plain LN, no RoPE, ungated residual
    c = layer_norm(xs, eps)
    qc = linear(c, W[p + "cross.q.weight"], W[p + "cross.q.bias"])
    wkv, bkv = W[p + "cross.kv.weight"], W[p + "cross.kv.bias"]
    kc = linear(ctx, wkv[:D], bkv[:D])
    vc = linear(ctx, wkv[D:], bkv[D:])
    xs = xs + linear(multihead_attention(qc, kc, vc, H), W[p + "cross.out.weight"],
                     W[p + "cross.out.bias"])
    # MLP half
    h2 = modulate(layer_norm(xs, eps), sh2, sc2)
    f = gelu_tanh(linear(h2, W[p + "mlp.fc1.weight"], W[p + "mlp.fc1.bias"]))
    return xs + g2 * linear(f, W[p + "mlp.fc2.weight"], W[p + "mlp.fc2.bias"])


def block_joint(x, xc, m, W, b: int, cfg: dict, grid, rows=None, angles=None):
    """One dual-stream joint-attention DiT block for one batch element [R11].

    x [N, D] image-token stream, xc [L, D] condition-token stream.  The joint
    sequence is [condition; image]; condition tokens take no rotation, image
    tokens take the grid RoPE.  Returns (x', xc').  rows: optional indices
    into the JOINT sequence (0..L-1 condition, L.. image) whose outputs are
    computed; then returns an array [len(rows), D] in that order.
    """
    D, H, eps = cfg["hidden"], cfg["heads"], cfg["ln_eps"]
    p = f"blocks.{b}."
    x, xc = np.asarray(x, F64), np.asarray(xc, F64)
    L, N = xc.shape[0], x.shape[0]
    if angles is None:
        angles = _rope_for(cfg, grid)
    mods = {"": block_modulation(m, W[p + "mod_table"], D),
            "ctx.": block_modulation(m, W[p + "ctx.mod_table"], D)}
    qs, ks, vs = [], [], []
    for st, xx in (("ctx.", xc), ("", x)):
        sh1, sc1 = mods[st][0], mods[st][1]
        h = modulate(layer_norm(xx, eps), sh1, sc1)
        w, bb = W[p + st + "attn.qkv.weight"], W[p + st + "attn.qkv.bias"]
        q, k, v = (linear(h, w[i * D:(i + 1) * D], bb[i * D:(i + 1) * D]) for i in range(3))
        if st == "" and angles is not None:
            q, k = apply_rope(q, angles), apply_rope(k, angles)
        qs.append(q); ks.append(k); vs.append(v)
    q, k, v = (np.concatenate(z, axis=0) for z in (qs, ks, vs))
    sel = np.arange(L + N) if rows is None else np.asarray(rows)
    a = multihead_attention(q[sel], k, v, H)
    xj = np.concatenate([xc, x], axis=0)[sel]
    out = np.empty_like(xj)
    for st, mask in (("ctx.", sel < L), ("", sel >= L)):
        if not mask.any():
            continue
        _, _, g1, sh2, sc2, g2 = mods[st]
        y = xj[mask] + g1 * linear(a[mask], W[p + st + "attn.out.weight"],
                                   W[p + st + "attn.out.bias"])
        h2 = modulate(layer_norm(y, eps), sh2, sc2)
        f = gelu_tanh(linear(h2, W[p + st + "mlp.fc1.weight"], W[p + st + "mlp.fc1.bias"]))
        out[mask] = y + g2 * linear(f, W[p + st + "mlp.fc2.weight"], W[p + st + "mlp.fc2.bias"])
    if rows is not None:
        return out
    return out[L:], out[:L]


def final_layer(x, m, W, cfg):
    """Head: (shift, scale) = m[:2D] + head table; LN, modulate, linear to the
    patch vector.  x [N, D] -> [N, C*pt*ph*pw]."""
    D = cfg["hidden"]
    mm = np.asarray(m, F64)[:2 * D].reshape(2, D) + np.asarray(W["head.mod_table"], F64)
    h = modulate(layer_norm(x, cfg["ln_eps"]), mm[0], mm[1])
    return linear(h, W["head.weight"], W["head.bias"])


def dit_forward(latent, t: float, ctx, W, cfg):
    """Velocity prediction v(latent, t, ctx) for one batch element.
    latent [C, T, H, W], ctx [L, Dc] -> v [C, T, H, W]."""
    grid = tuple(s // p for s, p in zip(latent.shape[1:], cfg["patch"]))
    angles = _rope_for(cfg, grid)
    m = timestep_modulation(t, W, cfg)
    x = patch_embed(latent, W, cfg)
    if cfg["cond_mode"] == 0:
        for b in range(cfg["depth"]):
            x = block_cross(x, m, ctx, W, b, cfg, grid, angles=angles)
    else:
        xc = np.asarray(ctx, F64)  # [R11] condition tokens enter the stream as given
        for b in range(cfg["depth"]):
            x, xc = block_joint(x, xc, m, W, b, cfg, grid, angles=angles)
    return unpatchify(final_layer(x, m, W, cfg), cfg["patch"], latent.shape)


# --------------------------------------------------------------------------
# guidance and the flow Euler step
# --------------------------------------------------------------------------
def cfg_combine(v_cond, v_uncond, g: float):
    """Classifier-free guidance: v = v_u + g (v_c - v_u)."""
    v_cond, v_uncond = np.asarray(v_cond, F64), np.asarray(v_uncond, F64)
    return v_uncond + g * (v_cond - v_uncond)


def euler_step(x, v, sigma: float, sigma_next: float):
    """Flow-matching Euler update x + (sigma_next - sigma) v."""
    return np.asarray(x, F64) + (sigma_next - sigma) * np.asarray(v, F64)


def denoise_loop(latent, cond, uncond, W, cfg, sigmas, guidance: float):
    """The denoiser stage for one request: for each step, velocity for the
    positive and (with CFG) the negative condition, guidance, Euler update.
    latent [C, T, H, W]; cond/uncond [L, Dc] (uncond None => no CFG);
    sigmas: n+1 already-shifted values.  Returns the final latent."""
    x = np.asarray(latent, F64).copy()
    ts = timesteps_from_sigmas(sigmas, cfg["timestep_scale"])
    for i in range(len(sigmas) - 1):
        vc = dit_forward(x, ts[i], cond, W, cfg)
        v = vc if uncond is None else cfg_combine(vc, dit_forward(x, ts[i], uncond, W, cfg), guidance)
        x = euler_step(x, v, sigmas[i], sigmas[i + 1])
    return x
