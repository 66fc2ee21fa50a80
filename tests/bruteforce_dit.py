"""A second, deliberately naive restatement of one DiT block written with
pure-Python scalar loops (lists and the math module, no numpy), used only on
tiny inputs to pin the oracle.  It is written token by token and channel by
channel so that a transposed operand, a dropped term or a wrong index in the
vectorised oracle shows up as a mismatch.
"""
import math


def _lin(vec, w, b):
    """w given as a list of rows [out][in]."""
    return [sum(w[o][i] * vec[i] for i in range(len(vec))) + b[o] for o in range(len(w))]


def _ln(vec, eps):
    n = len(vec)
    mu = sum(vec) / n
    var = sum((a - mu) * (a - mu) for a in vec) / n
    return [(a - mu) / math.sqrt(var + eps) for a in vec]


def _gelu(a):
    return 0.5 * a * (1.0 + math.tanh(math.sqrt(2.0 / math.pi) * (a + 0.044715 * a * a * a)))


def _rot(vec, pos, axes, theta, heads):
    """Rotate each head's channel pairs.  Pair p of a head belongs to the axis
    whose section contains channel 2p; its index inside that section is j."""
    d = len(vec) // heads
    out = list(vec)
    for h in range(heads):
        start = 0
        for a, da in enumerate(axes):
            for j in range(da // 2):
                ang = pos[a] * theta ** (-2.0 * j / da)
                i0 = h * d + start + 2 * j
                x0, x1 = vec[i0], vec[i0 + 1]
                out[i0] = x0 * math.cos(ang) - x1 * math.sin(ang)
                out[i0 + 1] = x0 * math.sin(ang) + x1 * math.cos(ang)
            start += da
    return out


def _attn(qs, ks, vs, heads):
    d = len(qs[0]) // heads
    out = []
    for q in qs:
        row = [0.0] * (heads * d)
        for h in range(heads):
            w = [math.exp(sum(q[h * d + c] * k[h * d + c] for c in range(d)) / math.sqrt(d)) for k in ks]
            z = sum(w)
            for c in range(d):
                row[h * d + c] = sum(w[j] * vs[j][h * d + c] for j in range(len(ks))) / z
        out.append(row)
    return out


def _tolist(a):
    return a.tolist() if hasattr(a, "tolist") else a


def _mods(m, table, D):
    m, table = _tolist(m), _tolist(table)
    return [[m[i * D + c] + table[i][c] for c in range(D)] for i in range(6)]


def _qkv_proj(xs, mod, W, pre, cfg):
    D = cfg["hidden"]
    w, b = _tolist(W[pre + "attn.qkv.weight"]), _tolist(W[pre + "attn.qkv.bias"])
    qs, ks, vs = [], [], []
    for x in xs:
        n = _ln(x, cfg["ln_eps"])
        h = [n[c] * (1.0 + mod[1][c]) + mod[0][c] for c in range(D)]
        y = _lin(h, w, b)
        qs.append(y[:D]); ks.append(y[D:2 * D]); vs.append(y[2 * D:])
    return qs, ks, vs


def _mlp_half(x, mod, W, pre, cfg):
    D = cfg["hidden"]
    n = _ln(x, cfg["ln_eps"])
    h = [n[c] * (1.0 + mod[4][c]) + mod[3][c] for c in range(D)]
    f = [_gelu(a) for a in _lin(h, _tolist(W[pre + "mlp.fc1.weight"]), _tolist(W[pre + "mlp.fc1.bias"]))]
    y = _lin(f, _tolist(W[pre + "mlp.fc2.weight"]), _tolist(W[pre + "mlp.fc2.bias"]))
    return [x[c] + mod[5][c] * y[c] for c in range(D)]


def block_cross(x, m, ctx, W, b, cfg, positions):
    """x: list of N token lists; ctx: list of L lists; positions: list of (t,h,w)."""
    D, H = cfg["hidden"], cfg["heads"]
    pre = f"blocks.{b}."
    x, ctx = _tolist(x), _tolist(ctx)
    mod = _mods(m, W[pre + "mod_table"], D)
    qs, ks, vs = _qkv_proj(x, mod, W, pre, cfg)
    qs = [_rot(q, positions[i], cfg["rope_axes"], cfg["rope_theta"], H) for i, q in enumerate(qs)]
    ks = [_rot(k, positions[i], cfg["rope_axes"], cfg["rope_theta"], H) for i, k in enumerate(ks)]
    a = _attn(qs, ks, vs, H)
    wo, bo = _tolist(W[pre + "attn.out.weight"]), _tolist(W[pre + "attn.out.bias"])
    x = [[x[i][c] + mod[2][c] * o for c, o in enumerate(_lin(a[i], wo, bo))] for i in range(len(x))]
    wkv, bkv = _tolist(W[pre + "cross.kv.weight"]), _tolist(W[pre + "cross.kv.bias"])
    kc = [_lin(t, wkv[:D], bkv[:D]) for t in ctx]
    vc = [_lin(t, wkv[D:], bkv[D:]) for t in ctx]
    wq, bq = _tolist(W[pre + "cross.q.weight"]), _tolist(W[pre + "cross.q.bias"])
    qc = [_lin(_ln(t, cfg["ln_eps"]), wq, bq) for t in x]
    ac = _attn(qc, kc, vc, H)
    wco, bco = _tolist(W[pre + "cross.out.weight"]), _tolist(W[pre + "cross.out.bias"])
    x = [[x[i][c] + o for c, o in enumerate(_lin(ac[i], wco, bco))] for i in range(len(x))]
    return [_mlp_half(t, mod, W, pre, cfg) for t in x]


def block_joint(x, xc, m, W, b, cfg, positions):
    """Dual-stream block; joint order [condition; image]; condition tokens unrotated."""
    D, H = cfg["hidden"], cfg["heads"]
    pre = f"blocks.{b}."
    x, xc = _tolist(x), _tolist(xc)
    mi = _mods(m, W[pre + "mod_table"], D)
    mc = _mods(m, W[pre + "ctx.mod_table"], D)
    qi, ki, vi = _qkv_proj(x, mi, W, pre, cfg)
    qc, kc, vc = _qkv_proj(xc, mc, W, pre + "ctx.", cfg)
    qi = [_rot(q, positions[i], cfg["rope_axes"], cfg["rope_theta"], H) for i, q in enumerate(qi)]
    ki = [_rot(k, positions[i], cfg["rope_axes"], cfg["rope_theta"], H) for i, k in enumerate(ki)]
    a = _attn(qc + qi, kc + ki, vc + vi, H)
    L = len(xc)
    outs = []
    for toks, mod, pre2, rows in ((xc, mc, pre + "ctx.", range(L)), (x, mi, pre, range(L, L + len(x)))):
        wo, bo = _tolist(W[pre2 + "attn.out.weight"]), _tolist(W[pre2 + "attn.out.bias"])
        res = []
        for t, r in zip(toks, rows):
            o = _lin(a[r], wo, bo)
            y = [t[c] + mod[2][c] * o[c] for c in range(D)]
            res.append(_mlp_half(y, mod, W, pre2, cfg))
        outs.append(res)
    return outs[1], outs[0]


def final_layer(x, m, W, cfg):
    D = cfg["hidden"]
    m, tab = _tolist(m), _tolist(W["head.mod_table"])
    sh = [m[c] + tab[0][c] for c in range(D)]
    sc = [m[D + c] + tab[1][c] for c in range(D)]
    w, b = _tolist(W["head.weight"]), _tolist(W["head.bias"])
    out = []
    for t in _tolist(x):
        n = _ln(t, cfg["ln_eps"])
        out.append(_lin([n[c] * (1.0 + sc[c]) + sh[c] for c in range(D)], w, b))
    return out


def timestep_modulation(t, W, cfg):
    half = cfg["freq_dim"] // 2
    e = [math.cos(t * 10000.0 ** (-k / half)) for k in range(half)] + \
        [math.sin(t * 10000.0 ** (-k / half)) for k in range(half)]
    h = _lin(e, _tolist(W["time_mlp.fc1.weight"]), _tolist(W["time_mlp.fc1.bias"]))
    h = [a / (1.0 + math.exp(-a)) for a in h]
    return _lin(h, _tolist(W["time_mlp.fc2.weight"]), _tolist(W["time_mlp.fc2.bias"]))


def dit_forward(lat, t, ctx, W, cfg):
    """Velocity for one latent [C][T][H][W] (nested lists or an array) at
    network timestep t: patch vectors gathered by index arithmetic, the
    blocks above, the head, and the velocity scattered back by index."""
    C = len(lat)
    T, H, Wd = len(lat[0]), len(lat[0][0]), len(lat[0][0][0])
    pt, ph, pw = cfg["patch"]
    gt, gh, gw = T // pt, H // ph, Wd // pw
    D = cfg["hidden"]
    w_pe, b_pe = _tolist(W["patch_embed.weight"]), _tolist(W["patch_embed.bias"])
    positions, toks = [], []
    for it in range(gt):
        for ih in range(gh):
            for iw in range(gw):
                vec = [lat[c][it * pt + a][ih * ph + b][iw * pw + e]
                       for c in range(C) for a in range(pt) for b in range(ph) for e in range(pw)]
                toks.append(_lin(vec, w_pe, b_pe))
                positions.append((it, ih, iw))
    m = timestep_modulation(t, W, cfg)
    if cfg["cond_mode"] == 0:
        for blk in range(cfg["depth"]):
            toks = block_cross(toks, m, ctx, W, blk, cfg, positions)
    else:
        xc = [list(r) for r in _tolist(ctx)]
        for blk in range(cfg["depth"]):
            toks, xc = block_joint(toks, xc, m, W, blk, cfg, positions)
    vt = final_layer(toks, m, W, cfg)
    v = [[[[0.0] * Wd for _ in range(H)] for _ in range(T)] for _ in range(C)]
    for n, (it, ih, iw) in enumerate(positions):
        k = 0
        for c in range(C):
            for a in range(pt):
                for b in range(ph):
                    for e in range(pw):
                        v[c][it * pt + a][ih * ph + b][iw * pw + e] = vt[n][k]
                        k += 1
    assert len(vt[0]) == k and len(vt[0]) == C * pt * ph * pw and D == len(toks[0])
    return v


def denoise_loop(lat, cond, uncond, W, cfg, sigmas, timesteps, g):
    """Flow-Euler loop with guidance, the timesteps given explicitly (so that
    the sigma -> timestep conversion is not restated here): per step the
    conditional and unconditional velocities, v = vu + g (vc - vu), then
    x += (sigma_{i+1} - sigma_i) v element by element."""
    x = [[[list(map(float, row)) for row in plane] for plane in ch] for ch in _tolist(lat)]
    for i in range(len(sigmas) - 1):
        vc = dit_forward(x, timesteps[i], cond, W, cfg)
        vu = dit_forward(x, timesteps[i], uncond, W, cfg)
        ds = sigmas[i + 1] - sigmas[i]
        for c in range(len(x)):
            for a in range(len(x[c])):
                for b in range(len(x[c][a])):
                    for e in range(len(x[c][a][b])):
                        u = vu[c][a][b][e]
                        x[c][a][b][e] += ds * (u + g * (vc[c][a][b][e] - u))
    return x
