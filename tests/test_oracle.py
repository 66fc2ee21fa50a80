"""Pins for the CPU oracle: each check ties it to something other than itself
(hand-worked fixtures, closed forms, invariants, library special functions,
or a naive scalar restatement on tiny inputs)."""
import inspect
import math
import os
import textwrap

import numpy as np
import pytest

from oracle import dit_oracle as O
from diffusion_transformer_denoising_gb300 import synth
from tests import bruteforce_dit as BF

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _rows(name):
    out = []
    with open(os.path.join(GOLD, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                out.append([float(v) for v in line.split()])
    return out


def small_cfg(mode=0, **kw):
    c = dict(in_channels=2, patch=(1, 2, 2), hidden=8, heads=2, head_dim=4, mlp=16,
             depth=1, cond_dim=6 if mode == 0 else 8, freq_dim=8, rope_axes=(0, 2, 2),
             cond_mode=mode, precision=1, ln_eps=1e-6, rope_theta=10.0,
             timestep_scale=1000.0)
    c.update(kw)
    return c


def rand_weights(cfg, seed=0, std=0.3):
    rng = np.random.default_rng(seed)
    return {n: rng.standard_normal(s) * std for n, s in synth.param_specs(cfg)}


# ---------------------------------------------------------------- schedule
def test_flow_shift_fixture():
    for s, sig, exp in _rows("flow_shift.txt"):
        assert abs(float(O.shift_sigma(sig, s)) - exp) < 1e-15


def test_schedule_endpoints_and_monotone():
    for n in (1, 4, 30, 50):
        for s in (1.0, 3.0, 5.0):
            sg = O.shift_sigma(O.sigma_schedule(n), s)
            assert len(sg) == n + 1 and sg[0] == 1.0 and sg[-1] == 0.0
            assert np.all(np.diff(sg) < 0)


def test_schedule_and_timesteps_fixture():
    # interior values, not only the endpoints: a curve through (0, 1) and
    # (n, 0) that is not linear in i fails here
    rows = np.array(_rows("schedule_n4.txt"))
    np.testing.assert_array_equal(O.sigma_schedule(4), rows[:, 1])
    np.testing.assert_allclose(O.shift_sigma(O.sigma_schedule(4), 3.0), rows[:, 2], rtol=0, atol=1e-15)
    np.testing.assert_allclose(O.timesteps_from_sigmas(rows[:, 2]), rows[:, 3], rtol=0, atol=1e-12)
    np.testing.assert_allclose(O.shift_sigma(O.sigma_schedule(4), 5.0), rows[:, 4], rtol=0, atol=1e-15)


def test_euler_constant_velocity_closed_form():
    # a constant field integrates exactly: the steps telescope to sigma_n - sigma_0 = -1
    rng = np.random.default_rng(3)
    x1, c = rng.standard_normal(100), rng.standard_normal(100)
    sg = O.shift_sigma(O.sigma_schedule(50), 5.0)
    x = x1.copy()
    for i in range(50):
        x = O.euler_step(x, c, sg[i], sg[i + 1])
    np.testing.assert_allclose(x, x1 - c, atol=1e-13)


def test_cfg_special_cases():
    rng = np.random.default_rng(4)
    vc, vu = rng.standard_normal(50), rng.standard_normal(50)
    # g=1 gives the conditional output and g=0 the unconditional one, up to
    # the rounding of vu + (vc - vu)
    np.testing.assert_allclose(O.cfg_combine(vc, vu, 1.0), vc, rtol=0, atol=1e-15)
    assert np.array_equal(O.cfg_combine(vc, vu, 0.0), vu)
    np.testing.assert_allclose(O.cfg_combine(vc, vu, 5.0), 5 * vc - 4 * vu, atol=1e-14)


# ---------------------------------------------------------------- layers
def test_timestep_embedding_fixture():
    for t, idx, val in _rows("timestep_embedding.txt"):
        assert abs(O.timestep_embedding(t, 256)[int(idx)] - val) < 1e-12


def test_layer_norm_moments_and_invariance():
    rng = np.random.default_rng(5)
    x = rng.standard_normal((7, 64)) * 3 + 2
    y = O.layer_norm(x, 1e-6)
    np.testing.assert_allclose(y.mean(-1), 0, atol=1e-12)
    np.testing.assert_allclose(y.var(-1), 1, atol=1e-5)
    np.testing.assert_allclose(O.layer_norm(4 * x + 9, 0.0), O.layer_norm(x, 0.0), atol=1e-12)


def test_gelu_tanh_against_erf_gelu():
    x = np.linspace(-8, 8, 2001)
    exact = np.array([0.5 * a * (1 + math.erf(a / math.sqrt(2))) for a in x])
    g = O.gelu_tanh(x)
    assert np.max(np.abs(g - exact)) < 1e-3     # known size of the tanh form's error
    assert O.gelu_tanh(np.array([0.0]))[0] == 0.0
    assert abs(O.gelu_tanh(np.array([30.0]))[0] - 30.0) < 1e-12
    assert abs(O.gelu_tanh(np.array([-30.0]))[0]) < 1e-12


# ---------------------------------------------------------------- attention
def test_softmax_rows_sum_to_one():
    rng = np.random.default_rng(6)
    p = O.softmax_rows(rng.standard_normal((9, 300)) * 10)
    np.testing.assert_allclose(p.sum(-1), 1.0, atol=1e-12)
    assert np.all(p >= 0)


def test_attention_against_scalar_loops():
    rng = np.random.default_rng(7)
    q, k, v = rng.standard_normal((5, 4)), rng.standard_normal((7, 4)), rng.standard_normal((7, 4))
    ref = np.zeros((5, 4))
    for i in range(5):
        w = [math.exp(sum(q[i, c] * k[j, c] for c in range(4)) / 2.0) for j in range(7)]
        for c in range(4):
            ref[i, c] = sum(w[j] * v[j, c] for j in range(7)) / sum(w)
    np.testing.assert_allclose(O.attention(q, k, v), ref, atol=1e-12)


def test_attention_special_cases():
    rng = np.random.default_rng(8)
    q, v = rng.standard_normal((6, 8)), rng.standard_normal((1, 8))
    k = rng.standard_normal((1, 8))
    np.testing.assert_allclose(O.attention(q, k, v), np.repeat(v, 6, 0), atol=1e-14)
    k = np.repeat(rng.standard_normal((1, 8)), 5, 0)   # equal keys -> mean of values
    v = rng.standard_normal((5, 8))
    np.testing.assert_allclose(O.attention(q, k, v), np.repeat(v.mean(0, keepdims=True), 6, 0), atol=1e-13)


# ---------------------------------------------------------------- rope
def test_rope_angles_fixture():
    ang = O.rope_angles(np.array([[1, 2, 3]]), (4, 2, 2), 100.0)[0]
    for p, a in _rows("rope_angles.txt"):
        assert abs(ang[int(p)] - a) < 1e-14


def test_rope_matches_complex_rotation():
    rng = np.random.default_rng(9)
    x = rng.standard_normal((10, 16))            # 2 heads of 8
    ang = rng.uniform(-5, 5, (10, 4))
    y = O.apply_rope(x, ang)
    for h in range(2):
        z = x[:, h * 8:(h + 1) * 8:2] + 1j * x[:, h * 8 + 1:(h + 1) * 8:2]
        z = z * np.exp(1j * ang)
        np.testing.assert_allclose(y[:, h * 8:(h + 1) * 8:2], z.real, atol=1e-13)
        np.testing.assert_allclose(y[:, h * 8 + 1:(h + 1) * 8:2], z.imag, atol=1e-13)


def test_rope_relative_position_and_norm():
    rng = np.random.default_rng(10)
    axes, th = (4, 6, 6), 1e4
    q, k = rng.standard_normal((1, 16)), rng.standard_normal((1, 16))
    def dot(pm, pn):
        a = O.apply_rope(q, O.rope_angles(np.array([pm]), axes, th))
        b = O.apply_rope(k, O.rope_angles(np.array([pn]), axes, th))
        return float((a * b).sum())
    assert abs(dot([3, 5, 7], [1, 2, 3]) - dot([12, 13, 14], [10, 10, 10])) < 1e-10
    r = O.apply_rope(q, O.rope_angles(np.array([[2, 9, 4]]), axes, th))
    assert abs(np.linalg.norm(r) - np.linalg.norm(q)) < 1e-12
    np.testing.assert_allclose(O.apply_rope(q, O.rope_angles(np.array([[0, 0, 0]]), axes, th)), q, atol=0)


# ---------------------------------------------------------------- packing
def test_patchify_fixture_and_roundtrip():
    lat = np.arange(32, dtype=np.float64).reshape(2, 1, 4, 4)
    tok = O.patchify(lat, (1, 2, 2))
    np.testing.assert_array_equal(tok, np.array(_rows("patchify_2x1x4x4.txt")))
    rng = np.random.default_rng(11)
    lat = rng.standard_normal((3, 4, 6, 10))
    np.testing.assert_array_equal(O.unpatchify(O.patchify(lat, (2, 2, 5)), (2, 2, 5), lat.shape), lat)


def test_token_positions_order():
    pos = O.token_positions((2, 3, 4))
    assert pos.shape == (24, 3)
    assert tuple(pos[0]) == (0, 0, 0) and tuple(pos[1]) == (0, 0, 1)
    assert tuple(pos[4]) == (0, 1, 0) and tuple(pos[12]) == (1, 0, 0) and tuple(pos[23]) == (1, 2, 3)


# ---------------------------------------------------------------- blocks
def test_cross_block_against_scalar_loops():
    cfg = small_cfg(0)
    W = rand_weights(cfg)
    rng = np.random.default_rng(12)
    grid = (1, 2, 3)
    x, ctx, m = rng.standard_normal((6, 8)), rng.standard_normal((3, 6)), rng.standard_normal(48) * 0.5
    pos = [tuple(p) for p in O.token_positions(grid)]
    ref = np.array(BF.block_cross(x, m, ctx, W, 0, cfg, pos))
    np.testing.assert_allclose(O.block_cross(x, m, ctx, W, 0, cfg, grid), ref, atol=1e-11)


def test_joint_block_against_scalar_loops():
    cfg = small_cfg(1)
    W = rand_weights(cfg)
    rng = np.random.default_rng(13)
    grid = (1, 2, 2)
    x, xc, m = rng.standard_normal((4, 8)), rng.standard_normal((3, 8)), rng.standard_normal(48) * 0.5
    pos = [tuple(p) for p in O.token_positions(grid)]
    rx, rc = BF.block_joint(x, xc, m, W, 0, cfg, pos)
    ox, oc = O.block_joint(x, xc, m, W, 0, cfg, grid)
    np.testing.assert_allclose(ox, np.array(rx), atol=1e-11)
    np.testing.assert_allclose(oc, np.array(rc), atol=1e-11)


def test_head_and_timestep_against_scalar_loops():
    cfg = small_cfg(0)
    W = rand_weights(cfg)
    rng = np.random.default_rng(14)
    x, m = rng.standard_normal((5, 8)), rng.standard_normal(48)
    np.testing.assert_allclose(O.final_layer(x, m, W, cfg), np.array(BF.final_layer(x, m, W, cfg)), atol=1e-12)
    np.testing.assert_allclose(O.timestep_modulation(321.5, W, cfg),
                               np.array(BF.timestep_modulation(321.5, W, cfg)), atol=1e-12)


def test_block_row_subset_matches_full():
    for mode in (0, 1):
        cfg = small_cfg(mode)
        W = rand_weights(cfg, seed=1)
        rng = np.random.default_rng(15)
        grid = (1, 2, 4)
        x, m = rng.standard_normal((8, 8)), rng.standard_normal(48)
        ctx = rng.standard_normal((3, cfg["cond_dim"]))
        if mode == 0:
            full = O.block_cross(x, m, ctx, W, 0, cfg, grid)
            np.testing.assert_allclose(O.block_cross(x, m, ctx, W, 0, cfg, grid, rows=[7, 0, 3]),
                                       full[[7, 0, 3]], atol=1e-13)
        else:
            fx, fc = O.block_joint(x, ctx, m, W, 0, cfg, grid)
            sub = O.block_joint(x, ctx, m, W, 0, cfg, grid, rows=[1, 3, 10])
            np.testing.assert_allclose(sub, np.stack([fc[1], fx[0], fx[7]]), atol=1e-13)


def test_block_identity_when_branches_closed():
    cfg = small_cfg(0)
    W = rand_weights(cfg, seed=2)
    W["blocks.0.mod_table"][[2, 5]] = 0.0          # gates 0 (with m = 0 below)
    W["blocks.0.cross.out.weight"][:] = 0.0
    W["blocks.0.cross.out.bias"][:] = 0.0
    rng = np.random.default_rng(16)
    x, ctx = rng.standard_normal((6, 8)), rng.standard_normal((3, 6))
    np.testing.assert_array_equal(O.block_cross(x, np.zeros(48), ctx, W, 0, cfg, (1, 2, 3)), x)


def test_block_token_permutation_equivariance_without_rope():
    for mode in (0, 1):
        cfg = small_cfg(mode, rope_axes=(0, 0, 0))
        W = rand_weights(cfg, seed=3)
        rng = np.random.default_rng(17)
        x, m = rng.standard_normal((8, 8)), rng.standard_normal(48)
        ctx = rng.standard_normal((3, cfg["cond_dim"]))
        perm = rng.permutation(8)
        if mode == 0:
            a = O.block_cross(x, m, ctx, W, 0, cfg, (1, 2, 4))
            b = O.block_cross(x[perm], m, ctx, W, 0, cfg, (1, 2, 4))
        else:
            a, _ = O.block_joint(x, ctx, m, W, 0, cfg, (1, 2, 4))
            b, _ = O.block_joint(x[perm], ctx, m, W, 0, cfg, (1, 2, 4))
        np.testing.assert_allclose(b, a[perm], atol=1e-12)


def test_loop_with_constant_velocity_head():
    # head weight 0 => v is the head bias broadcast over tokens: the loop must
    # land on x1 - v whatever the guidance and the rest of the network do.
    cfg = small_cfg(0, depth=2)
    W = rand_weights(cfg, seed=4)
    W["head.weight"][:] = 0.0
    rng = np.random.default_rng(18)
    lat = rng.standard_normal((2, 1, 4, 4))
    ctx = rng.standard_normal((3, 6))
    sg = O.shift_sigma(O.sigma_schedule(4), 3.0)
    out = O.denoise_loop(lat, ctx, np.zeros_like(ctx), W, cfg, sg, 5.0)
    v = O.unpatchify(np.tile(W["head.bias"], (4, 1)), (1, 2, 2), lat.shape)
    np.testing.assert_allclose(out, lat - v, atol=1e-12)


def test_dit_forward_composition_against_scalar_loops():
    cfg = small_cfg(0, depth=2)
    W = rand_weights(cfg, seed=5, std=0.2)
    rng = np.random.default_rng(19)
    lat, ctx = rng.standard_normal((2, 1, 4, 6)), rng.standard_normal((3, 6))
    grid = (1, 2, 3)
    pos = [tuple(p) for p in O.token_positions(grid)]
    m = BF.timestep_modulation(640.0, W, cfg)
    w_pe, b_pe = W["patch_embed.weight"], W["patch_embed.bias"]
    # patch vectors written out by index arithmetic, independently of patchify
    toks = []
    for ih in range(2):
        for iw in range(3):
            vec = [lat[c, 0, 2 * ih + jh, 2 * iw + jw] for c in range(2) for jh in range(2) for jw in range(2)]
            toks.append([sum(w_pe[o][i] * vec[i] for i in range(8)) + b_pe[o] for o in range(8)])
    for b in range(2):
        toks = BF.block_cross(toks, m, ctx, W, b, cfg, pos)
    vt = BF.final_layer(toks, m, W, cfg)
    v = np.zeros_like(lat)
    for n, (ih, iw) in enumerate([(a, b) for a in range(2) for b in range(3)]):
        for c in range(2):
            for jh in range(2):
                for jw in range(2):
                    v[c, 0, 2 * ih + jh, 2 * iw + jw] = vt[n][(c * 2 + jh) * 2 + jw]
    np.testing.assert_allclose(O.dit_forward(lat, 640.0, ctx, W, cfg), v, atol=1e-11)


def test_dit_forward_joint_composition_against_scalar_loops():
    # joint mode at depth 2: the condition stream must be carried from block
    # to block (block 1 reads block 0's condition-stream output)
    cfg = small_cfg(1, depth=2)
    W = rand_weights(cfg, seed=6, std=0.25)
    rng = np.random.default_rng(20)
    lat, ctx = rng.standard_normal((2, 1, 4, 4)), rng.standard_normal((3, 8))
    ref = np.array(BF.dit_forward(lat, 412.0, ctx, W, cfg))
    np.testing.assert_allclose(O.dit_forward(lat, 412.0, ctx, W, cfg), ref, atol=1e-11)


def _loop_case(mode, seed):
    cfg = small_cfg(mode, depth=2)
    W = rand_weights(cfg, seed=seed, std=0.25)
    rng = np.random.default_rng(seed + 100)
    lat = rng.standard_normal((2, 1, 4, 4))
    cond = rng.standard_normal((3, cfg["cond_dim"]))
    unc = rng.standard_normal((3, cfg["cond_dim"])) * 0.5   # a negative condition unlike the positive one
    return cfg, W, lat, cond, unc


@pytest.mark.parametrize("mode", [0, 1])
def test_loop_against_scalar_loops_with_hand_worked_timesteps(mode):
    # the full loop (guidance direction, sigma -> timestep wiring, Euler
    # increments) against the scalar restatement fed the hand-worked
    # schedule and timesteps of tests/golden/schedule_n4.txt (shift 3)
    cfg, W, lat, cond, unc = _loop_case(mode, 7 + mode)
    rows = np.array(_rows("schedule_n4.txt"))
    sig, ts = rows[:, 2], rows[:, 3]
    ref = np.array(BF.denoise_loop(lat, cond, unc, W, cfg, list(sig), list(ts), 4.0))
    np.testing.assert_allclose(O.denoise_loop(lat, cond, unc, W, cfg, sig, 4.0), ref, atol=1e-11)


@pytest.mark.parametrize("mode", [0, 1])
def test_loop_guidance_direction(mode):
    # one step from sigma 0.9 to 0.75 (timestep 900): guidance 0 must follow
    # the negative condition alone, guidance 1 the positive one
    cfg, W, lat, cond, unc = _loop_case(mode, 9 + mode)
    sig = np.array([0.9, 0.75])
    for g, which in ((0.0, unc), (1.0, cond)):
        v = np.array(BF.dit_forward(lat, 900.0, which, W, cfg))
        np.testing.assert_allclose(O.denoise_loop(lat, cond, unc, W, cfg, sig, g), lat - 0.15 * v, atol=1e-11)


# ---------------------------------------------------------------- the pins bite
def _source_mutant(fn_name, old, new):
    """The oracle function `fn_name` with the text `old` of its source
    replaced by `new` (a planted mistake), compiled against the oracle's
    module namespace."""
    src = textwrap.dedent(inspect.getsource(getattr(O, fn_name)))
    assert old in src, (fn_name, old)
    ns = dict(vars(O))
    exec(compile(src.replace(old, new), O.__file__, "exec"), ns)
    return ns[fn_name]


def _pin_block():
    cfg = small_cfg(0)
    W = rand_weights(cfg)
    rng = np.random.default_rng(12)
    grid = (1, 2, 3)
    x, ctx, m = rng.standard_normal((6, 8)), rng.standard_normal((3, 6)), rng.standard_normal(48) * 0.5
    pos = [tuple(p) for p in O.token_positions(grid)]
    ref = np.array(BF.block_cross(x, m, ctx, W, 0, cfg, pos))
    np.testing.assert_allclose(O.block_cross(x, m, ctx, W, 0, cfg, grid), ref, atol=1e-9)


def _pin_loops():
    for mode in (0, 1):
        test_loop_against_scalar_loops_with_hand_worked_timesteps(mode)
        test_loop_guidance_direction(mode)


# name -> (oracle function, replacement factory, the pin that must fail)
_MUTATIONS = {
    "rope_turns_backwards": ("apply_rope", lambda f: (lambda x, a: f(x, -a)), _pin_block),
    "modulate_without_one": ("modulate", lambda f: (lambda h, sh, sc: h * sc + sh), _pin_block),
    "gelu_erf_form": ("gelu_tanh", lambda f: (lambda x: 0.5 * x * (1 + np.vectorize(math.erf)(x / math.sqrt(2)))),
                      _pin_block),
    "attention_unscaled": ("attention", lambda f: (lambda q, k, v: O.softmax_rows(q @ k.T) @ v), _pin_block),
    "layer_norm_eps_outside": ("layer_norm", lambda f: (lambda x, eps: f(x, 0.0) + eps), _pin_block),
    # loop wiring
    "cfg_cond_uncond_swapped": ("denoise_loop", lambda f: _source_mutant(
        "denoise_loop", "cfg_combine(vc, dit_forward(x, ts[i], uncond, W, cfg), guidance)",
        "cfg_combine(dit_forward(x, ts[i], uncond, W, cfg), vc, guidance)"), _pin_loops),
    "timestep_not_scaled": ("timesteps_from_sigmas", lambda f: _source_mutant(
        "timesteps_from_sigmas", "np.asarray(sigmas, dtype=F64) * scale", "np.asarray(sigmas, dtype=F64)"),
        _pin_loops),
    "joint_condition_stream_not_carried": ("dit_forward", lambda f: _source_mutant(
        "dit_forward", "x, xc = block_joint(", "x, _ = block_joint("),
        test_dit_forward_joint_composition_against_scalar_loops),
    "schedule_squared": ("sigma_schedule", lambda f: _source_mutant(
        "sigma_schedule", "1.0 - i / n_steps", "(1.0 - i / n_steps) ** 2"), test_schedule_and_timesteps_fixture),
    "euler_step_reversed": ("euler_step", lambda f: (lambda x, v, s, sn: np.asarray(x) + (s - sn) * np.asarray(v)),
                            _pin_loops),
}


@pytest.mark.parametrize("name", sorted(_MUTATIONS))
def test_planted_oracle_mistakes_are_caught(name, monkeypatch):
    attr, mk, pin = _MUTATIONS[name]
    monkeypatch.setattr(O, attr, mk(getattr(O, attr)))
    with pytest.raises(AssertionError):
        pin()
