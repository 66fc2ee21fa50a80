"""Parity of the CUDA path (called through the C ABI) with the CPU oracle on
the same seeded inputs."""
import numpy as np
import pytest

from diffusion_transformer_denoising_gb300 import dit, synth
from oracle import dit_oracle as O
from tests.gpu_util import (COS_BF16_LOOP, TOL_F32, assert_block_close, cosine, dev, empty, host, make_model,
                            rel_max_err, small_bf16_cfg)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tiny():
    cfg = synth.config("tiny")
    W = synth.make_weights(cfg, seed=0)
    m = make_model(cfg, W)
    yield cfg, W, m
    m.close()


# ------------------------------------------------------------------ tiny, fp32
def test_tiny_timestep_modulation(tiny):
    cfg, W, m = tiny
    ts = np.array([0.0, 250.0, 700.0, 1000.0], np.float32)
    out = empty(4, 6 * cfg["hidden"])
    m.dit_timestep_modulation(ts, out)
    got = host(out)
    for i, t in enumerate(ts):
        ref = O.timestep_modulation(float(t), W, cfg)
        assert rel_max_err(got[i], ref) < TOL_F32


def test_tiny_patch_embed_and_final_layer(tiny):
    cfg, W, m = tiny
    lat = synth.make_latent(cfg, batch=2, seed=5)
    thw = cfg["latent"]
    x = empty(2, 64, cfg["hidden"])
    m.dit_patch_embed(dev(lat), 2, thw, x)
    gx = host(x)
    for b in range(2):
        assert rel_max_err(gx[b], O.patch_embed(lat[b], W, cfg)) < TOL_F32
    mod = dev(np.stack([O.timestep_modulation(t, W, cfg) for t in (300.0, 900.0)]))
    v = empty(2, *lat.shape[1:])
    m.dit_final_layer(x, mod, 2, thw, v)
    gv = host(v)
    for b, t in enumerate((300.0, 900.0)):
        mm = O.timestep_modulation(t, W, cfg)
        ref = O.unpatchify(O.final_layer(gx[b], mm, W, cfg), cfg["patch"], lat.shape[1:])
        assert rel_max_err(gv[b], ref) < TOL_F32


@pytest.mark.parametrize("block", [0, 1])
def test_tiny_block(tiny, block):
    cfg, W, m = tiny
    rng = np.random.default_rng(40 + block)
    x0 = rng.standard_normal((2, 64, cfg["hidden"])).astype(np.float32)
    ctx = synth.make_cond(cfg, batch=2, seed=7)
    mods = np.stack([O.timestep_modulation(t, W, cfg) for t in (123.0, 876.0)])
    x = dev(x0)
    m.dit_block_forward(block, x, None, dev(mods), dev(ctx), 2, (1, 8, 8), 16)
    got = host(x)
    for b in range(2):
        ref = O.block_cross(x0[b], mods[b], ctx[b], W, block, cfg, (1, 8, 8))
        assert rel_max_err(got[b], ref) < TOL_F32
        # the block's own update, not just the carried residual
        assert rel_max_err(got[b] - x0[b], ref - x0[b]) < 10 * TOL_F32


def test_tiny_denoise_loop(tiny):
    cfg, W, m = tiny
    lat = synth.make_latent(cfg, batch=1, seed=1)
    cond = synth.make_cond(cfg, batch=1, seed=2)
    unc = np.zeros_like(cond)
    sig = O.shift_sigma(O.sigma_schedule(cfg["steps"]), cfg["shift"]).astype(np.float32)
    x = dev(lat)
    m.dit_denoise_loop(x, 1, cfg["latent"], dev(cond), dev(unc), 16, sig, cfg["guidance"])
    m.dit_synchronize()
    got = host(x)[0]
    ref = O.denoise_loop(lat[0], cond[0], unc[0], W, cfg, sig.astype(np.float64), cfg["guidance"])
    assert rel_max_err(got, ref) < TOL_F32
    # the denoised latent moved away from the noise: compare the displacement too
    assert rel_max_err(got - lat[0], ref - lat[0]) < 10 * TOL_F32


def test_tiny_loop_twice_is_bitwise_identical(tiny):
    cfg, W, m = tiny
    lat = synth.make_latent(cfg, batch=1, seed=3)
    cond = dev(synth.make_cond(cfg, batch=1, seed=4))
    unc = dev(np.zeros((1, 16, 128), np.float32))
    sig = O.shift_sigma(O.sigma_schedule(4), 3.0).astype(np.float32)
    outs = []
    for _ in range(2):
        x = dev(lat)
        m.dit_denoise_loop(x, 1, cfg["latent"], cond, unc, 16, sig, 5.0)
        outs.append(host(x))
    assert np.array_equal(outs[0], outs[1])


# ------------------------------------------------------------------ guidance / Euler
@pytest.mark.parametrize("n", [1, 7, 4096, 100003])
def test_cfg_combine_and_euler(n):
    rng = np.random.default_rng(n)
    vc, vu, x = (rng.standard_normal(n).astype(np.float32) for _ in range(3))
    v = empty(n)
    dit.cfg_combine(dev(vc), dev(vu), 4.0, v, n)
    np.testing.assert_allclose(host(v), O.cfg_combine(vc, vu, 4.0), rtol=0, atol=1e-5)
    xd = dev(x)
    dit.flow_euler_step(xd, v, 0.75, 0.5, n)
    np.testing.assert_allclose(host(xd), O.euler_step(x, O.cfg_combine(vc, vu, 4.0), 0.75, 0.5), rtol=0, atol=1e-5)


def test_cfg_scale_one_gives_conditional():
    rng = np.random.default_rng(3)
    vc, vu = (rng.standard_normal(1000).astype(np.float32) for _ in range(2))
    v = empty(1000)
    dit.cfg_combine(dev(vc), dev(vu), 1.0, v, 1000)
    np.testing.assert_allclose(host(v), vc, rtol=0, atol=2e-7 * 8)


# ------------------------------------------------------------------ bf16, tensor cores
@pytest.fixture(scope="module")
def small_cross():
    cfg = small_bf16_cfg(synth.COND_CROSS)
    W = synth.make_weights(cfg, seed=11)
    m = make_model(cfg, W)
    yield cfg, W, m
    m.close()


@pytest.fixture(scope="module")
def small_joint():
    cfg = small_bf16_cfg(synth.COND_JOINT)
    W = synth.make_weights(cfg, seed=12)
    m = make_model(cfg, W)
    yield cfg, W, m
    m.close()


def test_bf16_patch_embed(small_cross):
    cfg, W, m = small_cross
    thw = (3, 20, 26)      # grid 3 x 10 x 13 = 390 tokens: ragged GEMM tail
    lat = synth.make_latent(cfg, batch=2, seed=8, latent=thw)
    x = empty(2, 390, cfg["hidden"])
    m.dit_patch_embed(dev(lat), 2, thw, x)
    m.dit_synchronize()
    gx = host(x)
    for b in range(2):
        lat_b = synth.round_bf16(lat[b]).astype(np.float64)   # the tensor-core path reads bf16 tokens
        assert rel_max_err(gx[b], O.patch_embed(lat_b, W, cfg)) < 1e-3


def test_bf16_final_layer(small_cross):
    cfg, W, m = small_cross
    thw = (3, 20, 26)
    rng = np.random.default_rng(9)
    x = rng.standard_normal((2, 390, cfg["hidden"])).astype(np.float32)
    mods = np.stack([O.timestep_modulation(t, W, cfg) for t in (100.0, 600.0)])
    v = empty(2, cfg["in_channels"], *thw)
    m.dit_final_layer(dev(x), dev(mods), 2, thw, v)
    m.dit_synchronize()
    gv = host(v)
    for b in range(2):
        ref = O.unpatchify(O.final_layer(x[b], mods[b], W, cfg), cfg["patch"], (cfg["in_channels"],) + thw)
        assert_block_close(gv[b], ref)


@pytest.mark.parametrize("grid,L", [((3, 10, 13), 77), ((1, 16, 16), 128), ((2, 9, 7), 5)])
def test_bf16_cross_block(small_cross, grid, L):
    cfg, W, m = small_cross
    N = int(np.prod(grid))
    rng = np.random.default_rng(N + L)
    x0 = (rng.standard_normal((2, N, cfg["hidden"])) * 0.5).astype(np.float32)
    ctx = synth.make_cond(cfg, batch=2, seed=L, length=L)
    mods = np.stack([O.timestep_modulation(t, W, cfg) for t in (200.0, 950.0)])
    x = dev(x0)
    m.dit_block_forward(1, x, None, dev(mods), dev(ctx), 2, grid, L)
    m.dit_synchronize()
    got = host(x)
    for b in range(2):
        ref = O.block_cross(x0[b], mods[b], ctx[b], W, 1, cfg, grid)
        assert_block_close(got[b], ref)
        assert_block_close(got[b] - x0[b], ref - x0[b], 5)


@pytest.mark.parametrize("grid,L", [((1, 12, 20), 64), ((1, 7, 9), 33)])
def test_bf16_joint_block(small_joint, grid, L):
    cfg, W, m = small_joint
    N = int(np.prod(grid))
    rng = np.random.default_rng(N + 3 * L)
    x0 = (rng.standard_normal((2, N, cfg["hidden"])) * 0.5).astype(np.float32)
    xc0 = synth.make_cond(cfg, batch=2, seed=L, length=L)
    mods = np.stack([O.timestep_modulation(t, W, cfg) for t in (333.0, 777.0)])
    x, xc = dev(x0), dev(xc0)
    m.dit_block_forward(0, x, xc, dev(mods), None, 2, grid, L)
    m.dit_synchronize()
    gx, gc = host(x), host(xc)
    for b in range(2):
        rx, rc = O.block_joint(x0[b], xc0[b], mods[b], W, 0, cfg, grid)
        assert_block_close(gx[b], rx)
        assert_block_close(gc[b], rc)


@pytest.mark.parametrize("mode", [synth.COND_CROSS, synth.COND_JOINT])
def test_bf16_denoise_loop(mode, small_cross, small_joint):
    cfg, W, m = small_cross if mode == synth.COND_CROSS else small_joint
    thw = (2, 12, 18) if mode == synth.COND_CROSS else (1, 24, 20)
    L = 40
    lat = synth.make_latent(cfg, batch=1, seed=21, latent=thw)
    cond = synth.make_cond(cfg, batch=1, seed=22, length=L)
    unc = np.zeros_like(cond)
    sig = O.shift_sigma(O.sigma_schedule(3), 3.0).astype(np.float32)
    x = dev(lat)
    m.dit_denoise_loop(x, 1, thw, dev(cond), dev(unc), L, sig, 4.0)
    m.dit_synchronize()
    got = host(x)[0]
    ref = O.denoise_loop(lat[0], cond[0], unc[0], W, cfg, sig.astype(np.float64), 4.0)
    assert cosine(got, ref) >= COS_BF16_LOOP
    assert cosine(got - lat[0], ref - lat[0]) >= 0.99


# ------------------------------------------------------------------ failure paths
def test_forward_before_load_is_rejected():
    cfg = synth.config("tiny")
    m = dit.DiT(cfg)
    with pytest.raises(dit.DitError) as e:
        m.dit_timestep_modulation(np.zeros(1, np.float32), empty(1, 768))
    assert e.value.status == dit.DIT_ERR_NOT_LOADED
    m.close()


def test_bad_schedule_and_missing_uncond(tiny):
    cfg, W, m = tiny
    x = dev(synth.make_latent(cfg))
    cond = dev(synth.make_cond(cfg))
    good = O.shift_sigma(O.sigma_schedule(4), 3.0).astype(np.float32)
    for sig, unc, g in ((good[::-1].copy(), cond, 5.0),          # reversed timesteps
                        (good, None, 5.0),                         # CFG on without negatives
                        (good[:-1].copy(), cond, 5.0)):            # does not end at 0
        with pytest.raises(dit.DitError) as e:
            m.dit_denoise_loop(x, 1, cfg["latent"], cond, unc, 16, sig, g)
        assert e.value.status == dit.DIT_ERR_INVALID_ARG
    with pytest.raises(dit.DitError) as e:
        m.dit_denoise_loop(x, 1, (1, 15, 16), cond, cond, 16, good, 5.0)   # not divisible by the patch
    assert e.value.status == dit.DIT_ERR_SHAPE
    # resuming part of a schedule is allowed with the flag
    m.dit_denoise_loop(x, 1, cfg["latent"], cond, cond, 16, good[1:].copy(), 5.0, flags=dit.LOOP_PARTIAL_SCHEDULE)
    m.dit_synchronize()


def test_strict_weight_loading():
    cfg = synth.config("tiny")
    W = synth.make_weights(cfg)
    m = dit.DiT(cfg)
    bad = dict(W)
    bad["head.bias"] = np.zeros(3, np.float32)
    with pytest.raises(dit.DitError) as e:
        m.load_weights(bad, chunk=10**6)
    assert e.value.status == dit.DIT_ERR_SHAPE
    with pytest.raises(dit.DitError) as e:
        m.load_weights({"blocks.9.attn.qkv.weight": np.zeros((384, 128), np.float32)})
    assert e.value.status == dit.DIT_ERR_SHAPE
    m.load_weights(W, chunk=10**6)           # nothing of the failed calls was kept
    with pytest.raises(dit.DitError):
        m.load_weights({"head.bias": W["head.bias"]})   # loaded twice
    m.close()


def test_injected_allocation_failure():
    cfg = synth.config("tiny")
    dit.dit_debug_fail_alloc_after(1)
    with pytest.raises(dit.DitError) as e:
        dit.DiT(cfg)
    assert e.value.status == dit.DIT_ERR_OOM
    dit.dit_debug_fail_alloc_after(0)
    dit.DiT(cfg).close()


def test_device_wait_timeout_is_reported_and_model_stays_usable(tiny):
    """A bounded device wait that nothing completes gives up after the wait
    limit: the failure surfaces as DIT_ERR_TIMEOUT at the next synchronize,
    the error word is cleared, and the same model keeps producing correct
    results (no fault, no hang, context intact)."""
    cfg, W, m = tiny
    m.dit_debug_stall()
    with pytest.raises(dit.DitError) as e:
        m.dit_synchronize()
    assert e.value.status == dit.DIT_ERR_TIMEOUT
    assert "site 99" in str(e.value)
    m.dit_synchronize()  # the word was cleared
    t = np.array([500.0], np.float32)
    out = empty(1, 6 * cfg["hidden"])
    m.dit_timestep_modulation(t, out)
    m.dit_synchronize()
    assert rel_max_err(host(out)[0], O.timestep_modulation(500.0, W, cfg)) < TOL_F32


# ------------------------------------------------------------------ more shapes and paths
def test_bf16_k_and_n_tails():
    """MLP width 648 and condition width 200 (multiples of 8, not of 64): the
    GEMMs' last K block and the FFN1 output's last column tile are partial
    (the tensor-map loads fill the missing K columns with zeros)."""
    cfg = small_bf16_cfg(synth.COND_CROSS, mlp=648, cond_dim=200, depth=1)
    W = synth.make_weights(cfg, seed=13)
    m = make_model(cfg, W)
    grid, L = (2, 9, 7), 37
    N = int(np.prod(grid))
    rng = np.random.default_rng(14)
    x0 = (rng.standard_normal((2, N, cfg["hidden"])) * 0.5).astype(np.float32)
    ctx = synth.make_cond(cfg, batch=2, seed=15, length=L)
    mods = np.stack([O.timestep_modulation(t, W, cfg) for t in (250.0, 650.0)])
    x = dev(x0)
    m.dit_block_forward(0, x, None, dev(mods), dev(ctx), 2, grid, L)
    m.dit_synchronize()
    got = host(x)
    for b in range(2):
        ref = O.block_cross(x0[b], mods[b], ctx[b], W, 0, cfg, grid)
        assert_block_close(got[b], ref, case=f"k_tails b{b}")
        assert_block_close(got[b] - x0[b], ref - x0[b], 5, case=f"k_tails update b{b}")
    m.close()


def test_bf16_attention_rescale_paths():
    """Peaked attention whose scores grow along the token order: the query and
    key projections are equal and scaled by 8 (exact in bf16), and the tokens
    lean more and more on one direction, so scores span ~180 log2 units and
    most rows' maxima grow by far more than 2^8 after the first key tile.
    This runs the attention kernel's slow paths (tile row max, rescale of O
    and l, redone rows; large tile sums) on most tiles."""
    cfg = small_bf16_cfg(synth.COND_CROSS, depth=1, rope_axes=(0, 0, 0))
    W = synth.make_weights(cfg, seed=51)
    D = cfg["hidden"]
    wqkv = W["blocks.0.attn.qkv.weight"].copy()
    wqkv[:D] *= 8.0
    wqkv[D:2 * D] = wqkv[:D]
    W["blocks.0.attn.qkv.weight"] = wqkv
    m = make_model(cfg, W)
    grid, L = (1, 20, 26), 64     # 520 tokens: 5 key tiles, the last one partial
    N = int(np.prod(grid))
    rng = np.random.default_rng(52)
    u = rng.standard_normal(D)
    x0 = (np.linspace(0.0, 4.0, N)[:, None] * u[None] + rng.standard_normal((N, D))).astype(np.float32)
    mod = O.timestep_modulation(600.0, W, cfg)
    # the case does what it claims: score span and growth along the key tiles
    sh1, sc1 = O.block_modulation(mod, W["blocks.0.mod_table"], D)[:2]
    h = O.modulate(O.layer_norm(x0, cfg["ln_eps"]), sh1, sc1)
    q = O.linear(h, wqkv[:D], W["blocks.0.attn.qkv.bias"][:D])
    k = O.linear(h, wqkv[D:2 * D], W["blocks.0.attn.qkv.bias"][D:2 * D])
    s = q[:, :128] @ k[:, :128].T * (np.log2(np.e) / np.sqrt(128))
    assert s.max() - s.min() > 20
    assert np.mean(s[:, 384:512].max(1) - s[:, :128].max(1) > 8) > 0.5
    ctx = synth.make_cond(cfg, batch=1, seed=53, length=L)
    x = dev(x0[None])
    m.dit_block_forward(0, x, None, dev(mod[None]), dev(ctx), 1, grid, L)
    m.dit_synchronize()
    got = host(x)[0]
    ref = O.block_cross(x0, mod, ctx[0], W, 0, cfg, grid)
    assert_block_close(got, ref, case="rescale")
    assert_block_close(got - x0, ref - x0, 5, case="rescale update")
    m.close()


@pytest.mark.parametrize("peaked", [False, True], ids=["flat", "peaked"])
def test_bf16_attention_long_key_range(peaked):
    """A key range long enough for the one-CTA-per-query-tile attention (more
    than 64 tiles of 128 keys): 8600 tokens = 45 key tiles of 192, the last
    one holding 152 keys (its third 64-key slice only 24), and a last query
    tile of 24 rows.  Flat: N(0, 0.02) weights, the fast path on almost every
    tile.  Peaked: the rescale case above at this length (query and key
    projections equal and scaled by 8, tokens leaning more and more on one
    direction), so the tile row max, the rescale of O and l and the redone
    rows run on most tiles.  Sampled rows of both batch items against the
    oracle."""
    cfg = small_bf16_cfg(synth.COND_CROSS, depth=1, rope_axes=(0, 0, 0) if peaked else (32, 48, 48))
    W = synth.make_weights(cfg, seed=61)
    D = cfg["hidden"]
    grid, L = (1, 86, 100), 40
    N = int(np.prod(grid))
    rng = np.random.default_rng(62)
    if peaked:
        wqkv = W["blocks.0.attn.qkv.weight"].copy()
        wqkv[:D] *= 8.0
        wqkv[D:2 * D] = wqkv[:D]
        W["blocks.0.attn.qkv.weight"] = wqkv
        u = rng.standard_normal(D)
        x0 = np.stack([np.linspace(0.0, 4.0, N)[:, None] * u[None] + rng.standard_normal((N, D)),
                       np.linspace(4.0, 0.0, N)[:, None] * u[None] + rng.standard_normal((N, D))])
    else:
        x0 = rng.standard_normal((2, N, D)) * 0.5
    x0 = x0.astype(np.float32)
    mods = np.stack([O.timestep_modulation(t, W, cfg) for t in (300.0, 800.0)])
    if peaked:
        # the case does what it claims: scores of sampled query rows span far
        # more than 2^8 and grow along the keys
        sh1, sc1 = O.block_modulation(mods[0], W["blocks.0.mod_table"], D)[:2]
        hh = O.modulate(O.layer_norm(x0[0], cfg["ln_eps"]), sh1, sc1)
        k = O.linear(hh, wqkv[D:2 * D], W["blocks.0.attn.qkv.bias"][D:2 * D])
        q = O.linear(hh[::97], wqkv[:D], W["blocks.0.attn.qkv.bias"][:D])
        sc = q[:, :128] @ k[:, :128].T * (np.log2(np.e) / np.sqrt(128))
        assert sc.max() - sc.min() > 20
        assert np.mean(sc[:, -192:].max(1) - sc[:, :192].max(1) > 8) > 0.5
    m = make_model(cfg, W)
    ctx = synth.make_cond(cfg, batch=2, seed=63, length=L)
    x = dev(x0)
    m.dit_block_forward(0, x, None, dev(mods), dev(ctx), 2, grid, L)
    m.dit_synchronize()
    got = host(x)
    rows = np.array(sorted(set(np.linspace(0, N - 1, 48).astype(int).tolist()) | set(range(N - 26, N))))
    angles = None if peaked else O.rope_angles(O.token_positions(grid), cfg["rope_axes"], cfg["rope_theta"])
    for b in range(2):
        ref = O.block_cross(x0[b], mods[b], ctx[b], W, 0, cfg, grid, rows=rows, angles=angles)
        case = f"long keys {'peaked' if peaked else 'flat'} b{b}"
        assert_block_close(got[b][rows], ref, case=case)
        assert_block_close(got[b][rows] - x0[b][rows], ref - x0[b][rows], 5, case=case + " update")
    m.close()


@pytest.mark.parametrize("which", ["tiny_fp32", "bf16_cross", "bf16_joint"])
def test_loop_two_requests(which, tiny, small_cross, small_joint):
    """dit_denoise_loop with batch = 2 requests, each with its own latent,
    positive and (non-zero) negative condition: the CFG batch runs as
    [cond(2); uncond(2)] and every request must match its own oracle loop."""
    if which == "tiny_fp32":
        cfg, W, m = tiny
        thw, L, g = cfg["latent"], cfg["cond_len"], cfg["guidance"]
    else:
        cfg, W, m = small_cross if which == "bf16_cross" else small_joint
        thw, L, g = ((2, 12, 16) if which == "bf16_cross" else (1, 16, 20)), 24, 4.0
    lat = synth.make_latent(cfg, batch=2, seed=61, latent=thw)
    cond = synth.make_cond(cfg, batch=2, seed=62, length=L)
    unc = synth.make_cond(cfg, batch=2, seed=63, length=L) * np.float32(0.5)
    sig = O.shift_sigma(O.sigma_schedule(3), 3.0).astype(np.float32)
    x = dev(lat)
    m.dit_denoise_loop(x, 2, thw, dev(cond), dev(unc), L, sig, g)
    m.dit_synchronize()
    got = host(x)
    for r in range(2):
        ref = O.denoise_loop(lat[r], cond[r], unc[r], W, cfg, sig.astype(np.float64), g)
        if which == "tiny_fp32":
            assert rel_max_err(got[r], ref) < TOL_F32
            assert rel_max_err(got[r] - lat[r], ref - lat[r]) < 10 * TOL_F32
        else:
            assert cosine(got[r], ref) >= COS_BF16_LOOP
            assert cosine(got[r] - lat[r], ref - lat[r]) >= 0.99


@pytest.mark.parametrize("which", ["tiny_fp32", "bf16_cross", "bf16_joint"])
def test_loop_cuda_graph_is_bitwise_eager(which, tiny, small_cross, small_joint):
    """DIT_LOOP_CUDA_GRAPH replays one captured step: the final latents are
    bitwise those of the eager launches, a second call reuses the capture,
    a changed guidance scale is captured again, and the launch counts of the
    replayed steps equal the eager ones."""
    if which == "tiny_fp32":
        cfg, W, m = tiny
        thw, L = cfg["latent"], cfg["cond_len"]
    else:
        cfg, W, m = small_cross if which == "bf16_cross" else small_joint
        thw, L = ((2, 12, 16) if which == "bf16_cross" else (1, 16, 20)), 24
    lat = synth.make_latent(cfg, batch=1, seed=91, latent=thw)
    cond = dev(synth.make_cond(cfg, batch=1, seed=92, length=L))
    unc = dev(np.zeros((1, L, cfg["cond_dim"]), np.float32))
    sig = O.shift_sigma(O.sigma_schedule(4), 3.0).astype(np.float32)
    x, x0 = dev(lat), dev(lat)

    def run(flags, g):
        x.copy_(x0)
        m.dit_profile_start(timing=False)
        m.dit_denoise_loop(x, 1, thw, cond, unc, L, sig, g, flags=flags)
        counts = m.dit_profile_stop()
        m.dit_synchronize()
        return host(x), counts

    eager, c_eager = run(0, 4.0)
    graph1, c_graph = run(dit.LOOP_CUDA_GRAPH, 4.0)
    graph2, _ = run(dit.LOOP_CUDA_GRAPH, 4.0)          # the capture is reused
    assert np.array_equal(eager, graph1) and np.array_equal(eager, graph2)
    assert {k: v[0] for k, v in c_eager.items()} == {k: v[0] for k, v in c_graph.items()}
    eager3, _ = run(0, 2.5)
    graph3, _ = run(dit.LOOP_CUDA_GRAPH, 2.5)          # new scalar: captured again
    assert np.array_equal(eager3, graph3) and not np.array_equal(eager3, eager)


# ------------------------------------------------------------------ fp8 precision
@pytest.mark.parametrize("mode,grid,L", [(synth.COND_CROSS, (3, 10, 13), 77), (synth.COND_CROSS, (2, 9, 7), 5),
                                         (synth.COND_JOINT, (1, 12, 20), 64), (synth.COND_JOINT, (1, 7, 9), 33)])
def test_fp8_block(mode, grid, L):
    """DIT_PREC_FP8: the same block as the bf16 tests with the LayerNorm-fed
    GEMMs in e4m3 (weights quantized at load, activations per row), against
    the oracle on the same bf16-valued weights."""
    from tests.gpu_util import assert_fp8_block_close
    cfg = small_bf16_cfg(mode, precision=synth.PREC_FP8, depth=1)
    W = synth.make_weights(cfg, seed=17)
    m = make_model(cfg, W)
    N = int(np.prod(grid))
    rng = np.random.default_rng(N + 7 * L)
    x0 = (rng.standard_normal((2, N, cfg["hidden"])) * 0.5).astype(np.float32)
    ctx = synth.make_cond(cfg, batch=2, seed=L + 1, length=L)
    mods = np.stack([O.timestep_modulation(t, W, cfg) for t in (300.0, 800.0)])
    x = dev(x0)
    if mode == synth.COND_CROSS:
        m.dit_block_forward(0, x, None, dev(mods), dev(ctx), 2, grid, L)
    else:
        xc = dev(ctx)
        m.dit_block_forward(0, x, xc, dev(mods), None, 2, grid, L)
    m.dit_synchronize()
    got = host(x)
    for b in range(2):
        if mode == synth.COND_CROSS:
            ref = O.block_cross(x0[b], mods[b], ctx[b], W, 0, cfg, grid)
        else:
            ref = O.block_joint(x0[b], ctx[b], mods[b], W, 0, cfg, grid)[0]
        assert_fp8_block_close(got[b], ref, x0[b], case=f"fp8 block mode {mode} grid {grid} L {L} b{b}")
    m.close()


@pytest.mark.parametrize("mode", [synth.COND_CROSS, synth.COND_JOINT])
def test_fp8_denoise_loop(mode):
    from tests.gpu_util import COS_FP8_LOOP, log_errors
    cfg = small_bf16_cfg(mode, precision=synth.PREC_FP8)
    W = synth.make_weights(cfg, seed=18)
    m = make_model(cfg, W)
    thw = (2, 12, 18) if mode == synth.COND_CROSS else (1, 24, 20)
    L = 40
    lat = synth.make_latent(cfg, batch=1, seed=23, latent=thw)
    cond = synth.make_cond(cfg, batch=1, seed=24, length=L)
    unc = np.zeros_like(cond)
    sig = O.shift_sigma(O.sigma_schedule(3), 3.0).astype(np.float32)
    x = dev(lat)
    m.dit_denoise_loop(x, 1, thw, dev(cond), dev(unc), L, sig, 4.0)
    m.dit_synchronize()
    got = host(x)[0]
    ref = O.denoise_loop(lat[0], cond[0], unc[0], W, cfg, sig.astype(np.float64), 4.0)
    c_all, c_upd = cosine(got, ref), cosine(got - lat[0], ref - lat[0])
    log_errors(f"fp8 loop mode {mode}", cos=c_all, cos_update=c_upd)
    assert c_all >= COS_FP8_LOOP and c_upd >= COS_FP8_LOOP - 0.01, (c_all, c_upd)
    m.close()


# ------------------------------------------------------------------ degenerate shapes
@pytest.mark.parametrize("prec", [synth.PREC_F32, synth.PREC_BF16])
@pytest.mark.parametrize("mode", [synth.COND_CROSS, synth.COND_JOINT])
@pytest.mark.parametrize("grid,L", [((1, 1, 1), 1), ((1, 1, 1), 3), ((1, 2, 1), 1)])
def test_degenerate_single_token_and_single_condition(prec, mode, grid, L):
    """One image/video token and/or one condition token: every GEMM has one
    partial row tile, the attention one partial key tile with a single valid
    key (cross mode, L = 1: the output row is that key's value row)."""
    if prec == synth.PREC_F32:
        cfg = synth.config("tiny", cond_mode=mode, depth=1, rope_axes=(0, 16, 16))
        if mode == synth.COND_JOINT:
            cfg["cond_dim"] = cfg["hidden"]
        tol = lambda got, ref, case: assert_f32_close(got, ref, case)
    else:
        cfg = small_bf16_cfg(mode, depth=1)
        tol = lambda got, ref, case: assert_block_close(got, ref, case=case)
    W = synth.make_weights(cfg, seed=29)
    m = make_model(cfg, W)
    N = int(np.prod(grid))
    rng = np.random.default_rng(77 + N + L)
    x0 = (rng.standard_normal((2, N, cfg["hidden"])) * 0.5).astype(np.float32)
    ctx = synth.make_cond(cfg, batch=2, seed=31 + L, length=L)
    mods = np.stack([O.timestep_modulation(t, W, cfg) for t in (150.0, 650.0)])
    x = dev(x0)
    if mode == synth.COND_CROSS:
        m.dit_block_forward(0, x, None, dev(mods), dev(ctx), 2, grid, L)
    else:
        xc = dev(ctx)
        m.dit_block_forward(0, x, xc, dev(mods), None, 2, grid, L)
    m.dit_synchronize()
    got = host(x)
    for b in range(2):
        if mode == synth.COND_CROSS:
            ref = O.block_cross(x0[b], mods[b], ctx[b], W, 0, cfg, grid)
        else:
            ref = O.block_joint(x0[b], ctx[b], mods[b], W, 0, cfg, grid)[0]
        tol(got[b], ref, f"degenerate {grid} L {L} mode {mode} prec {prec} b{b}")
    m.close()


def assert_f32_close(got, ref, case):
    e = rel_max_err(got, ref)
    assert e < TOL_F32, f"{case}: max error {e:.3e} of the reference RMS"


@pytest.mark.parametrize("which", ["tiny_fp32", "bf16_cross", "bf16_joint"])
def test_loop_resumed_from_a_sub_schedule_is_bitwise_the_same(which, tiny, small_cross, small_joint):
    """Resume: four steps in one call equal two calls over the sub-schedules
    sigmas[0:3] and sigmas[2:5] (DIT_LOOP_PARTIAL_SCHEDULE), bit for bit."""
    if which == "tiny_fp32":
        cfg, W, m = tiny
        thw, L = cfg["latent"], cfg["cond_len"]
    else:
        cfg, W, m = small_cross if which == "bf16_cross" else small_joint
        thw, L = ((2, 12, 16) if which == "bf16_cross" else (1, 16, 20)), 24
    lat = synth.make_latent(cfg, batch=1, seed=95, latent=thw)
    cond = dev(synth.make_cond(cfg, batch=1, seed=96, length=L))
    unc = dev(np.zeros((1, L, cfg["cond_dim"]), np.float32))
    sig = O.shift_sigma(O.sigma_schedule(4), 3.0).astype(np.float32)
    x_all = dev(lat)
    m.dit_denoise_loop(x_all, 1, thw, cond, unc, L, sig, 4.0)
    x_two = dev(lat)
    m.dit_denoise_loop(x_two, 1, thw, cond, unc, L, sig[0:3].copy(), 4.0, flags=dit.LOOP_PARTIAL_SCHEDULE)
    m.dit_denoise_loop(x_two, 1, thw, cond, unc, L, sig[2:5].copy(), 4.0, flags=dit.LOOP_PARTIAL_SCHEDULE)
    m.dit_synchronize()
    assert np.array_equal(host(x_all), host(x_two))


def test_two_models_on_unordered_streams_are_isolated():
    """Separate models share nothing: two models' loops enqueued on two
    streams with no ordering between them give, bit for bit, what each gives
    alone (tiny fp32 and small bf16 models, different weights and inputs)."""
    import torch
    cases = []
    for cfg, seed in ((synth.config("tiny"), 201), (small_bf16_cfg(synth.COND_CROSS), 202)):
        W = synth.make_weights(cfg, seed=seed)
        thw = cfg["latent"] if cfg["precision"] == synth.PREC_F32 else (2, 12, 16)
        L = 16
        lat = synth.make_latent(cfg, batch=1, seed=seed + 1, latent=thw)
        cond = dev(synth.make_cond(cfg, batch=1, seed=seed + 2, length=L))
        unc = dev(np.zeros((1, L, cfg["cond_dim"]), np.float32))
        cases.append((make_model(cfg, W), thw, L, lat, cond, unc))
    sig = O.shift_sigma(O.sigma_schedule(4), 3.0).astype(np.float32)
    alone = []
    for m, thw, L, lat, cond, unc in cases:
        x = dev(lat)
        m.dit_denoise_loop(x, 1, thw, cond, unc, L, sig, 5.0)
        m.dit_synchronize()
        alone.append(host(x))
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    xs = [dev(c[3]) for c in cases]
    torch.cuda.synchronize()
    for (m, thw, L, lat, cond, unc), x, st in zip(cases, xs, streams):
        m.dit_denoise_loop(x, 1, thw, cond, unc, L, sig, 5.0, stream=st)
    for (m, *_), st in zip(cases, streams):
        m.dit_synchronize(stream=st)
    for a, x in zip(alone, xs):
        assert np.array_equal(a, host(x))
    for m, *_ in cases:
        m.close()


# ------------------------------------------------------------------ GEMM CTA pairs
@pytest.mark.parametrize("prec,mode", [(synth.PREC_BF16, synth.COND_CROSS), (synth.PREC_FP8, synth.COND_CROSS),
                                       (synth.PREC_BF16, synth.COND_JOINT)])
def test_gemm_cta_pairs_match_single_ctas(prec, mode):
    """GEMMs of width a multiple of 256 can run on CTA pairs (one cta_group::2
    MMA of 256 x 256 per K step, each CTA holding half of the W tile) or on
    single CTAs (128 x 256).  Each output element is the same fp32 sum over
    the same K steps either way, so a block with pairs forced on (QKV,
    out-projections, cross-K/V, FFN2; in the joint block the two streams'
    problems share each launch) gives the same bits as with pairs off.  390
    (or 400) tokens x 2 = 7 row blocks: the last pair's second CTA reads rows
    past M; 5 condition rows: the whole second CTA does."""
    cfg = small_bf16_cfg(mode, precision=prec, depth=1)
    W = synth.make_weights(cfg, seed=19)
    grid, L = ((3, 10, 13) if mode == synth.COND_CROSS else (1, 20, 20)), 5
    N = int(np.prod(grid))
    rng = np.random.default_rng(5)
    x0 = (rng.standard_normal((2, N, cfg["hidden"])) * 0.5).astype(np.float32)
    ctx = synth.make_cond(cfg, batch=2, seed=6, length=L)
    mods = np.stack([O.timestep_modulation(t, W, cfg) for t in (250.0, 850.0)])
    out = {}
    try:
        for pairs in (2, 0):
            dit.dit_debug_gemm_cta_pairs(pairs)
            m = make_model(cfg, W)
            x = dev(x0)
            if mode == synth.COND_CROSS:
                m.dit_block_forward(0, x, None, dev(mods), dev(ctx), 2, grid, L)
                m.dit_synchronize()
                out[pairs] = host(x)
            else:
                xc = dev(ctx)
                m.dit_block_forward(0, x, xc, dev(mods), None, 2, grid, L)
                m.dit_synchronize()
                out[pairs] = np.concatenate([host(x).ravel(), host(xc).ravel()])
            m.close()
    finally:
        dit.dit_debug_gemm_cta_pairs(1)
    diff = float(np.max(np.abs(out[2] - out[0])))
    print(f"[gpu] cta pairs vs single, precision {prec} mode {mode}: max |diff| {diff:.3e}")
    assert np.isfinite(out[2]).all()
    assert np.array_equal(out[2], out[0]), diff
