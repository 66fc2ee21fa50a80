"""Parity at the full workload sizes, in the launch configuration the bench
times (batch 2 = conditional + unconditional pass): the CUDA path runs the
whole block; the oracle computes keys/values over every token and the block
output for a sample of rows (first, last, ragged-tail and spread rows)."""
import numpy as np
import pytest

from diffusion_transformer_denoising_gb300 import dit, synth
from oracle import dit_oracle as O
from tests.gpu_util import COS_BF16_LOOP, assert_block_close, cosine, dev, empty, host, make_model, rel_max_err

pytestmark = pytest.mark.gpu


def _rows(n, extra=()):
    r = set(np.linspace(0, n - 1, 40).astype(int).tolist()) | {0, 1, n - 1, n - 2} | set(extra)
    return np.array(sorted(x for x in r if 0 <= x < n))


@pytest.fixture(scope="module")
def video_block():
    cfg = synth.config("video", depth=1)
    W = synth.make_weights(cfg, seed=0)
    m = make_model(cfg, W)
    yield cfg, W, m
    m.close()


def test_video_block_full_size(video_block):
    """One video block: 32760 tokens (21 x 30 x 52 grid), 512 text tokens,
    batch 2 (condition / zero condition), timestep 700 (sigma 0.7)."""
    cfg, W, m = video_block
    grid = synth.grid(cfg)
    N, L = int(np.prod(grid)), cfg["cond_len"]
    lat = synth.make_latent(cfg, batch=1, seed=1)
    ctx = np.concatenate([synth.make_cond(cfg, batch=1, seed=2), np.zeros((1, L, cfg["cond_dim"]), np.float32)])
    # block input: the patch-embedded latent (both passes see the same latent)
    x0 = np.stack([O.patch_embed(lat[0], W, cfg)] * 2).astype(np.float32)
    mod = O.timestep_modulation(700.0, W, cfg)
    mods = np.stack([mod, mod]).astype(np.float32)
    x = dev(x0)
    m.dit_block_forward(0, x, None, dev(mods), dev(ctx), 2, grid, L)
    m.dit_synchronize()
    got = host(x)
    rows = _rows(N, extra=range(N - 120, N - 110))   # rows of the last (ragged) 128-row query tile
    angles = O.rope_angles(O.token_positions(grid), cfg["rope_axes"], cfg["rope_theta"])
    for b in range(2):
        ref = O.block_cross(x0[b], mods[b], ctx[b], W, 0, cfg, grid, rows=rows, angles=angles)
        assert_block_close(got[b][rows], ref)
        assert_block_close(got[b][rows] - x0[b][rows], ref - x0[b][rows], 5)


@pytest.fixture(scope="module")
def image_model():
    cfg = synth.config("image", depth=2)
    W = synth.make_weights(cfg, seed=0)
    m = make_model(cfg, W)
    yield cfg, W, m
    m.close()


def test_image_block_full_size(image_model):
    """One dual-stream image block: 4096 image tokens (64 x 64) jointly
    attending with 512 condition tokens, batch 2."""
    cfg, W, m = image_model
    grid = synth.grid(cfg)
    N, L, D = int(np.prod(grid)), cfg["cond_len"], cfg["hidden"]
    rng = np.random.default_rng(3)
    x0 = (rng.standard_normal((2, N, D)) * 0.2).astype(np.float32)
    xc0 = np.concatenate([synth.make_cond(cfg, batch=1, seed=4), np.zeros((1, L, D), np.float32)])
    mod = O.timestep_modulation(500.0, W, cfg)
    mods = np.stack([mod, mod]).astype(np.float32)
    x, xc = dev(x0), dev(xc0)
    m.dit_block_forward(1, x, xc, dev(mods), None, 2, grid, L)
    m.dit_synchronize()
    gx, gc = host(x), host(xc)
    rows = _rows(L + N, extra=range(L - 3, L + 3))   # both streams and their boundary
    angles = O.rope_angles(O.token_positions(grid), cfg["rope_axes"], cfg["rope_theta"])
    for b in range(2):
        ref = O.block_joint(x0[b], xc0[b], mods[b], W, 1, cfg, grid, rows=rows, angles=angles)
        got = np.concatenate([gc[b], gx[b]])[rows]
        assert_block_close(got, ref)


def _image_block_case(cfg, W, m, latent, batch, check, seed):
    """The dual-stream block at `latent` with `batch` rows of the CFG batch;
    sampled rows of the batch items in `check` against the oracle."""
    grid = synth.grid(cfg, latent)
    N, L, D = int(np.prod(grid)), cfg["cond_len"], cfg["hidden"]
    rng = np.random.default_rng(seed)
    x0 = (rng.standard_normal((batch, N, D)) * 0.2).astype(np.float32)
    xc0 = synth.round_bf16(rng.standard_normal((batch, L, D)).astype(np.float32))
    mods = np.stack([O.timestep_modulation(t, W, cfg) for t in np.linspace(900.0, 100.0, batch)]).astype(np.float32)
    x, xc = dev(x0), dev(xc0)
    m.dit_block_forward(1, x, xc, dev(mods), None, batch, grid, L)
    m.dit_synchronize()
    gx, gc = host(x), host(xc)
    rows = _rows(L + N, extra=range(L - 2, L + 2))
    angles = O.rope_angles(O.token_positions(grid), cfg["rope_axes"], cfg["rope_theta"])
    for b in check:
        ref = O.block_joint(x0[b], xc0[b], mods[b], W, 1, cfg, grid, rows=rows, angles=angles)
        assert_block_close(np.concatenate([gc[b], gx[b]])[rows], ref)


def test_image_block_sweep_batch4(image_model):
    """Sweep point: batch 4 (two requests' CFG pairs) at 4096 + 512 tokens;
    first and last batch items checked."""
    cfg, W, m = image_model
    _image_block_case(cfg, W, m, cfg["latent"], 4, (0, 3), seed=21)


def test_image_block_sweep_16384_tokens(image_model):
    """Sweep point: 16384 image tokens (128 x 128 grid) + 512 condition
    tokens, batch 2."""
    cfg, W, m = image_model
    _image_block_case(cfg, W, m, (1, 256, 256), 2, (1,), seed=22)


def test_image_loop_full_tokens_reduced_depth(image_model):
    """The whole denoise loop at the full 4096 + 512 token count, depth 2,
    two Euler steps with CFG: final latents against the full oracle loop."""
    cfg, W, m = image_model
    L = cfg["cond_len"]
    lat = synth.make_latent(cfg, batch=1, seed=5)
    cond = synth.make_cond(cfg, batch=1, seed=6)
    unc = np.zeros_like(cond)
    sig = O.shift_sigma(O.sigma_schedule(2), cfg["shift"]).astype(np.float32)
    x = dev(lat)
    m.dit_denoise_loop(x, 1, cfg["latent"], dev(cond), dev(unc), L, sig, cfg["guidance"])
    m.dit_synchronize()
    got = host(x)[0]
    ref = O.denoise_loop(lat[0], cond[0], unc[0], W, cfg, sig.astype(np.float64), cfg["guidance"])
    assert cosine(got, ref) >= COS_BF16_LOOP
    assert cosine(got - lat[0], ref - lat[0]) >= 0.99


def test_video_loop_bf16_tracks_fp32_path_full_tokens():
    """Transitive full-loop check at the video token count: the bf16
    production path against the fp32 test-precision path (itself pinned to
    the oracle at 1e-4 on complete loops), same bf16-rounded weights and
    condition, depth 4, two CFG + Euler steps over 32760 tokens."""
    cfg_b = synth.config("video", depth=4)
    cfg_f = dict(cfg_b, precision=synth.PREC_F32)
    W = synth.make_weights(cfg_b, seed=41)  # bf16-rounded values, read as fp32 by the test path
    L = cfg_b["cond_len"]
    lat = synth.make_latent(cfg_b, batch=1, seed=42)
    cond = synth.make_cond(cfg_b, batch=1, seed=43)
    unc = np.zeros_like(cond)
    sig = O.shift_sigma(O.sigma_schedule(cfg_b["steps"]), cfg_b["shift"])[:3].astype(np.float32)
    out = {}
    for name, cfg in (("bf16", cfg_b), ("fp32", cfg_f)):
        m = make_model(cfg, W)
        x = dev(lat)
        m.dit_denoise_loop(x, 1, cfg["latent"], dev(cond), dev(unc), L, sig, cfg["guidance"],
                           flags=dit.LOOP_PARTIAL_SCHEDULE)
        m.dit_synchronize()
        out[name] = host(x)[0]
        m.close()
    assert np.isfinite(out["bf16"]).all()
    assert cosine(out["bf16"], out["fp32"]) >= COS_BF16_LOOP
    assert cosine(out["bf16"] - lat[0], out["fp32"] - lat[0]) >= 0.99


def test_video_embed_head_and_cfg_euler_full_size(video_block):
    """Patch embedding, final layer and guidance + Euler at the full video
    latent size (16 x 21 x 60 x 104)."""
    cfg, W, m = video_block
    thw = cfg["latent"]
    grid = synth.grid(cfg)
    N, D = int(np.prod(grid)), cfg["hidden"]
    lat = synth.make_latent(cfg, batch=2, seed=7)
    x = empty(2, N, D)
    m.dit_patch_embed(dev(lat), 2, thw, x)
    m.dit_synchronize()
    gx = host(x)
    rows = _rows(N)
    for b in range(2):
        lat_b = synth.round_bf16(lat[b]).astype(np.float64)
        assert rel_max_err(gx[b][rows], O.patch_embed(lat_b, W, cfg)[rows]) < 1e-3
    mods = np.stack([O.timestep_modulation(t, W, cfg) for t in (900.0, 100.0)]).astype(np.float32)
    v = empty(2, cfg["in_channels"], *thw)
    xs = (gx * 0.5).astype(np.float32)
    m.dit_final_layer(dev(xs), dev(mods), 2, thw, v)
    m.dit_synchronize()
    gv = host(v)
    for b in range(2):
        ref = O.unpatchify(O.final_layer(xs[b], mods[b], W, cfg), cfg["patch"], (cfg["in_channels"],) + thw)
        assert_block_close(gv[b], ref)
    n = gv[0].size
    out = empty(n)
    dit.cfg_combine(dev(gv[0]), dev(gv[1]), 5.0, out, n)
    xl = dev(lat[0])
    dit.flow_euler_step(xl, out, 0.7, 0.65, n)
    ref = O.euler_step(lat[0], O.cfg_combine(gv[0], gv[1], 5.0), 0.7, 0.65)
    np.testing.assert_allclose(host(xl).reshape(ref.shape), ref, rtol=0, atol=1e-4)


def test_image_block_sweep_batch8(image_model):
    """Sweep point: batch 8 (four requests' CFG pairs) at 4096 + 512 tokens;
    first and last batch items checked."""
    cfg, W, m = image_model
    _image_block_case(cfg, W, m, cfg["latent"], 8, (0, 7), seed=23)


def test_image_block_sweep_1024_tokens(image_model):
    """Sweep point: 1024 image tokens (32 x 32 grid) + 512 condition tokens."""
    cfg, W, m = image_model
    _image_block_case(cfg, W, m, (1, 64, 64), 2, (0, 1), seed=24)


def test_image_block_sweep_65536_tokens(image_model):
    """Sweep point: 65536 image tokens (256 x 256 grid) + 512 condition tokens,
    batch 2: 344 key tiles of 192, so the attention runs the one-CTA-per-item
    kernel for long key ranges rather than the persistent walk used for short
    ones."""
    cfg, W, m = image_model
    _image_block_case(cfg, W, m, (1, 512, 512), 2, (0,), seed=25)


def test_fp8_video_block_full_size():
    """DIT_PREC_FP8 at the video block's full size (32760 tokens, batch 2),
    sampled rows against the oracle."""
    from tests.gpu_util import assert_fp8_block_close
    cfg = synth.config("video", depth=1, precision=synth.PREC_FP8)
    W = synth.make_weights(cfg, seed=0)
    m = make_model(cfg, W)
    grid = synth.grid(cfg)
    N, L = int(np.prod(grid)), cfg["cond_len"]
    lat = synth.make_latent(cfg, batch=1, seed=1)
    ctx = np.concatenate([synth.make_cond(cfg, batch=1, seed=2), np.zeros((1, L, cfg["cond_dim"]), np.float32)])
    x0 = np.stack([O.patch_embed(lat[0], W, cfg)] * 2).astype(np.float32)
    mod = O.timestep_modulation(700.0, W, cfg)
    mods = np.stack([mod, mod]).astype(np.float32)
    x = dev(x0)
    m.dit_block_forward(0, x, None, dev(mods), dev(ctx), 2, grid, L)
    m.dit_synchronize()
    got = host(x)
    rows = _rows(N, extra=range(N - 120, N - 110))
    angles = O.rope_angles(O.token_positions(grid), cfg["rope_axes"], cfg["rope_theta"])
    for b in range(2):
        ref = O.block_cross(x0[b], mods[b], ctx[b], W, 0, cfg, grid, rows=rows, angles=angles)
        assert_fp8_block_close(got[b][rows], ref, x0[b][rows], case=f"fp8 video block b{b}")
    m.close()


def test_fp8_video_loop_tracks_fp32_path_full_tokens():
    """The fp8 video loop at the full token count (depth 4, two CFG + Euler
    steps) against the fp32 test path with the same bf16-valued weights."""
    from tests.gpu_util import COS_FP8_LOOP, log_errors
    cfg_8 = synth.config("video", depth=4, precision=synth.PREC_FP8)
    cfg_f = dict(cfg_8, precision=synth.PREC_F32)
    W = synth.make_weights(cfg_8, seed=41)
    L = cfg_8["cond_len"]
    lat = synth.make_latent(cfg_8, batch=1, seed=42)
    cond = synth.make_cond(cfg_8, batch=1, seed=43)
    unc = np.zeros_like(cond)
    sig = O.shift_sigma(O.sigma_schedule(cfg_8["steps"]), cfg_8["shift"])[:3].astype(np.float32)
    out = {}
    for name, cfg in (("fp8", cfg_8), ("fp32", cfg_f)):
        m = make_model(cfg, W)
        x = dev(lat)
        m.dit_denoise_loop(x, 1, cfg["latent"], dev(cond), dev(unc), L, sig, cfg["guidance"],
                           flags=dit.LOOP_PARTIAL_SCHEDULE)
        m.dit_synchronize()
        out[name] = host(x)[0]
        m.close()
    c_all, c_upd = cosine(out["fp8"], out["fp32"]), cosine(out["fp8"] - lat[0], out["fp32"] - lat[0])
    log_errors("fp8 video loop depth 4", cos=c_all, cos_update=c_upd)
    assert c_all >= COS_FP8_LOOP and c_upd >= COS_FP8_LOOP - 0.01, (c_all, c_upd)


def test_fp8_image_block_full_size():
    """DIT_PREC_FP8 on the dual-stream image block at full size (4096 image +
    512 condition tokens, batch 2): the paired e4m3 GEMMs carry their own row
    scales per stream; sampled rows of both streams against the oracle."""
    from tests.gpu_util import assert_fp8_block_close
    cfg = synth.config("image", depth=1, precision=synth.PREC_FP8)
    W = synth.make_weights(cfg, seed=0)
    m = make_model(cfg, W)
    grid = synth.grid(cfg)
    N, L, D = int(np.prod(grid)), cfg["cond_len"], cfg["hidden"]
    rng = np.random.default_rng(33)
    x0 = (rng.standard_normal((2, N, D)) * 0.2).astype(np.float32)
    xc0 = np.concatenate([synth.make_cond(cfg, batch=1, seed=34), np.zeros((1, L, D), np.float32)])
    mod = O.timestep_modulation(400.0, W, cfg)
    mods = np.stack([mod, mod]).astype(np.float32)
    x, xc = dev(x0), dev(xc0)
    m.dit_block_forward(0, x, xc, dev(mods), None, 2, grid, L)
    m.dit_synchronize()
    gx, gc = host(x), host(xc)
    rows = _rows(L + N, extra=range(L - 3, L + 3))
    angles = O.rope_angles(O.token_positions(grid), cfg["rope_axes"], cfg["rope_theta"])
    for b in range(2):
        ref = O.block_joint(x0[b], xc0[b], mods[b], W, 0, cfg, grid, rows=rows, angles=angles)
        got = np.concatenate([gc[b], gx[b]])[rows]
        inp = np.concatenate([xc0[b], x0[b]])[rows]
        assert_fp8_block_close(got, ref, inp, case=f"fp8 image block b{b}")
    m.close()
