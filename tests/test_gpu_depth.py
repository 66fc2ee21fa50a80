"""Parity at the full depth of the two large workloads.

The 30-block video loop (32760 tokens, 50 steps) is far beyond what the
float64 oracle can run on host cores, so it is checked teacher-forced: at
steps 0, 24 and 49 of the shift-5 schedule the GPU runs the step block by
block through the C ABI (dit_timestep_modulation, dit_patch_embed,
dit_block_forward), and at every one of the 30 blocks the oracle takes the
GPU's block input (all tokens, for the keys and values) and computes the
block output for 64 sampled rows.  Between the checked steps the latent
advances through dit_denoise_loop itself.

The 30-block image loop (4096 + 512 joint tokens) runs complete, in bf16 and
in fp8 precision, against the fp32 test-precision path (pinned to the oracle
at 1e-4 on complete loops), with the same bf16-valued weights.
"""
import time

import numpy as np
import pytest

from diffusion_transformer_denoising_gb300 import dit, synth
from oracle import dit_oracle as O
from tests.gpu_util import COS_BF16_LOOP, assert_block_close, cosine, dev, empty, host, log_errors, make_model

pytestmark = pytest.mark.gpu


def _sample_rows(n, k=64):
    r = set(np.linspace(0, n - 1, k - 6).astype(int).tolist()) | {0, 1, n - 1, n - 2, n - 60, n - 100}
    return np.array(sorted(r))


def test_video_loop_teacher_forced_every_block():
    import torch
    cfg = synth.config("video")
    W = synth.make_weights(cfg, seed=71)
    m = make_model(cfg, W)
    grid = synth.grid(cfg)
    thw, L, D, C = cfg["latent"], cfg["cond_len"], cfg["hidden"], cfg["in_channels"]
    N = int(np.prod(grid))
    lat0 = synth.make_latent(cfg, batch=1, seed=72)
    cond = synth.make_cond(cfg, batch=1, seed=73)
    unc = np.zeros_like(cond)
    ctx2 = dev(np.concatenate([cond, unc]))
    sig = O.shift_sigma(O.sigma_schedule(cfg["steps"]), cfg["shift"]).astype(np.float32)
    angles = O.rope_angles(O.token_positions(grid), cfg["rope_axes"], cfg["rope_theta"])
    rows = _sample_rows(N)
    lat = dev(lat0)
    x = empty(2, N, D)
    mods = empty(2, 6 * D)
    done = 0
    worst = 0.0
    for step, b in ((0, 0), (24, 1), (49, 0)):
        if step > done:   # advance the latent through the loop itself
            m.dit_denoise_loop(lat, 1, thw, dev(cond), dev(unc), L, sig[done:step + 1].copy(), cfg["guidance"],
                               flags=dit.LOOP_PARTIAL_SCHEDULE)
            done = step
        t = float(cfg["timestep_scale"] * sig[step])
        m.dit_timestep_modulation(np.array([t, t], np.float32), mods)
        lat2 = torch.cat([lat, lat])
        m.dit_patch_embed(lat2, 2, thw, x)
        mo = O.timestep_modulation(t, W, cfg)
        ctx_b = cond[0] if b == 0 else unc[0]
        for blk in range(cfg["depth"]):
            x_in = host(x[b])
            m.dit_block_forward(blk, x, None, mods, ctx2, 2, grid, L)
            m.dit_synchronize()
            got = host(x[b])[rows]
            ref = O.block_cross(x_in, mo, ctx_b, W, blk, cfg, grid, rows=rows, angles=angles)
            assert_block_close(got, ref, case=f"video step {step} block {blk} pass {b}")
            worst = max(worst, float(np.sqrt(np.mean((got - ref) ** 2) / np.mean(ref ** 2))))
        # the step itself through the loop (the block-by-block pass above only checked it)
        m.dit_denoise_loop(lat, 1, thw, dev(cond), dev(unc), L, sig[step:step + 2].copy(), cfg["guidance"],
                           flags=dit.LOOP_PARTIAL_SCHEDULE)
        done = step + 1
    m.dit_synchronize()
    assert done == cfg["steps"]
    out = host(lat)
    assert np.isfinite(out).all()
    log_errors("video teacher-forced worst block", rms=worst)
    m.close()


def test_image_loop_full_depth_all_steps_tracks_fp32_path():
    """The complete image loop: 30 dual-stream blocks, 30 steps of the shift-3
    schedule, CFG scale 4, 4096 + 512 tokens; bf16 production path against
    the fp32 test-precision path, final latents cosine >= 0.999; the fp8
    precision against the same fp32 result, cosine >= 0.99."""
    import torch
    from tests.gpu_util import COS_FP8_LOOP
    cfg_b = synth.config("image")
    cfg_f = dict(cfg_b, precision=synth.PREC_F32)
    cfg_8 = dict(cfg_b, precision=synth.PREC_FP8)
    Wt = synth.make_weights_torch(cfg_b, seed=81, device="cuda")   # bf16 values; the fp32 model widens them
    L = cfg_b["cond_len"]
    lat = synth.make_latent(cfg_b, batch=1, seed=82)
    cond = synth.make_cond(cfg_b, batch=1, seed=83)
    unc = np.zeros_like(cond)
    sig = O.shift_sigma(O.sigma_schedule(cfg_b["steps"]), cfg_b["shift"]).astype(np.float32)
    out, secs = {}, {}
    for name, cfg in (("bf16", cfg_b), ("fp8", cfg_8), ("fp32", cfg_f)):
        m = dit.DiT(cfg)
        m.load_weights(Wt)
        x = dev(lat)
        t0 = time.perf_counter()
        m.dit_denoise_loop(x, 1, cfg["latent"], dev(cond), dev(unc), L, sig, cfg["guidance"])
        m.dit_synchronize()
        secs[name] = time.perf_counter() - t0
        out[name] = host(x)[0]
        m.close()
        torch.cuda.empty_cache()
    del Wt
    c_all, c_upd = cosine(out["bf16"], out["fp32"]), cosine(out["bf16"] - lat[0], out["fp32"] - lat[0])
    f_all, f_upd = cosine(out["fp8"], out["fp32"]), cosine(out["fp8"] - lat[0], out["fp32"] - lat[0])
    log_errors("image full loop", cos=c_all, cos_update=c_upd, fp8_cos=f_all, fp8_cos_update=f_upd,
               bf16_s=secs["bf16"], fp8_s=secs["fp8"], fp32_s=secs["fp32"])
    assert np.isfinite(out["bf16"]).all() and np.isfinite(out["fp8"]).all()
    assert c_all >= COS_BF16_LOOP, (c_all, c_upd)
    assert c_upd >= 0.99, (c_all, c_upd)
    # fp8 precision over the complete loop (reading R16's loop bound)
    assert f_all >= COS_FP8_LOOP and f_upd >= COS_FP8_LOOP - 0.01, (f_all, f_upd)
