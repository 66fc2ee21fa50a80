"""The debug build (libdit_debug.so, compiled with -DDIT_DEBUG_BOUNDS) checks
tile coordinates and indices on the device (GEMM tiles and head-major store
boxes, attention items and key tiles, LayerNorm rows and modulation entries)
and records the first failure in the model's error word instead of touching
memory; dit_synchronize then reports it.  Run over the small odd shapes of
the CPU comparisons (ragged token counts, a single token, short and
single-token conditions, K and N tails, both conditioning modes, GEMMs on
single CTAs and on CTA pairs, a key range long enough for the 192-key-tile
attention, complete loops), every check must pass and every result must still match the oracle.  Runs in a child process because
the library a process loads is fixed at its first use."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

_CHILD = r"""
import sys
import numpy as np
import torch
sys.path.insert(0, sys.argv[1])
from diffusion_transformer_denoising_gb300 import dit, synth
from oracle import dit_oracle as O
from tests.gpu_util import (COS_BF16_LOOP, TOL_F32, assert_block_close, assert_fp8_block_close, cosine, dev, host,
                            rel_max_err, small_bf16_cfg)

assert dit.LIB_PATH.endswith("libdit_debug.so"), dit.LIB_PATH
torch.cuda.set_device(0)
n_checked = 0

def model(cfg, W):
    m = dit.DiT(cfg)
    m.load_weights(W)
    return m

# blocks: ragged grids, short conditions, K/N tails, both modes; GEMMs of
# width a multiple of 256 on CTA pairs by main-loop length (these short K
# give single CTAs) and then with pairs forced on
import itertools
for pairs, (mode, grid, L, kw) in itertools.product((1, 2), (
        (synth.COND_CROSS, (2, 9, 7), 5, {}), (synth.COND_CROSS, (3, 10, 13), 77, {}),
        (synth.COND_CROSS, (1, 6, 11), 37, dict(mlp=648, cond_dim=200)),
        (synth.COND_JOINT, (1, 7, 9), 33, {}), (synth.COND_JOINT, (1, 12, 20), 64, {}),
        (synth.COND_CROSS, (1, 1, 1), 1, {}), (synth.COND_JOINT, (1, 1, 1), 1, {}),
        (synth.COND_CROSS, (3, 10, 13), 77, dict(precision=synth.PREC_FP8)),
        (synth.COND_JOINT, (1, 7, 9), 33, dict(precision=synth.PREC_FP8)))):
    dit.dit_debug_gemm_cta_pairs(pairs)
    cfg = small_bf16_cfg(mode, depth=1, **kw)
    W = synth.make_weights(cfg, seed=101)
    m = model(cfg, W)
    N = int(np.prod(grid))
    rng = np.random.default_rng(N + L)
    x0 = (rng.standard_normal((2, N, cfg["hidden"])) * 0.5).astype(np.float32)
    mods = np.stack([O.timestep_modulation(t, W, cfg) for t in (210.0, 840.0)])
    ctx = synth.make_cond(cfg, batch=2, seed=L, length=L)
    x = dev(x0)
    if mode == synth.COND_CROSS:
        m.dit_block_forward(0, x, None, dev(mods), dev(ctx), 2, grid, L)
    else:
        xc = dev(ctx)
        m.dit_block_forward(0, x, xc, dev(mods), None, 2, grid, L)
    m.dit_synchronize()          # raises DitError if a bounds check failed
    got = host(x)
    for b in range(2):
        if mode == synth.COND_CROSS:
            ref = O.block_cross(x0[b], mods[b], ctx[b], W, 0, cfg, grid)
        else:
            ref = O.block_joint(x0[b], ctx[b], mods[b], W, 0, cfg, grid)[0]
        if cfg["precision"] == synth.PREC_FP8:
            assert_fp8_block_close(got[b], ref, x0[b], case=f"debug build fp8 block {mode} {grid} {L}")
        else:
            assert_block_close(got[b], ref, case=f"debug build block {mode} {grid} {L}")
        n_checked += 1
    m.close()

# a key range long enough for the one-CTA-per-query-tile attention (8600
# tokens: 45 key tiles of 192, the last one partial), sampled rows
dit.dit_debug_gemm_cta_pairs(1)
cfg = small_bf16_cfg(synth.COND_CROSS, depth=1)
W = synth.make_weights(cfg, seed=105)
m = model(cfg, W)
grid, L = (1, 86, 100), 40
N = int(np.prod(grid))
rng = np.random.default_rng(106)
x0 = (rng.standard_normal((2, N, cfg["hidden"])) * 0.5).astype(np.float32)
mods = np.stack([O.timestep_modulation(t, W, cfg) for t in (330.0, 770.0)])
ctx = synth.make_cond(cfg, batch=2, seed=107, length=L)
x = dev(x0)
m.dit_block_forward(0, x, None, dev(mods), dev(ctx), 2, grid, L)
m.dit_synchronize()
got = host(x)
rows = np.array(sorted(set(np.linspace(0, N - 1, 24).astype(int).tolist()) | set(range(N - 26, N))))
for b in range(2):
    ref = O.block_cross(x0[b], mods[b], ctx[b], W, 0, cfg, grid, rows=rows)
    assert_block_close(got[b][rows], ref, case="debug build long key range")
    n_checked += 1
m.close()

# complete loops: tiny fp32 and bf16 in both modes
for name, thw, L in (("tiny", None, 16), ("cross", (2, 12, 18), 40), ("joint", (1, 24, 20), 40)):
    if name == "tiny":
        cfg = synth.config("tiny")
        thw = cfg["latent"]
    else:
        cfg = small_bf16_cfg(synth.COND_CROSS if name == "cross" else synth.COND_JOINT)
    W = synth.make_weights(cfg, seed=102)
    m = model(cfg, W)
    lat = synth.make_latent(cfg, batch=1, seed=103, latent=thw)
    cond = synth.make_cond(cfg, batch=1, seed=104, length=L)
    unc = np.zeros_like(cond)
    sig = O.shift_sigma(O.sigma_schedule(3), 3.0).astype(np.float32)
    x = dev(lat)
    m.dit_denoise_loop(x, 1, thw, dev(cond), dev(unc), L, sig, 4.0)
    m.dit_synchronize()
    got = host(x)[0]
    ref = O.denoise_loop(lat[0], cond[0], unc[0], W, cfg, sig.astype(np.float64), 4.0)
    if name == "tiny":
        assert rel_max_err(got, ref) < TOL_F32
    else:
        assert cosine(got, ref) >= COS_BF16_LOOP
    n_checked += 1
    m.close()
print("debug build checked", n_checked)
"""


def test_debug_bounds_build_on_odd_shapes():
    from diffusion_transformer_denoising_gb300 import build
    srcs = [os.path.join(build.CSRC, f) for f in os.listdir(build.CSRC)]
    if not os.path.exists(build.LIB_DEBUG) or \
            os.path.getmtime(build.LIB_DEBUG) < max(os.path.getmtime(f) for f in srcs):
        build.build(debug=True)
    env = dict(os.environ, DIT_LIB=build.LIB_DEBUG)
    r = subprocess.run([sys.executable, "-c", _CHILD, ROOT], cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=900)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    assert "debug build checked 41" in r.stdout, r.stdout[-2000:]
