"""Helpers shared by the GPU tests: device upload, model construction from
seeded weights, and the tolerance checks against the oracle."""
import numpy as np

from diffusion_transformer_denoising_gb300 import dit, synth


def torch():
    import torch as t
    return t


def dev(a):
    t = torch()
    return t.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def host(t):
    torch().cuda.synchronize()
    return t.detach().float().cpu().numpy().astype(np.float64)


def empty(*shape):
    t = torch()
    return t.full(shape, float("nan"), dtype=t.float32, device="cuda")


def make_model(cfg, W):
    m = dit.DiT(cfg)
    m.load_weights(W)
    return m


def rel_max_err(got, ref):
    """max |got - ref| / RMS(ref)."""
    ref = np.asarray(ref, np.float64)
    return float(np.max(np.abs(np.asarray(got, np.float64) - ref)) / np.sqrt(np.mean(ref ** 2)))


def cosine(a, b):
    a, b = np.ravel(a).astype(np.float64), np.ravel(b).astype(np.float64)
    return float(a @ b / np.sqrt((a @ a) * (b @ b)))


def rel_rms_err(got, ref):
    """RMS(got - ref) / RMS(ref)."""
    ref = np.asarray(ref, np.float64)
    d = np.asarray(got, np.float64) - ref
    return float(np.sqrt(np.mean(d ** 2)) / np.sqrt(np.mean(ref ** 2)))


# tolerances (fp32-accumulate test precision / bf16 production precision).
# fp32 test mode: max abs error <= 1e-4 of the output RMS.  bf16 production
# mode: the per-block output error, taken as the RMS of the error, <= 2e-2 of
# the output RMS; single elements are also held to TOL_BF16_MAX so that an
# isolated wrong value still fails (bf16 rounding of the activations alone
# puts the largest element error near 1e-2 of the RMS on 3072-wide blocks).
TOL_F32 = 1e-4
TOL_BF16_BLOCK = 2e-2
TOL_BF16_MAX = 5e-2
COS_BF16_LOOP = 0.999


def assert_block_close(got, ref, scale=1.0):
    """bf16 per-block criterion (RMS error and element bound), both scaled by `scale`."""
    rms, mx = rel_rms_err(got, ref), rel_max_err(got, ref)
    assert rms < scale * TOL_BF16_BLOCK and mx < scale * TOL_BF16_MAX, (rms, mx)


def small_bf16_cfg(mode=synth.COND_CROSS, **kw):
    """Smallest bf16 configuration the tensor-core path serves: head_dim 128,
    two heads, several GEMM and attention tiles with ragged tails."""
    c = synth.config("video" if mode == synth.COND_CROSS else "image", hidden=256, heads=2, head_dim=128,
                     mlp=640, depth=2, cond_dim=256 if mode == synth.COND_JOINT else 192,
                     rope_axes=(32, 48, 48) if mode == synth.COND_CROSS else (0, 64, 64))
    c.update(kw)
    return c
