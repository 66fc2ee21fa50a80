"""Host-side checks of the C ABI that need no GPU: the library loads, exports
every function include/dit.h declares, enumerates the same parameter list as
the input generator, and rejects bad arguments before touching a device."""
import ctypes as C
import os
import re

import numpy as np
import pytest

from diffusion_transformer_denoising_gb300 import dit, synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    if not os.path.exists(dit.LIB_PATH):
        from diffusion_transformer_denoising_gb300 import build
        build.build()
    return dit.lib()


def _declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(\w+)\s*\(", src, flags=re.M))
    return names


def test_library_exports_every_declared_function(L):
    declared = _declared_functions()
    assert {"dit_create", "dit_denoise_loop", "cfg_combine", "flow_euler_step"} <= declared
    for name in declared:
        assert hasattr(L, name), name
    assert set(dit.EXPORTS) == declared


@pytest.mark.parametrize("name", ["tiny", "video", "image"])
def test_param_list_matches_generator(L, name):
    cfg = synth.config(name)
    specs = synth.param_specs(cfg)
    assert dit.dit_num_params(cfg) == len(specs)
    for i in (0, 1, 5, 6, len(specs) // 2, len(specs) - 3, len(specs) - 1):
        assert dit.dit_param_info(cfg, i) == (specs[i][0], tuple(specs[i][1]))


def test_param_count_matches_model_scale():
    n = lambda c: sum(int(np.prod(s)) for _, s in synth.param_specs(synth.config(c)))
    assert 1.3e9 < n("video") < 1.5e9      # ~1.3B video DiT
    assert 6.5e9 < n("image") < 7.2e9      # ~7B image DiT


@pytest.mark.parametrize("field,value,status", [
    ("heads", 5, dit.DIT_ERR_SHAPE),              # heads * head_dim != hidden
    ("rope_axes", (2, 2, 2), dit.DIT_ERR_INVALID_ARG),  # axes do not sum to head_dim
    ("rope_axes", (1, 15, 16), dit.DIT_ERR_INVALID_ARG),  # odd axis
    ("cond_mode", 7, dit.DIT_ERR_INVALID_ARG),
    ("precision", 3, dit.DIT_ERR_INVALID_ARG),
    ("freq_dim", 255, dit.DIT_ERR_INVALID_ARG),
    ("depth", 0, dit.DIT_ERR_INVALID_ARG),
])
def test_create_rejects_bad_config_before_gpu(L, field, value, status):
    cfg = synth.config("tiny", **{field: value})
    with pytest.raises(dit.DitError) as e:
        dit.DiT(cfg)
    assert e.value.status == status


def test_bf16_needs_head_dim_128(L):
    with pytest.raises(dit.DitError) as e:
        dit.DiT(synth.config("tiny", precision=synth.PREC_BF16))
    assert e.value.status == dit.DIT_ERR_SHAPE


def test_joint_mode_needs_cond_dim_equal_hidden(L):
    with pytest.raises(dit.DitError) as e:
        dit.DiT(synth.config("image", cond_dim=1024))
    assert e.value.status == dit.DIT_ERR_SHAPE


def test_elementwise_calls_reject_bad_arguments_on_host(L):
    with pytest.raises(dit.DitError) as e:
        dit.cfg_combine(None, None, 5.0, None, 10)
    assert e.value.status == dit.DIT_ERR_INVALID_ARG
    with pytest.raises(dit.DitError) as e:
        dit.flow_euler_step(1024, 2048, float("nan"), 0.0, 4)
    assert e.value.status == dit.DIT_ERR_INVALID_ARG
    with pytest.raises(dit.DitError):
        dit.cfg_combine(1024, 2048, float("inf"), 4096, 4)
    # empty input is a valid no-op
    dit.cfg_combine(None, None, 5.0, None, 0)


def test_status_strings(L):
    for s in range(7):
        assert L.dit_status_string(s)
