"""dit_timestep_modulation_noalloc: the entry point for callers that may not
allocate device memory during a call (a serving thread that must not trigger
the implicit synchronisation of cudaMalloc/cudaFree, or a process whose
device memory all belongs to its own pool).

Checked on two calls in a row (the fixed scratch keeps the previous call's
contents, and the second call is the smaller one): the result against the
CPU oracle and against the allocating dit_timestep_modulation, and that the
calls take no device memory at all.  The memory check runs in a fresh
process, so that the first no-allocation call of that process is the one
measured (module loading would show up there), whether this file runs alone
or after the rest of the suite.  Collected last so that a failure here
cannot hide the rest of the suite."""
import json
import os
import subprocess
import sys

import numpy as np
import pytest

from diffusion_transformer_denoising_gb300 import dit, synth
from tests.gpu_util import TOL_F32, empty, make_model

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

_CHILD = r"""
import json, sys
import numpy as np
import torch
sys.path.insert(0, sys.argv[1])
from diffusion_transformer_denoising_gb300 import dit, synth
from oracle import dit_oracle as O
from tests.gpu_util import host, rel_max_err, small_bf16_cfg

which = sys.argv[2]
torch.cuda.set_device(0)
cfg = synth.config("tiny") if which == "tiny_fp32" else small_bf16_cfg(depth=1)
W = synth.make_weights(cfg, seed=31)
m = dit.DiT(cfg)
m.load_weights(W)
calls = [np.array([0.0, 250.0, 700.0, 1000.0], np.float32), np.array([999.5, 3.25], np.float32)]
outs = [torch.full((len(t), 6 * cfg["hidden"]), float("nan"), device="cuda") for t in calls]
torch.cuda.synchronize()
free_before = torch.cuda.mem_get_info()[0]
dit.dit_debug_fail_alloc_after(1)          # any allocation by the library would now fail the call
for t, o in zip(calls, outs):
    m.dit_timestep_modulation_noalloc(t, o)
m.dit_synchronize()
torch.cuda.synchronize()
free_after = torch.cuda.mem_get_info()[0]
dit.dit_debug_fail_alloc_after(0)
err_oracle, err_alloc = [], []
for t, o in zip(calls, outs):
    got = host(o)
    ref = torch.full_like(o, float("nan"))
    m.dit_timestep_modulation(t, ref)
    m.dit_synchronize()
    err_alloc.append(rel_max_err(got, host(ref)))
    err_oracle.append(max(rel_max_err(got[i], O.timestep_modulation(float(t[i]), W, cfg)) for i in range(len(t))))
m.close()
print(json.dumps(dict(free_before=free_before, free_after=free_after, err_oracle=err_oracle, err_alloc=err_alloc)))
"""


@pytest.mark.parametrize("which", ["tiny_fp32", "bf16"])
def test_noalloc_two_calls_match_oracle_and_allocate_nothing(which):
    r = subprocess.run([sys.executable, "-c", _CHILD, ROOT, which], cwd=ROOT, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    res = json.loads(r.stdout.strip().splitlines()[-1])
    # the device's free memory is unchanged across the first two calls of the process
    assert res["free_after"] == res["free_before"], res
    for e in res["err_oracle"]:
        assert e < TOL_F32, res
    for e in res["err_alloc"]:
        assert e < TOL_F32, res


def test_noalloc_rejects_sizes_beyond_the_fixed_scratch():
    cfg = synth.config("tiny")
    m = make_model(cfg, synth.make_weights(cfg, seed=32))
    t = np.zeros(dit.NOALLOC_MAX_BATCH + 1, np.float32)
    with pytest.raises(dit.DitError) as e:
        m.dit_timestep_modulation_noalloc(t, empty(len(t), 6 * cfg["hidden"]))
    assert e.value.status == dit.DIT_ERR_INVALID_ARG
    assert "scratch limit" in str(e.value)
    m.close()
