"""dit_timestep_modulation_noalloc: the entry point for callers that may not
allocate device memory during a call.  It must give the result of the
allocating dit_timestep_modulation on the same inputs, on consecutive calls
(its fixed scratch keeps the previous call's contents), and must not grow the
library's device memory.  Collected last so a failure here cannot hide the
rest of the suite."""
import numpy as np
import pytest

from diffusion_transformer_denoising_gb300 import dit, synth
from tests.gpu_util import TOL_F32, empty, host, make_model, rel_max_err, small_bf16_cfg

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("which", ["tiny_fp32", "bf16"])
def test_noalloc_matches_allocating_call_twice(which):
    cfg = synth.config("tiny") if which == "tiny_fp32" else small_bf16_cfg(depth=1)
    m = make_model(cfg, synth.make_weights(cfg, seed=31))
    D6 = 6 * cfg["hidden"]
    for ts in ([0.0, 250.0, 700.0, 1000.0], [999.5, 3.25]):      # second call is smaller: stale tail must not matter
        t = np.array(ts, np.float32)
        got = empty(len(t), D6)
        bytes_before = m.device_bytes()
        m.dit_timestep_modulation_noalloc(t, got)
        m.dit_synchronize()
        assert m.device_bytes() == bytes_before      # the no-allocation call grew nothing
        ref = empty(len(t), D6)
        m.dit_timestep_modulation(t, ref)
        m.dit_synchronize()
        assert rel_max_err(host(got), host(ref)) < TOL_F32
    m.close()


def test_noalloc_rejects_batches_beyond_the_fixed_scratch():
    cfg = synth.config("tiny")
    m = make_model(cfg, synth.make_weights(cfg, seed=32))
    t = np.zeros(dit.NOALLOC_MAX_BATCH + 1, np.float32)
    with pytest.raises(dit.DitError) as e:
        m.dit_timestep_modulation_noalloc(t, empty(len(t), 6 * cfg["hidden"]))
    assert e.value.status == dit.DIT_ERR_INVALID_ARG
    assert "scratch limit" in str(e.value)
    m.close()
