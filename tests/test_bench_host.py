"""Host-side logic of bench.py: FLOP accounting and the multi-rank aggregation
(world size 2 over gloo on CPU; one request per rank, no data-path collective)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from diffusion_transformer_denoising_gb300 import synth


def test_video_step_flops():
    cfg = synth.config("video")
    fl = bench.step_flops(cfg, 2, 32760, 512)
    assert abs(fl["total"] - 5.66e14) / 5.66e14 < 0.01
    assert abs(fl["attn_self"] / fl["total"] - 0.70) < 0.01      # attention dominates the video step
    img = bench.step_flops(synth.config("image"), 2, 4096, 512)
    assert abs(img["total"] - 7.83e13) / 7.83e13 < 0.02


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    elapsed = [2.0, 3.0][rank]
    t, v = bench.aggregate(elapsed, 10, world, dist)
    q.put((rank, t, v))
    dist.barrier()
    dist.destroy_process_group()


def test_aggregate_max_over_ranks_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for _, t, v in res:
        assert t == 3.0                 # slowest rank sets the time
        assert v == pytest.approx(10 * 2 / 3.0)   # whole-job steps / max time


def test_single_rank_aggregate_is_identity():
    t, v = bench.aggregate(2.5, 5, 1, None)
    assert t == 2.5 and v == pytest.approx(2.0)


def test_reference_line_states_its_extrapolation(monkeypatch, capsys):
    """The reference arm's line: `config` is the GPU arm's object, the value
    is labelled extrapolated, `steps` counts the samples that ran and
    `ms_per_step` is their measured wall time (so steps x ms_per_step is the
    time the arm actually spent), with the extrapolated full step beside it."""
    import argparse
    import json
    calls = []

    def fake_sample(workload):
        calls.append(workload)
        return dict(t_block=1.0, t_step=60.0, sample_s=0.001, sample="s", cores=4)

    monkeypatch.setattr(bench, "cpu_oracle_sample", fake_sample)
    monkeypatch.setattr(bench, "_oracle_block_weights", lambda w: None)
    bench.run_reference(argparse.Namespace(gpus=1, steps=3, warmup=1, workload="video"))
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["extrapolated"] is True
    assert line["config"] == bench.workload_config("video", 3, 1)
    assert line["steps"] == 3 and len(calls) == 4            # warm-up + timed samples
    assert line["ms_per_step"] * line["steps"] < 1e3         # the time that ran, not the extrapolation
    assert line["ms_per_full_step_extrapolated"] == pytest.approx(60.0e3)
    assert line["value"] == pytest.approx(1 / 60.0)
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["extrapolated"] is True


def test_measured_peaks_carry_the_clock_of_the_sustained_figure(tmp_path, monkeypatch):
    """The roofline's clock-scaled fraction needs the median SM clock under
    which the sustained bf16 peak was measured; without the file the
    fallback figures carry none (and the fraction is then left out)."""
    import json
    import bench
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps(
        {"hbm_gbs": 6000.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
         "clocks_under_load": {"sm_mhz_median": 1455.0}}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    p = bench.measured_peaks()
    assert p["source"] == "measured" and p["sustained_sm_mhz"] == 1455.0
    (tmp_path / "MEASURED_PEAKS.json").unlink()
    p = bench.measured_peaks()
    assert p["source"] == "fallback" and p["sustained_sm_mhz"] is None
