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
