#!/usr/bin/env python
"""Throughput of the denoiser stage (DiT forward loop + CFG + flow-Euler) on
GB300, printed as one JSON line.

A step is one denoising step of the whole hot path: timestep MLP and
modulation tables, patch embedding, every DiT block for the conditional and
unconditional passes (batch 2), the final layer, guidance and the Euler
update.  Default workload: the 30-block Wan2.1-1.3B-shaped video DiT on an
81-frame 480x832 request (16 x 21 x 60 x 104 latent, 32760 tokens, 512 text
tokens), random bf16 weights, synthetic inputs.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload video|image]
  python bench.py --impl reference ...   # the CPU oracle on a bounded sample

The headline loop is timed with one CUDA event pair around the whole call
(launches are counted, nothing else is recorded on the stream); the
per-kernel breakdown and the roofline figure come from a second, separately
timed pass with an event pair around every launch.  On one GPU the default
line also carries the 30-block image loop (`image_loop`), the video and image
workloads in fp8 precision (`fp8_loop`, `fp8_image_loop`), the seven points of the image block
batch/sequence sweep (`sweep`) and the CPU oracle timings (`cpu_baseline`).

With N > 1 (torchrun), each rank denoises its own request on its own GPU
(independent replicas, no collective on the data path); the timing is the
maximum over ranks and the value counts every rank's steps.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from diffusion_transformer_denoising_gb300 import synth  # noqa: E402

METRIC = "denoise steps/s per config; attention+GEMM TFLOP/s as % of GB300 BF16 peak"
# The pages' only figure for this path: 50 denoising steps of Wan2.1-T2V-1.3B
# (81 frames, 832x480) in 312.8 s on one H200 with layerwise offload.
PAGES_STEPS_PER_S = {"video": 50 / 312.8}

WORKLOADS = {
    "video": dict(cfg="video", desc="30-block video DiT (hidden 1536, 12x128 heads, MLP 8960), "
                                    "latent 16x21x60x104 -> 32760 tokens, 512 text tokens, CFG pair (batch 2)"),
    "image": dict(cfg="image", desc="30-block dual-stream image DiT (hidden 3072, 24x128 heads, MLP 12288), "
                                    "latent 16x128x128 -> 4096 tokens + 512 joint condition tokens, CFG pair"),
}

# ncu DRAM traffic (read + write bytes per launch) of the dominant kernel,
# valid only for the exact kernel source it was captured on.
TRAFFIC = {
    # kernel source file -> (sha256 prefix of the source, workload, bytes per launch).
    # attn_tc.cu: dram__bytes_read.sum + dram__bytes_write.sum = 606.4 + 187.2 MB
    # for one batch-2 video self-attention launch (attn_wide_kernel, the launch
    # the step runs), from an ncu capture of the block case (one launch,
    # --clock-control none).
    "attn_tc.cu": ("8782399015da528d", "video", 606381312 + 187175168),
}


def step_flops(cfg: dict, B: int, N: int, L: int, loop: bool = True) -> dict:
    """Algorithmic FLOPs of one step: 2*MACs of every block GEMM plus QK^T and
    PV of attention, split by kind.  Cross-attention keys/values are computed
    once per loop call and are not part of a step.  loop=False counts a
    stand-alone block forward (every output of both streams computed)."""
    D, F, H, hd, depth = cfg["hidden"], cfg["mlp"], cfg["heads"], cfg["head_dim"], cfg["depth"]
    if cfg["cond_mode"] == synth.COND_CROSS:
        gemm = 2 * B * N * D * (3 * D + D + D + D + 2 * F)
        attn_self = 4 * B * H * N * N * hd
        attn_cross = 4 * B * H * N * L * hd
    else:
        S = N + L
        gemm = 2 * B * S * D * (3 * D + D + 2 * F)
        attn_self = 4 * B * H * S * S * hd
        attn_cross = 0
    total_gemm = depth * gemm
    if loop and cfg["cond_mode"] != synth.COND_CROSS:
        # in the loop the last block's condition stream skips its
        # out-projection and MLP (their output is never read): not counted
        total_gemm -= 2 * B * L * D * (D + 2 * F)
    return dict(gemm=total_gemm, attn_self=depth * attn_self, attn_cross=depth * attn_cross,
                total=total_gemm + depth * (attn_self + attn_cross), attn_self_per_launch=attn_self)


def workload_config(workload: str, steps: int, world: int) -> dict:
    """The `config` object of the JSON line, identical for both arms."""
    cfg = synth.config(WORKLOADS[workload]["cfg"])
    N = int(np.prod(synth.grid(cfg)))
    return {"workload": WORKLOADS[workload]["desc"], "tokens": N, "cond_tokens": cfg["cond_len"], "cfg_batch": 2,
            "schedule": f"first {steps} of {cfg['steps']} flow steps, shift {cfg['shift']}",
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
            "l2": "inputs larger than L2 (activations >= 400 MB per step)"}


def measured_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return dict(hbm=d["hbm_gbs"], bf16=d["bf16_tflops"], bf16_sustained=d["bf16_tflops_sustained"],
                    source="measured", sustained_sm_mhz=(d.get("clocks_under_load") or {}).get("sm_mhz_median"))
    return dict(hbm=6800.0, bf16=1900.0, bf16_sustained=1700.0, source="fallback", sustained_sm_mhz=None)


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.p = None
        try:
            self.p = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                       "-lms", "200", "-i", gpu_id], stdout=subprocess.PIPE,
                                      stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.p = None

    def stop(self) -> dict:
        if self.p is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.3)
        self.p.terminate()
        out, _ = self.p.communicate(timeout=10)
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
                power.append(float(f[3]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        busy = [s for s in sm if s > 0.5 * max(sm)] or sm
        return {"sm_mhz": statistics.median(busy), "sm_max_mhz": max(smax), "samples": len(sm),
                "power_w_max": max(power) if power else None, "reasons": sorted(reasons)}


# ------------------------------------------------------------------ CPU oracle baseline
_ORACLE_WEIGHTS = {}


def _oracle_block_weights(workload: str):
    if workload not in _ORACLE_WEIGHTS:
        cfg = synth.config(WORKLOADS[workload]["cfg"])
        _ORACLE_WEIGHTS[workload] = (cfg, synth.make_weights(cfg, seed=0, blocks=[0]))
    return _ORACLE_WEIGHTS[workload]


def cpu_oracle_sample(workload: str) -> dict:
    """Time the CPU oracle on a bounded sample of one step: one block at two
    sampled query-row counts (keys/values over all tokens), split into a fixed
    and a per-row cost, extrapolated to a full step (all rows, every block,
    both CFG passes).  Returns seconds per block and per step (extrapolated),
    the seconds actually spent, and the description."""
    from oracle import dit_oracle as O
    cfg, W = _oracle_block_weights(workload)
    grid = synth.grid(cfg)
    N, L, D = int(np.prod(grid)), cfg["cond_len"], cfg["hidden"]
    rng = np.random.default_rng(0)
    x = rng.standard_normal((N, D)).astype(np.float32) * 0.5
    ctx = synth.make_cond(cfg, seed=2)[0]
    m = O.timestep_modulation(700.0, W, cfg)
    angles = O.rope_angles(O.token_positions(grid), cfg["rope_axes"], cfg["rope_theta"])
    r1, r2 = 128, 384
    times = {}
    for r in (r1, r2):
        rows = np.linspace(0, N - 1, r).astype(np.int64)
        t0 = time.perf_counter()
        if cfg["cond_mode"] == synth.COND_CROSS:
            O.block_cross(x, m, ctx, W, 0, cfg, grid, rows=rows, angles=angles)
        else:
            O.block_joint(x, ctx, m, W, 0, cfg, grid, rows=rows + L, angles=angles)
        times[r] = time.perf_counter() - t0
    per_row = max((times[r2] - times[r1]) / (r2 - r1), 0.0)
    fixed = max(times[r1] - r1 * per_row, 0.0)
    rows_all = N if cfg["cond_mode"] == synth.COND_CROSS else N + L
    t_block = fixed + rows_all * per_row
    t_step = 2 * cfg["depth"] * t_block
    sample = (f"oracle (numpy float64) on one {workload} block at {r1} and {r2} sampled query rows "
              f"(keys/values over all {rows_all} tokens), split into fixed + per-row cost and extrapolated "
              f"x{rows_all} rows x{cfg['depth']} blocks x2 CFG passes")
    return dict(t_block=t_block, t_step=t_step, sample_s=times[r1] + times[r2], sample=sample,
                cores=os.cpu_count())


def cpu_oracle_tiny_loop() -> dict:
    """The whole tiny loop (2 blocks, 64 tokens, 4 CFG + Euler steps) on the
    CPU oracle: nothing extrapolated."""
    from oracle import dit_oracle as O
    cfg = synth.config("tiny")
    W = synth.make_weights(cfg, seed=0)
    lat, cond = synth.make_latent(cfg, seed=1)[0], synth.make_cond(cfg, seed=2)[0]
    sig = O.shift_sigma(O.sigma_schedule(cfg["steps"]), cfg["shift"])
    t0 = time.perf_counter()
    O.denoise_loop(lat, cond, np.zeros_like(cond), W, cfg, sig, cfg["guidance"])
    t = time.perf_counter() - t0
    return dict(loop_s=t, steps_per_s=cfg["steps"] / t)


def cpu_baseline_leg(workload: str) -> dict:
    """The `cpu_baseline` object: the headline workload's extrapolated step
    rate, with the tiny loop (complete) and one block of each large workload
    (extrapolated from sampled rows) beside it."""
    main = cpu_oracle_sample(workload)
    other = "image" if workload == "video" else "video"
    oth = cpu_oracle_sample(other)
    tiny = cpu_oracle_tiny_loop()
    return {"value": 1.0 / main["t_step"], "unit": "steps/s", "cores": main["cores"], "kind": "oracle",
            "sample": main["sample"], "extrapolated": True,
            "sample_seconds": main["sample_s"] + oth["sample_s"] + tiny["loop_s"],
            "cases": {"tiny_loop": {"seconds": tiny["loop_s"], "steps_per_s": tiny["steps_per_s"],
                                    "extrapolated": False, "what": "complete 4-step CFG loop of the tiny config"},
                      f"{workload}_block": {"seconds": main["t_block"], "extrapolated": True,
                                            "sample_seconds": main["sample_s"]},
                      f"{other}_block": {"seconds": oth["t_block"], "extrapolated": True,
                                         "sample_seconds": oth["sample_s"], "sample": oth["sample"]}}}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if rank != 0:
        return
    _oracle_block_weights(args.workload)       # set-up outside the timed samples
    for _ in range(args.warmup):
        cpu_oracle_sample(args.workload)
    ts, walls = [], []
    for _ in range(args.steps):
        w0 = time.perf_counter()
        r = cpu_oracle_sample(args.workload)
        walls.append(time.perf_counter() - w0)
        ts.append(r["t_step"])
    t_step = statistics.median(ts)
    v = 1.0 / t_step
    wall = sum(walls)
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "steps/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": wall / args.steps * 1e3,
            "extrapolated": True,
            "step_is": "one bounded oracle sample: one block at two sampled query-row counts; `value` is the "
                       "full denoising step rate extrapolated from it",
            "ms_per_full_step_extrapolated": t_step * 1e3, "sample_seconds_total": wall,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(args.workload, args.steps, world),
            "cpu_baseline": {"value": v, "unit": "steps/s", "cores": r["cores"], "kind": "oracle",
                             "sample": r["sample"], "extrapolated": True},
            "e2e": {"value": v, "unit": "steps/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ GPU run
def aggregate(elapsed_s: float, steps: int, world: int, dist=None) -> tuple:
    """Maximum time over ranks and the whole-job step rate."""
    t = elapsed_s
    if dist is not None and world > 1:
        import torch
        tt = torch.tensor([t], dtype=torch.float64)
        if dist.get_backend() == "nccl":
            tt = tt.cuda()
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        t = float(tt.item())
    return t, steps * world / t


def file_sha(path: str) -> str:
    with open(path, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def _schedule(cfg: dict, k: int) -> np.ndarray:
    """The first k steps of the workload's shifted schedule (a longer linear
    one if k exceeds it)."""
    full = np.array([1.0 - i / cfg["steps"] for i in range(cfg["steps"] + 1)])
    full = (cfg["shift"] * full / (1 + (cfg["shift"] - 1) * full)).astype(np.float32)
    if k <= cfg["steps"]:
        return full[:k + 1].copy()
    return np.linspace(1.0, 1e-3, k + 1).astype(np.float32)


def run_image_loop(args, clocks_gpu: str) -> dict:
    """Steps/s of the 30-block image DiT loop (4096 + 512 joint tokens, CFG
    pair), device-timed over --steps steps after --warmup, no per-launch
    instrumentation."""
    import torch
    from diffusion_transformer_denoising_gb300 import dit
    cfg = synth.config("image")
    L, C = cfg["cond_len"], cfg["in_channels"]
    N = int(np.prod(synth.grid(cfg)))
    m = dit.DiT(cfg)
    W = synth.make_weights_torch(cfg, seed=0, device="cuda")
    m.load_weights(W)
    del W
    torch.cuda.empty_cache()
    g = torch.Generator(device="cuda")
    g.manual_seed(2000)
    lat0 = torch.randn((1, C) + cfg["latent"], generator=g, device="cuda")
    cond = torch.randn((1, L, cfg["cond_dim"]), generator=g, device="cuda").to(torch.bfloat16).float()
    unc = torch.zeros_like(cond)
    flags = dit.LOOP_PARTIAL_SCHEDULE
    lat = lat0.clone()
    m.dit_denoise_loop(lat, 1, cfg["latent"], cond, unc, L, _schedule(cfg, args.warmup), cfg["guidance"], flags)
    m.dit_synchronize()
    lat = lat0.clone()
    stream = torch.cuda.current_stream()
    torch.cuda.synchronize()
    clocks = ClockSampler(clocks_gpu)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    m.dit_denoise_loop(lat, 1, cfg["latent"], cond, unc, L, _schedule(cfg, args.steps), cfg["guidance"], flags)
    e1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    m.dit_synchronize()
    t_step = e0.elapsed_time(e1) / 1e3 / args.steps
    # the same steps replayed from one captured step (DIT_LOOP_CUDA_GRAPH); the
    # capture is made by an untimed call with the same buffers and step count
    sched = _schedule(cfg, args.steps)
    gflags = flags | dit.LOOP_CUDA_GRAPH
    lat_g = lat0.clone()
    m.dit_denoise_loop(lat_g, 1, cfg["latent"], cond, unc, L, sched, cfg["guidance"], gflags)
    m.dit_synchronize()
    lat_g.copy_(lat0)
    torch.cuda.synchronize()
    g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    g0.record(stream)
    m.dit_denoise_loop(lat_g, 1, cfg["latent"], cond, unc, L, sched, cfg["guidance"], gflags)
    g1.record(stream)
    torch.cuda.synchronize()
    m.dit_synchronize()
    t_graph = g0.elapsed_time(g1) / 1e3 / args.steps
    fl = step_flops(cfg, 2, N, L)
    peaks = measured_peaks()
    out = {"what": WORKLOADS["image"]["desc"] + f", first {args.steps} of {cfg['steps']} steps, shift {cfg['shift']}",
           "steps_per_s": 1.0 / t_step, "ms_per_step": t_step * 1e3, "steps": args.steps,
           "attn_gemm_tflops": fl["total"] / t_step / 1e12,
           "pct_bf16_peak": 100 * fl["total"] / t_step / 1e12 / peaks["bf16"],
           "graph_steps_per_s": 1.0 / t_graph, "graph_ms_per_step": t_graph * 1e3,
           "graph_bitwise_equal": bool(torch.equal(lat_g, lat)),
           "finite": bool(torch.isfinite(lat).all().item()), "clocks": clk}
    del lat_g
    m.close()
    del lat, lat0, cond, unc
    torch.cuda.empty_cache()
    return out


def run_fp8_loop(args, clocks_gpu: str, workload: str = "video") -> dict:
    """Steps/s of a workload in fp8 precision (the LayerNorm-fed GEMMs -- Q/K/V,
    cross-attention Q, MLP up-projection -- in e4m3), timed like the headline;
    then a separate per-launch pass for the fp8 GEMMs' rate, given against the
    fp8 peak taken as twice the measured bf16 peak (the nominal dense fp8 :
    bf16 ratio, 4.5 : 2.25 PFLOP/s)."""
    import torch
    from diffusion_transformer_denoising_gb300 import dit
    cfg = synth.config(WORKLOADS[workload]["cfg"], precision=synth.PREC_FP8)
    L, C, D, F = cfg["cond_len"], cfg["in_channels"], cfg["hidden"], cfg["mlp"]
    N = int(np.prod(synth.grid(cfg)))
    m = dit.DiT(cfg)
    W = synth.make_weights_torch(cfg, seed=0, device="cuda")
    m.load_weights(W)
    del W
    torch.cuda.empty_cache()
    g = torch.Generator(device="cuda")
    g.manual_seed(3000)
    lat0 = torch.randn((1, C) + cfg["latent"], generator=g, device="cuda")
    cond = torch.randn((1, L, cfg["cond_dim"]), generator=g, device="cuda").to(torch.bfloat16).float()
    unc = torch.zeros_like(cond)
    flags = dit.LOOP_PARTIAL_SCHEDULE
    lat = lat0.clone()
    m.dit_denoise_loop(lat, 1, cfg["latent"], cond, unc, L, _schedule(cfg, args.warmup), cfg["guidance"], flags)
    m.dit_synchronize()
    lat = lat0.clone()
    stream = torch.cuda.current_stream()
    torch.cuda.synchronize()
    clocks = ClockSampler(clocks_gpu)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    m.dit_denoise_loop(lat, 1, cfg["latent"], cond, unc, L, _schedule(cfg, args.steps), cfg["guidance"], flags)
    e1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    m.dit_synchronize()
    t_step = e0.elapsed_time(e1) / 1e3 / args.steps
    k_prof = max(1, min(args.steps, 3))
    lat_p = lat0.clone()
    m.dit_profile_start(timing=True)
    m.dit_denoise_loop(lat_p, 1, cfg["latent"], cond, unc, L, _schedule(cfg, k_prof), cfg["guidance"], flags)
    prof = m.dit_profile_stop()
    m.dit_synchronize()
    fl = step_flops(cfg, 2, N, L)
    peaks = measured_peaks()
    if cfg["cond_mode"] == synth.COND_CROSS:
        f8_flops = 2 * 2 * N * D * (3 * D + D + F) * cfg["depth"]      # Q/K/V, cross Q, FFN1 per step
    else:
        # Q/K/V and FFN1 of both streams; the last block's condition stream
        # skips its MLP (its output is never read)
        f8_flops = 2 * 2 * (N + L) * D * (3 * D + F) * cfg["depth"] - 2 * 2 * L * D * F
    f8_ms = sum(prof[k][1] for k in ("gemm_qkv", "gemm_cross_q", "gemm_ffn1")) / k_prof
    f8_tflops = f8_flops / (f8_ms / 1e3) / 1e12
    out = {"what": f"{workload} workload with the LayerNorm-fed GEMMs in e4m3 (per-row / per-output-channel "
                   f"scales), first {args.steps} of {cfg['steps']} steps",
           "steps_per_s": 1.0 / t_step, "ms_per_step": t_step * 1e3, "steps": args.steps,
           "attn_gemm_tflops": fl["total"] / t_step / 1e12,
           "fp8_gemm_tflops": f8_tflops, "fp8_peak_tflops": 2 * peaks["bf16_sustained"],
           "fp8_gemm_frac": f8_tflops / (2 * peaks["bf16_sustained"]),
           "fp8_peak_kind": f"2 x measured bf16 sustained ({peaks['source']}), nominal fp8:bf16 ratio",
           "kernel_ms_per_step": {k: v[1] / k_prof for k, v in prof.items()},
           "finite": bool(torch.isfinite(lat).all().item()), "clocks": clk}
    m.close()
    del lat, lat0, lat_p, cond, unc
    torch.cuda.empty_cache()
    return out


def run_gpu(args):
    import torch
    from diffusion_transformer_denoising_gb300 import dit

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    dev_idx = torch.cuda.current_device()
    stream = torch.cuda.current_stream()
    uuid = str(torch.cuda.get_device_properties(dev_idx).uuid)
    gpu_id = uuid if uuid.startswith("GPU-") else "GPU-" + uuid

    wl = WORKLOADS[args.workload]
    cfg = synth.config(wl["cfg"])
    N = int(np.prod(synth.grid(cfg)))
    L = cfg["cond_len"]
    C = cfg["in_channels"]
    m = dit.DiT(cfg, device=dev_idx)
    W = synth.make_weights_torch(cfg, seed=0, device=f"cuda:{dev_idx}")
    m.load_weights(W)
    del W
    torch.cuda.empty_cache()
    g = torch.Generator(device=f"cuda:{dev_idx}")
    g.manual_seed(1000 + rank)
    lat0 = torch.randn((1, C) + cfg["latent"], generator=g, device="cuda", dtype=torch.float32)
    cond = torch.randn((1, L, cfg["cond_dim"]), generator=g, device="cuda", dtype=torch.float32)
    cond = cond.to(torch.bfloat16).float()
    unc = torch.zeros_like(cond)
    flags = dit.LOOP_PARTIAL_SCHEDULE

    # warm-up
    lat = lat0.clone()
    m.dit_denoise_loop(lat, 1, cfg["latent"], cond, unc, L, _schedule(cfg, args.warmup), cfg["guidance"], flags)
    m.dit_synchronize()

    # timed region: exactly K steps in one loop call; launches are counted,
    # nothing else is recorded on the stream
    st = _schedule(cfg, args.steps)
    lat = lat0.clone()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(gpu_id)
    m.dit_profile_start(timing=False)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    m.dit_denoise_loop(lat, 1, cfg["latent"], cond, unc, L, st, cfg["guidance"], flags)
    e1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    counts = m.dit_profile_stop()
    m.dit_synchronize()
    elapsed = e0.elapsed_time(e1) / 1e3
    if dist is not None:
        dist.barrier()
    t_max, value = aggregate(elapsed, args.steps, world, dist)
    ok = bool(torch.isfinite(lat).all().item())

    # per-kernel breakdown: a separate pass over the same steps with a CUDA
    # event pair around every launch on the launching stream
    k_prof = max(1, min(args.steps, 3))
    lat_p = lat0.clone()
    m.dit_profile_start(timing=True)
    m.dit_denoise_loop(lat_p, 1, cfg["latent"], cond, unc, L, _schedule(cfg, k_prof), cfg["guidance"], flags)
    prof = m.dit_profile_stop()
    m.dit_synchronize()
    del lat_p

    # end to end through the public API with host buffers: every step copies
    # its inputs host->device and reads the latent back
    pin_lat = lat0.cpu().pin_memory()
    pin_cond = cond.cpu().pin_memory()
    pin_unc = unc.cpu().pin_memory()
    out_host = torch.empty_like(pin_lat).pin_memory()
    d_lat, d_cond, d_unc = torch.empty_like(lat0), torch.empty_like(cond), torch.empty_like(unc)
    k_e2e = max(1, min(args.steps, 3))
    full = _schedule(cfg, cfg["steps"])
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    f0.record(stream)
    for i in range(k_e2e):
        d_lat.copy_(pin_lat if i == 0 else out_host, non_blocking=True)
        d_cond.copy_(pin_cond, non_blocking=True)
        d_unc.copy_(pin_unc, non_blocking=True)
        m.dit_denoise_loop(d_lat, 1, cfg["latent"], d_cond, d_unc, L, full[i:i + 2].copy(), cfg["guidance"], flags)
        out_host.copy_(d_lat, non_blocking=True)
    f1.record(stream)
    torch.cuda.synchronize()
    e2e_t, e2e_value = aggregate(f0.elapsed_time(f1) / 1e3, k_e2e, world, dist)
    h2d = (pin_lat.numel() + pin_cond.numel() + pin_unc.numel()) * 4
    d2h = out_host.numel() * 4

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return

    fl = step_flops(cfg, 2, N, L)
    peaks = measured_peaks()
    ms_step = t_max / args.steps * 1e3
    tflops = fl["total"] / (t_max / args.steps) / 1e12
    n_self, ms_self = prof["attn_self"]
    attn_ms = ms_self / max(n_self, 1)
    attn_achieved = fl["attn_self_per_launch"] / (attn_ms / 1e3) / 1e12
    src = os.path.join(ROOT, "diffusion_transformer_denoising_gb300", "csrc", "attn_tc.cu")
    tr = TRAFFIC.get("attn_tc.cu")
    traffic = tr[2] if tr and tr[0] == file_sha(src) and tr[1] == args.workload else None
    gemm_ms = sum(prof[k][1] for k in prof if k.startswith("gemm"))
    kern_ms = sum(v[1] for v in prof.values())
    n_ce, ms_ce = prof["cfg_euler"]
    ce_bytes = 16 * C * int(np.prod(cfg["latent"]))    # both passes' velocity read, latent read + write (fp32)
    line = {
        "metric": METRIC, "value": value, "unit": "steps/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": (value / world / PAGES_STEPS_PER_S[args.workload]) if args.workload in PAGES_STEPS_PER_S
        else None,
        "dtype": "bf16", "data": "synthetic (seeded N(0,1) latents/condition, N(0,0.02) bf16 weights)",
        "config": workload_config(args.workload, args.steps, world),
        "attn_gemm_tflops": tflops,
        "pct_bf16_peak": 100 * tflops / peaks["bf16"],
        "pct_bf16_peak_sustained": 100 * tflops / peaks["bf16_sustained"],
        "roofline": {"kernel": "attn_wide_kernel (self-attention)", "bound": "tensor",
                     "achieved": attn_achieved, "peak": peaks["bf16_sustained"], "unit": "TFLOP/s",
                     "frac": attn_achieved / peaks["bf16_sustained"], "traffic": traffic,
                     # the sustained peak was measured at a lower median SM clock than
                     # this run's: the same fraction with the peak scaled to this clock
                     "frac_at_run_clock": (attn_achieved / (peaks["bf16_sustained"] * clk["sm_mhz"]
                                                            / peaks["sustained_sm_mhz"])
                                           if clk.get("sm_mhz") and peaks.get("sustained_sm_mhz") else None),
                     "peak_sm_mhz": peaks.get("sustained_sm_mhz"), "run_sm_mhz": clk.get("sm_mhz"),
                     "peak_kind": f"bf16 sustained ({peaks['source']}), kernel timed inside a long step",
                     "per_launch_flops": fl["attn_self_per_launch"], "avg_launch_ms": attn_ms,
                     "timed_by": f"event pair per launch, separate {k_prof}-step pass after the headline"},
        "breakdown_steps": k_prof,
        "kernel_ms_per_step": {k: v[1] / k_prof for k, v in prof.items()},
        "kernel_share": {k: v[1] / kern_ms for k, v in prof.items()} if kern_ms > 0 else None,
        "gemm_tflops": fl["gemm"] / (gemm_ms / k_prof / 1e3) / 1e12 if gemm_ms > 0 else None,
        "cfg_euler": {"us_per_launch": ms_ce / max(n_ce, 1) * 1e3, "bytes_per_launch": ce_bytes,
                      "gbs": ce_bytes / (ms_ce / max(n_ce, 1) / 1e3) / 1e9 if ms_ce > 0 else None,
                      "hbm_peak_gbs": peaks["hbm"]},
        "gpu_launches": int(sum(v[0] for v in counts.values())),
        "clocks": clk,
        "finite": ok,
        "e2e": {"value": e2e_value, "unit": "steps/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "steps": k_e2e, "note": "one dit_denoise_loop call per step from pinned host buffers; "
                                        "includes the per-call condition key/value projection"},
    }
    if world == 1 and not args.no_extras and args.workload == "video":
        m.close()
        del lat, lat0, cond, unc, d_lat, d_cond, d_unc
        torch.cuda.empty_cache()
        line["image_loop"] = run_image_loop(args, gpu_id)
        line["fp8_loop"] = run_fp8_loop(args, gpu_id)
        line["fp8_image_loop"] = run_fp8_loop(args, gpu_id, "image")
        line["sweep"] = sweep_points(args, steps=3, warmup=1)
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_leg(args.workload)
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def run_block_case(args):
    """One DiT block of the workload (depth-1 model, CFG batch 2, full token
    count, batch --batch) run warmup + steps times: the small case for kernel
    profiling."""
    import torch
    from diffusion_transformer_denoising_gb300 import dit
    torch.cuda.set_device(0)
    prec = {"bf16": synth.PREC_BF16, "fp8": synth.PREC_FP8}[args.precision]
    cfg = synth.config(WORKLOADS[args.workload]["cfg"], depth=1, precision=prec)
    grid = synth.grid(cfg)
    N, L, D = int(np.prod(grid)), cfg["cond_len"], cfg["hidden"]
    m = dit.DiT(cfg)
    W = synth.make_weights_torch(cfg, seed=0, device="cuda")
    m.load_weights(W)
    del W
    g = torch.Generator(device="cuda")
    g.manual_seed(7)
    B = args.batch
    x0 = torch.randn((B, N, D), generator=g, device="cuda") * 0.5
    cond = torch.randn((B, L, cfg["cond_dim"]), generator=g, device="cuda").to(torch.bfloat16).float()
    mod = torch.randn((B, 6 * D), generator=g, device="cuda") * 0.1
    joint = cfg["cond_mode"] == synth.COND_JOINT
    x = x0.clone()
    xc = cond.clone() if joint else None
    for _ in range(args.warmup):
        m.dit_block_forward(0, x, xc, mod, None if joint else cond, B, grid, L)
    m.dit_synchronize()
    m.dit_profile_start(timing=True)
    for _ in range(args.steps):
        m.dit_block_forward(0, x, xc, mod, None if joint else cond, B, grid, L)
    prof = m.dit_profile_stop()
    m.dit_synchronize()
    fl = step_flops(cfg, B, N, L, loop=False)   # dit_block_forward computes both streams' outputs
    n, ms = prof["attn_self"]
    out = {"case": f"one {args.workload} block, batch {B}, {args.precision}", "per_kernel_ms": {k: v[1] / args.steps for k, v in prof.items()},
           "attn_self_tflops": fl["attn_self_per_launch"] / (ms / max(n, 1) / 1e3) / 1e12,
           "block_tflops": fl["total"] / (sum(v[1] for v in prof.values()) / args.steps / 1e3) / 1e12}
    print(json.dumps(out), flush=True)


SWEEP_POINTS = [(1, 4096), (2, 4096), (4, 4096), (8, 4096), (1, 1024), (1, 16384), (1, 65536)]


def sweep_points(args, steps: int, warmup: int) -> list:
    """Batch/sequence sweep of the image DiT block: a depth-1 image model
    (hidden 3072, 24x128 heads, MLP 12288) at batch 1/2/4/8 with 4096 image
    tokens and at 1024/16384/65536 tokens with batch 1, always jointly with
    512 condition tokens.  Each point times one denoising step (timestep MLP,
    patch embed, the block on the CFG pair, final layer, guidance + Euler)
    through dit_denoise_loop, device-timed over `steps` calls."""
    import torch
    from diffusion_transformer_denoising_gb300 import dit
    base = synth.config("image", depth=1)
    L, C = base["cond_len"], base["in_channels"]
    _, ph, pw = base["patch"]
    W = synth.make_weights_torch(base, seed=0, device="cuda")
    sig = np.array([1.0, 1.0 - 1.0 / base["steps"]])
    sig = (base["shift"] * sig / (1 + (base["shift"] - 1) * sig)).astype(np.float32)
    g = torch.Generator(device="cuda")
    g.manual_seed(11)
    stream = torch.cuda.current_stream()
    peaks = measured_peaks()
    points = []
    for batch, ntok in SWEEP_POINTS:
        side = int(round(ntok ** 0.5))
        cfg = synth.config("image", depth=1, latent=(1, side * ph, side * pw))
        m = dit.DiT(cfg)
        m.load_weights(W)
        lat0 = torch.randn((batch, C) + cfg["latent"], generator=g, device="cuda")
        cond = torch.randn((batch, L, cfg["cond_dim"]), generator=g, device="cuda").to(torch.bfloat16).float()
        unc = torch.zeros_like(cond)
        lat = lat0.clone()
        for _ in range(max(1, warmup)):
            m.dit_denoise_loop(lat, batch, cfg["latent"], cond, unc, L, sig, cfg["guidance"], dit.LOOP_PARTIAL_SCHEDULE)
        m.dit_synchronize()
        lat = lat0.clone()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            m.dit_denoise_loop(lat, batch, cfg["latent"], cond, unc, L, sig, cfg["guidance"], dit.LOOP_PARTIAL_SCHEDULE)
        e1.record(stream)
        torch.cuda.synchronize()
        t_step = e0.elapsed_time(e1) / 1e3 / steps
        fl = step_flops(cfg, 2 * batch, side * side, L)
        tf = fl["total"] / t_step / 1e12
        points.append({"batch": batch, "image_tokens": side * side, "cond_tokens": L,
                       "steps_per_s": 1.0 / t_step, "ms_per_step": t_step * 1e3, "tflops": tf,
                       "pct_bf16_peak": 100 * tf / peaks["bf16"],
                       "finite": bool(torch.isfinite(lat).all().item())})
        m.close()
        del lat, lat0, cond, unc
        torch.cuda.empty_cache()
    del W
    torch.cuda.empty_cache()
    return points


def run_sweep(args):
    import torch
    torch.cuda.set_device(0)
    points = sweep_points(args, steps=args.steps, warmup=args.warmup)
    print(json.dumps({"case": "image DiT block sweep: depth 1, one CFG + Euler step per point", "dtype": "bf16",
                      "data": "synthetic (seeded N(0,1) latents/condition, N(0,0.02) bf16 weights)",
                      "steps": args.steps, "warmup": args.warmup, "peak_bf16_tflops": measured_peaks()["bf16"],
                      "points": points}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default="video", choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the image loop and the sweep points that the default video line also carries")
    ap.add_argument("--batch", type=int, default=2, help="batch of the block case")
    ap.add_argument("--precision", default="bf16", choices=["bf16", "fp8"], help="precision of the block case")
    ap.add_argument("--case", default="step", choices=["step", "block", "sweep"],
                    help="block: one DiT block repeatedly (small case for kernel profiling); "
                         "sweep: image block batch/sequence sweep")
    ap.add_argument("--gemm-cta-pairs", type=int, default=1, choices=[0, 1, 2],
                    help="GEMMs of width a multiple of 256 on CTA pairs (cta_group::2, 256 x 256 tiles): "
                         "0 never (single CTAs, 128 x 256), 1 when the main loop has >= 16 K blocks, 2 always")
    args = ap.parse_args()
    if args.impl != "reference" and args.gemm_cta_pairs != 1:
        from diffusion_transformer_denoising_gb300 import dit
        dit.dit_debug_gemm_cta_pairs(args.gemm_cta_pairs)
    if args.case == "block":
        run_block_case(args)
    elif args.case == "sweep":
        run_sweep(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
