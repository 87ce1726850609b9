"""Throughput of the exact-attention hot path on GB300, one JSON line on stdout.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Workload (the configuration the headline metric is quoted on): bf16 attention,
B=4, H=16, N=2048, d=128, scale 1/sqrt(d), non-causal, Q, K, V, dO ~ N(0,1) from
seed 2.  One step = one pass of the whole hot path over that batch, six
launches: the bf16 forward (fa_fwd), the backward's three stages (fa_bwd_prep,
fa_bwd_main, fa_bwd_dq), and the FP8 path on the same Q, K, V (fa_fp8_prepare
with seeded rotation signs, fa_fwd_fp8).  TFLOP/s counts 4*B*H*N^2*d per forward
(bf16 or FP8) and 2.5 times that per backward.  `frac_of_peak` is the time the
step's work would take at the measured peaks (bf16 FLOPs at the bf16 peak, FP8
FLOPs at twice it, the nominal ratio) over the measured time.  Each stage is
bracketed by its own CUDA events, which give the per-kernel rooflines.

Timing: W untimed warm-up steps, then exactly K steps bracketed by a barrier and
torch.cuda.synchronize() on both sides.  L2 (129 MB) is flushed before every
step by writing a 256 MB buffer outside the per-step CUDA-event pairs; device
time is the sum of the per-step event pairs on the launching stream, max over
ranks.  `e2e` repeats the step through the same public calls with the inputs in
pinned host memory: every step copies Q, K, V and dO in and O, LSE, dQ, dK, dV and the
FP8 O and LSE out, all inside its timed region.  The copies run on their own streams
and overlap the neighbouring steps' kernels (double-buffered), as a serving or
training loop would overlap them.

Under torchrun (N > 1) every rank runs the same independent replica (the heads
shard with no exchange, so there is no collective on the data path) and rank 0
prints the aggregate.  `--impl reference` times the float64 CPU oracle on a
bounded row sample of the same workload instead (rank 0 only).
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = {"workload": "bf16 attention forward + backward, B=4 H=16 N=2048 d=128, non-causal, scale=1/sqrt(d)",
            "B": 4, "H": 16, "N": 2048, "d": 128, "causal": False, "seed": 2}
METRIC = "attention fwd/bwd TFLOP/s on 1 GB300 and % of dense BF16/FP8 tensor peak"
FALLBACK_BF16_TFLOPS = 1900.0


def fwd_flops(B, H, N, d, causal):
    f = 4.0 * B * H * N * N * d
    return f / 2 if causal else f


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        return {"bf16_tflops": j.get("bf16_tflops"), "bf16_tflops_sustained": j.get("bf16_tflops_sustained"),
                "hbm_gbs": j.get("hbm_gbs"), "source": "measured"}
    return {"bf16_tflops": FALLBACK_BF16_TFLOPS, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0,
            "source": "fallback"}


def profile_traffic(profile: str, source: str):
    """DRAM bytes per launch from a committed ncu summary, or None.

    The summary records the sha256 prefix of the kernel source it was captured
    from; if that source has changed since, the counters no longer describe the
    kernel and None is returned.
    """
    import hashlib

    path = os.path.join(ROOT, "profiles", profile)
    if not os.path.exists(path):
        return None
    meta = {}
    for line in open(path):
        if ":" in line and not line.startswith(("|", "#", " ")):
            key, _, val = line.partition(":")
            meta[key.strip()] = val.strip()
    want = meta.get("kernel_source_sha256_16")
    src = os.path.join(ROOT, meta.get("kernel_source", source))
    if not want or not os.path.exists(src):
        return None
    have = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    if have != want:
        return None
    try:
        return float(meta["traffic_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def max_over_ranks(ms: float, device) -> float:
    """The slowest rank's time: every rank gets the maximum (a no-op for one process)."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return ms
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.barrier()
    return float(t.item())


def whole_job_tflops(flops_per_rank_step: float, steps: int, world: int, max_ms: float) -> float:
    """Whole-job throughput: the work of every rank over the slowest rank's time."""
    return flops_per_rank_step * steps * world / (max_ms * 1e-3) / 1e12


def dist_env():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), int(
        os.environ.get("LOCAL_RANK", "0"))


class ClockSampler:
    """nvidia-smi clock / throttle samples while the timed region runs."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.path = os.path.join(ROOT, "gpurun_out", f"clocks_{os.getpid()}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def mark(self, which: str):
        setattr(self, which, time.time())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        import datetime

        t0, t1 = getattr(self, "t0", None), getattr(self, "t1", None)
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                if t0 is not None and t1 is not None and not (t0 <= ts <= t1):
                    continue  # outside the timed region
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


def run_ours(args):
    import torch

    import io_aware_exact_fwd_gb300 as fa
    from synth import normal_qkv, rotation_signs

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl")
    fa.load_library()
    w = WORKLOAD
    B, H, N, d, causal = w["B"], w["H"], w["N"], w["d"], w["causal"]
    scale = d ** -0.5
    x = normal_qkv(B, H, N, d, w["seed"] + rank, with_do=True)
    q, k, v, g = (x[n].to(torch.bfloat16).cuda() for n in ("q", "k", "v", "do"))
    o = torch.empty_like(q)
    lse = torch.empty(B, H, N, dtype=torch.float32, device="cuda")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(fa.fa_bwd_workspace_size(B, H, N, d), dtype=torch.uint8, device="cuda")
    ws8 = torch.empty(fa.fa_fp8_workspace_size(B, H, N, d), dtype=torch.uint8, device="cuda")
    signs = rotation_signs(d, w["seed"]).cuda()
    o8 = torch.empty_like(q)
    lse8 = torch.empty_like(lse)
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    stages = ("fwd", "bwd_prep", "bwd_main", "bwd_dq", "fp8_prep", "fwd_fp8")
    calls = {
        "fwd": lambda: fa.fa_fwd(q, k, v, o=o, lse=lse, causal=causal, scale=scale),
        "bwd_prep": lambda: fa.fa_bwd_prep(o, g, lse, ws),
        "bwd_main": lambda: fa.fa_bwd_main(q, k, v, g, dk, dv, ws, causal=causal, scale=scale),
        "bwd_dq": lambda: fa.fa_bwd_dq(ws, dq, scale=scale),
        "fp8_prep": lambda: fa.fa_fp8_prepare(q, k, v, signs, ws8),
        "fwd_fp8": lambda: fa.fa_fwd_fp8(ws8, (B, H, N, d), o=o8, lse=lse8, causal=causal, scale=scale),
    }
    launches_per_step = 6

    for _ in range(args.warmup):
        flush.zero_()
        for st in stages:
            calls[st]()
    fa.fa_sync_check()

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(stages) + 1)] for _ in range(args.steps)]
    sampler = ClockSampler(local) if rank == 0 else None
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    if sampler:
        sampler.start()
        time.sleep(0.3)
    t_wall0 = time.perf_counter()
    if sampler:
        sampler.mark("t0")
    for i in range(args.steps):
        flush.zero_()
        ev[i][0].record(stream)
        for j, st in enumerate(stages):
            calls[st]()
            ev[i][j + 1].record(stream)
    torch.cuda.synchronize()
    if sampler:
        sampler.mark("t1")
    t_wall = time.perf_counter() - t_wall0
    clocks = sampler.stop() if sampler else None
    fa.fa_sync_check()
    stage_ms = {st: sum(ev[i][j].elapsed_time(ev[i][j + 1]) for i in range(args.steps)) / args.steps
                for j, st in enumerate(stages)}
    dev_ms = sum(ev[i][0].elapsed_time(ev[i][-1]) for i in range(args.steps))
    dev_ms = max_over_ranks(dev_ms, "cuda")
    f_fwd = fwd_flops(B, H, N, d, causal)
    flops_step = 4.5 * f_fwd  # bf16 forward + backward (2.5x) + FP8 forward
    ms_per_step = dev_ms / args.steps
    value = whole_job_tflops(flops_step, args.steps, world, dev_ms)

    # End to end through the public calls: pinned host inputs in, every output back
    # out, every step.  Pipelined over three streams: while step i computes, the
    # inputs of step i + 1 are copied in and the outputs of step i - 1 copied out
    # (two sets of device inputs, device outputs and pinned host outputs; events
    # order each set's reuse).  The timed region runs from the first step's first
    # input copy to the last step's last output copy.
    hq, hk, hv, hg = (t.cpu().pin_memory() for t in (q, k, v, g))
    h_in = (hq, hk, hv, hg)
    e2e_steps = max(3, min(args.steps, 50))
    s_h2d, s_comp, s_d2h = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    sets = []
    for _ in range(2):
        din = [torch.empty_like(t) for t in (q, k, v, g)]
        dout = [torch.empty_like(q), torch.empty_like(lse), torch.empty_like(q), torch.empty_like(k),
                torch.empty_like(v), torch.empty_like(q), torch.empty_like(lse)]  # o, lse, dq, dk, dv, o8, lse8
        hout = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in dout]
        ev = {n: torch.cuda.Event() for n in ("in_ready", "in_free", "out_ready", "out_free")}
        sets.append((din, dout, hout, ev))

    def e2e_step(i):
        din, dout, hout, ev = sets[i % 2]
        with torch.cuda.stream(s_h2d):
            if i >= 2:
                s_h2d.wait_event(ev["in_free"])  # step i - 2 has finished reading these inputs
            for dst, src in zip(din, h_in):
                dst.copy_(src, non_blocking=True)
            ev["in_ready"].record(s_h2d)
        s_comp.wait_event(ev["in_ready"])
        if i >= 2:
            s_comp.wait_event(ev["out_free"])  # step i - 2's outputs have been copied out
        qi, ki, vi, gi = din
        o_, lse_, dq_, dk_, dv_, o8_, lse8_ = dout
        fa.fa_fwd(qi, ki, vi, o=o_, lse=lse_, causal=causal, scale=scale, stream=s_comp)
        fa.fa_bwd(qi, ki, vi, o_, gi, lse_, dq_, dk_, dv_, ws, causal=causal, scale=scale, stream=s_comp)
        fa.fa_fp8_prepare(qi, ki, vi, signs, ws8, stream=s_comp)
        fa.fa_fwd_fp8(ws8, (B, H, N, d), o=o8_, lse=lse8_, causal=causal, scale=scale, stream=s_comp)
        ev["in_free"].record(s_comp)
        ev["out_ready"].record(s_comp)
        with torch.cuda.stream(s_d2h):
            s_d2h.wait_event(ev["out_ready"])
            for dst, src in zip(hout, dout):
                dst.copy_(src, non_blocking=True)
            ev["out_free"].record(s_d2h)

    for i in range(2):
        e2e_step(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_h2d)
    for i in range(2, 2 + e2e_steps):
        e2e_step(i)
    e1.record(s_d2h)
    torch.cuda.synchronize()
    fa.fa_sync_check()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, "cuda")
    h2d = sum(t.numel() * t.element_size() for t in h_in)
    d2h = sum(t.numel() * t.element_size() for t in sets[0][2])

    nxt = (next_rows(fa, q, k, v, g, o, lse, dq, dk, dv, ws, causal, scale, stage_ms, (ws8, signs, o8, lse8))
           if rank == 0 else None)

    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return None

    peaks = load_peaks()
    peak = peaks["bf16_tflops"]
    hbm = peaks["hbm_gbs"]
    elems = B * H * N * d
    npad = (N + 63) // 64 * 64
    stage_info = {
        "fwd": {"bound": "tensor", "flops": f_fwd, "bytes": 8 * elems + 4 * B * H * N,
                "kernel": "fwd_bf16_kernel<128,false>", "profile": "fwd_bf16_B4H16N2048d128.md",
                "source": "io_aware_exact_fwd_gb300/csrc/fa_fwd.cu"},
        "bwd_prep": {"bound": "hbm", "flops": 2.0 * elems,
                     "bytes": 4 * elems + 4 * B * H * N + 8 * B * H * npad + 4 * elems,
                     "kernel": "bwd_preprocess_kernel"},
        "bwd_main": {"bound": "tensor", "flops": 2.5 * f_fwd,
                     "bytes": 10 * elems + 8 * B * H * npad + 4 * elems + 4 * elems,
                     "kernel": "bwd_main_kernel<false>", "profile": "bwd_main_B4H16N2048d128.md",
                     "source": "io_aware_exact_fwd_gb300/csrc/fa_bwd.cu"},
        "bwd_dq": {"bound": "hbm", "flops": 0.0, "bytes": 4 * elems + 2 * elems, "kernel": "bwd_dq_convert_kernel"},
        "fp8_prep": {"bound": "hbm", "flops": 0.0, "bytes": 3 * 2 * elems + 3 * elems, "kernel": "fp8_prepare_kernel<128>"},
        "fwd_fp8": {"bound": "tensor_fp8", "flops": f_fwd, "bytes": 3 * elems + 2 * elems + 4 * B * H * N,
                    "kernel": "fwd_kernel<128,false,fp8>"},
    }
    per_stage = {}
    for st in stages:
        info, ms = stage_info[st], stage_ms[st]
        tf = info["flops"] / (ms * 1e-3) / 1e12
        gbs = info["bytes"] / (ms * 1e-3) / 1e9
        if info["bound"] in ("tensor", "tensor_fp8"):
            pk = peak if info["bound"] == "tensor" else 2.0 * peak
            per_stage[st] = {"ms": round(ms, 5), "bound": info["bound"], "achieved": round(tf, 1),
                             "unit": "TFLOP/s", "frac": round(tf / pk, 4), "peak": pk, "gbs": round(gbs, 1)}
        else:
            per_stage[st] = {"ms": round(ms, 5), "bound": "hbm", "achieved": round(gbs, 1), "unit": "GB/s",
                             "frac": round(gbs / hbm, 4)}
    dom = max(stages, key=lambda st: stage_ms[st])
    di = stage_info[dom]
    dom_ach = per_stage[dom]["achieved"]
    dom_peak = {"tensor": peak, "tensor_fp8": 2.0 * peak, "hbm": hbm}[di["bound"]]
    traffic = None
    if args.traffic is not None:
        traffic = args.traffic
    elif "profile" in di:
        traffic = profile_traffic(di["profile"], di["source"])
    roofline = {
        "bound": di["bound"], "kernel": di["kernel"], "achieved": dom_ach, "peak": dom_peak,
        "peak_source": {"tensor": f"{peaks['source']} bf16_tflops (burst, cuBLAS)",
                        "tensor_fp8": f"2 x {peaks['source']} bf16_tflops (FP8/BF16 nominal ratio)",
                        "hbm": f"{peaks['source']} hbm_gbs (copy)"}[di["bound"]],
        "unit": per_stage[dom]["unit"], "frac": round(dom_ach / dom_peak, 4), "traffic": traffic,
        "traffic_unit": "bytes per launch (ncu dram__bytes_read.sum + dram__bytes_write.sum)",
        "algorithmic_flops_per_launch": di["flops"], "algorithmic_bytes_per_launch": di["bytes"],
    }
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        cpu = cpu_baseline(seconds=args.cpu_seconds)
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": dict(WORKLOAD, l2="flushed before every step (256 MB write, outside the timed event pairs)",
                       parallelism=f"replicas x{world}" if world > 1 else "single GPU",
                       flops_per_step=flops_step),
        "frac_of_peak": round((3.5 * f_fwd / peak + f_fwd / (2.0 * peak)) / 1e12 / (ms_per_step * 1e-3), 4),
        "roofline": roofline,
        "stages": per_stage,
        "e2e": {"value": round(flops_step / (e2e_ms * 1e-3) / 1e12 * world, 2), "unit": "TFLOP/s",
                "ms_per_step": round(e2e_ms, 4), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": launches_per_step * args.steps,
        "wall_s_timed_region": round(t_wall, 3),
        "clocks": clocks,
        "cpu_baseline": cpu,
        "next": finish_next_rows(nxt, peaks),
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return line


# Rows past the hot path, timed after the step (not part of `value`): the split-KV
# decode forward and the 4-bit-weight GEMV on their own workloads; the
# deterministic backward and the FP8 backward on the step's.
DECODE = {"B": 8, "H": 16, "Nq": 1, "Nk": 32768, "d": 128, "causal": False, "seed": 5}
W4A16 = {"M": 1, "N": 28672, "K": 8192, "seed": 6}


def _median_ms(fn, reps, flush=None):
    import torch

    ts = []
    for _ in range(reps):
        if flush is not None:
            flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        ts.append((a, b))
    torch.cuda.synchronize()
    return sorted(x.elapsed_time(y) for x, y in ts)[reps // 2]


def next_rows(fa, q, k, v, g, o, lse, dq, dk, dv, ws, causal, scale, stage_ms, fp8):
    import torch

    from synth import normal_qkv, w4a16_inputs

    out = {}
    w = DECODE
    B, H, Nq, Nk, d = w["B"], w["H"], w["Nq"], w["Nk"], w["d"]
    kv = normal_qkv(B, H, Nk, d, w["seed"])
    qd = normal_qkv(B, H, Nq, d, w["seed"] + 1)["q"].to(torch.bfloat16).cuda()
    kd, vd = kv["k"].to(torch.bfloat16).cuda(), kv["v"].to(torch.bfloat16).cuda()
    del kv
    n = fa.fa_splitkv_default_splits(B, H, Nq, Nk, d)
    wsd = torch.empty(fa.fa_splitkv_workspace_size(B, H, Nq, d, n), dtype=torch.uint8, device="cuda")
    od = torch.empty_like(qd)
    lsed = torch.empty(B, H, Nq, dtype=torch.float32, device="cuda")
    call = lambda: fa.fa_fwd_splitkv(qd, kd, vd, od, lsed, wsd, n_split=n, causal=w["causal"])
    for _ in range(3):
        call()
    ms = _median_ms(call, 20)  # K and V (2.1 GB) are far larger than L2
    byts = 4 * B * H * Nk * d + 4 * B * H * Nq * d + 8 * n * B * H * Nq * (d + 1)
    out["splitkv_decode"] = {"config": dict(w, n_split=n), "ms": round(ms, 5), "bytes": byts, "gbs": byts / ms / 1e6,
                             "launches": 2}
    del kd, vd
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device="cuda")
    det = lambda: fa.fa_bwd(q, k, v, o, g, lse, dq, dk, dv, ws, causal=causal, scale=scale, deterministic=True)
    for _ in range(3):
        det()
    ms_det = _median_ms(det, 20, flush)
    fa.fa_sync_check()
    out["bwd_deterministic"] = {"ms": round(ms_det, 5),
                                "ms_atomic": round(stage_ms["bwd_prep"] + stage_ms["bwd_main"] + stage_ms["bwd_dq"], 5),
                                "launches": 4}
    # FP8 backward on the step's FP8 workspace and dO, both modes.
    ws8, signs, o8, lse8 = fp8
    B, H, N, d = q.shape
    wsb = torch.empty(fa.fa_bwd_fp8_workspace_size(B, H, N, d), dtype=torch.uint8, device="cuda")
    for rec in (False, True):
        call = lambda: fa.fa_bwd_fp8(ws8, signs, o8, g, lse8, dq, dk, dv, wsb, causal=causal, scale=scale,
                                     recompute_forward=rec)
        for _ in range(3):
            call()
        out["bwd_fp8_recompute" if rec else "bwd_fp8"] = {"ms": round(_median_ms(call, 20, flush), 5),
                                                          "launches": 6 if rec else 5}
    fa.fa_sync_check()
    del wsb
    # W4A16 decode GEMV: 28672 x 8192 packed weights (117 MB, beyond L2) times one activation row.
    w = W4A16
    xin = w4a16_inputs(w["M"], w["N"], w["K"], w["seed"])
    x, wq, sc, zr = (xin[n].cuda() for n in ("x", "wq", "scales", "zeros"))
    nsp = fa.fa_w4a16_default_splits(w["M"], w["N"], w["K"])
    wsw = torch.empty(max(fa.fa_w4a16_workspace_size(w["M"], w["N"], w["K"], nsp), 1), dtype=torch.uint8,
                      device="cuda")
    y = torch.empty(w["M"], w["N"], dtype=torch.float16, device="cuda")
    call = lambda: fa.fa_w4a16_gemm(x, wq, sc, zr, y, wsw, n_split=nsp)
    for _ in range(3):
        call()
    ms_w = _median_ms(call, 20, flush)
    fa.fa_sync_check()
    M_, N_, K_ = w["M"], w["N"], w["K"]
    byts = N_ * K_ // 2 + 3 * N_ * K_ // 128 + 2 * M_ * K_ + 2 * M_ * N_
    out["w4a16_gemv"] = {"config": dict(w, n_split=nsp), "ms": round(ms_w, 5), "bytes": byts,
                         "gbs": byts / ms_w / 1e6, "launches": 2 if nsp > 1 else 1}
    return out


def finish_next_rows(nxt, peaks):
    if nxt is None:
        return None
    w = WORKLOAD
    sk = nxt["splitkv_decode"]
    f_bwd = 2.5 * fwd_flops(w["B"], w["H"], w["N"], w["d"], w["causal"])
    bd = nxt["bwd_deterministic"]
    return {
        "splitkv_decode": {"workload": "split-KV decode forward + merge", "config": sk["config"], "ms": sk["ms"],
                           "bound": "hbm", "achieved": round(sk["gbs"], 1), "unit": "GB/s",
                           "peak": peaks["hbm_gbs"], "frac": round(sk["gbs"] / peaks["hbm_gbs"], 4),
                           "algorithmic_bytes": sk["bytes"], "gpu_launches": sk["launches"]},
        "bwd_deterministic": {"workload": "bf16 backward with order-free dQ, the step's configuration",
                              "ms": bd["ms"], "tflops": round(f_bwd / (bd["ms"] * 1e-3) / 1e12, 1),
                              "ms_atomic_dq": bd["ms_atomic"], "gpu_launches": bd["launches"]},
        "bwd_fp8": {"workload": "FP8 backward (straight-through; dequantise, bf16 backward, inverse rotation), "
                                "the step's configuration, with fa_fwd_fp8's O and LSE",
                    "ms": nxt["bwd_fp8"]["ms"], "tflops": round(f_bwd / (nxt["bwd_fp8"]["ms"] * 1e-3) / 1e12, 1),
                    "ms_recompute_forward": nxt["bwd_fp8_recompute"]["ms"],
                    "tflops_recompute_forward": round(f_bwd / (nxt["bwd_fp8_recompute"]["ms"] * 1e-3) / 1e12, 1),
                    "gpu_launches": nxt["bwd_fp8"]["launches"]},
        "w4a16_gemv": {"workload": "W4A16 dequantising GEMV (4-bit weights, group 128, fp16 activations)",
                       "config": nxt["w4a16_gemv"]["config"], "ms": nxt["w4a16_gemv"]["ms"], "bound": "hbm",
                       "achieved": round(nxt["w4a16_gemv"]["gbs"], 1), "unit": "GB/s", "peak": peaks["hbm_gbs"],
                       "frac": round(nxt["w4a16_gemv"]["gbs"] / peaks["hbm_gbs"], 4),
                       "algorithmic_bytes": nxt["w4a16_gemv"]["bytes"],
                       "gpu_launches": nxt["w4a16_gemv"]["launches"]},
    }


def _oracle_step_sample(q, k, v, g, scale, causal, head, r0, rows_per_step):
    """The oracle on one row block of one head: forward rows plus that block's backward share."""
    import numpy as np

    from oracle import attention_backward_rows, attention_forward_rows

    N = q.shape[2]
    rows = np.arange(r0, min(N, r0 + rows_per_step))
    attention_forward_rows(q[0, head], k[0, head], v[0, head], scale, causal, rows)
    attention_backward_rows(q[0, head], k[0, head], v[0, head], g[0, head], scale, causal, rows)
    return len(rows)


def _oracle_inputs():
    import torch

    from synth import normal_qkv, rotation_signs

    w = WORKLOAD
    x = normal_qkv(1, 2, w["N"], w["d"], w["seed"], with_do=True)
    return [x[n].to(torch.bfloat16).to(torch.float64).numpy() for n in ("q", "k", "v", "do")]


def cpu_baseline(seconds: float = 10.0):
    """The float64 oracle, as it stands, on a bounded row sample of the workload (fwd + bwd)."""
    w = WORKLOAD
    N, d, causal = w["N"], w["d"], w["causal"]
    q, k, v, g = _oracle_inputs()
    rows_per_call = 256
    done_rows, t0, i = 0, time.perf_counter(), 0
    while time.perf_counter() - t0 < seconds:
        done_rows += _oracle_step_sample(q, k, v, g, d ** -0.5, causal, i % 2, (i * rows_per_call) % N,
                                         rows_per_call)
        i += 1
    dt = time.perf_counter() - t0
    flops = 3.5 * 4.0 * done_rows * N * d / (2 if causal else 1)
    cores = len(os.sched_getaffinity(0))
    return {"value": round(flops / dt / 1e12, 6), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": f"{done_rows} query rows x {N} keys (forward rows + their backward share) of 2 heads "
                      f"(d={d}) in {dt:.1f} s, float64 numpy, BLAS threads = {cores}"}


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return None
    w = WORKLOAD
    N, d, causal = w["N"], w["d"], w["causal"]
    q, k, v, g = _oracle_inputs()
    rows_per_step = 32

    def step(i):
        return _oracle_step_sample(q, k, v, g, d ** -0.5, causal, i % 2, (i * rows_per_step) % N, rows_per_step)

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    rows = 0
    for i in range(args.steps):
        rows += step(i)
    dt = time.perf_counter() - t0
    flops = 3.5 * 4.0 * rows * N * d / (2 if causal else 1)
    value = flops / dt / 1e12
    cores = len(os.sched_getaffinity(0))
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": dict(WORKLOAD),
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": f"{rows_per_step} query rows x {N} keys of one head per step "
                                   f"(forward rows + their backward share)"},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return line


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--traffic", type=float, default=None,
                    help="DRAM bytes per launch of the dominant kernel from an ncu capture of this kernel version")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
