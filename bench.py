"""Throughput of the exact-attention hot path on GB300, one JSON line on stdout.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Headline workload: bf16 attention, B=2, H=16, N=8192, d=128, scale 1/sqrt(d),
non-causal, Q, K, V, dO ~ N(0,1) from seed 2 (the shape shared by the sequence
sweep, the backward configuration and the FP8 configuration, inside the N >= 4096
regime the throughput targets are stated for).  One step = one forward and one
backward pass over that batch, four launches: fa_fwd, then the backward's three
stages (fa_bwd_prep, fa_bwd_main, fa_bwd_dq).  TFLOP/s counts 4*B*H*N^2*d for
the forward and 2.5 times that for the backward; `frac_of_peak` divides by the
measured dense bf16 peak.  Each stage is bracketed by its own CUDA events, which
give the per-kernel rooflines.

Timed the same way after the headline, and reported beside it (not in `value`):
the causal forward and backward at the same shape, and the FP8 path on the FP8
workload (B=2, H=16, N=8192, d=128, fp32 inputs with 0.1 % x20 outliers, seeded
rotation signs): fa_fp8_prepare and fa_fwd_fp8, non-causal and causal, each
against its own roofline (the FP8 forward against twice the measured bf16 peak,
the nominal FP8/bf16 ratio).

Timing: W untimed warm-up steps, then exactly K steps bracketed by a barrier and
torch.cuda.synchronize() on both sides.  L2 (129 MB) is flushed before every
step by writing a 256 MB buffer outside the per-step CUDA-event pairs (the
inputs, 268 MB, are larger than L2 as well); device time is the sum of the
per-step event pairs on the launching stream, max over ranks.  SM clocks and
throttle reasons are polled through NVML every 2 ms during the timed region.
`e2e` repeats the step through the public calls (fa_fwd, fa_bwd) with the inputs
in pinned host memory: every step copies Q, K, V and dO in and O, LSE, dQ, dK and
dV out, all inside its timed region; the copies run on their own streams and
overlap the neighbouring steps' kernels (double-buffered).

Under torchrun (N > 1) every rank runs the same independent replica (the heads
shard with no exchange, so there is no collective on the data path) and rank 0
prints the aggregate.  `--impl reference` times the float64 CPU oracle on a
bounded row sample of the same workload instead (rank 0 only).
"""

from __future__ import annotations

import argparse
import ctypes
import json
import os
import statistics
import subprocess
import sys
import tempfile
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = {"workload": "bf16 attention forward + backward (fa_fwd, fa_bwd_prep, fa_bwd_main, fa_bwd_dq), "
                        "B=2 H=16 N=8192 d=128, non-causal, scale=1/sqrt(d)",
            "B": 2, "H": 16, "N": 8192, "d": 128, "causal": False, "seed": 2}
FP8_WORKLOAD = {"workload": "FP8 e4m3 attention forward (fa_fp8_prepare + fa_fwd_fp8), B=2 H=16 N=8192 d=128, fp32 "
                            "Q/K/V ~ N(0,1) with 0.1% x20 outliers, seeded +-1 Hadamard rotation, bf16 O",
                "B": 2, "H": 16, "N": 8192, "d": 128, "seed": 5}
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


# NVML clock-event reason bits (nvml.h, nvmlClocksEventReason*).
_NVML_REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
                 0x80: "hw_power_brake_slowdown"}


class ClockSampler:
    """SM clock and throttle reasons of one GPU, polled while the timed region runs.

    NVML (the library behind nvidia-smi) is read from a thread every 2 ms, so even
    a region of a few tens of milliseconds gets samples; without NVML, nvidia-smi
    is sampled every 100 ms into a temporary file.  Reading clocks changes no
    setting of the GPU.
    """

    def __init__(self, cuda_index: int):
        self.cuda_index = cuda_index
        self.samples = []  # (time, sm_mhz, reasons bitmask)
        self.max_mhz = None
        self._stop = threading.Event()
        self._thread = None
        self._smi = None
        self._nvml = None
        self._dev = None

    def _open_nvml(self):
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
        except OSError:
            return False
        if nv.nvmlInit_v2() != 0:
            return False
        dev = ctypes.c_void_p()
        bus = None
        try:
            import torch

            props = torch.cuda.get_device_properties(self.cuda_index)
            dom, b, dv = (getattr(props, a, None) for a in ("pci_domain_id", "pci_bus_id", "pci_device_id"))
            if None not in (dom, b, dv):
                bus = f"{dom:08x}:{b:02x}:{dv:02x}.0".encode()
        except Exception:
            bus = None
        ok = bus is not None and nv.nvmlDeviceGetHandleByPciBusId_v2(ctypes.c_char_p(bus), ctypes.byref(dev)) == 0
        if not ok and nv.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(self.cuda_index), ctypes.byref(dev)) != 0:
            return False
        mx = ctypes.c_uint()
        if nv.nvmlDeviceGetMaxClockInfo(dev, 1, ctypes.byref(mx)) == 0:  # 1 = NVML_CLOCK_SM
            self.max_mhz = float(mx.value)
        self._reasons = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or getattr(
            nv, "nvmlDeviceGetCurrentClocksThrottleReasons")
        self._nvml, self._dev = nv, dev
        return True

    def _poll(self):
        nv, dev = self._nvml, self._dev
        mhz, rs = ctypes.c_uint(), ctypes.c_ulonglong()
        while not self._stop.is_set():
            if nv.nvmlDeviceGetClockInfo(dev, 1, ctypes.byref(mhz)) == 0 and self._reasons(dev, ctypes.byref(rs)) == 0:
                self.samples.append((time.time(), float(mhz.value), int(rs.value)))
            time.sleep(0.002)

    def start(self):
        if self._open_nvml():
            self._thread = threading.Thread(target=self._poll, daemon=True)
            self._thread.start()
            return
        try:
            self._fh = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self._smi = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.cuda_index), "--query-gpu=timestamp,clocks.sm,clocks.max.sm,"
                 "clocks_event_reasons.active", "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self._fh, stderr=subprocess.DEVNULL)
        except Exception:
            self._smi = None

    def mark(self, which: str):
        setattr(self, which, time.time())

    def stop(self):
        if self._thread is not None:
            self._stop.set()
            self._thread.join(timeout=5)
            self._nvml.nvmlShutdown()
            source = "nvml"
        elif self._smi is not None:
            import datetime

            self._smi.terminate()
            try:
                self._smi.wait(timeout=5)
            except Exception:
                self._smi.kill()
            self._fh.seek(0)
            for line in self._fh:
                parts = [p.strip() for p in line.split(",")]
                try:
                    ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                    self.samples.append((ts, float(parts[1]), int(parts[3], 16)))
                    self.max_mhz = float(parts[2])
                except (ValueError, IndexError):
                    continue
            self._fh.close()
            os.unlink(self._fh.name)
            source = "nvidia-smi"
        else:
            return None
        t0, t1 = getattr(self, "t0", None), getattr(self, "t1", None)
        inside = [s for s in self.samples if t0 is None or t1 is None or t0 <= s[0] <= t1]
        if not inside:
            return None
        reasons = set()
        for _, _, bits in inside:
            for b, name in _NVML_REASONS.items():
                if bits & b:
                    reasons.add(name)
        return {"sm_mhz": statistics.median(s[1] for s in inside), "sm_max_mhz": self.max_mhz,
                "samples": len(inside), "reasons": sorted(reasons), "source": source}


def _median_ms(fn, reps, flush=None, stream=None):
    import torch

    stream = stream or torch.cuda.current_stream()
    ts = []
    for _ in range(reps):
        if flush is not None:
            flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        ts.append((a, b))
    torch.cuda.synchronize()
    return sorted(x.elapsed_time(y) for x, y in ts)[reps // 2]


def _tensor_stage(ms, flops, peak, kernel, bound="tensor"):
    tf = flops / (ms * 1e-3) / 1e12
    return {"ms": round(ms, 5), "bound": bound, "kernel": kernel, "achieved": round(tf, 1), "unit": "TFLOP/s",
            "peak": peak, "frac": round(tf / peak, 4)}


def _hbm_stage(ms, byts, hbm, kernel):
    gbs = byts / (ms * 1e-3) / 1e9
    return {"ms": round(ms, 5), "bound": "hbm", "kernel": kernel, "achieved": round(gbs, 1), "unit": "GB/s",
            "peak": hbm, "frac": round(gbs / hbm, 4), "algorithmic_bytes": byts}


def run_ours(args):
    import torch

    import io_aware_exact_fwd_gb300 as fa
    from synth import normal_qkv

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl")
    fa.load_library()
    peaks = load_peaks()
    peak, hbm = peaks["bf16_tflops"], peaks["hbm_gbs"]
    w = WORKLOAD
    B, H, N, d, causal = w["B"], w["H"], w["N"], w["d"], w["causal"]
    scale = d ** -0.5
    x = normal_qkv(B, H, N, d, w["seed"] + rank, with_do=True)
    q, k, v, g = (x[n].to(torch.bfloat16).cuda() for n in ("q", "k", "v", "do"))
    del x
    o = torch.empty_like(q)
    lse = torch.empty(B, H, N, dtype=torch.float32, device="cuda")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(fa.fa_bwd_workspace_size(B, H, N, d), dtype=torch.uint8, device="cuda")
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()

    def step_calls(c):
        return {
            "fwd": lambda: fa.fa_fwd(q, k, v, o=o, lse=lse, causal=c, scale=scale),
            "bwd_prep": lambda: fa.fa_bwd_prep(o, g, lse, ws),
            "bwd_main": lambda: fa.fa_bwd_main(q, k, v, g, dk, dv, ws, causal=c, scale=scale),
            "bwd_dq": lambda: fa.fa_bwd_dq(ws, dq, scale=scale),
        }

    stages = ("fwd", "bwd_prep", "bwd_main", "bwd_dq")
    calls = step_calls(causal)
    launches_per_step = 4

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
        time.sleep(0.05)
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
    flops_step = 3.5 * f_fwd  # bf16 forward + backward (2.5x)
    ms_per_step = dev_ms / args.steps
    value = whole_job_tflops(flops_step, args.steps, world, dev_ms)

    elems = B * H * N * d
    npad = (N + 63) // 64 * 64
    # Algorithmic bytes and FLOPs of each stage (per launch).
    stage_info = {
        "fwd": {"bound": "tensor", "flops": f_fwd, "bytes": 8 * elems + 4 * B * H * N,
                "kernel": "fwd_kernel<128,false,bf16>", "profile": "fwd_bf16_B2H16N8192d128.md",
                "source": "io_aware_exact_fwd_gb300/csrc/fa_fwd.cu"},
        # prep: O, dO and LSE read; the LSE/D operand rows (64 B per padded query row) written;
        # the fp32 dQ accumulator zeroed.
        "bwd_prep": {"bound": "hbm", "bytes": 4 * elems + 4 * B * H * N + 64 * B * H * npad + 4 * elems,
                     "kernel": "bwd_preprocess_kernel"},
        # main: Q, K, V, dO read once; dK, dV written; the dQ accumulator read and written once;
        # the LSE/D operand rows read once.
        "bwd_main": {"bound": "tensor", "flops": 2.5 * f_fwd,
                     "bytes": 8 * elems + 4 * elems + 8 * elems + 64 * B * H * npad,
                     "kernel": "bwd_main_kernel<false>", "profile": "bwd_main_B2H16N8192d128.md",
                     "source": "io_aware_exact_fwd_gb300/csrc/fa_bwd.cu"},
        "bwd_dq": {"bound": "hbm", "bytes": 4 * elems + 2 * elems, "kernel": "bwd_dq_convert_kernel"},
    }

    def stage_report(st, ms):
        info = stage_info[st]
        if info["bound"] == "tensor":
            r = _tensor_stage(ms, info["flops"], peak, info["kernel"])
            r["gbs"] = round(info["bytes"] / (ms * 1e-3) / 1e9, 1)
            return r
        return _hbm_stage(ms, info["bytes"], hbm, info["kernel"])

    per_stage = {st: stage_report(st, stage_ms[st]) for st in stages}
    dom = max(stages, key=lambda st: stage_ms[st])
    di = stage_info[dom]
    traffic = args.traffic if args.traffic is not None else (
        profile_traffic(di["profile"], di["source"]) if "profile" in di else None)
    roofline = {
        "bound": di["bound"], "kernel": di["kernel"], "achieved": per_stage[dom]["achieved"],
        "peak": per_stage[dom]["peak"],
        "peak_source": (f"{peaks['source']} bf16_tflops (burst, cuBLAS): the kernel runs a few ms at a time"
                        if di["bound"] == "tensor" else f"{peaks['source']} hbm_gbs (copy)"),
        "unit": per_stage[dom]["unit"], "frac": per_stage[dom]["frac"], "traffic": traffic,
        "traffic_unit": "bytes per launch (ncu dram__bytes_read.sum + dram__bytes_write.sum)",
        "algorithmic_flops_per_launch": di.get("flops"), "algorithmic_bytes_per_launch": di["bytes"],
    }

    extra = None
    if not args.step_only:
        extra = extra_rows(fa, args, q, k, v, g, o, lse, dq, dk, dv, ws, scale, flush, peaks, stage_info, rank)

    # End to end through the public calls: pinned host inputs in, every output back
    # out, every step.  Pipelined over three streams: while step i computes, the
    # inputs of step i + 1 are copied in and the outputs of step i - 1 copied out
    # (two sets of device inputs, device outputs and pinned host outputs; events
    # order each set's reuse).  The timed region runs from the first step's first
    # input copy to the last step's last output copy.
    e2e = None
    if not args.step_only:
        e2e = run_e2e(fa, args, q, k, v, g, lse, ws, causal, scale, flops_step, world)

    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return None

    cpu = None
    if not args.no_cpu_baseline and world == 1 and not args.step_only:
        cpu = cpu_baseline(seconds=args.cpu_seconds)
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": dict(WORKLOAD, l2="flushed before every step (256 MB write, outside the timed event pairs); "
                                    "inputs (268 MB) also exceed L2",
                       parallelism=f"replicas x{world}" if world > 1 else "single GPU",
                       flops_per_step=flops_step),
        "frac_of_peak": round(flops_step / 1e12 / (ms_per_step * 1e-3) / peak, 4),
        "roofline": roofline,
        "stages": per_stage,
        "e2e": e2e,
        "gpu_launches": launches_per_step * args.steps,
        "wall_s_timed_region": round(t_wall, 4),
        "clocks": clocks,
        "cpu_baseline": cpu,
    }
    if extra is not None:
        line.update(extra)
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return line


def gpu_local_cpus(cuda_index):
    """The host CPUs NVML names as closest to this GPU (nvmlDeviceGetCpuAffinity), or None.

    Pinned host buffers are placed on the NUMA node of the thread that first touches
    them; allocated from one of these CPUs they sit next to the GPU's host link.
    """
    import ctypes

    try:
        import torch

        nv = ctypes.CDLL("libnvidia-ml.so.1")
        if nv.nvmlInit_v2() != 0:
            return None
        try:
            props = torch.cuda.get_device_properties(cuda_index)
            bus = f"{props.pci_domain_id:08x}:{props.pci_bus_id:02x}:{props.pci_device_id:02x}.0".encode()
            dev = ctypes.c_void_p()
            if nv.nvmlDeviceGetHandleByPciBusId_v2(ctypes.c_char_p(bus), ctypes.byref(dev)) != 0:
                return None
            words = 64
            mask = (ctypes.c_ulong * words)()
            if nv.nvmlDeviceGetCpuAffinity(dev, ctypes.c_uint(words), mask) != 0:
                return None
            bits = ctypes.sizeof(ctypes.c_ulong) * 8
            cpus = {w * bits + b for w in range(words) for b in range(bits) if (mask[w] >> b) & 1}
            return cpus or None
        finally:
            nv.nvmlShutdown()
    except Exception:
        return None


def run_e2e(fa, args, q, k, v, g, lse, ws, causal, scale, flops_step, world):
    import torch

    # Allocate and drive the pinned host buffers from CPUs next to the GPU (restored after).
    saved_affinity = os.sched_getaffinity(0) if hasattr(os, "sched_getaffinity") else None
    local = gpu_local_cpus(torch.cuda.current_device())
    host_cpus = None
    if saved_affinity and local and (local & saved_affinity):
        host_cpus = sorted(local & saved_affinity)
        os.sched_setaffinity(0, host_cpus)
    try:
        return _run_e2e(fa, args, q, k, v, g, lse, ws, causal, scale, flops_step, world, host_cpus)
    finally:
        if host_cpus is not None:
            os.sched_setaffinity(0, saved_affinity)


def _run_e2e(fa, args, q, k, v, g, lse, ws, causal, scale, flops_step, world, host_cpus):
    import torch

    hq, hk, hv, hg = (t.cpu().pin_memory() for t in (q, k, v, g))
    h_in = (hq, hk, hv, hg)
    e2e_steps = max(3, min(args.steps, 50))
    s_h2d, s_comp, s_d2h = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    sets = []
    for _ in range(2):
        din = [torch.empty_like(t) for t in (q, k, v, g)]
        dout = [torch.empty_like(q), torch.empty_like(lse), torch.empty_like(q), torch.empty_like(k),
                torch.empty_like(v)]  # o, lse, dq, dk, dv
        hout = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in dout]
        evs = {n: torch.cuda.Event() for n in ("in_ready", "in_free", "out_ready", "out_free")}
        sets.append((din, dout, hout, evs))

    def e2e_step(i):
        din, dout, hout, evs = sets[i % 2]
        with torch.cuda.stream(s_h2d):
            if i >= 2:
                s_h2d.wait_event(evs["in_free"])  # step i - 2 has finished reading these inputs
            for dst, src in zip(din, h_in):
                dst.copy_(src, non_blocking=True)
            evs["in_ready"].record(s_h2d)
        s_comp.wait_event(evs["in_ready"])
        if i >= 2:
            s_comp.wait_event(evs["out_free"])  # step i - 2's outputs have been copied out
        qi, ki, vi, gi = din
        o_, lse_, dq_, dk_, dv_ = dout
        fa.fa_fwd(qi, ki, vi, o=o_, lse=lse_, causal=causal, scale=scale, stream=s_comp)
        fa.fa_bwd(qi, ki, vi, o_, gi, lse_, dq_, dk_, dv_, ws, causal=causal, scale=scale, stream=s_comp)
        evs["in_free"].record(s_comp)
        evs["out_ready"].record(s_comp)
        with torch.cuda.stream(s_d2h):
            s_d2h.wait_event(evs["out_ready"])
            for dst, src in zip(hout, dout):
                dst.copy_(src, non_blocking=True)
            evs["out_free"].record(s_d2h)

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
    return {"value": round(flops_step / (e2e_ms * 1e-3) / 1e12 * world, 2), "unit": "TFLOP/s",
            "ms_per_step": round(e2e_ms, 4), "steps": e2e_steps, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h,
            "calls": "fa_fwd + fa_bwd per step; H2D of q, k, v, dO and D2H of o, lse, dq, dk, dv inside the "
                     "timed region, overlapped with the neighbouring steps' kernels",
            "host_cpus": (f"{len(host_cpus)} CPUs local to the GPU (NVML affinity)" if host_cpus
                          else "process affinity unchanged")}


# Rows past the headline, timed after it (not part of `value`): the causal step
# and the FP8 forward as stage objects; the split-KV decode forward and the
# 4-bit-weight GEMV on their own workloads; the deterministic backward and the
# FP8 backward on the headline / FP8 shapes.
DECODE = {"B": 8, "H": 16, "Nq": 1, "Nk": 32768, "d": 128, "causal": False, "seed": 5}
W4A16 = {"M": 1, "N": 28672, "K": 8192, "seed": 6}


def extra_rows(fa, args, q, k, v, g, o, lse, dq, dk, dv, ws, scale, flush, peaks, stage_info, rank):
    import torch

    from synth import normal_qkv, outlier_qkv, rotation_signs, w4a16_inputs

    peak, hbm = peaks["bf16_tflops"], peaks["hbm_gbs"]
    reps = max(5, min(args.steps, 20))
    B, H, N, d = q.shape
    out = {}

    # Causal forward and backward at the headline shape.
    calls = {
        "fwd": lambda: fa.fa_fwd(q, k, v, o=o, lse=lse, causal=True, scale=scale),
        "bwd_prep": lambda: fa.fa_bwd_prep(o, g, lse, ws),
        "bwd_main": lambda: fa.fa_bwd_main(q, k, v, g, dk, dv, ws, causal=True, scale=scale),
        "bwd_dq": lambda: fa.fa_bwd_dq(ws, dq, scale=scale),
    }
    for _ in range(3):
        for c in calls.values():
            c()
    cs = {}
    for st, c in calls.items():
        # Each stage reads what the previous ones wrote; they are timed one by one,
        # L2 flushed before each repetition.
        ms = _median_ms(c, reps, flush)
        info = stage_info[st]
        if info["bound"] == "tensor":
            cs[st] = _tensor_stage(ms, info["flops"] / 2, peak, info["kernel"].replace("false", "true"))
        else:
            cs[st] = _hbm_stage(ms, info["bytes"], hbm, info["kernel"])
    fa.fa_sync_check()
    f_c = fwd_flops(B, H, N, d, True)
    tot = sum(s["ms"] for s in cs.values())
    out["causal"] = {"workload": WORKLOAD["workload"].replace("non-causal", "causal"),
                     "tflops": round(3.5 * f_c / (tot * 1e-3) / 1e12, 1),
                     "frac_of_peak": round(3.5 * f_c / (tot * 1e-3) / 1e12 / peak, 4), "ms": round(tot, 5),
                     "stages": cs}

    # FP8 path on the FP8 workload.
    w8 = FP8_WORKLOAD
    B8, H8, N8, d8 = w8["B"], w8["H"], w8["N"], w8["d"]
    x8 = outlier_qkv(B8, H8, N8, d8, w8["seed"])
    q8, k8, v8 = (x8[n].cuda() for n in ("q", "k", "v"))
    del x8
    signs = rotation_signs(d8, w8["seed"]).cuda()
    ws8 = torch.empty(fa.fa_fp8_workspace_size(B8, H8, N8, d8), dtype=torch.uint8, device="cuda")
    o8 = torch.empty(B8, H8, N8, d8, dtype=torch.bfloat16, device="cuda")
    lse8 = torch.empty(B8, H8, N8, dtype=torch.float32, device="cuda")
    prep = lambda: fa.fa_fp8_prepare(q8, k8, v8, signs, ws8)
    for _ in range(3):
        prep()
    ms_prep = _median_ms(prep, reps, flush)
    el8 = B8 * H8 * N8 * d8
    fp8 = {"workload": w8["workload"], "config": {kk: w8[kk] for kk in ("B", "H", "N", "d", "seed")},
           "fp8_prepare": _hbm_stage(ms_prep, 3 * 4 * el8 + 3 * el8 + 3 * 4 * B8 * H8 * ((N8 + 63) // 64), hbm,
                                     "fp8_prepare_kernel<128>")}
    for c8 in (False, True):
        call = lambda: fa.fa_fwd_fp8(ws8, (B8, H8, N8, d8), o=o8, lse=lse8, causal=c8, scale=d8 ** -0.5)
        for _ in range(3):
            call()
        ms = _median_ms(call, reps, flush)
        r = _tensor_stage(ms, fwd_flops(B8, H8, N8, d8, c8), 2.0 * peak, f"fwd_kernel<128,{str(c8).lower()},fp8>",
                          bound="tensor_fp8")
        r["peak_source"] = f"2 x {peaks['source']} bf16_tflops (the nominal FP8/bf16 ratio)"
        r["tflops_with_prepare"] = round(fwd_flops(B8, H8, N8, d8, c8) / ((ms + ms_prep) * 1e-3) / 1e12, 1)
        fp8["fwd_fp8_causal" if c8 else "fwd_fp8"] = r
    fa.fa_sync_check()
    out["fp8"] = fp8

    if rank != 0:
        return out
    nxt = {}
    # Split-KV decode: one query row against 32768 keys (K and V, 2.1 GB, far beyond L2).
    wd = DECODE
    Bd, Hd, Nq, Nk, dd = wd["B"], wd["H"], wd["Nq"], wd["Nk"], wd["d"]
    kv = normal_qkv(Bd, Hd, Nk, dd, wd["seed"])
    qd = normal_qkv(Bd, Hd, Nq, dd, wd["seed"] + 1)["q"].to(torch.bfloat16).cuda()
    kd, vd = kv["k"].to(torch.bfloat16).cuda(), kv["v"].to(torch.bfloat16).cuda()
    del kv
    n = fa.fa_splitkv_default_splits(Bd, Hd, Nq, Nk, dd)
    wsd = torch.empty(fa.fa_splitkv_workspace_size(Bd, Hd, Nq, dd, n), dtype=torch.uint8, device="cuda")
    od = torch.empty_like(qd)
    lsed = torch.empty(Bd, Hd, Nq, dtype=torch.float32, device="cuda")
    call = lambda: fa.fa_fwd_splitkv(qd, kd, vd, od, lsed, wsd, n_split=n, causal=wd["causal"])
    for _ in range(3):
        call()
    ms = _median_ms(call, 20)
    byts = 4 * Bd * Hd * Nk * dd + 4 * Bd * Hd * Nq * dd + 8 * n * Bd * Hd * Nq * (dd + 1)
    r = _hbm_stage(ms, byts, hbm, "fwd_kernel<128,false,bf16,split> + merge_kernel<128>")
    r.update(workload="split-KV decode forward + merge", config=dict(wd, n_split=n), gpu_launches=2)
    nxt["splitkv_decode"] = r
    del kd, vd
    f_bwd = 2.5 * fwd_flops(B, H, N, d, False)
    det = lambda: fa.fa_bwd(q, k, v, o, g, lse, dq, dk, dv, ws, causal=False, scale=scale, deterministic=True)
    fa.fa_fwd(q, k, v, o=o, lse=lse, causal=False, scale=scale)
    for _ in range(3):
        det()
    ms_det = _median_ms(det, reps, flush)
    plain = lambda: fa.fa_bwd(q, k, v, o, g, lse, dq, dk, dv, ws, causal=False, scale=scale)
    ms_plain = _median_ms(plain, reps, flush)
    fa.fa_sync_check()
    nxt["bwd_deterministic"] = {"workload": "bf16 backward with order-free dQ, the headline shape (non-causal)",
                                "ms": round(ms_det, 5), "tflops": round(f_bwd / (ms_det * 1e-3) / 1e12, 1),
                                "ms_atomic_dq": round(ms_plain, 5), "gpu_launches": 4}
    # FP8 backward on the FP8 workspace (FP8 workload) with a seeded dO.
    g8 = normal_qkv(B8, H8, N8, d8, w8["seed"] + 1)["q"].to(torch.bfloat16).cuda()
    fa.fa_fwd_fp8(ws8, (B8, H8, N8, d8), o=o8, lse=lse8, causal=False, scale=d8 ** -0.5)
    wsb = torch.empty(fa.fa_bwd_fp8_workspace_size(B8, H8, N8, d8), dtype=torch.uint8, device="cuda")
    dq8, dk8, dv8 = (torch.empty_like(o8) for _ in range(3))
    f_bwd8 = 2.5 * fwd_flops(B8, H8, N8, d8, False)
    res = {}
    for rec in (False, True):
        call = lambda: fa.fa_bwd_fp8(ws8, signs, o8, g8, lse8, dq8, dk8, dv8, wsb, causal=False, scale=d8 ** -0.5,
                                     recompute_forward=rec)
        for _ in range(3):
            call()
        res[rec] = _median_ms(call, reps, flush)
    fa.fa_sync_check()
    nxt["bwd_fp8"] = {"workload": "FP8 backward (straight-through: dequantise, bf16 backward, inverse rotation), "
                                  "the FP8 workload, with fa_fwd_fp8's O and LSE",
                      "ms": round(res[False], 5), "tflops": round(f_bwd8 / (res[False] * 1e-3) / 1e12, 1),
                      "ms_recompute_forward": round(res[True], 5),
                      "tflops_recompute_forward": round(f_bwd8 / (res[True] * 1e-3) / 1e12, 1), "gpu_launches": 5}
    del wsb, dq8, dk8, dv8, g8
    # W4A16 decode GEMV: 28672 x 8192 packed weights (117 MB, beyond L2) times one activation row.
    ww = W4A16
    xin = w4a16_inputs(ww["M"], ww["N"], ww["K"], ww["seed"])
    xw, wq, sc, zr = (xin[nn].cuda() for nn in ("x", "wq", "scales", "zeros"))
    nsp = fa.fa_w4a16_default_splits(ww["M"], ww["N"], ww["K"])
    wsw = torch.empty(max(fa.fa_w4a16_workspace_size(ww["M"], ww["N"], ww["K"], nsp), 1), dtype=torch.uint8,
                      device="cuda")
    y = torch.empty(ww["M"], ww["N"], dtype=torch.float16, device="cuda")
    call = lambda: fa.fa_w4a16_gemm(xw, wq, sc, zr, y, wsw, n_split=nsp)
    for _ in range(3):
        call()
    ms_w = _median_ms(call, 20, flush)
    fa.fa_sync_check()
    M_, N_, K_ = ww["M"], ww["N"], ww["K"]
    byts = N_ * K_ // 2 + 3 * N_ * K_ // 128 + 2 * M_ * K_ + 2 * M_ * N_
    r = _hbm_stage(ms_w, byts, hbm, "w4a16_gemv_kernel")
    r.update(workload="W4A16 dequantising GEMV (4-bit weights, group 128, fp16 activations)",
             config=dict(ww, n_split=nsp), gpu_launches=2 if nsp > 1 else 1)
    nxt["w4a16_gemv"] = r
    out["next"] = nxt
    return out


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

    from synth import normal_qkv

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


SWEEP_FWD = ([(1, 2, 128, 64), (4, 16, 2048, 128)]
             + [(16384 // n, 32, n, 64) for n in (512, 1024, 2048, 4096, 8192, 16384)]
             + [(16384 // n, 16, n, 128) for n in (512, 1024, 2048, 4096, 8192, 16384)])
SWEEP_BWD = [(8, 16, 2048, 128), (2, 16, 8192, 128), (8, 32, 2048, 64), (2, 32, 8192, 64)]
SWEEP_DECODE = [(8, 16, 1, 32768, 128), (1, 16, 1, 131072, 128), (8, 32, 1, 32768, 64), (4, 16, 16, 32768, 128),
                (1, 16, 128, 65536, 128)]
SWEEP_W4A16 = [(1, 28672, 8192), (16, 28672, 8192), (64, 28672, 8192), (128, 28672, 8192), (1, 8192, 28672)]


def run_sweep(args):
    """Every configuration of the forward sweep, the backward, FP8, decode and W4A16 rows, one JSON line each.

    Each row is the median of `reps` launches of the public call, with L2 flushed
    (256 MB write) before each launch, outside the event pair.  Inputs are seeded
    and synthetic, shaped as the workload names them.  --sweep-filter keeps the
    rows whose tags (the row's words and key=value pairs of its configuration)
    contain every token of the filter.
    """
    import torch

    import io_aware_exact_fwd_gb300 as fa
    from synth import normal_qkv, outlier_qkv, rotation_signs, w4a16_inputs

    fa.load_library()
    peaks = load_peaks()
    peak, hbm = peaks["bf16_tflops"], peaks["hbm_gbs"]
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    reps = max(5, min(args.steps, 20))
    tokens = (args.sweep_filter or "").split()

    def want(row, cfg):
        tags = row.split() + [f"{k}={int(v) if isinstance(v, bool) else v}" for k, v in cfg.items()]
        return all(t in tags for t in tokens)

    def emit(row, cfg, ms, amount, unit, pk, **kw):
        ach = amount / (ms * 1e-3) / (1e12 if unit == "TFLOP/s" else 1e9)
        line = {"row": row, "config": cfg, "ms": round(ms, 5), "achieved": round(ach, 1), "unit": unit, "peak": pk,
                "frac": round(ach / pk, 4)}
        line.update(kw)
        print(json.dumps(line), flush=True)

    def timed(call):
        for _ in range(3):
            call()
        ms = _median_ms(call, reps, flush)
        fa.fa_sync_check()
        return ms

    def bf16_inputs(B, H, N, d, seed, with_do=False):
        x = normal_qkv(B, H, N, d, seed, with_do=with_do)
        return {n: t.to(torch.bfloat16).cuda() for n, t in x.items()}

    for (B, H, N, d) in SWEEP_FWD:
        cfgs = [{"B": B, "H": H, "N": N, "d": d, "causal": c} for c in (False, True)]
        cfgs = [c for c in cfgs if want("bf16 forward", c)]
        if not cfgs:
            continue
        x = bf16_inputs(B, H, N, d, 2)
        o = torch.empty_like(x["q"])
        lse = torch.empty(B, H, N, dtype=torch.float32, device="cuda")
        for cfg in cfgs:
            c = cfg["causal"]
            ms = timed(lambda: fa.fa_fwd(x["q"], x["k"], x["v"], o=o, lse=lse, causal=c))
            emit("bf16 forward", cfg, ms, fwd_flops(B, H, N, d, c), "TFLOP/s", peak)
        del x, o, lse

    for (B, H, N, d) in SWEEP_BWD:
        rows = [("bf16 backward" + (" deterministic" if det else ""), {"B": B, "H": H, "N": N, "d": d, "causal": c},
                 det) for c in (False, True) for det in (False, True)]
        rows = [r for r in rows if want(r[0], r[1])]
        if not rows:
            continue
        x = bf16_inputs(B, H, N, d, 3, with_do=True)
        q, k, v, g = x["q"], x["k"], x["v"], x["do"]
        o = torch.empty_like(q)
        lse = torch.empty(B, H, N, dtype=torch.float32, device="cuda")
        dq, dk, dv = (torch.empty_like(q) for _ in range(3))
        ws = torch.empty(fa.fa_bwd_workspace_size(B, H, N, d), dtype=torch.uint8, device="cuda")
        for row, cfg, det in rows:
            c = cfg["causal"]
            fa.fa_fwd(q, k, v, o=o, lse=lse, causal=c)
            ms = timed(lambda: fa.fa_bwd(q, k, v, o, g, lse, dq, dk, dv, ws, causal=c, deterministic=det))
            emit(row, cfg, ms, 2.5 * fwd_flops(B, H, N, d, c), "TFLOP/s", peak, launches=4 if det else 3)
        del x, q, k, v, g, o, lse, dq, dk, dv, ws

    w8 = FP8_WORKLOAD
    for d8 in (w8["d"],):
        B8, H8, N8 = w8["B"], w8["H"], w8["N"]
        cfg8 = {"B": B8, "H": H8, "N": N8, "d": d8}
        fwd_cfgs = [dict(cfg8, causal=c) for c in (False, True) if want("FP8 forward", dict(cfg8, causal=c))]
        if not (want("FP8 prepare (fp32 in)", cfg8) or fwd_cfgs):
            continue
        x8 = outlier_qkv(B8, H8, N8, d8, w8["seed"])
        q8, k8, v8 = (x8[n].cuda() for n in ("q", "k", "v"))
        del x8
        signs = rotation_signs(d8, w8["seed"]).cuda()
        ws8 = torch.empty(fa.fa_fp8_workspace_size(B8, H8, N8, d8), dtype=torch.uint8, device="cuda")
        o8 = torch.empty(B8, H8, N8, d8, dtype=torch.bfloat16, device="cuda")
        lse8 = torch.empty(B8, H8, N8, dtype=torch.float32, device="cuda")
        el8 = B8 * H8 * N8 * d8
        ms_prep = timed(lambda: fa.fa_fp8_prepare(q8, k8, v8, signs, ws8))
        if want("FP8 prepare (fp32 in)", cfg8):
            emit("FP8 prepare (fp32 in)", cfg8, ms_prep,
                 3 * 4 * el8 + 3 * el8 + 3 * 4 * B8 * H8 * ((N8 + 63) // 64), "GB/s", hbm)
        for cfg in fwd_cfgs:
            c = cfg["causal"]
            ms = timed(lambda: fa.fa_fwd_fp8(ws8, (B8, H8, N8, d8), o=o8, lse=lse8, causal=c, scale=d8 ** -0.5))
            f = fwd_flops(B8, H8, N8, d8, c)
            emit("FP8 forward", cfg, ms, f, "TFLOP/s", 2.0 * peak,
                 tflops_with_prepare=round(f / ((ms + ms_prep) * 1e-3) / 1e12, 1))
        del q8, k8, v8, ws8, o8, lse8

    for (B, H, Nq, Nk, d) in SWEEP_DECODE:
        cfg = {"B": B, "H": H, "Nq": Nq, "Nk": Nk, "d": d}
        if not want("split-KV decode + merge", cfg):
            continue
        kv = normal_qkv(B, H, Nk, d, 5)
        k, v = kv["k"].to(torch.bfloat16).cuda(), kv["v"].to(torch.bfloat16).cuda()
        del kv
        q = normal_qkv(B, H, Nq, d, 6)["q"].to(torch.bfloat16).cuda()
        n = fa.fa_splitkv_default_splits(B, H, Nq, Nk, d)
        ws = torch.empty(fa.fa_splitkv_workspace_size(B, H, Nq, d, n), dtype=torch.uint8, device="cuda")
        o = torch.empty_like(q)
        lse = torch.empty(B, H, Nq, dtype=torch.float32, device="cuda")
        ms = timed(lambda: fa.fa_fwd_splitkv(q, k, v, o, lse, ws, n_split=n))
        byts = 4 * B * H * Nk * d + 4 * B * H * Nq * d + 8 * n * B * H * Nq * (d + 1)
        emit("split-KV decode + merge", dict(cfg, n_split=n), ms, byts, "GB/s", hbm)
        del k, v, q, ws, o, lse

    for (M, N, K) in SWEEP_W4A16:
        cfg = {"M": M, "N": N, "K": K}
        if not want("W4A16 GEMM", cfg):
            continue
        xin = w4a16_inputs(M, N, K, 6)
        xw, wq, sc, zr = (xin[nn].cuda() for nn in ("x", "wq", "scales", "zeros"))
        nsp = fa.fa_w4a16_default_splits(M, N, K)
        wsw = torch.empty(max(fa.fa_w4a16_workspace_size(M, N, K, nsp), 1), dtype=torch.uint8, device="cuda")
        y = torch.empty(M, N, dtype=torch.float16, device="cuda")
        ms = timed(lambda: fa.fa_w4a16_gemm(xw, wq, sc, zr, y, wsw, n_split=nsp))
        byts = N * K // 2 + 3 * N * K // 128 + 2 * M * K + 2 * M * N
        emit("W4A16 GEMM", dict(cfg, n_split=nsp), ms, byts, "GB/s", hbm,
             tflops=round(2.0 * M * N * K / (ms * 1e-3) / 1e12, 1))
        del xw, wq, sc, zr, wsw, y


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--step-only", action="store_true",
                    help="time the headline step alone (for profiler captures): no e2e, extra rows or CPU baseline")
    ap.add_argument("--sweep", action="store_true",
                    help="time every configuration of the sweep tables (one JSON line per row) instead of the step")
    ap.add_argument("--sweep-filter", default=None,
                    help="with --sweep: only the rows whose tags contain every token, e.g. 'forward N=8192 d=64'")
    ap.add_argument("--traffic", type=float, default=None,
                    help="DRAM bytes per launch of the dominant kernel from an ncu capture of this kernel version")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    elif args.sweep:
        run_sweep(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
