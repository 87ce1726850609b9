"""Helpers shared by the GPU parity tests (input marshalling, error metrics and a per-head thread pool)."""

from __future__ import annotations

import concurrent.futures as cf
import os

import numpy as np
import torch

# Tolerances of the bf16 paths, as stated for this library's parity contract.
FWD_O_ATOL = 1e-2
FWD_LSE_ATOL = 1e-3
BWD_REL = 2e-2

# Measured error metrics of the parity tests, printed in pytest's terminal summary
# (tests/conftest.py) so that a GPU run records them next to pass/fail.
REPORT: dict[str, dict] = {}


def report(name: str, **values):
    REPORT[name] = {k: (float(v) if isinstance(v, (float, np.floating)) else v) for k, v in values.items()}


def to_dev_bf16(x: dict, names=("q", "k", "v")):
    """bf16 device copies of fp32 CPU tensors; the oracle is evaluated on these same bf16 values."""
    return [x[n].to(torch.bfloat16).cuda() for n in names]


def host_f64(t) -> np.ndarray:
    """Exact float64 host copy of a (device or host) tensor."""
    return t.detach().to("cpu", torch.float64).numpy() if isinstance(t, torch.Tensor) else np.asarray(t, np.float64)


def _f64(a):
    return host_f64(a)


def bf16_half_ulp(x):
    """Half the spacing of bf16 numbers around each |x| (8 significant bits): 2^(floor(log2|x|) - 8)."""
    ax = np.abs(np.asarray(x, dtype=np.float64))
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(ax > 0, ax, 1.0)))
    return np.where(ax > 0, 2.0 ** (e - 8), 0.0)


def o_excess(o, o_ref) -> float:
    """max over elements of |O - O_ref| beyond the rounding of O_ref itself to the bf16 output.

    O is returned in bf16, so even the exact result carries up to half a bf16 ulp
    of error (0.0156 for |O| in [4, 8)), which alone can exceed an absolute 1e-2.
    The forward tolerance therefore applies to the kernel's error on top of that
    unavoidable output rounding: max(0, |O - O_ref| - half_ulp_bf16(O_ref)).
    """
    a, b = _f64(o), _f64(o_ref)
    if a.size == 0:
        return 0.0
    return float(np.maximum(np.abs(a - b) - bf16_half_ulp(b), 0.0).max())


def max_abs(a, b) -> float:
    a, b = _f64(a), _f64(b)
    return float(np.abs(a - b).max()) if a.size else 0.0


def rel_max(x, ref, floor: float = 1e-4) -> float:
    """max|x - ref| / max|ref| (the backward's metric); the reference magnitude is floored at ``floor``."""
    x, ref = _f64(x), _f64(ref)
    return float(np.abs(x - ref).max() / max(np.abs(ref).max(), floor))


def rel_rmse(x, ref) -> float:
    """RMSE(x - ref) / RMS(ref) over all elements."""
    x, ref = _f64(x), _f64(ref)
    return float(np.sqrt(((x - ref) ** 2).mean()) / np.sqrt((ref ** 2).mean()))


def map_heads(fn, heads, workers: int | None = None):
    """[fn(b, h) for (b, h) in heads], evaluated on a thread pool.

    The oracle is numpy; its matrix products and element-wise kernels release the
    GIL, so heads evaluated on threads use the host's cores.  Threads (not
    processes) keep this safe after the CUDA context exists.
    """
    heads = list(heads)
    workers = workers or min(len(heads), max(1, len(os.sched_getaffinity(0))))
    if workers <= 1:
        return [fn(b, h) for b, h in heads]
    with cf.ThreadPoolExecutor(max_workers=workers) as ex:
        return list(ex.map(lambda bh: fn(*bh), heads))


def all_heads(B: int, H: int):
    return [(b, h) for b in range(B) for h in range(H)]


def edge_heads(B: int, H: int):
    """The first and the last head (b, h), plus one from the middle when there are more than two."""
    heads = [(0, 0), (B - 1, H - 1)]
    mid = ((B * H) // 2 // H, (B * H) // 2 % H)
    if B * H > 2 and mid not in heads:
        heads.insert(1, mid)
    return heads
