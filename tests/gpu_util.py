"""Helpers shared by the GPU parity tests (input marshalling and error metrics only)."""

from __future__ import annotations

import numpy as np
import torch

# Tolerances of the bf16 paths, as stated for this library's parity contract.
FWD_O_ATOL = 1e-2
FWD_LSE_ATOL = 1e-3
BWD_REL = 2e-2


def to_dev_bf16(x: dict, names=("q", "k", "v")):
    """bf16 device copies of fp32 CPU tensors; the oracle is evaluated on these same bf16 values."""
    return [x[n].to(torch.bfloat16).cuda() for n in names]


def _f64(a):
    return (a.float().cpu().numpy() if isinstance(a, torch.Tensor) else np.asarray(a)).astype(np.float64)


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
    a = a.float().cpu().numpy() if isinstance(a, torch.Tensor) else np.asarray(a)
    b = b.float().cpu().numpy() if isinstance(b, torch.Tensor) else np.asarray(b)
    return float(np.abs(a.astype(np.float64) - b.astype(np.float64)).max()) if a.size else 0.0
