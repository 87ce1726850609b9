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


def max_abs(a, b) -> float:
    a = a.float().cpu().numpy() if isinstance(a, torch.Tensor) else np.asarray(a)
    b = b.float().cpu().numpy() if isinstance(b, torch.Tensor) else np.asarray(b)
    return float(np.abs(a.astype(np.float64) - b.astype(np.float64)).max()) if a.size else 0.0
