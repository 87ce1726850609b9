"""Seeded synthetic inputs for the attention workloads.

This module only draws random numbers and arranges them into tensors; it holds
none of the attention arithmetic, so both the CUDA path's tests and the oracle's
tests can take their inputs from it.  Every draw uses a CPU
``torch.Generator`` seeded explicitly, in a fixed order (Q, K, V, dO, then the
outlier positions of Q, K, V; the rotation signs come from a generator of
their own), so the same seed gives
the same tensors on every machine.
"""

from __future__ import annotations

import torch


def normal_qkv(B: int, H: int, N: int, d: int, seed: int, with_do: bool = False):
    """Q, K, V (and dO) ~ N(0, 1), fp32 CPU tensors of shape [B, H, N, d]."""
    g = torch.Generator().manual_seed(seed)
    shape = (B, H, N, d)
    out = {name: torch.randn(shape, generator=g, dtype=torch.float32) for name in ("q", "k", "v")}
    if with_do:
        out["do"] = torch.randn(shape, generator=g, dtype=torch.float32)
    return out


def outlier_qkv(B: int, H: int, N: int, d: int, seed: int, frac: float = 0.001,
                factor: float = 20.0):
    """Q, K, V ~ N(0, 1) with exactly round(frac * numel) entries per tensor multiplied by ``factor``.

    The outlier positions of each tensor are the first round(frac * numel) entries
    of a seeded random permutation (uniform, without replacement).  Returns fp32
    CPU tensors [B, H, N, d] and the positions used.
    """
    g = torch.Generator().manual_seed(seed)
    shape = (B, H, N, d)
    t = {name: torch.randn(shape, generator=g, dtype=torch.float32) for name in ("q", "k", "v")}
    numel = B * H * N * d
    count = int(round(frac * numel))
    positions = {}
    for name in ("q", "k", "v"):
        idx = torch.randperm(numel, generator=g)[:count]
        flat = t[name].view(-1)
        flat[idx] *= factor
        positions[name] = idx
    t["positions"] = positions
    return t


def rotation_signs(d: int, seed: int) -> torch.Tensor:
    """A seeded vector of d random signs (+1 / -1) as int8, from its own generator derived from ``seed``."""
    g = torch.Generator().manual_seed(seed * 7919 + 17)
    bits = torch.randint(0, 2, (d,), generator=g)
    return (bits * 2 - 1).to(torch.int8)


def w4a16_inputs(M: int, N: int, K: int, seed: int, group: int = 128):
    """Seeded inputs of the 4-bit-weight GEMM: activations and random packed weights.

    x: fp16 [M, K] ~ N(0, 1).  wq: int32 [N, K / 8] of uniformly random bits (so
    every 4-bit code is uniform on 0..15; how the bits map to codes is the
    kernel's interface, not this module's).  scales: fp16 [K / group, N], uniform
    on [0.005, 0.02].  zeros: uint8 [K / group, N], uniform integers 0..15.
    CPU tensors.
    """
    g = torch.Generator().manual_seed(seed)
    x = torch.randn((M, K), generator=g, dtype=torch.float32).to(torch.float16)
    wq = torch.randint(-(2 ** 31), 2 ** 31, (N, K // 8), generator=g, dtype=torch.int64).to(torch.int32)
    scales = (0.005 + 0.015 * torch.rand((K // group, N), generator=g)).to(torch.float16)
    zeros = torch.randint(0, 16, (K // group, N), generator=g, dtype=torch.int64).to(torch.uint8)
    return {"x": x, "wq": wq, "scales": scales, "zeros": zeros}
