"""4-bit-weight, 16-bit-activation matrix product (W4A16), float64 numpy (test infrastructure).

What the pages describe ("FlashAttention-Skalierung, Multi-GPU-Training und
Gewichtsquantisierung", section 3, "Wie spezielle CUDA-Kernels während der
Ausführung dequantisieren (W4A16)"): weights are stored as 4-bit integers, eight
per 32-bit word, and read from memory in that packed form; the kernel takes them
apart with shifts and masks, applies stored scale and zero-point factors to turn
them back into fp16 values, and feeds those with fp16 activations to the tensor
cores, never writing the unpacked weights back to memory.

This module restates that computation directly:

    q[n, k]  = 4-bit code of weight (n, k)                       (0 .. 15)
    W[n, k]  = fp16( (q[n, k] - z[g, n]) * s[g, n] ),  g = k // 128
    Y[m, n]  = sum_k X[m, k] * W[n, k]                            (exact here)

Readings (the pages name the ingredients but fix no format):
* group size 128 along K, one fp16 scale s and one integer zero point z (0..15)
  per (group, output row), stored group-major: s, z of shape [K / 128, N];
* packing: word w of row n holds k = 8w .. 8w+7; the code of k = 8w + 2i sits in
  bits 4i .. 4i+3 and that of k = 8w + 2i + 1 in bits 4i+16 .. 4i+19 (i = 0..3),
  so one shift and one mask deliver the codes of a consecutive pair;
* the dequantised weight is the fp16 rounding of the exact (q - z) s: the pages
  have the kernel build fp16 weights, and (q - z) is an exact small integer.
"""

from __future__ import annotations

import numpy as np

GROUP = 128


def _np(x):
    if hasattr(x, "detach"):
        x = x.detach().cpu().numpy()
    return np.asarray(x)


def w4a16_unpack(wq) -> np.ndarray:
    """Codes q [N, K] (int64, 0..15) from packed words [N, K / 8] (any 32-bit integer dtype)."""
    w = _np(wq).astype(np.int64) & 0xFFFFFFFF
    N, W = w.shape
    q = np.empty((N, 8 * W), dtype=np.int64)
    for i in range(4):
        q[:, 2 * i::8] = (w >> (4 * i)) & 0xF           # k = 8w + 2i
        q[:, 2 * i + 1::8] = (w >> (4 * i + 16)) & 0xF  # k = 8w + 2i + 1
    return q


def w4a16_dequant(wq, scales, zeros) -> np.ndarray:
    """Dequantised weights W [N, K]: fp16((q - z) s), returned as float64 values."""
    q = w4a16_unpack(wq)
    s = _np(scales).astype(np.float64)          # [K / 128, N]
    z = _np(zeros).astype(np.int64)             # [K / 128, N]
    g = np.arange(q.shape[1]) // GROUP          # group of every k
    exact = (q - z.T[:, g]) * s.T[:, g]         # (q - z) exact, one product
    return exact.astype(np.float16).astype(np.float64)


def w4a16_gemm(x, wq, scales, zeros) -> np.ndarray:
    """Y [M, N] = X W^T in float64 (the products of fp16 values are exact)."""
    xd = _np(x).astype(np.float64)
    return xd @ w4a16_dequant(wq, scales, zeros).T


def w4a16_abs_sum(x, wq, scales, zeros) -> np.ndarray:
    """sum_k |X[m, k] W[n, k]| (for the floating-point error bound of a kernel's sum)."""
    xd = np.abs(_np(x).astype(np.float64))
    return xd @ np.abs(w4a16_dequant(wq, scales, zeros)).T


__all__ = ["GROUP", "w4a16_unpack", "w4a16_dequant", "w4a16_gemm", "w4a16_abs_sum"]
