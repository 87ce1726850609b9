"""Backward pass of the FP8 attention, float64 numpy (test infrastructure).

Source of the forward it differentiates: "FlashAttention-Skalierung,
Multi-GPU-Training und Gewichtsquantisierung", section 1, bullet "Unterstützung
geringer FP8-Präzision" (block-quantised FP8 operands, Q and K multiplied by a
random orthogonal matrix first).  The pages give FP8 for the forward only; the
readings taken for its backward are:

* Straight-through quantisation.  The derivative of the rounding to e4m3 is taken
  as 1 (its true derivative is zero almost everywhere), so the gradient is that of
  exact attention on the dequantised operands, carried back through the rotation.
  With the unnormalised rotation M = diag(s) H_d of the forward (the 1/d it leaves
  in Q' K'^T is folded into the scores' scale):

      Q' ~ Q M,  K' ~ K M,  S = (scale / d) Q' K'^T,  O = softmax(S) V'
      dQ = dQ' M^T = (dQ' H_d) * s,   dK = (dK' H_d) * s,   dV = dV'

  where dQ', dK', dV' are the textbook attention gradients with respect to the
  operands Q', K', V' (``attention_backward``).
* Operand precision.  The backward's products take the dequantised operands as
  bf16 values: decode(code) times the tile's fp32 scale as one fp32 product, then
  rounded to the nearest bf16 (ties to even).  This is a rounding the kernel
  performs, so the oracle performs the same one and both sides see the same
  operand values.
"""

from __future__ import annotations

import numpy as np

from .attention import attention_backward, attention_backward_sampled, attention_forward
from .fp8 import e4m3_decode, sylvester_hadamard


def bf16_round(x) -> np.ndarray:
    """Round fp32 values to the nearest bf16 (ties to even); returned as float64.

    bf16 keeps the upper 16 bits of the fp32 pattern.  Round to nearest even on
    the 16 dropped bits: add 0x7FFF plus the lowest kept bit, then truncate.  An
    overflow of the exponent field gives infinity, as IEEE rounding does.  NaN
    stays NaN.
    """
    x32 = np.asarray(x, dtype=np.float32)
    u = x32.view(np.uint32).astype(np.uint64)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000).astype(np.uint32)
    out = r.view(np.float32).astype(np.float64)
    return np.where(np.isnan(x32), np.nan, out)


def fp8_dequantize_bf16(codes, sigma, tile: int = 64) -> np.ndarray:
    """bf16(fp32(decode(code)) * sigma) per element, sigma the fp32 scale of the row's tile.

    codes: uint8 e4m3 [..., N, d]; sigma: float32 [..., ceil(N / tile)].
    """
    vals = e4m3_decode(codes).astype(np.float32)      # exact: e4m3 values fit fp32
    N = np.asarray(codes).shape[-2]
    sig = np.asarray(sigma, dtype=np.float32)[..., np.arange(N) // tile][..., None]
    return bf16_round(vals * sig)                      # one fp32 product, then RNE to bf16


def fp8_operands(prep: dict, tile: int = 64):
    """The backward's operands (Q', K', V') from ``fp8_prepare``'s codes and scales."""
    return (fp8_dequantize_bf16(prep["q8"], prep["sq"], tile),
            fp8_dequantize_bf16(prep["k8"], prep["sk"], tile),
            fp8_dequantize_bf16(prep["v8"], prep["sv"], tile))


def fp8_backward_from_operands(qr, kr, v, do, signs, scale: float, causal: bool):
    """(dQ, dK, dV) with respect to the unrotated inputs, from rotated operands Q', K', V.

    qr, kr, v, do: [B, H, N, d]; signs: [d] of +-1; ``scale`` is the softmax scale
    of the unrotated problem (the operands' scores carry scale / d).
    """
    qr = np.asarray(qr, dtype=np.float64)
    d = qr.shape[-1]
    dqr, dkr, dv = attention_backward(qr, kr, v, do, scale / d, causal)
    hd = sylvester_hadamard(d)
    s = np.asarray(signs, dtype=np.float64).reshape(-1)
    return (dqr @ hd) * s, (dkr @ hd) * s, dv


def fp8_backward(prep: dict, signs, do, scale: float, causal: bool, tile: int = 64):
    """Straight-through backward of the FP8 attention from the prepared codes.

    Returns (dQ, dK, dV, O, LSE); O and LSE are the exact forward on the same
    operands (what the backward's softmax recomputation is relative to).
    """
    qr, kr, vr = fp8_operands(prep, tile)
    d = qr.shape[-1]
    o, lse = attention_forward(qr, kr, vr, scale / d, causal)
    dq, dk, dv = fp8_backward_from_operands(qr, kr, vr, do, signs, scale, causal)
    return dq, dk, dv, o, lse


def fp8_backward_sampled(qr_head, kr_head, v_head, do_head, signs, scale: float, causal: bool, rows, keys):
    """dQ at selected rows and dK, dV at selected keys of ONE head, from its operands.

    The same definition as ``fp8_backward_from_operands`` evaluated for the chosen
    rows and keys only (``attention_backward_sampled``), then carried back through
    the rotation.  Returns (dQ[len(rows), d], dK[len(keys), d], dV[len(keys), d]).
    """
    d = np.asarray(qr_head).shape[-1]
    dqr, dkr, dv = attention_backward_sampled(qr_head, kr_head, v_head, do_head, scale / d, causal, rows, keys)
    hd = sylvester_hadamard(d)
    s = np.asarray(signs, dtype=np.float64).reshape(-1)
    return (dqr @ hd) * s, (dkr @ hd) * s, dv


__all__ = ["bf16_round", "fp8_dequantize_bf16", "fp8_operands", "fp8_backward_from_operands", "fp8_backward",
           "fp8_backward_sampled"]
