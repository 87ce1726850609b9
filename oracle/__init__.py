"""Plain CPU oracle for exact attention (test infrastructure only).

This package is test infrastructure.  It is a slow, deliberately simple float64
restatement of what the attention path computes, written so that a reader can
check it against the pages by eye:

* ``attention``  -- the textbook definition O = softmax(scale * Q K^T [+causal]) V,
  the per-row logsumexp, and the analytic backward (dQ, dK, dV).  Source of the
  definition: "FlashAttention-2 (DE)", section "Hintergrund: Das Attention-Problem
  in Transformern" (standard self-attention, O(N^2) time and memory); the
  article's lead and its section "Leistung und Effizienz" state that the tiled
  method loses no accuracy against it (the same result up to rounding, and a
  deterministic one).  So the oracle is the definition itself, never an online or
  tiled softmax.
* ``brute``      -- a scalar triple-loop twin of ``attention`` for tiny inputs.
* ``splitkv``    -- attention partials over key ranges and their exact merge
  (LSE = ln sum_s exp LSE_s, O = sum_s exp(LSE_s - LSE) O_s), with causal
  queries aligned to the last keys when Nq < Nk.  Source of the setting:
  "FlashAttention-Skalierung, Multi-GPU-Training und Gewichtsquantisierung",
  section 3 (token-by-token inference is bandwidth-bound); the merge itself is
  the softmax definition split over key ranges.
* ``w4a16``      -- the 4-bit-weight GEMM of "FlashAttention-Skalierung, Multi-GPU-Training
  und Gewichtsquantisierung", section 3 (W4A16): unpack eight 4-bit codes per
  32-bit word, dequantise with per-group scale and zero point to fp16, multiply
  with fp16 activations.
* ``fp8``        -- the FP8 input preparation: random-sign Walsh-Hadamard rotation
  of Q and K (incoherent processing) and per-tile block quantisation to OCP e4m3.
  Source: "FlashAttention-Skalierung, Multi-GPU-Training und
  Gewichtsquantisierung", section 1, bullet "Unterstützung geringer
  FP8-Präzision".
* ``fp8_backward`` -- the straight-through backward of that FP8 attention: the
  textbook gradient on the dequantised operands (rounded to bf16), carried back
  through the rotation (dQ = (dQ' H) * s, dK likewise).  The pages give FP8 for
  the forward only; this is the plainest reading of its backward.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package.  The product
path (``io_aware_exact_fwd_gb300``) never imports it, and this package imports
nothing from the product path.  Every function here is pinned by CPU tests
against closed forms, invariants, brute force or library special cases; none is
"parity unpinned".
"""

from .attention import (
    attention_forward,
    attention_forward_rows,
    attention_backward,
    attention_backward_sampled,
    attention_backward_rows,
)
from .brute import attention_forward_brute
from .splitkv import (
    split_key_ranges,
    attention_partial,
    attention_splitkv,
    merge_partials,
    attention_general,
    splitkv_flops,
)
from .w4a16 import w4a16_unpack, w4a16_dequant, w4a16_gemm, w4a16_abs_sum
from .fp8 import (
    sylvester_hadamard,
    fwht_f32,
    e4m3_encode,
    e4m3_decode,
    e4m3_round,
    fp8_prepare,
    fp8_dequantize,
    pow2_scale_exponent,
    splitmix64,
    seeded_rotation_signs,
    E4M3_MAX,
)
from .fp8_backward import (
    bf16_round,
    fp8_dequantize_bf16,
    fp8_operands,
    fp8_backward_from_operands,
    fp8_backward,
)

__all__ = [
    "attention_forward",
    "attention_forward_rows",
    "attention_backward",
    "attention_backward_sampled",
    "attention_backward_rows",
    "attention_forward_brute",
    "split_key_ranges",
    "attention_partial",
    "attention_splitkv",
    "merge_partials",
    "attention_general",
    "splitkv_flops",
    "w4a16_unpack",
    "w4a16_dequant",
    "w4a16_gemm",
    "w4a16_abs_sum",
    "sylvester_hadamard",
    "fwht_f32",
    "e4m3_encode",
    "e4m3_decode",
    "e4m3_round",
    "fp8_prepare",
    "fp8_dequantize",
    "pow2_scale_exponent",
    "splitmix64",
    "seeded_rotation_signs",
    "E4M3_MAX",
    "bf16_round",
    "fp8_dequantize_bf16",
    "fp8_operands",
    "fp8_backward_from_operands",
    "fp8_backward",
]
