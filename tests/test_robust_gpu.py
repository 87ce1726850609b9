"""Failure detection without a GPU fault: a bounded in-kernel wait expires and
the host reads an error status; the CUDA context stays usable afterwards.

The fault is injected on the host side of the pipeline (the TMA producer
withholds one K block), never by a trap, an invalid address or an unbounded
wait.  Every wait in the kernel polls a deadline (50 ms here) and the CTA-wide
abort flag, drains its own in-flight copies, frees TMEM and exits.
"""

import pytest
import torch

import io_aware_exact_fwd_gb300 as fa
from oracle import attention_forward
from synth import normal_qkv

from gpu_util import FWD_LSE_ATOL, FWD_O_ATOL, max_abs, o_excess, to_dev_bf16

pytestmark = pytest.mark.gpu


def test_expired_wait_reports_timeout_and_context_survives():
    fa.load_library()
    x = normal_qkv(1, 2, 512, 128, 9)
    q, k, v = to_dev_bf16(x)
    fa.fa_debug_set_wait_limit_ns(50_000_000)
    fa.fa_debug_set_fault(1)
    try:
        fa.fa_fwd(q, k, v, causal=False)
        with pytest.raises(fa.FAError) as err:
            fa.fa_sync_check()
        assert err.value.status == 5
        site = fa.fa_last_error_site()
        assert site & 0x80000000 and ((site >> 8) & 0xF) in (1, 2, 3)
    finally:
        fa.fa_debug_set_fault(0)
        fa.fa_debug_set_wait_limit_ns(0)
    # The error word was cleared and the context still works.
    o, lse = fa.fa_fwd(q, k, v, causal=False)
    fa.fa_sync_check()
    o_ref, lse_ref = attention_forward(q, k, v, 128 ** -0.5, False)
    assert o_excess(o, o_ref) <= FWD_O_ATOL and max_abs(lse, lse_ref) <= FWD_LSE_ATOL
    assert torch.cuda.is_available()
