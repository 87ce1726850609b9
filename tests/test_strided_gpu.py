"""Strided layouts: fa_fwd_strided / fa_bwd_strided (through the C ABI) on [B, N, H, d]
views and padded rows, against the dense calls on the same values.

The kernels address every tensor through the same 4-D map {d, N, H, B} whatever its
strides, so the results must be bitwise those of the dense layout (dQ of the default
backward up to its atomic summation order; the deterministic backward bitwise).
"""

import numpy as np
import pytest
import torch

import io_aware_exact_fwd_gb300 as fa
from oracle import attention_forward
from synth import normal_qkv

from gpu_util import FWD_LSE_ATOL, FWD_O_ATOL, max_abs, o_excess

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    fa.load_library()
    fa.fa_debug_set_fault(0)
    fa.fa_debug_set_wait_limit_ns(0)


def _bnhd(t):
    """The same values in [B, N, H, d] memory, seen as [B, H, N, d]."""
    B, H, N, d = t.shape
    return t.transpose(1, 2).contiguous().transpose(1, 2)


def _padded(t, pad=64):
    """The same values with each row padded to d + pad elements."""
    B, H, N, d = t.shape
    buf = torch.zeros((B, H, N, d + pad), dtype=t.dtype, device=t.device)
    buf[..., :d] = t
    return buf[..., :d]


def _inputs(B, H, N, d, seed):
    x = normal_qkv(B, H, N, d, seed, with_do=True)
    return [x[n].to(torch.bfloat16).cuda() for n in ("q", "k", "v", "do")]


@pytest.mark.parametrize("layout", ["bnhd", "padded"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
def test_forward_strided_equals_dense(layout, causal, d):
    B, H, N = 2, 3, 333
    q, k, v, _ = _inputs(B, H, N, d, 7)
    view = _bnhd if layout == "bnhd" else _padded
    qs, ks, vs = view(q), view(k), view(v)
    assert not qs.is_contiguous()
    o_ref, l_ref = fa.fa_fwd(q, k, v, causal=causal)
    os_ = view(torch.empty_like(q))
    o, l = fa.fa_fwd(qs, ks, vs, o=os_, causal=causal)
    fa.fa_sync_check()
    assert torch.equal(o, o_ref) and torch.equal(l, l_ref)


def test_forward_bnhd_matches_oracle():
    B, H, N, d = 2, 4, 500, 128
    q, k, v, _ = _inputs(B, H, N, d, 11)
    o, lse = fa.fa_fwd(_bnhd(q), _bnhd(k), _bnhd(v), causal=True)
    fa.fa_sync_check()
    o_ref, lse_ref = attention_forward(q, k, v, d ** -0.5, True)
    assert o_excess(o, o_ref) <= FWD_O_ATOL and max_abs(lse, lse_ref) <= FWD_LSE_ATOL


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("layout", ["bnhd", "padded"])
@pytest.mark.parametrize("causal", [False, True])
def test_backward_strided_equals_dense(layout, causal, d):
    B, H, N = 2, 2, 400
    q, k, v, g = _inputs(B, H, N, d, 13)
    view = _bnhd if layout == "bnhd" else _padded
    o, lse = fa.fa_fwd(q, k, v, causal=causal)
    for det in (False, True):
        ref = fa.fa_bwd(q, k, v, o, g, lse, causal=causal, deterministic=det)
        outs = [view(torch.empty_like(q)) for _ in range(3)]
        got = fa.fa_bwd(view(q), view(k), view(v), view(o), view(g), lse, *outs, causal=causal, deterministic=det)
        fa.fa_sync_check()
        assert torch.equal(got[1], ref[1]) and torch.equal(got[2], ref[2])
        if det:
            assert torch.equal(got[0], ref[0])
        else:
            assert float((got[0].float() - ref[0].float()).abs().max()) <= 1e-2 * float(ref[0].float().abs().max())


def test_bad_strides_are_refused():
    q, k, v, _ = _inputs(1, 2, 64, 128, 3)
    with pytest.raises(ValueError):
        fa.fa_fwd(q[..., ::2], k[..., ::2], v[..., ::2])  # d not contiguous
    bad = torch.zeros((1, 2, 64, 132), dtype=torch.bfloat16, device="cuda")[..., :128]  # rows of 132: not 16-byte aligned
    with pytest.raises(fa.FAError) as e:
        fa.fa_fwd(bad, k, v)
    assert e.value.status == 3
