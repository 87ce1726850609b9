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


# ------------------------------------------------------------ FP8 prepare, split-KV
#
# fa_fp8_prepare_strided reads its inputs at the strides and writes the dense
# workspace: the whole workspace (codes and scales) must be bitwise that of the
# dense call.  fa_fwd_splitkv_strided addresses q, k, v through the same TMA maps
# and o through the merge kernel's strides: O and LSE bitwise those of dense.

from oracle import attention_general  # noqa: E402
from synth import outlier_qkv, rotation_signs  # noqa: E402


def _padded_f32(t, pad=32):
    B, H, N, d = t.shape
    buf = torch.zeros((B, H, N, d + pad), dtype=t.dtype, device=t.device)
    buf[..., :d] = t
    return buf[..., :d]


@pytest.mark.parametrize("layout", ["bnhd", "padded"])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("d", [64, 128])
def test_fp8_prepare_strided_equals_dense(layout, dtype, d):
    B, H, N = 2, 3, 333
    x = outlier_qkv(B, H, N, d, seed=40 + d)
    dense = [x[n].to(dtype).cuda() for n in ("q", "k", "v")]
    view = [_bnhd(t) if layout == "bnhd" else _padded_f32(t) for t in dense]
    assert not any(t.is_contiguous() for t in view)
    s = rotation_signs(d, seed=41).cuda()
    # Zeroed workspaces: the alignment gaps between regions are never written.
    zws = lambda: torch.zeros(fa.fa_fp8_workspace_size(B, H, N, d), dtype=torch.uint8, device="cuda")
    ws_dense = fa.fa_fp8_prepare(*dense, s, workspace=zws())
    ws_view = fa.fa_fp8_prepare(*view, s, workspace=zws())
    ws_seed_dense = fa.fa_fp8_prepare_seeded(*dense, 1234567, workspace=zws())
    ws_seed_view = fa.fa_fp8_prepare_seeded(*view, 1234567, workspace=zws())
    fa.fa_sync_check()
    assert torch.equal(ws_dense, ws_view)
    assert torch.equal(ws_seed_dense, ws_seed_view)


@pytest.mark.parametrize("layout", ["bnhd", "padded"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("Nq", [5, 1])  # one query row at d = 64: the CUDA-core partials
def test_splitkv_strided_equals_dense(layout, causal, d, Nq):
    B, H, Nk = 2, 3, 1500
    kv = normal_qkv(B, H, Nk, d, 50)
    k, v = (kv[n].to(torch.bfloat16).cuda() for n in ("k", "v"))
    q = normal_qkv(B, H, Nq, d, 51)["q"].to(torch.bfloat16).cuda()
    conv = _bnhd if layout == "bnhd" else _padded
    qv, kvv, vv = conv(q), conv(k), conv(v)
    o_view = conv(torch.zeros_like(q))
    o, lse = fa.fa_fwd_splitkv(q, k, v, n_split=4, causal=causal)
    o2, lse2 = fa.fa_fwd_splitkv(qv, kvv, vv, o=o_view, n_split=4, causal=causal)
    fa.fa_sync_check()
    # K and V are strided views in both layouts; with one query row a [B, 1, H, d]
    # view of q or o is contiguous as far as torch is concerned.
    assert not kvv.is_contiguous() and not vv.is_contiguous()
    assert Nq == 1 or not o_view.is_contiguous()
    assert torch.equal(o, o2.contiguous())
    assert torch.equal(lse, lse2)
    # Sanity against the oracle on one head (queries are the last Nq positions).
    ref_o, ref_l = attention_general(q[:1, :1], k[:1, :1], v[:1, :1], d ** -0.5, causal)
    assert o_excess(o2[:1, :1], ref_o) <= FWD_O_ATOL
    assert max_abs(lse2[:1, :1], ref_l) <= FWD_LSE_ATOL


def test_fp8_prepare_and_splitkv_bad_strides_are_refused():
    q = torch.zeros((1, 2, 64, 136), dtype=torch.bfloat16, device="cuda")[..., :128]  # rows of 136: 16-byte multiples
    bad = torch.zeros((1, 2, 64, 132), dtype=torch.bfloat16, device="cuda")[..., :128]  # rows of 132: not
    s = rotation_signs(128, seed=1).cuda()
    fa.fa_fp8_prepare(q, q, q, s)
    with pytest.raises(fa.FAError) as e:
        fa.fa_fp8_prepare(bad, q, q, s)
    assert e.value.status == 3
    with pytest.raises(fa.FAError) as e:
        fa.fa_fwd_splitkv(q[:, :, :1], bad, q, n_split=2)
    assert e.value.status == 3
    fa.fa_sync_check()
