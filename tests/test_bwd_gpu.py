"""Backward parity: fa_bwd (through the C ABI) against the float64 oracle.

Tolerance, per tensor X in {Q, K, V}: max|dX - dX_ref| <= 2e-2 * max|dX_ref|.
O and LSE come from the library's own forward (as a training step would use
them); the oracle works from the bf16 inputs alone.
"""

import numpy as np
import pytest
import torch

import io_aware_exact_fwd_gb300 as fa
from oracle import attention_backward
from synth import normal_qkv

from gpu_util import BWD_REL, all_heads, edge_heads, host_f64, map_heads, rel_max, report

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    fa.load_library()
    fa.fa_debug_set_fault(0)
    fa.fa_debug_set_wait_limit_ns(0)


def _inputs(B, H, N, d, seed):
    x = normal_qkv(B, H, N, d, seed, with_do=True)
    return [x[n].to(torch.bfloat16).cuda() for n in ("q", "k", "v", "do")]


def _run(q, k, v, g, causal, scale):
    o, lse = fa.fa_fwd(q, k, v, causal=causal, scale=scale)
    dq, dk, dv = fa.fa_bwd(q, k, v, o, g, lse, causal=causal, scale=scale)
    fa.fa_sync_check()
    return dq, dk, dv


def _rel_err(x, ref):
    # The reference magnitude is floored at 1e-4: where a gradient is exactly 0 in
    # exact arithmetic (N = 1: P = 1, so dS = P (dP - D) = 0 and dQ = dK = 0), the
    # kernel returns rounding noise of order 1e-7 (dP from the tensor core and D
    # from the bf16 O are fp32 sums in different orders), which a relative test
    # against 0 cannot accept.
    x = x.float().cpu().numpy().astype(np.float64) if isinstance(x, torch.Tensor) else np.asarray(x)
    return float(np.abs(x - ref).max() / max(np.abs(ref).max(), 1e-4))


def _check_full(B, H, N, d, causal, seed, scale=None):
    scale = d ** -0.5 if scale is None else scale
    q, k, v, g = _inputs(B, H, N, d, seed)
    dq, dk, dv = _run(q, k, v, g, causal, scale)
    rq, rk, rv = attention_backward(q, k, v, g, scale, causal)
    errs = (_rel_err(dq, rq), _rel_err(dk, rk), _rel_err(dv, rv))
    assert max(errs) <= BWD_REL, (B, H, N, d, causal, errs)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 63, 64, 65, 127, 128, 129, 200, 1000])
def test_backward_ragged_lengths(N, causal, d):
    _check_full(1, 2, N, d, causal, seed=200 + N + d)


def _compare_backward_heads(q, k, v, g, dq, dk, dv, scale, causal, heads):
    """Every row of dQ, dK, dV of the given heads against the oracle: the three relative errors."""
    qc, kc, vc, gc = (t.cpu() for t in (q, k, v, g))
    gq, gk, gv = host_f64(dq), host_f64(dk), host_f64(dv)

    def one(b, h):
        sl = (slice(b, b + 1), slice(h, h + 1))
        rq, rk, rv = attention_backward(qc[sl], kc[sl], vc[sl], gc[sl], scale, causal)
        return rel_max(gq[sl], rq), rel_max(gk[sl], rk), rel_max(gv[sl], rv)

    errs = map_heads(one, heads)
    return tuple(max(e[i] for e in errs) for i in range(3))


@pytest.mark.parametrize("causal", [False, True])
def test_backward_config_n2048_all_heads(causal):
    # B=8, H=16, N=2048, d=128 at full size; every head compared in full by the oracle.
    B, H, N, d = 8, 16, 2048, 128
    scale = d ** -0.5
    q, k, v, g = _inputs(B, H, N, d, 4)
    dq, dk, dv = _run(q, k, v, g, causal, scale)
    errs = _compare_backward_heads(q, k, v, g, dq, dk, dv, scale, causal, all_heads(B, H))
    report(f"bwd B=8 H=16 N=2048 d=128 causal={int(causal)}", heads=B * H, dq=errs[0], dk=errs[1], dv=errs[2])
    assert max(errs) <= BWD_REL, errs
    _check_sum_rules(dk, dv, g)


@pytest.mark.parametrize("causal", [False, True])
def test_backward_d64_sweep_n2048_all_heads(causal):
    # The sweep's d = 64 shape at N = 2048 (B=8, H=32): every head compared in full.
    B, H, N, d = 8, 32, 2048, 64
    scale = d ** -0.5
    q, k, v, g = _inputs(B, H, N, d, 14)
    dq, dk, dv = _run(q, k, v, g, causal, scale)
    errs = _compare_backward_heads(q, k, v, g, dq, dk, dv, scale, causal, all_heads(B, H))
    report(f"bwd B=8 H=32 N=2048 d=64 causal={int(causal)}", heads=B * H, dq=errs[0], dk=errs[1], dv=errs[2])
    assert max(errs) <= BWD_REL, errs
    _check_sum_rules(dk, dv, g)


@pytest.mark.parametrize("causal", [False, True])
def test_backward_d64_sweep_n8192_whole_heads(causal):
    # The sweep's d = 64 shape at N = 8192 (B=2, H=32): every row of three heads.
    B, H, N, d = 2, 32, 8192, 64
    scale = d ** -0.5
    q, k, v, g = _inputs(B, H, N, d, 15)
    dq, dk, dv = _run(q, k, v, g, causal, scale)
    heads = edge_heads(B, H)
    errs = _compare_backward_heads(q, k, v, g, dq, dk, dv, scale, causal, heads)
    report(f"bwd B=2 H=32 N=8192 d=64 causal={int(causal)}", heads=len(heads), dq=errs[0], dk=errs[1], dv=errs[2])
    assert max(errs) <= BWD_REL, errs
    _check_sum_rules(dk, dv, g)


@pytest.mark.parametrize("causal", [False, True])
def test_backward_config_n8192_whole_heads(causal):
    # B=2, H=16, N=8192, d=128 at full size; every query row (dQ) and every key
    # (dK, dV) of the first, a middle and the last head.
    B, H, N, d = 2, 16, 8192, 128
    scale = d ** -0.5
    q, k, v, g = _inputs(B, H, N, d, 4)
    dq, dk, dv = _run(q, k, v, g, causal, scale)
    heads = edge_heads(B, H)
    errs = _compare_backward_heads(q, k, v, g, dq, dk, dv, scale, causal, heads)
    report(f"bwd B=2 H=16 N=8192 d=128 causal={int(causal)}", heads=len(heads), dq=errs[0], dk=errs[1],
           dv=errs[2])
    assert max(errs) <= BWD_REL, errs
    _check_sum_rules(dk, dv, g)


def _check_sum_rules(dk, dv, g):
    # Exact identities of the gradient: sum over keys of dK is 0 (each row of dS
    # sums to 0) and sum over keys of dV equals the sum over queries of dO.  They
    # hold for every head at any size; bf16 rounding bounds the mismatch.
    sk = dk.double().sum(dim=2)
    sv = dv.double().sum(dim=2)
    sg = g.double().sum(dim=2)
    n = dk.shape[2]
    assert float(sk.abs().max()) <= 2e-2 * float(dk.double().abs().max()) * n ** 0.5
    assert float((sv - sg).abs().max()) <= 2e-2 * float(sg.abs().max()) + 1e-2 * n ** 0.5


@pytest.mark.parametrize("d", [64, 128])
def test_backward_other_scale(d):
    _check_full(2, 2, 300, d, True, seed=7, scale=0.2)


def test_backward_dk_dv_deterministic():
    q, k, v, g = _inputs(1, 4, 1500, 128, 9)
    a = _run(q, k, v, g, True, 128 ** -0.5)
    b = _run(q, k, v, g, True, 128 ** -0.5)
    assert torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])
    rq = a[0].float()
    assert float((rq - b[0].float()).abs().max()) <= 1e-2 * float(rq.abs().max())


def test_backward_rejects_bad_arguments():
    q, k, v, g = _inputs(1, 1, 128, 128, 10)
    o, lse = fa.fa_fwd(q, k, v)
    with pytest.raises(fa.FAError) as e:
        fa.fa_bwd(q, k, v, o, g, lse, workspace=torch.empty(16, dtype=torch.uint8, device="cuda"))
    assert e.value.status == 6
    fa.fa_sync_check()


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_staged_backward_equals_fa_bwd(causal, d):
    # fa_bwd is fa_bwd_prep + fa_bwd_main + fa_bwd_dq on one stream.
    q, k, v, g = _inputs(2, 2, 700, d, 12)
    o, lse = fa.fa_fwd(q, k, v, causal=causal)
    ref = fa.fa_bwd(q, k, v, o, g, lse, causal=causal)
    ws = torch.empty(fa.fa_bwd_workspace_size(2, 2, 700, d), dtype=torch.uint8, device="cuda")
    dq, dk, dv = (torch.empty_like(q) for _ in range(3))
    fa.fa_bwd_prep(o, g, lse, ws)
    fa.fa_bwd_main(q, k, v, g, dk, dv, ws, causal=causal)
    fa.fa_bwd_dq(ws, dq)
    fa.fa_sync_check()
    assert torch.equal(dk, ref[1]) and torch.equal(dv, ref[2])
    assert _rel_err(dq, ref[0].double().cpu().numpy()) <= 1e-2
