"""Deterministic backward (fa_bwd_deterministic) against the float64 oracle, and its
bitwise reproducibility.

Tolerance as for fa_bwd: max|dX - dX_ref| <= 2e-2 * max|dX_ref| per tensor.  dQ
must be the same bits on every run; dK and dV must equal fa_bwd's bits (the
deterministic mode changes only how dQ is summed).
"""

import numpy as np
import pytest
import torch

import io_aware_exact_fwd_gb300 as fa
from oracle import attention_backward
from synth import normal_qkv, outlier_qkv

from gpu_util import BWD_REL, edge_heads, host_f64, map_heads, rel_max, report

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    fa.load_library()
    fa.fa_debug_set_fault(0)
    fa.fa_debug_set_wait_limit_ns(0)


def _inputs(B, H, N, d, seed, outliers=False):
    x = normal_qkv(B, H, N, d, seed, with_do=True)
    if outliers:
        x.update({n: t for n, t in outlier_qkv(B, H, N, d, seed).items() if n in ("q", "k", "v")})
    return [x[n].to(torch.bfloat16).cuda() for n in ("q", "k", "v", "do")]


def _rel_err(x, ref):
    x = x.float().cpu().numpy().astype(np.float64)
    return float(np.abs(x - ref).max() / max(np.abs(ref).max(), 1e-4))


def _bwd(q, k, v, g, causal, det=True, scale=None):
    scale = q.shape[-1] ** -0.5 if scale is None else scale
    o, lse = fa.fa_fwd(q, k, v, causal=causal, scale=scale)
    out = fa.fa_bwd(q, k, v, o, g, lse, causal=causal, scale=scale, deterministic=det)
    fa.fa_sync_check()
    return out


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 63, 65, 128, 200, 1000])
def test_deterministic_matches_oracle(N, causal, d):
    q, k, v, g = _inputs(1, 2, N, d, 300 + N + d)
    dq, dk, dv = _bwd(q, k, v, g, causal)
    rq, rk, rv = attention_backward(q, k, v, g, d ** -0.5, causal)
    errs = (_rel_err(dq, rq), _rel_err(dk, rk), _rel_err(dv, rv))
    assert max(errs) <= BWD_REL, errs


@pytest.mark.parametrize("causal", [False, True])
def test_outliers_and_a_large_row(causal):
    # x20 outliers raise the bound; one dO row scaled by 1000 raises its own block's
    # bound only.  Both stay within the tolerance.
    q, k, v, g = _inputs(1, 2, 700, 128, 41, outliers=True)
    g[0, 1, 333] *= 1000
    dq, dk, dv = _bwd(q, k, v, g, causal)
    rq, rk, rv = attention_backward(q, k, v, g, 128 ** -0.5, causal)
    errs = (_rel_err(dq, rq), _rel_err(dk, rk), _rel_err(dv, rv))
    assert max(errs) <= BWD_REL, errs
    # Rows of other blocks keep their accuracy relative to their own magnitude.
    other = np.r_[0:320, 384:700]
    assert _rel_err(dq[0, 1, other], rq[0, 1, other]) <= BWD_REL


@pytest.mark.parametrize("causal", [False, True])
def test_dq_bits_identical_across_runs(causal):
    q, k, v, g = _inputs(1, 4, 1500, 128, 9)
    o, lse = fa.fa_fwd(q, k, v, causal=causal)
    ref = fa.fa_bwd(q, k, v, o, g, lse, causal=causal, deterministic=True)
    # Other work on a second stream changes the timing of the atomics, not the bits.
    side = torch.cuda.Stream()
    for _ in range(3):
        with torch.cuda.stream(side):
            x = torch.randn(2048, 2048, device="cuda")
            for _ in range(4):
                x = x @ x * 1e-3
        out = fa.fa_bwd(q, k, v, o, g, lse, causal=causal, deterministic=True)
        torch.cuda.synchronize()
        assert torch.equal(out[0], ref[0]) and torch.equal(out[1], ref[1]) and torch.equal(out[2], ref[2])
    fa.fa_sync_check()


@pytest.mark.parametrize("causal", [False, True])
def test_dk_dv_equal_fa_bwd_and_dq_close(causal):
    q, k, v, g = _inputs(2, 2, 777, 128, 13)
    o, lse = fa.fa_fwd(q, k, v, causal=causal)
    a = fa.fa_bwd(q, k, v, o, g, lse, causal=causal)
    b = fa.fa_bwd(q, k, v, o, g, lse, causal=causal, deterministic=True)
    fa.fa_sync_check()
    assert torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])
    d = (a[0].float() - b[0].float()).abs().max()
    assert float(d) <= 1e-2 * float(a[0].float().abs().max())


@pytest.mark.parametrize("causal", [False, True])
def test_deterministic_config_n8192_whole_heads(causal):
    # B=2, H=16, N=8192, d=128 at full size, twice; every row and key of three heads.
    B, H, N, d = 2, 16, 8192, 128
    scale = d ** -0.5
    q, k, v, g = _inputs(B, H, N, d, 4)
    dq, dk, dv = _bwd(q, k, v, g, causal)
    dq2, _, _ = _bwd(q, k, v, g, causal)
    assert torch.equal(dq, dq2)
    qc, kc, vc, gc = (t.cpu() for t in (q, k, v, g))
    gq, gk, gv = host_f64(dq), host_f64(dk), host_f64(dv)

    def one(b, h):
        sl = (slice(b, b + 1), slice(h, h + 1))
        rq, rk, rv = attention_backward(qc[sl], kc[sl], vc[sl], gc[sl], scale, causal)
        return rel_max(gq[sl], rq), rel_max(gk[sl], rk), rel_max(gv[sl], rv)

    errs = map_heads(one, edge_heads(B, H))
    worst = tuple(max(e[i] for e in errs) for i in range(3))
    report(f"bwd deterministic B=2 H=16 N=8192 d=128 causal={int(causal)}", heads=len(errs), dq=worst[0],
           dk=worst[1], dv=worst[2])
    assert max(worst) <= BWD_REL, worst
