"""Forward parity: the CUDA path (through the C ABI) against the float64 oracle.

Tolerances: max|LSE - LSE_ref| <= 1e-3, and for O the 1e-2 bound applied to
the error beyond the rounding of the exact result to the bf16 output format
(``o_excess``; the raw max|O - O_ref| is at most that plus half a bf16 ulp of
|O|).  The oracle is evaluated on the same bf16 input values the GPU receives.
"""

import numpy as np
import pytest
import torch

import io_aware_exact_fwd_gb300 as fa
from oracle import attention_forward
from synth import normal_qkv

from gpu_util import (FWD_LSE_ATOL, FWD_O_ATOL, all_heads, edge_heads, host_f64, map_heads, max_abs, o_excess,
                      report, to_dev_bf16)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    fa.load_library()
    fa.fa_debug_set_fault(0)
    fa.fa_debug_set_wait_limit_ns(0)


def _run_and_compare(B, H, N, d, causal, seed, scale=None, o_atol=FWD_O_ATOL, name=None):
    x = normal_qkv(B, H, N, d, seed)
    q, k, v = to_dev_bf16(x)
    scale = d ** -0.5 if scale is None else scale
    o, lse = fa.fa_fwd(q, k, v, causal=causal, scale=scale)
    fa.fa_sync_check()
    if B * H > 4:
        qc, kc, vc = (t.cpu() for t in (q, k, v))
        eo, el, raw = _compare_heads(o, lse, qc, kc, vc, scale, causal, all_heads(B, H))
    else:
        o_ref, lse_ref = attention_forward(q, k, v, scale, causal)
        eo, el, raw = o_excess(o, o_ref), max_abs(lse, lse_ref), max_abs(o, o_ref)
    if name:
        report(name, heads=B * H, o_excess=eo, lse=el, o_raw=raw)
    assert eo <= o_atol and el <= FWD_LSE_ATOL, (B, H, N, d, causal, eo, el)
    return o, lse


@pytest.mark.parametrize("causal", [False, True])
def test_tiny_config(causal):
    # B=1, H=2, N=128, d=64, fp32 N(0,1) draws from seed 1, cast to bf16 at the boundary.
    _run_and_compare(1, 2, 128, 64, causal, seed=1, name=f"fwd tiny B=1 H=2 N=128 d=64 causal={int(causal)}")


@pytest.mark.parametrize("causal", [False, True])
def test_bf16_config_all_heads(causal):
    # B=4, H=16, N=2048, d=128, seed 2: every head compared in full.
    _run_and_compare(4, 16, 2048, 128, causal, seed=2, name=f"fwd B=4 H=16 N=2048 d=128 causal={int(causal)}")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N", [1, 63, 65, 127, 129, 200, 1000])
@pytest.mark.parametrize("causal", [False, True])
def test_ragged_lengths(N, d, causal):
    _run_and_compare(1, 3, N, d, causal, seed=100 + N)


@pytest.mark.parametrize("scale", [0.05, 0.5])
def test_other_scales(scale):
    # Away from 1/sqrt(d) the softmax can be nearly one-hot, so |O| approaches
    # max|V| and the rounding of P to bf16 (half-ulp, relative 2^-9, and the same
    # mismatch between the fp32 row sum and the rounded P) bounds the kernel's
    # error by 2 * 2^-9 * max|V| = 2^-8 * max|V| on top of the output rounding.
    x = normal_qkv(2, 2, 300, 128, 7)
    vmax = float(x["v"].to(torch.bfloat16).abs().max())
    _run_and_compare(2, 2, 300, 128, True, seed=7, scale=scale, o_atol=max(FWD_O_ATOL, 2.0 ** -8 * vmax))


# Sequence sweep at 16384 tokens and hidden 2048: (d=64, H=32) and (d=128, H=16).
SWEEP = [(n, d) for n in (512, 1024, 2048, 4096, 8192, 16384) for d in (64, 128)]


def _compare_heads(o, lse, q, k, v, scale, causal, heads):
    """Every row of the given heads against the oracle: (max o_excess, max LSE error, raw max |O - O_ref|)."""
    oh, lh = host_f64(o), host_f64(lse)

    def one(b, h):
        sl = (slice(b, b + 1), slice(h, h + 1))
        o_ref, lse_ref = attention_forward(q[sl], k[sl], v[sl], scale, causal)
        return (o_excess(oh[sl], o_ref), float(np.abs(lh[sl] - lse_ref).max()),
                float(np.abs(oh[sl] - o_ref).max()))

    errs = map_heads(one, heads)
    return max(e[0] for e in errs), max(e[1] for e in errs), max(e[2] for e in errs)


@pytest.mark.parametrize("N,d", SWEEP)
@pytest.mark.parametrize("causal", [False, True])
def test_sequence_sweep(N, d, causal):
    # Full-size launch.  N <= 2048: every head compared in full; N >= 4096: every
    # row of the first, a middle and the last head.
    H = 32 if d == 64 else 16
    B = 16384 // N
    x = normal_qkv(B, H, N, d, 3)
    q, k, v = to_dev_bf16(x)
    scale = d ** -0.5
    o, lse = fa.fa_fwd(q, k, v, causal=causal, scale=scale)
    fa.fa_sync_check()
    assert torch.isfinite(o).all() and torch.isfinite(lse).all()
    heads = all_heads(B, H) if N <= 2048 else edge_heads(B, H)
    qc, kc, vc = (t.cpu() for t in (q, k, v))
    eo, el, raw = _compare_heads(o, lse, qc, kc, vc, scale, causal, heads)
    report(f"fwd sweep N={N} d={d} causal={int(causal)}", heads=len(heads), o_excess=eo, lse=el, o_raw=raw)
    assert eo <= FWD_O_ATOL and el <= FWD_LSE_ATOL, (N, d, causal, eo, el)


def test_identical_keys_give_column_mean():
    B, H, N, d = 1, 2, 300, 128
    x = normal_qkv(B, H, N, d, 41)
    q, _, v = to_dev_bf16(x)
    k = x["k"][:, :, :1].expand(B, H, N, d).contiguous().to(torch.bfloat16).cuda()
    for causal in (False, True):
        o, lse = fa.fa_fwd(q, k, v, causal=causal)
        fa.fa_sync_check()
        vf = v.double().cpu()
        counts = torch.arange(1, N + 1, dtype=torch.float64)[:, None]
        ref = vf.cumsum(2) / counts if causal else vf.mean(2, keepdim=True).expand_as(vf)
        assert o_excess(o, ref) <= FWD_O_ATOL


def test_causal_row_zero_is_v0():
    x = normal_qkv(2, 2, 333, 64, 42)
    q, k, v = to_dev_bf16(x)
    o, lse = fa.fa_fwd(q, k, v, causal=True)
    fa.fa_sync_check()
    assert torch.equal(o[:, :, 0], v[:, :, 0])
    ref = (q[:, :, 0].double() * k[:, :, 0].double()).sum(-1) * 64 ** -0.5
    assert max_abs(lse[:, :, 0], ref) <= FWD_LSE_ATOL


def test_dominant_score_selects_value_row():
    N, d = 256, 128
    k = torch.zeros(1, 1, N, d)
    k[0, 0, torch.arange(d), torch.arange(d)] = 1.0      # keys 0..127 orthonormal
    k[0, 0, d:, :] = 0.0                                 # keys 128..255 are zero
    v = normal_qkv(1, 1, N, d, 43)["v"]
    target = torch.randperm(d, generator=torch.Generator().manual_seed(1))
    q = torch.zeros(1, 1, N, d)
    q[0, 0, torch.arange(d), target] = 64.0               # row i picks key target[i]
    qd, kd, vd = (t.to(torch.bfloat16).cuda() for t in (q, k, v))
    o, _ = fa.fa_fwd(qd, kd, vd, causal=False, scale=1.0)
    fa.fa_sync_check()
    assert o_excess(o[0, 0, :d], vd[0, 0, target]) <= FWD_O_ATOL


def _shared_tail(B, H, N):
    # Whether fa_fwd deals its partial last pass out as shared tiles on this device
    # (non-causal; 0 < R = units mod SMs, 2R <= SMs, at most 4 full passes, N > 128).
    units = B * H * ((N + 255) // 256)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    rem = units % sms
    return N > 128 and rem > 0 and 2 * rem <= sms and units // sms <= 4


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("B,H,N", [(1, 160, 512), (2, 44, 1536), (3, 20, 700)])
def test_shared_tail_tiles_all_heads(B, H, N, d):
    # Launches whose last pass runs as shared tiles after one to four full passes of
    # whole units (and a ragged N = 700): every head against the oracle, the
    # softmax of each shared tile being split over two warpgroups (even and odd key
    # blocks) and merged; then bitwise reproducible.
    if not _shared_tail(B, H, N):
        pytest.skip("this device's SM count gives no shared last pass for the shape")
    o, lse = _run_and_compare(B, H, N, d, False, seed=46 + d,
                              name=f"fwd shared tail B={B} H={H} N={N} d={d}")
    x = normal_qkv(B, H, N, d, 46 + d)
    q, k, v = to_dev_bf16(x)
    o2, l2 = fa.fa_fwd(q, k, v)
    fa.fa_sync_check()
    assert torch.equal(o, o2) and torch.equal(lse, l2)


def test_forward_is_bitwise_deterministic():
    x = normal_qkv(2, 4, 1500, 128, 44)
    q, k, v = to_dev_bf16(x)
    for causal in (False, True):
        o1, l1 = fa.fa_fwd(q, k, v, causal=causal)
        o2, l2 = fa.fa_fwd(q, k, v, causal=causal)
        fa.fa_sync_check()
        assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_outputs_do_not_spill_outside_their_buffers():
    B, H, N, d = 1, 2, 777, 64
    x = normal_qkv(B, H, N, d, 45)
    q, k, v = to_dev_bf16(x)
    pad = 4096
    n_o, n_l = B * H * N * d, B * H * N
    obuf = torch.full((n_o + 2 * pad,), float("nan"), dtype=torch.bfloat16, device="cuda")
    lbuf = torch.full((n_l + 2 * pad,), float("nan"), dtype=torch.float32, device="cuda")
    o = obuf[pad:pad + n_o].view(B, H, N, d)
    lse = lbuf[pad:pad + n_l].view(B, H, N)
    fa.fa_fwd(q, k, v, o=o, lse=lse, causal=True)
    fa.fa_sync_check()
    assert torch.isnan(obuf[:pad]).all() and torch.isnan(obuf[pad + n_o:]).all()
    assert torch.isnan(lbuf[:pad]).all() and torch.isnan(lbuf[pad + n_l:]).all()
    o_ref, lse_ref = attention_forward(q, k, v, d ** -0.5, True)
    assert o_excess(o, o_ref) <= FWD_O_ATOL and max_abs(lse, lse_ref) <= FWD_LSE_ATOL


def test_runs_on_a_side_stream():
    x = normal_qkv(1, 2, 500, 128, 46)
    q, k, v = to_dev_bf16(x)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        o, lse = fa.fa_fwd(q, k, v, causal=False)
    fa.fa_sync_check(s)
    o_ref, _ = attention_forward(q, k, v, 128 ** -0.5, False)
    assert o_excess(o, o_ref) <= FWD_O_ATOL


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("growth", [4.0, 40.0])
def test_row_max_jumps_between_key_blocks(growth, causal):
    # Later key blocks carry much larger scores, so exponentials taken against the
    # running maximum of earlier blocks grow beyond the kernel's bound (growth 4)
    # or overflow to inf (growth 40): the kernel must redo those blocks with their
    # own maximum and rescale O.
    B, H, N, d = 1, 2, 640, 128
    x = normal_qkv(B, H, N, d, 47)
    for j in range(N // 128):
        x["k"][:, :, j * 128:(j + 1) * 128] *= 1.0 + growth * j
    q, k, v = to_dev_bf16(x)
    o, lse = fa.fa_fwd(q, k, v, causal=causal)
    fa.fa_sync_check()
    o_ref, lse_ref = attention_forward(q, k, v, d ** -0.5, causal)
    assert torch.isfinite(o).all()
    assert o_excess(o, o_ref) <= FWD_O_ATOL
    assert max_abs(lse, lse_ref) <= FWD_LSE_ATOL * max(1.0, float(np.abs(lse_ref).max()) / 100.0)
