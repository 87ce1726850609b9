"""Pins of the FP8 backward oracle: bf16 rounding, operand dequantisation, the rotation
and scale of the straight-through gradient, and finite differences of the composed
function."""

import numpy as np
import pytest
import torch

from oracle import attention_backward, attention_forward, fp8_prepare, sylvester_hadamard
from oracle.fp8_backward import (
    bf16_round,
    fp8_backward,
    fp8_backward_from_operands,
    fp8_dequantize_bf16,
    fp8_operands,
)
from synth import normal_qkv, outlier_qkv, rotation_signs


def test_bf16_round_golden_values():
    # bf16 keeps 8 significant bits: the spacing at 1 is 2^-7.
    cases = [
        (1.0 + 2.0 ** -8, 1.0),                          # tie, lower neighbour even
        (1.0 + 2.0 ** -8 + 2.0 ** -20, 1.0 + 2.0 ** -7),  # above the tie
        (1.0 + 3 * 2.0 ** -8, 1.0 + 2.0 ** -6),          # tie, upper neighbour even
        (-(1.0 + 3 * 2.0 ** -8), -(1.0 + 2.0 ** -6)),
        (1.0 + 2.0 ** -8 - 2.0 ** -23, 1.0),              # just below the tie
        (0.0, 0.0),
        (2.0 ** -133, 2.0 ** -133),                       # fp32 subnormal with few bits
        (float(np.finfo(np.float32).max), np.inf),        # rounds past bf16's largest finite
        (3.3895313892515355e38, 3.3895313892515355e38),   # bf16's largest finite itself
    ]
    for x, want in cases:
        got = float(bf16_round(np.float32(x)))
        assert got == want, (x, got, want)
    assert np.isnan(bf16_round(np.float32(np.nan)))


def test_bf16_round_agrees_with_torch_cast():
    rng = np.random.default_rng(5)
    x = (rng.standard_normal(200000) * np.exp(rng.uniform(-60, 60, 200000))).astype(np.float32)
    want = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(bf16_round(x), want)


def test_dequantize_bf16_agrees_with_torch_fp8_decode():
    # torch decodes e4m3fn bytes itself; fp32 multiply then bf16 cast is the same
    # two roundings.  Every code, several tile scales including awkward ones.
    codes = np.arange(256, dtype=np.uint8)
    codes = codes[(codes & 0x7F) != 0x7F]                         # drop the two NaN codes
    N = 64 * 4
    c = np.resize(codes, (N, 8)).astype(np.uint8)
    sigma = np.array([1.0, 1.0 / 3.0, 448.0 / 437.1, 2.0 ** -20], dtype=np.float32)
    got = fp8_dequantize_bf16(c, sigma)
    dec = torch.from_numpy(c).view(torch.float8_e4m3fn).to(torch.float32)
    sig = torch.from_numpy(sigma).repeat_interleave(64)[:, None]
    want = (dec * sig).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(got, want)


def test_dequantize_bf16_short_last_tile():
    c = np.full((70, 4), 0x38, dtype=np.uint8)                    # e4m3 1.0
    got = fp8_dequantize_bf16(c, np.array([0.5, 4.0], dtype=np.float32))
    assert (got[:64] == 0.5).all() and (got[64:] == 4.0).all()


@pytest.mark.parametrize("causal", [False, True])
def test_rotation_direction_and_scale(causal):
    # With exact (unquantised) rotated operands the straight-through gradient must be
    # the gradient of the unrotated problem: (Q M)(K M)^T / d = Q K^T for M = diag(s) H.
    # Using M instead of M^T, or dropping the 1/d, fails this (signs are not all +1).
    B, H, N, d = 1, 2, 40, 64
    x = normal_qkv(B, H, N, d, seed=12, with_do=True)
    q, k, v, do = (x[n].numpy().astype(np.float64) for n in ("q", "k", "v", "do"))
    s = rotation_signs(d, seed=12).numpy().astype(np.float64)
    assert (s < 0).any() and (s > 0).any()
    m = np.diag(s) @ sylvester_hadamard(d)
    scale = 0.3
    got = fp8_backward_from_operands(q @ m, k @ m, v, do, s, scale, causal)
    want = attention_backward(q, k, v, do, scale, causal)
    for g, w in zip(got, want):
        assert np.abs(g - w).max() <= 1e-10 * np.abs(w).max()


@pytest.mark.parametrize("causal", [False, True])
def test_composed_gradient_matches_central_finite_differences(causal):
    # L(Q, K, V) = <dO, attention((Q M), (K M), V, scale / d)> with M = diag(s) H;
    # the oracle's gradient in Q, K, V against central differences in float64.
    B, H, N, d = 1, 1, 6, 8
    rng = np.random.default_rng(3)
    q, k, v, do = (rng.standard_normal((B, H, N, d)) for _ in range(4))
    s = np.where(rng.random(d) < 0.5, -1.0, 1.0)
    m = np.diag(s) @ sylvester_hadamard(d)
    scale = 0.7

    def loss(q_, k_, v_):
        o, _ = attention_forward(q_ @ m, k_ @ m, v_, scale / d, causal)
        return float((o * do).sum())

    dq, dk, dv = fp8_backward_from_operands(q @ m, k @ m, v, do, s, scale, causal)
    h = 1e-6
    for name, t, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        for idx in [(0, 0, 0, 0), (0, 0, N - 1, d - 1), (0, 0, 2, 5), (0, 0, 4, 1)]:
            tp, tm = t.copy(), t.copy()
            tp[idx] += h
            tm[idx] -= h
            args_p = {"q": q, "k": k, "v": v}
            args_m = dict(args_p)
            args_p[name], args_m[name] = tp, tm
            fd = (loss(args_p["q"], args_p["k"], args_p["v"]) - loss(args_m["q"], args_m["k"], args_m["v"])) / (2 * h)
            assert abs(fd - g[idx]) <= 1e-6 * max(1.0, abs(fd)), (name, idx, fd, g[idx])


def test_fp8_backward_uses_the_dequantised_operands():
    # fp8_backward = forward and straight-through backward on fp8_operands(prep).
    B, H, N, d = 1, 1, 70, 64
    x = outlier_qkv(B, H, N, d, seed=8)
    do = torch.randn(B, H, N, d, generator=torch.Generator().manual_seed(1)).numpy().astype(np.float64)
    s = rotation_signs(d, seed=8).numpy()
    prep = fp8_prepare(x["q"], x["k"], x["v"], s)
    dq, dk, dv, o, lse = fp8_backward(prep, s, do, d ** -0.5, True)
    qr, kr, vr = fp8_operands(prep)
    o2, lse2 = attention_forward(qr, kr, vr, d ** -0.5 / d, True)
    np.testing.assert_array_equal(o, o2)
    np.testing.assert_array_equal(lse, lse2)
    dq2, dk2, dv2 = fp8_backward_from_operands(qr, kr, vr, do, s, d ** -0.5, True)
    np.testing.assert_array_equal(dq, dq2)
    # The operands are close to the unquantised rotated inputs (e4m3: 2^-4 relative
    # per element at most, bf16 adds 2^-9), and the gradient is close to the exact one.
    m = np.diag(s.astype(np.float64)) @ sylvester_hadamard(d)
    qx = x["q"].numpy().astype(np.float64) @ m
    assert np.abs(qr - qx).max() <= (2.0 ** -4 + 2.0 ** -8) * np.abs(qx).max()
    dqx, _, dvx = attention_backward(x["q"].numpy().astype(np.float64), x["k"].numpy().astype(np.float64),
                                     x["v"].numpy().astype(np.float64), do, d ** -0.5, True)
    assert np.abs(dv - dvx).max() <= 0.2 * np.abs(dvx).max()
    assert np.abs(dq - dqx).max() <= 0.5 * np.abs(dqx).max()


def test_operands_are_the_exact_dequantised_values():
    # Power-of-two tile scales: decode(code) * sigma has at most 4 significant bits,
    # so its bf16 rounding is exact and the backward sees the forward's operands.
    from oracle import fp8_dequantize

    x = outlier_qkv(2, 2, 300, 128, seed=21)
    s = rotation_signs(128, seed=21).numpy()
    prep = fp8_prepare(x["q"], x["k"], x["v"], s)
    for name, op in zip(("q", "k", "v"), fp8_operands(prep)):
        np.testing.assert_array_equal(op, fp8_dequantize(prep[name + "8"], prep["s" + name]))


@pytest.mark.parametrize("causal", [False, True])
def test_sampled_equals_full(causal):
    from oracle.fp8_backward import fp8_backward_sampled

    B, H, N, d = 1, 1, 150, 64
    x = outlier_qkv(B, H, N, d, seed=30)
    do = torch.randn(B, H, N, d, generator=torch.Generator().manual_seed(2)).numpy().astype(np.float64)
    s = rotation_signs(d, seed=30).numpy()
    prep = fp8_prepare(x["q"], x["k"], x["v"], s)
    dq, dk, dv, _, _ = fp8_backward(prep, s, do, 0.2, causal)
    qr, kr, vr = fp8_operands(prep)
    idx = np.array([0, 5, 63, 64, 149])
    sq, sk, sv = fp8_backward_sampled(qr[0, 0], kr[0, 0], vr[0, 0], do[0, 0], s, 0.2, causal, idx, idx)
    for got, full in ((sq, dq), (sk, dk), (sv, dv)):
        np.testing.assert_allclose(got, full[0, 0, idx], rtol=1e-10, atol=1e-12 * np.abs(full).max())
