"""Pins of the backward oracle: finite differences, autograd, and exact sum rules."""

import numpy as np
import pytest
import torch

from oracle import attention_backward, attention_backward_rows, attention_backward_sampled, attention_forward
from synth import normal_qkv


def _loss(q, k, v, g, scale, causal):
    o, _ = attention_forward(q, k, v, scale, causal)
    return float((o * g).sum())


@pytest.mark.parametrize("causal", [False, True])
def test_backward_matches_central_finite_differences(causal):
    x = normal_qkv(1, 2, 7, 4, seed=21, with_do=True)
    q, k, v, g = (x[n].numpy().astype(np.float64) for n in ("q", "k", "v", "do"))
    scale, h = 0.55, 1e-6
    dq, dk, dv = attention_backward(q, k, v, g, scale, causal)
    for name, arr, grad in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.zeros_like(arr)
        it = np.nditer(arr, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            plus, minus = arr.copy(), arr.copy()
            plus[idx] += h
            minus[idx] -= h
            args = {"q": q, "k": k, "v": v}
            args[name] = plus
            lp = _loss(args["q"], args["k"], args["v"], g, scale, causal)
            args[name] = minus
            lm = _loss(args["q"], args["k"], args["v"], g, scale, causal)
            num[idx] = (lp - lm) / (2 * h)
        err = np.abs(num - grad).max() / max(1e-12, np.abs(grad).max())
        assert err < 1e-6, (name, err)


@pytest.mark.parametrize("causal", [False, True])
def test_backward_matches_torch_autograd_of_textbook_formula(causal):
    x = normal_qkv(2, 2, 29, 8, seed=22, with_do=True)
    q, k, v, g = (x[n].to(torch.float64) for n in ("q", "k", "v", "do"))
    scale = 0.42
    qq, kk, vv = (t.clone().requires_grad_(True) for t in (q, k, v))
    s = scale * qq @ kk.transpose(-1, -2)
    if causal:
        s = s.masked_fill(torch.ones(29, 29, dtype=torch.bool).triu(1), float("-inf"))
    o = torch.softmax(s, dim=-1) @ vv
    (o * g).sum().backward()
    dq, dk, dv = attention_backward(q, k, v, g, scale, causal)
    np.testing.assert_allclose(dq, qq.grad.numpy(), rtol=0, atol=1e-10)
    np.testing.assert_allclose(dk, kk.grad.numpy(), rtol=0, atol=1e-10)
    np.testing.assert_allclose(dv, vv.grad.numpy(), rtol=0, atol=1e-10)


@pytest.mark.parametrize("causal", [False, True])
def test_backward_sum_rules(causal):
    # Each row of dS sums to zero, so dK sums to zero over keys; dV sums to the sum of dO rows.
    x = normal_qkv(1, 3, 45, 8, seed=23, with_do=True)
    q, k, v, g = (x[n].numpy().astype(np.float64) for n in ("q", "k", "v", "do"))
    dq, dk, dv = attention_backward(q, k, v, g, 0.3, causal)
    np.testing.assert_allclose(dk.sum(axis=2), 0.0, rtol=0, atol=1e-12)
    np.testing.assert_allclose(dv.sum(axis=2), g.sum(axis=2), rtol=0, atol=1e-12)


def test_backward_chunking_is_a_plain_sum():
    x = normal_qkv(1, 1, 37, 8, seed=24, with_do=True)
    q, k, v, g = (x[n].numpy().astype(np.float64) for n in ("q", "k", "v", "do"))
    for causal in (False, True):
        a = attention_backward(q, k, v, g, 0.5, causal, row_chunk=1024)
        b = attention_backward(q, k, v, g, 0.5, causal, row_chunk=5)
        for x1, x2 in zip(a, b):
            np.testing.assert_allclose(x1, x2, rtol=0, atol=1e-12)


def test_causal_last_key_gets_gradient_only_from_last_query():
    # Key N-1 is visible to query N-1 only: dV[N-1] = P[N-1, N-1] * dO[N-1].
    x = normal_qkv(1, 1, 12, 4, seed=25, with_do=True)
    q, k, v, g = (x[n].numpy().astype(np.float64) for n in ("q", "k", "v", "do"))
    scale = 0.7
    _, lse = attention_forward(q, k, v, scale, True)
    p_last = np.exp(scale * q[0, 0, -1] @ k[0, 0, -1] - lse[0, 0, -1])
    _, _, dv = attention_backward(q, k, v, g, scale, True)
    np.testing.assert_allclose(dv[0, 0, -1], p_last * g[0, 0, -1], rtol=0, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_sampled_backward_equals_full_backward(causal):
    x = normal_qkv(1, 1, 150, 16, seed=26, with_do=True)
    q, k, v, g = (x[n].numpy().astype(np.float64) for n in ("q", "k", "v", "do"))
    dq, dk, dv = attention_backward(q, k, v, g, 0.45, causal)
    rows = [0, 1, 77, 149]
    keys = [0, 64, 148, 149]
    sq, sk, sv = attention_backward_sampled(q[0, 0], k[0, 0], v[0, 0], g[0, 0], 0.45, causal, rows, keys,
                                            row_chunk=37)
    np.testing.assert_allclose(sq, dq[0, 0, rows], rtol=0, atol=1e-12)
    np.testing.assert_allclose(sk, dk[0, 0, keys], rtol=0, atol=1e-12)
    np.testing.assert_allclose(sv, dv[0, 0, keys], rtol=0, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_row_block_parts_sum_to_full_backward(causal):
    x = normal_qkv(1, 1, 90, 8, seed=27, with_do=True)
    q, k, v, g = (x[n].numpy().astype(np.float64)[0, 0] for n in ("q", "k", "v", "do"))
    dq, dk, dv = attention_backward(q[None, None], k[None, None], v[None, None], g[None, None], 0.6, causal)
    sk, sv = np.zeros_like(k), np.zeros_like(v)
    for r0 in (0, 31, 60):
        rows = np.arange(r0, {0: 31, 31: 60, 60: 90}[r0])
        pq, pk, pv = attention_backward_rows(q, k, v, g, 0.6, causal, rows)
        np.testing.assert_allclose(pq, dq[0, 0, rows], rtol=0, atol=1e-12)
        sk += pk
        sv += pv
    np.testing.assert_allclose(sk, dk[0, 0], rtol=0, atol=1e-12)
    np.testing.assert_allclose(sv, dv[0, 0], rtol=0, atol=1e-12)
