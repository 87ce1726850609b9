"""Pins of the forward oracle against facts fixed by the definition, not by itself.

Each test would fail for a plausible mistake in the oracle: a dropped or doubled
``scale``, a transposed operand, the causal mask on the wrong side, a natural/base-2
mix-up in LSE, a missing max subtraction (overflow), or chunking that mixes rows.
"""

import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import attention_forward, attention_forward_rows, attention_forward_brute
from synth import normal_qkv

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _num(x):
    if isinstance(x, str):
        return {"ln3": math.log(3.0), "ln4": math.log(4.0), "ln2": math.log(2.0)}[x]
    return float(x)


def _arr(nested):
    return np.array([[_num(x) for x in row] for row in nested], dtype=np.float64)


@pytest.mark.parametrize("causal", [False, True])
def test_hand_derived_two_token_example(causal):
    g = json.load(open(os.path.join(GOLDEN, "hand_two_tokens.json")))
    q, k, v = (_arr(g[n])[None, None] for n in ("q", "k", "v"))
    o, lse = attention_forward(q, k, v, g["scale"], causal)
    ref = g["causal" if causal else "noncausal"]
    np.testing.assert_allclose(o[0, 0], _arr(ref["o"]), rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse[0, 0], [_num(x) for x in ref["lse"]], rtol=0, atol=1e-14)


@pytest.mark.parametrize("causal", [False, True])
def test_rows_are_probability_distributions(causal):
    # With V = identity (d = N), O is exactly the probability matrix P.
    N = 24
    x = normal_qkv(1, 1, N, N, seed=11)
    v = np.eye(N)[None, None]
    p, _ = attention_forward(x["q"].numpy() * 3.0, x["k"].numpy(), v, 0.7, causal)
    p = p[0, 0]
    assert (p >= 0).all()
    np.testing.assert_allclose(p.sum(axis=1), 1.0, rtol=0, atol=1e-12)
    if causal:
        assert np.all(p[np.triu_indices(N, 1)] == 0.0)


@pytest.mark.parametrize("causal", [False, True])
def test_identical_keys_give_column_means(causal):
    N, d, scale = 40, 8, 0.3
    x = normal_qkv(1, 1, N, d, seed=12)
    q, v = x["q"].numpy().astype(np.float64), x["v"].numpy().astype(np.float64)
    krow = np.linspace(-1.0, 2.0, d)
    k = np.broadcast_to(krow, (1, 1, N, d)).copy()
    o, lse = attention_forward(q, k, v, scale, causal)
    counts = np.arange(1, N + 1) if causal else np.full(N, N)
    if causal:
        ref_o = np.cumsum(v[0, 0], axis=0) / counts[:, None]
    else:
        ref_o = np.broadcast_to(v[0, 0].mean(axis=0), (N, d))
    ref_lse = scale * (q[0, 0] @ krow) + np.log(counts)
    np.testing.assert_allclose(o[0, 0], ref_o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse[0, 0], ref_lse, rtol=0, atol=1e-12)


def test_dominant_score_selects_value_row_closed_form():
    # Orthonormal keys e_0..e_{N-1}; q_i = c * e_{j(i)}; scores are c*scale at j(i), 0 elsewhere.
    N, d, scale, c = 16, 16, 1.0, 50.0
    k = np.eye(N, d)[None, None]
    rng = np.random.default_rng(5)
    v = rng.standard_normal((1, 1, N, d))
    target = rng.permutation(N)
    q = (c * np.eye(N, d)[target])[None, None]
    o, lse = attention_forward(q, k, v, scale, False)
    w = math.exp(c * scale)
    vs = v[0, 0]
    for i, j in enumerate(target):
        ref = (w * vs[j] + (vs.sum(axis=0) - vs[j])) / (w + N - 1)
        np.testing.assert_allclose(o[0, 0, i], ref, rtol=0, atol=1e-12)
        np.testing.assert_allclose(o[0, 0, i], vs[j], rtol=0, atol=1e-12)
        assert abs(lse[0, 0, i] - (c * scale + math.log1p((N - 1) / w))) < 1e-12


def test_causal_row_zero_and_single_token():
    x = normal_qkv(2, 3, 33, 8, seed=13)
    q, k, v = (x[n].numpy().astype(np.float64) for n in ("q", "k", "v"))
    scale = 0.45
    o, lse = attention_forward(q, k, v, scale, True)
    np.testing.assert_array_equal(o[:, :, 0], v[:, :, 0])
    np.testing.assert_allclose(lse[:, :, 0], scale * np.einsum("bhd,bhd->bh", q[:, :, 0], k[:, :, 0]),
                               rtol=0, atol=1e-12)
    for causal in (False, True):
        o1, l1 = attention_forward(q[:, :, :1], k[:, :, :1], v[:, :, :1], scale, causal)
        np.testing.assert_array_equal(o1, v[:, :, :1])
        np.testing.assert_allclose(l1[..., 0], scale * np.einsum("bhd,bhd->bh", q[:, :, 0], k[:, :, 0]),
                                   rtol=0, atol=1e-12)


def test_noncausal_permutation_equivariance():
    x = normal_qkv(1, 2, 30, 8, seed=14)
    q, k, v = (x[n].numpy().astype(np.float64) for n in ("q", "k", "v"))
    o, lse = attention_forward(q, k, v, 0.4, False)
    rng = np.random.default_rng(0)
    pk = rng.permutation(30)
    o2, lse2 = attention_forward(q, k[:, :, pk], v[:, :, pk], 0.4, False)
    np.testing.assert_allclose(o2, o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse2, lse, rtol=0, atol=1e-12)
    pq = rng.permutation(30)
    o3, lse3 = attention_forward(q[:, :, pq], k, v, 0.4, False)
    np.testing.assert_allclose(o3, o[:, :, pq], rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse3, lse[:, :, pq], rtol=0, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_constant_score_shift(causal):
    # Appending a feature 1 to every query and a to every key adds scale*a to every score.
    x = normal_qkv(1, 1, 20, 6, seed=15)
    q, k, v = (x[n].numpy().astype(np.float64) for n in ("q", "k", "v"))
    scale, a = 0.8, 3.25
    o, lse = attention_forward(q, k, v, scale, causal)
    q2 = np.concatenate([q, np.ones(q.shape[:-1] + (1,))], axis=-1)
    k2 = np.concatenate([k, np.full(k.shape[:-1] + (1,), a)], axis=-1)
    o2, lse2 = attention_forward(q2, k2, v, scale, causal)
    np.testing.assert_allclose(o2, o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse2, lse + scale * a, rtol=0, atol=1e-12)


def test_large_scores_do_not_overflow():
    # Scores near 1e4 would overflow a softmax without the row-max subtraction.
    x = normal_qkv(1, 1, 16, 4, seed=16)
    q, k, v = (x[n].numpy().astype(np.float64) for n in ("q", "k", "v"))
    o, lse = attention_forward(q * 100.0, k * 100.0, v, 1.0, False)
    assert np.isfinite(o).all() and np.isfinite(lse).all()


@pytest.mark.parametrize("causal", [False, True])
def test_vectorised_matches_scalar_brute_force(causal):
    x = normal_qkv(2, 2, 13, 5, seed=17)
    q, k, v = (x[n].numpy().astype(np.float64) for n in ("q", "k", "v"))
    o, lse = attention_forward(q, k, v, 0.6, causal)
    ob, lb = attention_forward_brute(q.tolist(), k.tolist(), v.tolist(), 0.6, causal)
    np.testing.assert_allclose(o, np.array(ob), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, np.array(lb), rtol=0, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_matches_torch_sdpa_math_path(causal):
    x = normal_qkv(2, 3, 50, 16, seed=18)
    q, k, v = (x[n].to(torch.float64) for n in ("q", "k", "v"))
    scale = 0.37
    o, lse = attention_forward(q, k, v, scale, causal)
    ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=causal, scale=scale)
    np.testing.assert_allclose(o, ref.numpy(), rtol=0, atol=1e-12)
    s = scale * q @ k.transpose(-1, -2)
    if causal:
        s = s.masked_fill(torch.ones(50, 50, dtype=torch.bool).triu(1), float("-inf"))
    np.testing.assert_allclose(lse, torch.logsumexp(s, dim=-1).numpy(), rtol=0, atol=1e-12)


def test_row_chunking_is_exact_and_rows_helper_agrees():
    x = normal_qkv(1, 2, 70, 8, seed=19)
    q, k, v = (x[n].numpy().astype(np.float64) for n in ("q", "k", "v"))
    for causal in (False, True):
        o, lse = attention_forward(q, k, v, 0.5, causal, row_chunk=1024)
        o7, lse7 = attention_forward(q, k, v, 0.5, causal, row_chunk=7)
        np.testing.assert_array_equal(o, o7)
        np.testing.assert_array_equal(lse, lse7)
        rows = [0, 5, 63, 69]
        orow, lrow = attention_forward_rows(q[0, 1], k[0, 1], v[0, 1], 0.5, causal, rows)
        np.testing.assert_allclose(orow, o[0, 1, rows], rtol=0, atol=1e-13)
        np.testing.assert_allclose(lrow, lse[0, 1, rows], rtol=0, atol=1e-13)


def test_oracle_imports_nothing_from_the_product_path():
    import re
    import sys

    for name, mod in list(sys.modules.items()):
        if name.startswith("oracle"):
            src = open(mod.__file__).read() if getattr(mod, "__file__", None) else ""
            assert not re.search(r"^\s*(from|import)\s+io_aware_exact_fwd_gb300", src, re.M)
    assert oracle.__doc__ and "test infrastructure" in oracle.__doc__
