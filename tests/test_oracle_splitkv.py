"""Pins of the split-KV oracle (partials over key ranges and their merge).

Each pin comes from outside the code under test: the unsplit attention oracle
(itself pinned in test_oracle_forward.py), a scalar loop on tiny inputs, or a closed
form.  A dropped merge weight, a merge in base 2 instead of e, a causal offset on
the wrong side, or a split rule that skips or repeats keys fails one of them.
"""

import math

import numpy as np
import pytest

from oracle import (
    attention_forward,
    attention_general,
    attention_partial,
    attention_splitkv,
    merge_partials,
    split_key_ranges,
    splitkv_flops,
)
from synth import normal_qkv


def _qkv(B, H, Nq, Nk, d, seed):
    x = normal_qkv(B, H, Nk, d, seed)
    q = normal_qkv(B, H, Nq, d, seed + 1000)["q"].numpy().astype(np.float64)
    return q, x["k"].numpy().astype(np.float64), x["v"].numpy().astype(np.float64)


@pytest.mark.parametrize("Nk,n", [(1, 1), (127, 2), (128, 1), (129, 2), (1000, 3), (1280, 6), (4096, 7), (300, 40)])
def test_split_rule_partitions_keys(Nk, n):
    r = split_key_ranges(Nk, n)
    assert len(r) == n
    assert r[0][0] == 0 and r[-1][1] == Nk
    for (a, b), (c, _) in zip(r, r[1:]):
        assert b == c and a <= b
    for a, b in r:
        assert a % 128 == 0 or a == Nk
    nonempty = [b - a for a, b in r if b > a]
    assert all(x % 128 == 0 for x in nonempty[:-1])  # only the last nonempty split can be ragged


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("n_split", [1, 2, 3, 5])
def test_merge_of_splits_equals_unsplit_attention(causal, n_split):
    q, k, v = _qkv(1, 2, 300, 300, 16, 3)
    op, lp = attention_splitkv(q, k, v, 0.25, causal, n_split)
    o, lse = merge_partials(op, lp)
    o_ref, lse_ref = attention_forward(q, k, v, 0.25, causal)
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lse_ref, rtol=0, atol=1e-12)


def test_bottom_right_causal_equals_scalar_loop():
    # Nq < Nk: query i sees keys j <= i + Nk - Nq.  Scalar reference on a tiny head.
    q, k, v = _qkv(1, 1, 5, 9, 3, 11)
    scale = 0.7
    o, lse = attention_general(q, k, v, scale, True)
    Nq, Nk = 5, 9
    for i in range(Nq):
        keys = [j for j in range(Nk) if j <= i + Nk - Nq]
        s = [scale * sum(q[0, 0, i, c] * k[0, 0, j, c] for c in range(3)) for j in keys]
        m = max(s)
        e = [math.exp(x - m) for x in s]
        tot = sum(e)
        for c in range(3):
            ref = sum(e[t] * v[0, 0, keys[t], c] for t in range(len(keys))) / tot
            assert abs(o[0, 0, i, c] - ref) < 1e-12
        assert abs(lse[0, 0, i] - (m + math.log(tot))) < 1e-12


def test_single_query_causal_sees_every_key():
    q, k, v = _qkv(2, 2, 1, 333, 8, 5)
    oc, lc = attention_general(q, k, v, 0.3, True)
    on, ln_ = attention_general(q, k, v, 0.3, False)
    np.testing.assert_array_equal(oc, on)
    np.testing.assert_array_equal(lc, ln_)


def test_duplicated_keys_closed_form():
    # Keys [K; K] with values [V; V]: the weights are unchanged, so O is the one-copy
    # output and LSE grows by exactly ln 2; the two splits are the two copies.
    q, k, v = _qkv(1, 2, 64, 128, 16, 7)
    k2, v2 = np.concatenate([k, k], axis=2), np.concatenate([v, v], axis=2)
    op, lp = attention_splitkv(q, k2, v2, 0.5, False, 2)
    np.testing.assert_allclose(lp[0], lp[1], rtol=0, atol=0)
    o, lse = merge_partials(op, lp)
    o_ref, lse_ref = attention_general(q, k, v, 0.5, False)
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, lse_ref + math.log(2.0), rtol=0, atol=1e-13)


def test_empty_and_masked_splits_carry_no_weight():
    # Causal, Nq = Nk: split 1 (keys 128..255) is invisible to rows 0..127.
    q, k, v = _qkv(1, 1, 256, 256, 8, 9)
    op, lp = attention_splitkv(q, k, v, 0.4, True, 2)
    assert np.all(np.isneginf(lp[1, 0, 0, :128]))
    assert np.all(op[1, 0, 0, :128] == 0)
    # Garbage in an empty split's O must not reach the merge.
    op_bad = op.copy()
    op_bad[1, 0, 0, :128] = np.nan
    o, lse = merge_partials(op_bad, lp)
    o_ref, lse_ref = attention_forward(q, k, v, 0.4, True)
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lse_ref, rtol=0, atol=1e-12)
    # A trailing split past the last key is empty.
    op2, lp2 = attention_splitkv(q, k, v, 0.4, False, 3)
    assert split_key_ranges(256, 3)[2] == (256, 256)
    assert np.all(np.isneginf(lp2[2]))
    # All splits empty: O = 0, LSE = -inf.
    o0, l0 = merge_partials(np.full((2, 1, 1, 3, 4), np.nan), np.full((2, 1, 1, 3), -np.inf))
    assert np.all(o0 == 0) and np.all(np.isneginf(l0))


def test_merge_is_order_free_and_uses_natural_log():
    q, k, v = _qkv(1, 1, 32, 640, 16, 13)
    op, lp = attention_splitkv(q, k, v, 0.25, False, 5)
    o1, l1 = merge_partials(op, lp)
    perm = [3, 0, 4, 2, 1]
    o2, l2 = merge_partials(op[perm], lp[perm])
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-13)
    np.testing.assert_allclose(l1, l2, rtol=0, atol=1e-13)
    # Two splits with equal LSE: the merged LSE is that value + ln 2 and O their mean.
    o3, l3 = merge_partials(np.stack([op[0], op[1]]), np.stack([lp[0], lp[0]]))
    np.testing.assert_allclose(l3, lp[0] + math.log(2.0), rtol=0, atol=1e-13)
    np.testing.assert_allclose(o3, 0.5 * (op[0] + op[1]), rtol=0, atol=1e-13)


def test_partial_of_full_range_is_the_forward():
    q, k, v = _qkv(1, 2, 200, 200, 16, 17)
    for causal in (False, True):
        o, lse = attention_partial(q, k, v, 0.3, causal, 0, 200)
        o_ref, lse_ref = attention_forward(q, k, v, 0.3, causal)
        np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-13)
        np.testing.assert_allclose(lse, lse_ref, rtol=0, atol=1e-13)


def test_flop_count():
    assert splitkv_flops(1, 1, 4, 4, 8, False) == 4 * 8 * 16
    assert splitkv_flops(1, 1, 4, 4, 8, True) == 4 * 8 * 10       # 1+2+3+4 visible pairs
    assert splitkv_flops(1, 1, 2, 5, 8, True) == 4 * 8 * (4 + 5)  # rows see 4 and 5 keys
