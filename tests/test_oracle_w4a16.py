"""Pins of the W4A16 oracle: hand-derived packed words, exact dequantisation cases,
a scalar triple loop, and closed forms.  A swapped nibble order, a missing zero
point, scales applied per column instead of per group, or a transposed product
fails one of them."""

import json
import os

import numpy as np
import pytest
import torch

from oracle import w4a16_abs_sum, w4a16_dequant, w4a16_gemm, w4a16_unpack
from synth import w4a16_inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_hand_derived_words():
    g = json.load(open(os.path.join(GOLDEN, "w4a16_words.json")))
    for c in g["cases"]:
        w = np.array([[int(c["word"], 16)]], dtype=np.uint32).view(np.int32)
        assert w4a16_unpack(w)[0].tolist() == c["codes"], c["word"]


def test_unpack_covers_every_bit_once():
    rng = np.random.default_rng(0)
    w = rng.integers(0, 2 ** 32, (3, 5), dtype=np.uint64).astype(np.uint32)
    q = w4a16_unpack(w.view(np.int32))
    # Re-pack by the reading's positions and recover the words exactly.
    back = np.zeros_like(w, dtype=np.uint64)
    for i in range(4):
        back |= (q[:, 2 * i::8].astype(np.uint64) << (4 * i)) | (q[:, 2 * i + 1::8].astype(np.uint64) << (4 * i + 16))
    assert np.array_equal(back.astype(np.uint32), w)


def test_dequant_exact_cases():
    # One row, one group (K = 128): codes chosen per k, scale and zero point fixed.
    codes = np.zeros(128, dtype=np.int64)
    codes[0], codes[1], codes[2], codes[3] = 15, 8, 0, 7
    words = np.zeros((1, 16), dtype=np.uint64)
    for k, c in enumerate(codes):
        wi, j = divmod(k, 8)
        shift = 4 * (j // 2) + 16 * (j % 2)
        words[0, wi] |= np.uint64(c) << np.uint64(shift)
    wq = words.astype(np.uint32).view(np.int32)
    s = np.array([[0.5]], dtype=np.float16)
    z = np.array([[8]], dtype=np.uint8)
    w = w4a16_dequant(wq, s, z)[0]
    assert w[0] == 3.5 and w[1] == 0.0 and w[2] == -4.0 and w[3] == -0.5
    assert np.all(w[4:] == -4.0)
    # fp16 rounding of an inexact product: 7 * fp16(0.1).
    s2 = np.array([[0.1]], dtype=np.float16)
    z2 = np.array([[8]], dtype=np.uint8)
    w2 = w4a16_dequant(wq, s2, z2)[0]
    assert w2[0] == float(np.float16(7 * float(np.float16(0.1))))


def test_gemm_matches_scalar_loop():
    d = w4a16_inputs(2, 3, 256, 5)
    y = w4a16_gemm(d["x"], d["wq"], d["scales"], d["zeros"])
    wq = d["wq"].numpy().astype(np.int64) & 0xFFFFFFFF
    x = d["x"].float().numpy().astype(np.float64)
    s, z = d["scales"].float().numpy().astype(np.float64), d["zeros"].numpy().astype(np.int64)
    for m in range(2):
        for n in range(3):
            acc = 0.0
            for k in range(256):
                j = k % 8
                code = (wq[n, k // 8] >> (4 * (j // 2) + 16 * (j % 2))) & 0xF
                wv = float(np.float16((code - z[k // 128, n]) * s[k // 128, n]))
                acc += x[m, k] * wv
            assert abs(y[m, n] - acc) <= 1e-12 * max(1.0, abs(acc))


def test_closed_form_constant_weights():
    # Every code 9, zero point 1, scale 0.25: every weight is 2, so Y = 2 * row sums of X.
    M, N, K = 3, 4, 384
    word = 0
    for j in range(8):
        word |= 9 << (4 * (j // 2) + 16 * (j % 2))
    wq = np.full((N, K // 8), word, dtype=np.uint32).view(np.int32)
    s = np.full((K // 128, N), 0.25, dtype=np.float16)
    z = np.ones((K // 128, N), dtype=np.uint8)
    x = torch.randn(M, K, generator=torch.Generator().manual_seed(3)).to(torch.float16)
    y = w4a16_gemm(x, wq, s, z)
    ref = 2.0 * x.double().sum(dim=1, keepdim=True).numpy()
    np.testing.assert_allclose(y, np.repeat(ref, N, axis=1), rtol=0, atol=1e-12)
    # Codes equal to the zero point give zero weights.
    z9 = np.full((K // 128, N), 9, dtype=np.uint8)
    assert np.all(w4a16_gemm(x, wq, s, z9) == 0)


def test_groups_use_their_own_scale_and_zero():
    M, N, K = 1, 2, 256
    d = w4a16_inputs(M, N, K, 9)
    s = d["scales"].clone()
    s[1] = s[1] * 2  # second group of every row doubled
    w0 = w4a16_dequant(d["wq"], d["scales"], d["zeros"])
    w1 = w4a16_dequant(d["wq"], s, d["zeros"])
    assert np.array_equal(w0[:, :128], w1[:, :128])
    assert np.array_equal(w1[:, 128:], 2 * w0[:, 128:])  # a power-of-two scale commutes with fp16 rounding
    assert np.all(w4a16_abs_sum(d["x"], d["wq"], d["scales"], d["zeros"]) >=
                  np.abs(w4a16_gemm(d["x"], d["wq"], d["scales"], d["zeros"])))
