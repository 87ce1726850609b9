"""Split-KV attention partials and their exact merge, float64 numpy (test infrastructure).

What is computed.  Attention of Nq queries against Nk keys, with the keys cut into
consecutive ranges ("splits").  For one head and one split covering keys
[a, b):

    S_ij   = scale * q_i . k_j                       for a <= j < b
    S_ij   = -inf  where key j is not visible to query i
    LSE_i  = ln sum_j exp(S_ij)                       (-inf if row i sees no key)
    O_i    = sum_j exp(S_ij - LSE_i) v_j              (0 if row i sees no key)

and the merge of the splits s = 0 .. n-1 of one row is

    LSE = ln sum_s exp(LSE_s)
    O   = sum_s exp(LSE_s - LSE) O_s

which is exactly the softmax over the union of the key ranges: exp(LSE_s) is the
partial row sum of exp(S) over split s, so the weights exp(LSE_s - LSE) put every
split's normalised output back on the common denominator.  The pages state the
inference setting this serves ("FlashAttention-Skalierung, Multi-GPU-Training und
Gewichtsquantisierung", section 3: generating one token at a time is bound by
memory bandwidth, not arithmetic) but print no split-KV algorithm; the formulas
above are the plain reading of "softmax over all keys" cut into key ranges.

Causal masking with Nq <= Nk aligns the queries with the LAST Nq keys: query i
(0-based) sees key j iff j <= i + (Nk - Nq).  With Nq == Nk this is the usual
causal mask (key j visible to query i iff j <= i).

Split rule (part of the library's interface, restated here): keys are grouped in
blocks of 128; with nkb = ceil(Nk / 128) blocks and kbps = ceil(nkb / n_split)
blocks per split, split s covers keys [128 s kbps, min(128 (s+1) kbps, Nk)).  Trailing
splits may be empty.

Shapes: q [B, H, Nq, d]; k, v [B, H, Nk, d]; partial O [n, B, H, Nq, d]; partial
LSE [n, B, H, Nq].
"""

from __future__ import annotations

import numpy as np

from .attention import _as_f64

KEY_BLOCK = 128


def split_key_ranges(Nk: int, n_split: int, block: int = KEY_BLOCK):
    """Key ranges [a, b) of the n_split splits (trailing ones may be empty)."""
    nkb = -(-Nk // block)
    kbps = -(-nkb // n_split)
    out = []
    for s in range(n_split):
        a = min(s * kbps * block, Nk)
        b = min((s + 1) * kbps * block, Nk)
        out.append((a, b))
    return out


def _visible(Nq: int, Nk: int, causal: bool, a: int, b: int) -> np.ndarray:
    """Boolean [Nq, b - a]: key a + j visible to query i."""
    keys = np.arange(a, b)
    if not causal:
        return np.ones((Nq, b - a), dtype=bool)
    limit = np.arange(Nq) + (Nk - Nq)
    return keys[None, :] <= limit[:, None]


def attention_partial(q, k, v, scale: float, causal: bool, a: int, b: int):
    """Partial (O_s, LSE_s) of keys [a, b) for every (batch, head).

    Returns (O [B, H, Nq, d] float64, LSE [B, H, Nq] float64); rows that see no
    key of the range get O = 0 and LSE = -inf.
    """
    q, k, v = _as_f64(q), _as_f64(k), _as_f64(v)
    B, H, Nq, _ = q.shape
    Nk = k.shape[2]
    dv = v.shape[-1]
    o = np.zeros((B, H, Nq, dv))
    lse = np.full((B, H, Nq), -np.inf)
    if b <= a:
        return o, lse
    vis = _visible(Nq, Nk, causal, a, b)
    any_vis = vis.any(axis=1)
    for bb in range(B):
        for h in range(H):
            s = scale * (q[bb, h] @ k[bb, h, a:b].T)
            s = np.where(vis, s, -np.inf)
            rows = np.nonzero(any_vis)[0]
            if rows.size == 0:
                continue
            sr = s[rows]
            m = sr.max(axis=1, keepdims=True)
            e = np.exp(sr - m)
            l = e.sum(axis=1, keepdims=True)
            o[bb, h, rows] = (e / l) @ v[bb, h, a:b]
            lse[bb, h, rows] = m[:, 0] + np.log(l[:, 0])
    return o, lse


def attention_splitkv(q, k, v, scale: float, causal: bool, n_split: int):
    """All partials of the split rule: (O [n, B, H, Nq, d], LSE [n, B, H, Nq])."""
    k_ = _as_f64(k)
    ranges = split_key_ranges(k_.shape[2], n_split)
    parts = [attention_partial(q, k, v, scale, causal, a, b) for a, b in ranges]
    return np.stack([p[0] for p in parts]), np.stack([p[1] for p in parts])


def merge_partials(o_parts, lse_parts):
    """Exact merge of partials along axis 0: returns (O, LSE).

    Splits with LSE = -inf carry no weight and their O is not read.  A row whose
    every split is empty gets O = 0 and LSE = -inf.
    """
    o_parts, lse_parts = _as_f64(o_parts), _as_f64(lse_parts)
    m = lse_parts.max(axis=0)
    finite = np.isfinite(m)
    m_safe = np.where(finite, m, 0.0)
    w = np.where(np.isfinite(lse_parts), np.exp(lse_parts - m_safe[None]), 0.0)
    tot = w.sum(axis=0)
    lse = np.where(finite, m_safe + np.log(np.where(finite, tot, 1.0)), -np.inf)
    o_sum = np.zeros(o_parts.shape[1:])
    with np.errstate(invalid="ignore"):
        for s in range(o_parts.shape[0]):
            ws = w[s][..., None]
            o_sum += np.where(ws > 0, ws * o_parts[s], 0.0)
    o = np.where(finite[..., None], o_sum / np.where(finite, tot, 1.0)[..., None], 0.0)
    return o, lse


def attention_general(q, k, v, scale: float, causal: bool):
    """Unsplit attention of Nq queries against Nk keys (the single-split partial)."""
    Nk = _as_f64(k).shape[2]
    return attention_partial(q, k, v, scale, causal, 0, Nk)


def splitkv_flops(B: int, H: int, Nq: int, Nk: int, d: int, causal: bool) -> float:
    """Matmul flops of the visible (query, key) pairs: 4 d per pair (Q K^T and P V)."""
    if not causal:
        pairs = Nq * Nk
    else:
        off = Nk - Nq
        pairs = sum(min(Nk, i + off + 1) for i in range(Nq))
    return 4.0 * d * B * H * pairs


__all__ = [
    "KEY_BLOCK",
    "split_key_ranges",
    "attention_partial",
    "attention_splitkv",
    "merge_partials",
    "attention_general",
    "splitkv_flops",
]
