"""Exact attention, forward and backward, in float64 numpy (test infrastructure).

Definition followed ("FlashAttention-2 (DE)", section "Hintergrund: Das
Attention-Problem in Transformern"; "FlashAttention-Skalierung, Multi-GPU-Training
und Gewichtsquantisierung", section 1): standard self-attention builds the full
score matrix of every (batch, head) and normalises each row with a softmax.  For
one head with Q, K, V in R^{N x d}:

    S   = scale * Q K^T                      (N x N)
    S_ij = -inf  for j > i                   (causal only; key j visible iff j <= i)
    m_i = max_j S_ij
    E   = exp(S - m)        l_i = sum_j E_ij        P = E / l
    O   = P V               LSE_i = m_i + ln(l_i)   (natural log)

Subtracting the row maximum before ``exp`` does not change P (it cancels in E/l)
and keeps ``exp`` finite; it is part of the textbook softmax, not a tiling trick.
Rows are processed in independent chunks only to bound memory: every row of S is
complete before its softmax is taken.

The backward follows from the chain rule with an upstream gradient dO on O and
none on LSE:

    dV = P^T dO
    dP = dO V^T
    D_i = sum_j P_ij dP_ij          (= sum_c dO_ic O_ic)
    dS = P * (dP - D 1^T)
    dQ = scale * dS K
    dK = scale * dS^T Q

Inputs are taken as exact float64 up-casts of whatever values are passed (bf16
values stay the bf16 values).  Shapes are [B, H, N, d] (a head is an N x d
matrix); LSE is [B, H, N].
"""

from __future__ import annotations

import numpy as np


def _as_f64(x) -> np.ndarray:
    """Exact float64 copy of a numpy array or a (CPU or device) torch tensor."""
    if hasattr(x, "detach"):
        import torch

        x = x.detach().to("cpu", torch.float64).numpy()
    return np.asarray(x, dtype=np.float64)


def _scores(q_rows: np.ndarray, k: np.ndarray, rows: np.ndarray, scale: float,
            causal: bool) -> np.ndarray:
    """Scaled scores for the given query rows against every key, causal mask applied."""
    s = scale * (q_rows @ k.T)
    if causal:
        keys = np.arange(k.shape[0])
        s = np.where(keys[None, :] > rows[:, None], -np.inf, s)
    return s


def _softmax_rows(s: np.ndarray):
    """Row softmax of a score block: returns (P, m, l)."""
    m = s.max(axis=1, keepdims=True)
    e = np.exp(s - m)
    l = e.sum(axis=1, keepdims=True)
    return e / l, m[:, 0], l[:, 0]


def attention_forward(q, k, v, scale: float, causal: bool, row_chunk: int = 1024):
    """Exact O and LSE for every (batch, head).

    q, k, v: [B, H, N, d].  Returns (O [B,H,N,d] float64, LSE [B,H,N] float64).
    """
    q, k, v = _as_f64(q), _as_f64(k), _as_f64(v)
    B, H, N, d = q.shape
    out = np.empty((B, H, N, v.shape[-1]), dtype=np.float64)
    lse = np.empty((B, H, N), dtype=np.float64)
    for b in range(B):
        for h in range(H):
            for r0 in range(0, N, row_chunk):
                rows = np.arange(r0, min(N, r0 + row_chunk))
                s = _scores(q[b, h, rows], k[b, h], rows, scale, causal)
                p, m, l = _softmax_rows(s)
                out[b, h, rows] = p @ v[b, h]
                lse[b, h, rows] = m + np.log(l)
    return out, lse


def attention_forward_rows(q_head, k_head, v_head, scale: float, causal: bool, rows):
    """Exact O and LSE of selected query rows of ONE head.

    q_head, k_head, v_head: [N, d].  ``rows``: 1-D integer indices.  Each row is
    computed against all N keys exactly as in :func:`attention_forward`, so a
    sample of rows of a large head can be checked without the whole N x N matrix.
    Returns (O [len(rows), d], LSE [len(rows)]).
    """
    q_head, k_head, v_head = _as_f64(q_head), _as_f64(k_head), _as_f64(v_head)
    rows = np.asarray(rows, dtype=np.int64)
    s = _scores(q_head[rows], k_head, rows, scale, causal)
    p, m, l = _softmax_rows(s)
    return p @ v_head, m + np.log(l)


def attention_backward(q, k, v, do, scale: float, causal: bool, row_chunk: int = 1024):
    """Exact dQ, dK, dV for every (batch, head) given the upstream gradient dO.

    P is formed from the definition (not from a stored logsumexp), and D from
    P and dP, so the result does not depend on any forward output.  Rows are
    processed in chunks; dK and dV accumulate over the chunks (a plain sum of the
    per-row contributions).  Returns (dQ, dK, dV), each [B, H, N, d] float64.
    """
    q, k, v, do = _as_f64(q), _as_f64(k), _as_f64(v), _as_f64(do)
    B, H, N, d = q.shape
    dq = np.empty_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for b in range(B):
        for h in range(H):
            for r0 in range(0, N, row_chunk):
                rows = np.arange(r0, min(N, r0 + row_chunk))
                s = _scores(q[b, h, rows], k[b, h], rows, scale, causal)
                p, _, _ = _softmax_rows(s)
                g = do[b, h, rows]
                dv[b, h] += p.T @ g
                dp = g @ v[b, h].T
                dsum = (p * dp).sum(axis=1, keepdims=True)
                ds = p * (dp - dsum)
                dq[b, h, rows] = scale * (ds @ k[b, h])
                dk[b, h] += scale * (ds.T @ q[b, h, rows])
    return dq, dk, dv


def attention_backward_sampled(q_head, k_head, v_head, do_head, scale: float, causal: bool, rows, keys,
                               row_chunk: int = 1024):
    """Exact dQ at selected query rows and dK, dV at selected keys of ONE head.

    The same definition as :func:`attention_backward`, evaluated element by
    element: LSE_i and D_i = sum_j P_ij dP_ij are formed for every row (in row
    chunks, from complete rows of S), then
      dQ_i = scale * sum_j P_ij (dP_ij - D_i) k_j      for i in rows
      dV_j = sum_i P_ij dO_i                            for j in keys
      dK_j = scale * sum_i P_ij (dP_ij - D_i) q_i       for j in keys
    with P_ij = exp(scale q_i.k_j - LSE_i) (0 where masked) and dP_ij = dO_i . v_j.
    Returns (dQ[len(rows), d], dK[len(keys), d], dV[len(keys), d]).
    """
    q, k, v, g = (_as_f64(t) for t in (q_head, k_head, v_head, do_head))
    N = q.shape[0]
    rows = np.asarray(rows, dtype=np.int64)
    keys = np.asarray(keys, dtype=np.int64)
    lse = np.empty(N)
    dsum = np.empty(N)
    for r0 in range(0, N, row_chunk):
        rr = np.arange(r0, min(N, r0 + row_chunk))
        s = _scores(q[rr], k, rr, scale, causal)
        p, m, l = _softmax_rows(s)
        lse[rr] = m + np.log(l)
        dsum[rr] = (p * (g[rr] @ v.T)).sum(axis=1)
    # rows of P for dQ
    s = _scores(q[rows], k, rows, scale, causal)
    p = np.exp(s - lse[rows][:, None])
    ds = p * (g[rows] @ v.T - dsum[rows][:, None])
    dq = scale * (ds @ k)
    # columns of P for dK, dV
    allr = np.arange(N)
    sc = scale * (q @ k[keys].T)                          # [N, len(keys)]
    if causal:
        sc = np.where(keys[None, :] > allr[:, None], -np.inf, sc)
    pc = np.exp(sc - lse[:, None])
    dpc = g @ v[keys].T
    dsc = pc * (dpc - dsum[:, None])
    dv = pc.T @ g
    dk = scale * (dsc.T @ q)
    return dq, dk, dv


def attention_backward_rows(q_head, k_head, v_head, do_head, scale: float, causal: bool, rows):
    """One row block's share of the backward of ONE head (the loop body of attention_backward).

    For the query rows ``rows``: returns (dQ[rows], dK_part, dV_part), where dK_part
    and dV_part are the contributions of those rows to dK and dV ([N, d] each);
    summing the parts over any partition of the rows gives attention_backward's
    dK and dV.
    """
    q, k, v, g = (_as_f64(t) for t in (q_head, k_head, v_head, do_head))
    rows = np.asarray(rows, dtype=np.int64)
    s = _scores(q[rows], k, rows, scale, causal)
    p, _, _ = _softmax_rows(s)
    gr = g[rows]
    dp = gr @ v.T
    ds = p * (dp - (p * dp).sum(axis=1, keepdims=True))
    return scale * (ds @ k), scale * (ds.T @ q[rows]), p.T @ gr
