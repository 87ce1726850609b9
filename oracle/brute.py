"""Scalar triple-loop attention for tiny inputs (test infrastructure).

The same definition as ``oracle.attention`` ("FlashAttention-2 (DE)", section
"Hintergrund: Das Attention-Problem in Transformern"), written with Python
floats and ``math.exp`` one score at a time, so that the vectorised oracle can be
checked against code that shares none of its numpy expressions.  Use only for
N <= 32 and d <= 16: it is O(B*H*N^2*d) Python operations.
"""

from __future__ import annotations

import math


def attention_forward_brute(q, k, v, scale: float, causal: bool):
    """q, k, v: nested lists (or arrays) [B][H][N][d].  Returns (O, LSE) as nested lists."""
    B, H = len(q), len(q[0])
    out, lse = [], []
    for b in range(B):
        ob, lb = [], []
        for h in range(H):
            Q, K, V = q[b][h], k[b][h], v[b][h]
            N, dv = len(Q), len(V[0])
            oh, lh = [], []
            for i in range(N):
                scores = []
                for j in range(N):
                    if causal and j > i:
                        continue
                    acc = 0.0
                    for c in range(len(Q[i])):
                        acc += float(Q[i][c]) * float(K[j][c])
                    scores.append((j, scale * acc))
                mx = max(sc for _, sc in scores)
                weights = [(j, math.exp(sc - mx)) for j, sc in scores]
                total = sum(w for _, w in weights)
                row = []
                for c in range(dv):
                    row.append(sum(w * float(V[j][c]) for j, w in weights) / total)
                oh.append(row)
                lh.append(mx + math.log(total))
            ob.append(oh)
            lb.append(lh)
        out.append(ob)
        lse.append(lb)
    return out, lse
