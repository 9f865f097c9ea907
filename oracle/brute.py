"""Dense brute force of the DeepSeekMoE layer -- TEST INFRASTRUCTURE ONLY.

A second, structurally different statement of the layer for tiny inputs:
every token runs through EVERY expert, and the routed outputs are then masked
by g'_{i,t} (zero for unselected experts) and normalised -- the equations of
ai.flicky.cc "06 - DeepSeek-V3 reading" section 2.1.2 and xyznot.com
"DeepSeek-V3 technical report" Method 2, taken literally:

  h'_t = u_t + sum_{i<=N_s} FFN^(s)_i(u_t) + sum_{i<=N_r} g_{i,t} FFN^(r)_i(u_t)
  s_{i,t} = sigmoid(u_t^T e_i)
  g'_{i,t} = s_{i,t} if s_{i,t} + b_i is among the K_r largest, else 0
  g_{i,t} = g'_{i,t} / sum_j g'_{j,t}

The selection uses Python's sorted() on (-score, index) -- a library sort
instead of the C oracle's repeated arg-max -- and the matrix products are
numpy fp64 matmuls.  Shares no code with moe_oracle.c.
"""
from __future__ import annotations

import math

import numpy as np


def _silu(a: np.ndarray) -> np.ndarray:
    return a / (1.0 + np.exp(-a))


def dense_layer(u: np.ndarray, cent: np.ndarray, bias: np.ndarray, k: int, routed, shared) -> dict:
    """u [T,d], cent [E,d] fp64; bias [E]; routed/shared: lists of (W1, W3, W2) fp64.

    Returns dict(out [T,d], g [T,E] dense normalised gates, sel list of sets).
    """
    T, d = u.shape
    E = cent.shape[0]
    logits = u @ cent.T
    s = 1.0 / (1.0 + np.exp(-logits))
    g = np.zeros((T, E))
    sel = []
    for t in range(T):
        order = sorted(range(E), key=lambda i: (-(s[t, i] + float(bias[i])), i))
        chosen = set(order[:k])
        sel.append(chosen)
        for i in chosen:
            g[t, i] = s[t, i]
        g[t] /= g[t].sum()
    out = u.copy()
    for (w1, w3, w2) in shared:
        out += (_silu(u @ w1.T) * (u @ w3.T)) @ w2.T
    for i, (w1, w3, w2) in enumerate(routed):
        y = (_silu(u @ w1.T) * (u @ w3.T)) @ w2.T    # every token, every expert
        out += g[:, i:i + 1] * y                    # masked by g (zero where unselected)
    return dict(out=out, g=g, sel=sel, s=s)


def e4m3_value_table() -> dict:
    """All finite E4M3 values by enumeration of sign, exponent and mantissa (pure Python).

    Format: 1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits; field
    exponent 0 is subnormal (m/8 * 2^-6); S.1111.111 is NaN; no infinities.
    """
    table = {}
    for code in range(256):
        sgn, e, m = code >> 7, (code >> 3) & 15, code & 7
        if e == 15 and m == 7:
            continue
        mag = (m / 8.0) * 2.0 ** -6 if e == 0 else (1.0 + m / 8.0) * 2.0 ** (e - 7)
        table[code] = -mag if sgn else mag
    return table


def nearest_e4m3(x: float) -> float:
    """Nearest finite E4M3 value to x by exhaustive search; ties to the even code; saturating."""
    if math.isnan(x):
        return float("nan")
    a = min(abs(x), 448.0)
    best = None
    for code, v in e4m3_value_table().items():
        if v < 0 or (v == 0 and code != 0):
            continue
        dist = abs(v - a)
        if best is None or dist < best[0] or (dist == best[0] and (code & 1) == 0):
            best = (dist, code, v)
    return math.copysign(best[2], x)
