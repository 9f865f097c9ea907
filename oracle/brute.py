"""Dense brute force of the DeepSeekMoE layer -- TEST INFRASTRUCTURE ONLY.

A second, structurally different statement of the layer for tiny inputs, in
bf16-exact fp64 (dense_layer) and with the FP8 operands of the main GEMMs
(dense_layer_fp8):
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


def _silu_and_mul(xw1: np.ndarray, xw3: np.ndarray) -> np.ndarray:
    return _silu(xw1) * xw3


# ----------------------------------------------------------------------------
# FP8 statement of the layer (ai.flicky.cc "06 - DeepSeek-V3 reading",
# section 3.3 "FP8 training": the inputs of the main GEMMs are E4M3 with one
# scale per 1 x 128 activation tile and per 128 x 128 weight block; the router
# stays in high precision).  Written from the format and the scale rule alone:
# the values of the format come from enumerating its bit fields, rounding is a
# nearest-value search in that table, and the products are numpy fp64 matmuls
# of the dequantised operands -- the exact limit that the FP32 promotion every
# 128 elements of K approaches.  Shares no code with moe_oracle.c.
def _e4m3_sorted_positive():
    """The non-negative finite E4M3 values in code order (codes 0x00..0x7E),
    which is also ascending value order."""
    table = e4m3_value_table()
    codes = sorted(c for c, v in table.items() if c < 0x80)
    vals = np.array([table[c] for c in codes])
    assert codes == list(range(127)) and (np.diff(vals) > 0).all()
    return vals


_E4M3_POS = None


def e4m3_round(x: np.ndarray) -> np.ndarray:
    """Nearest finite E4M3 value of every element (ties to the even code,
    saturating at +-448), by a search in the enumerated value table."""
    global _E4M3_POS
    if _E4M3_POS is None:
        _E4M3_POS = _e4m3_sorted_positive()
    vals = _E4M3_POS
    x = np.asarray(x, np.float64)
    a = np.minimum(np.abs(x), vals[-1])
    hi = np.clip(np.searchsorted(vals, a, side="left"), 0, len(vals) - 1)
    lo = np.maximum(hi - 1, 0)
    d_lo, d_hi = a - vals[lo], vals[hi] - a
    pick = np.where(d_lo < d_hi, lo, np.where(d_hi < d_lo, hi, np.where(lo % 2 == 0, lo, hi)))
    return np.copysign(vals[pick], x)


def pow2_at_least(s: np.ndarray) -> np.ndarray:
    """The smallest power of two >= s, for positive fp32 s (numpy's frexp:
    s = m 2^e with m in [0.5, 1); s is a power of two exactly when m = 0.5)."""
    m, e = np.frexp(np.asarray(s, np.float32))
    return np.where(m == 0.5, s, np.ldexp(np.float32(1.0), e)).astype(np.float32)


def quant_dequant(x: np.ndarray, group_rows: int, group_cols: int, pow2: bool = False,
                  recip: bool = False) -> np.ndarray:
    """Quantise x [R, C] in groups of group_rows x group_cols elements and
    return the dequantised values: scale = amax / 448 in fp32 (1 for an
    all-zero group) -- rounded up to a power of two for UE8M0 scales (pow2) --,
    element = nearest E4M3 of (x / scale) taken in fp32 -- or, recip, of
    x * (1 / scale) with both operations in fp32 --, times scale."""
    x = np.asarray(x, np.float64)
    R, C = x.shape
    g = x.reshape(R // group_rows, group_rows, C // group_cols, group_cols)
    amax = np.abs(g).max(axis=(1, 3), keepdims=True)
    scale = np.where(amax > 0, amax.astype(np.float32) / np.float32(448.0), np.float32(1.0)).astype(np.float32)
    if pow2:
        scale = pow2_at_least(scale)
    if recip:
        ratio = (g.astype(np.float32) * (np.float32(1.0) / scale).astype(np.float32)).astype(np.float64)
    else:
        ratio = (g.astype(np.float32) / scale).astype(np.float64)
    return (e4m3_round(ratio) * scale.astype(np.float64)).reshape(R, C)


def dense_layer_fp8(u: np.ndarray, cent: np.ndarray, bias: np.ndarray, k: int, routed, shared,
                    pow2: bool = False) -> dict:
    """The layer of dense_layer with the FP8 operands of the main GEMMs
    (pow2: every scale a power of two, the UE8M0 scales of DeepSeek-V3.1).

    Routing (affinities, selection, gates) uses the unquantised u; every
    expert, shared or routed, multiplies the 1 x 128-quantised u by its
    128 x 128-quantised W1 and W3, quantises h per 1 x 128 tile along I and
    multiplies by its 128 x 128-quantised W2; the residual is u itself.
    """
    T, d = u.shape
    E = cent.shape[0]
    s = 1.0 / (1.0 + np.exp(-(u @ cent.T)))
    g = np.zeros((T, E))
    for t in range(T):
        order = sorted(range(E), key=lambda i: (-(s[t, i] + float(bias[i])), i))
        for i in order[:k]:
            g[t, i] = s[t, i]
        g[t] /= g[t].sum()
    xq = quant_dequant(u, 1, 128, pow2)

    def expert(w1, w3, w2):
        w1q, w3q, w2q = (quant_dequant(w, 128, 128, pow2) for w in (w1, w3, w2))
        h = _silu_and_mul(xq @ w1q.T, xq @ w3q.T)
        return quant_dequant(h, 1, 128, pow2) @ w2q.T

    out = u.copy()
    for ws in shared:
        out += expert(*ws)
    for i, ws in enumerate(routed):
        out += g[:, i:i + 1] * expert(*ws)      # every token through every expert, masked by g
    return dict(out=out, g=g)


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


def node_limited_topk(score: np.ndarray, k: int, groups: int, limit: int) -> list:
    """The k selected experts of one token when its experts may span at most
    `limit` of `groups` nodes (E/groups consecutive experts per node), written
    as: rank the nodes by their best expert (ties: the node of the lower expert
    index), keep the first `limit`, then take the k best experts on those nodes
    (ties: lower index).  Python sorts only."""
    E = len(score)
    gs = E // groups
    best = [max(range(n * gs, (n + 1) * gs), key=lambda i: (score[i], -i)) for n in range(groups)]
    nodes = sorted(range(groups), key=lambda n: (-score[best[n]], best[n]))[:limit]
    allowed = [i for i in range(E) if i // gs in nodes]
    return sorted(allowed, key=lambda i: (-score[i], i))[:k]
