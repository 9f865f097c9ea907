"""Backward pass of the DeepSeekMoE layer in fp64 -- TEST INFRASTRUCTURE ONLY.

Only the test suite and the bench's CPU leg use this module; it shares no code
with the CUDA library.  It differentiates the layer of ai.flicky.cc "06 -
DeepSeek-V3 reading" section 2.1.2 (and xyznot.com "DeepSeek-V3 technical
report", Method 2):

  h'_t    = u_t + sum_s FFN_s(u_t) + sum_j g_{t,j} FFN_{e_j}(u_t)
  g_{t,j} = s_{t,e_j} / sum_j' s_{t,e_j'},   s_{t,i} = sigmoid(u_t . c_i)
  FFN(x)  = W2 (SiLU(W1 x) * (W3 x))

given dL/dh' = G.  Readings where the pages are silent:
  * the selection {e_j} is held fixed (it is a discrete choice; the gradient
    flows through the gate values only -- "straight through" the top-k);
  * the bias b never receives a gradient: it enters the selection only, and
    the pages update it by the sign rule, not by gradient descent (section
    2.1.2, and its quiz question 4);
  * weight gradients are kept in high precision (section 3.3, item 1: master
    weights and weight gradients are stored in higher precision).
Matrix products are numpy fp64 matmuls, expert by expert.
"""
from __future__ import annotations

import numpy as np

from . import bf16_to_f64


def _sigmoid(a):
    return 1.0 / (1.0 + np.exp(-a))


def swiglu_backward(x, w1, w3, w2, dy):
    """One SwiGLU expert y = W2 (SiLU(W1 x) * (W3 x)) on rows x [n, d]:
    returns (dx [n, d], dW1 [I, d], dW3 [I, d], dW2 [d, I], y [n, d]) for the
    output gradient dy [n, d].  With a = W1 x, b = W3 x, sg = sigmoid(a):
    h = a sg b, dh = dy W2, da = dh b sg (1 + a (1 - sg)), db = dh a sg."""
    a = x @ w1.T
    b = x @ w3.T
    sg = _sigmoid(a)
    h = a * sg * b
    y = h @ w2.T
    dh = dy @ w2
    da = dh * b * sg * (1.0 + a * (1.0 - sg))
    db = dh * a * sg
    dx = da @ w1 + db @ w3
    return dx, da.T @ x, db.T @ x, dy.T @ h, y


def layer_backward(u_bits, cent_bits, idx, G, routed_weights, shared_weights, n_shared: int, E: int) -> dict:
    """Gradients of the layer for dL/dh' = G [T, d], the selection idx [T, k]
    held fixed.  routed_weights(e) / shared_weights(s) return bf16 bit patterns
    (W1, W3, W2).  Returns dict(du [T, d], dcent [E, d], dw_routed {e: (dW1,
    dW3, dW2)} for every selected expert, dw_shared [(dW1, dW3, dW2)] per
    shared expert, gate [T, k], dgate [T, k])."""
    x = bf16_to_f64(u_bits)
    cent = bf16_to_f64(cent_bits)
    G = np.asarray(G, np.float64)
    T, d = x.shape
    k = idx.shape[1]
    idx = np.asarray(idx, np.int64)
    s_sel = _sigmoid(np.einsum("td,tjd->tj", x, cent[idx]))
    S = s_sel.sum(1, keepdims=True)
    gate = s_sel / S
    du = G.copy()                                    # the residual
    dw_shared = []
    for s in range(n_shared):
        w1, w3, w2 = (bf16_to_f64(w) for w in shared_weights(s))
        dx, dw1, dw3, dw2, _ = swiglu_backward(x, w1, w3, w2, G)
        du += dx
        dw_shared.append((dw1, dw3, dw2))
    dgate = np.zeros((T, k))
    dw_routed = {}
    for e in range(E):
        rows, js = np.nonzero(idx == e)
        if rows.size == 0:
            continue
        w1, w3, w2 = (bf16_to_f64(w) for w in routed_weights(e))
        dy = gate[rows, js][:, None] * G[rows]
        dx, dw1, dw3, dw2, y = swiglu_backward(x[rows], w1, w3, w2, dy)
        np.add.at(du, rows, dx)
        dgate[rows, js] = (G[rows] * y).sum(1)
        dw_routed[e] = (dw1, dw3, dw2)
    # g_j = s_j / S:  ds_j = (dg_j - sum_j' g_j' dg_j') / S;  s = sigmoid(z): dz = ds s (1 - s)
    ds = (dgate - (gate * dgate).sum(1, keepdims=True)) / S
    dz = ds * s_sel * (1.0 - s_sel)
    du += np.einsum("tj,tjd->td", dz, cent[idx])
    dcent = np.zeros((E, d))
    np.add.at(dcent, idx.ravel(), dz.ravel()[:, None] * np.repeat(x, k, axis=0))
    return dict(du=du, dcent=dcent, dw_routed=dw_routed, dw_shared=dw_shared, gate=gate, dgate=dgate)
