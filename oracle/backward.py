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

fp8=True / "ue8m0": the fine-grained FP8 scheme of section 3.3 on all three
GEMMs of every expert linear layer -- the forward product, the data gradient
and the weight gradient (item 1) -- with E4M3 for every operand (item 4),
weights in 128 x 128 blocks and activations and gradients in 1 x 128 tiles
(item 2).  The pages do not say along which axis a gradient GEMM's tiles
run; here, as in the forward, an activation or gradient operand is
quantised along that GEMM's contraction axis (so one scale covers each
promoted 128-long K block, item 3):
  forward   x = Q_row(u) (along d), h' = Q_row(h) (along I), weights Q_blk(W);
  dgrad     dh = Q_row(dy) Q_blk(W2), dx = Q_row(da) Q_blk(W1) + Q_row(db) Q_blk(W3);
  wgrad     dW2 = Q_tok(dy)^T Q_tok(h), dW1 = Q_tok(da)^T Q_tok(u), dW3 = Q_tok(db)^T Q_tok(u),
where Q_tok quantises each column in blocks of 128 consecutive tokens of the
expert (token-ascending, the first block starting at the expert's first
token; a short last block is padded with zeros) and the wgrad operands are
the unquantised activations.  The quantisation is straight-through: the
gradient of Q(x) is taken as that of x.  The router (affinities, gates,
centroid gradient) stays in high precision (item 1).  Products of the
dequantised operands are exact (fp64).

The codes of the quantised intermediates (h before the down product, dy
and [da db] before the data-gradient products, and every weight-gradient
operand) are taken from x * (1/s), one correctly rounded fp32 reciprocal per
tile: these values are known only to the kernels' accuracy, and a product
costs the kernels far less than a division.  The codes of u in the forward
are taken from u / s, as in the forward's gather.

act_bf16=True: every intermediate the kernels keep in bf16 is rounded to
bf16 here too (a and b, h, y, dy, dh, da and db, dx, and the dequantised
weight-gradient operands), so that the floats that decide the E4M3 codes
are taken in the kernels' precision; without it the intermediates are fp64.
Rounding: to fp32, then to bf16, both round-to-nearest-even (round_bf16).
"""
from __future__ import annotations

import numpy as np

from . import bf16_to_f64, fp8_roundtrip_1x128, fp8_roundtrip_128x128


def _sigmoid(a):
    return 1.0 / (1.0 + np.exp(-a))


def round_bf16(x: np.ndarray) -> np.ndarray:
    """fp64 -> fp32 -> bf16 (round-to-nearest-even each time) -> fp64, for
    finite values: the bf16 value a kernel stores for an fp32 result."""
    b = np.ascontiguousarray(np.asarray(x, np.float64).astype(np.float32)).view(np.uint32).astype(np.uint64)
    b = (b + 0x7FFF + ((b >> 16) & 1)) & 0xFFFF0000
    return b.astype(np.uint32).view(np.float32).astype(np.float64)


def _identity(x):
    return x


def swiglu_backward(x, w1, w3, w2, dy, rb=_identity):
    """One SwiGLU expert y = W2 (SiLU(W1 x) * (W3 x)) on rows x [n, d]:
    returns (dx [n, d], dW1 [I, d], dW3 [I, d], dW2 [d, I], y [n, d]) for the
    output gradient dy [n, d].  With a = W1 x, b = W3 x, sg = sigmoid(a):
    h = a sg b, dh = dy W2, da = dh b sg (1 + a (1 - sg)), db = dh a sg.
    rb rounds the stored intermediates (identity, or round_bf16)."""
    a = rb(x @ w1.T)
    b = rb(x @ w3.T)
    sg = _sigmoid(a)
    h = rb(a * sg * b)
    y = rb(h @ w2.T)
    dy = rb(dy)
    dh = rb(dy @ w2)
    da = rb(dh * b * sg * (1.0 + a * (1.0 - sg)))
    db = rb(dh * a * sg)
    dx = rb(da @ w1 + db @ w3)
    return dx, da.T @ x, db.T @ x, dy.T @ h, y


def _q_tok(m: np.ndarray, pow2: bool) -> np.ndarray:
    """Q_tok: 1 x 128 tiles along the token axis (axis 0) of m [n, C], blocks of
    128 consecutive rows from row 0, a short last block padded with zeros."""
    n, C = m.shape
    n_pad = -(-n // 128) * 128
    t = np.zeros((C, n_pad))
    t[:, :n] = m.T
    return fp8_roundtrip_1x128(t, pow2, recip=True)[:, :n].T


def _expert_backward_fp8(x, w1, w3, w2, dy, pow2, rb=_identity):
    """swiglu_backward in the FP8 scheme (module docstring): x [n, d] the
    unquantised input rows, w* the unquantised weights, dy [n, d]."""
    q_row = lambda m: fp8_roundtrip_1x128(m, pow2, recip=True)
    w1q, w3q, w2q = (fp8_roundtrip_128x128(w, pow2) for w in (w1, w3, w2))
    xq = fp8_roundtrip_1x128(x, pow2)
    a = rb(xq @ w1q.T)
    b = rb(xq @ w3q.T)
    sg = _sigmoid(a)
    h = rb(a * sg * b)
    y = rb(q_row(h) @ w2q.T)
    dy = rb(dy)
    dh = rb(q_row(dy) @ w2q)
    da = rb(dh * b * sg * (1.0 + a * (1.0 - sg)))
    db = rb(dh * a * sg)
    dx = rb(q_row(da) @ w1q + q_row(db) @ w3q)
    ut = rb(_q_tok(x, pow2))
    dyt, ht, dat, dbt = (rb(_q_tok(m, pow2)) for m in (dy, h, da, db))
    return dx, dat.T @ ut, dbt.T @ ut, dyt.T @ ht, y


def layer_backward(u_bits, cent_bits, idx, G, routed_weights, shared_weights, n_shared: int, E: int,
                   fp8=False, act_bf16: bool = False, keep_dw=None) -> dict:
    """Gradients of the layer for dL/dh' = G [T, d], the selection idx [T, k]
    held fixed.  routed_weights(e) / shared_weights(s) return bf16 bit patterns
    (W1, W3, W2).  Returns dict(du [T, d], dcent [E, d], dw_routed {e: (dW1,
    dW3, dW2)} for every selected expert, dw_shared [(dW1, dW3, dW2)] per
    shared expert, gate [T, k], dgate [T, k]).  fp8: False, True (amax/448
    scales) or "ue8m0" (power-of-two scales): the FP8 scheme of the module
    docstring, whose forward is that of oracle.layer_output(fp8=...).
    act_bf16: the kernels' bf16 intermediates (module docstring).  keep_dw:
    the routed experts whose weight gradients dw_routed keeps (None: all; a
    V3-sized expert's three fp64 gradients take 350 MB)."""
    x = bf16_to_f64(u_bits)
    cent = bf16_to_f64(cent_bits)
    G = np.asarray(G, np.float64)
    T, d = x.shape
    k = idx.shape[1]
    idx = np.asarray(idx, np.int64)
    pow2 = fp8 == "ue8m0"
    rb = round_bf16 if act_bf16 else _identity

    def expert(xr, ws, dy):
        w1, w3, w2 = (bf16_to_f64(w) for w in ws)
        if fp8:
            return _expert_backward_fp8(xr, w1, w3, w2, dy, pow2, rb)
        return swiglu_backward(xr, w1, w3, w2, dy, rb)

    s_sel = _sigmoid(np.einsum("td,tjd->tj", x, cent[idx]))
    S = s_sel.sum(1, keepdims=True)
    gate = s_sel / S
    du = G.copy()                                    # the residual
    dw_shared = []
    for s in range(n_shared):
        dx, dw1, dw3, dw2, _ = expert(x, shared_weights(s), G)
        du += dx
        dw_shared.append((dw1, dw3, dw2))
    dgate = np.zeros((T, k))
    dw_routed = {}
    for e in range(E):
        rows, js = np.nonzero(idx == e)               # token-ascending
        if rows.size == 0:
            continue
        dy = gate[rows, js][:, None] * G[rows]
        dx, dw1, dw3, dw2, y = expert(x[rows], routed_weights(e), dy)
        np.add.at(du, rows, dx)
        dgate[rows, js] = (G[rows] * y).sum(1)
        if keep_dw is None or e in keep_dw:
            dw_routed[e] = (dw1, dw3, dw2)
    # g_j = s_j / S:  ds_j = (dg_j - sum_j' g_j' dg_j') / S;  s = sigmoid(z): dz = ds s (1 - s)
    ds = (dgate - (gate * dgate).sum(1, keepdims=True)) / S
    dz = ds * s_sel * (1.0 - s_sel)
    du += np.einsum("tj,tjd->td", dz, cent[idx])
    dcent = np.zeros((E, d))
    np.add.at(dcent, idx.ravel(), dz.ravel()[:, None] * np.repeat(x, k, axis=0))
    return dict(du=du, dcent=dcent, dw_routed=dw_routed, dw_shared=dw_shared, gate=gate, dgate=dgate)
