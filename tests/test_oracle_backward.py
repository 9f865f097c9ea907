"""Pins of the backward oracle (oracle/backward.py, no GPU) against two
statements that share no code with it: a dense all-experts-then-mask forward
in float64 torch differentiated by autograd, and central finite differences of
a dense numpy forward.  The selection is held fixed (the gradient flows through
the gate values, not the top-k choice), and the bias gets no gradient."""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
import synth
from oracle import backward as ob


def _setup(name, seed=7):
    cfg = synth.get_config(name)
    u, c = synth.tokens(cfg), synth.centroids(cfg)
    b = np.asarray(synth.normal_f32(4245, (cfg.E,), 0.02))
    routed = [synth.expert_weights(cfg, e) for e in range(cfg.E)]
    shared = [synth.expert_weights(cfg, s, shared=True) for s in range(cfg.n_shared)]
    r = oracle.route(synth.bf16_bits(u), synth.bf16_bits(c), b, cfg.k)
    G = np.random.default_rng(seed).standard_normal((cfg.T, cfg.d))
    bits = lambda ws: tuple(synth.bf16_bits(w) for w in ws)
    res = ob.layer_backward(synth.bf16_bits(u), synth.bf16_bits(c), r["idx"], G, lambda e: bits(routed[e]),
                            lambda s: bits(shared[s]), cfg.n_shared, cfg.E)
    return cfg, u, c, routed, shared, r["idx"], G, res


def _dense_torch(u, c, routed, shared, mask):
    """h' with every token through every expert, routed outputs masked by the
    fixed selection's normalised gates (float64 torch)."""
    s = torch.sigmoid(u @ c.T) * mask
    g = s / s.sum(1, keepdim=True)
    out = u
    for w1, w3, w2 in shared:
        out = out + (F.silu(u @ w1.T) * (u @ w3.T)) @ w2.T
    for i, (w1, w3, w2) in enumerate(routed):
        out = out + g[:, i:i + 1] * ((F.silu(u @ w1.T) * (u @ w3.T)) @ w2.T)
    return out


@pytest.mark.parametrize("name", ["tiny", "ragged"])
def test_backward_equals_autograd_of_dense_statement(name):
    cfg, u, c, routed, shared, idx, G, res = _setup(name)
    ut = u.double().requires_grad_()
    ct = c.double().requires_grad_()
    rt = [tuple(w.double().requires_grad_() for w in ws) for ws in routed]
    st = [tuple(w.double().requires_grad_() for w in ws) for ws in shared]
    mask = torch.zeros((cfg.T, cfg.E), dtype=torch.float64)
    mask[torch.arange(cfg.T)[:, None], torch.from_numpy(idx.astype(np.int64))] = 1.0
    out = _dense_torch(ut, ct, rt, st, mask)
    (out * torch.from_numpy(G)).sum().backward()
    tol = lambda ref: 1e-10 * max(1.0, float(np.abs(ref).max()))
    np.testing.assert_allclose(res["du"], ut.grad.numpy(), rtol=0, atol=tol(ut.grad.numpy()))
    np.testing.assert_allclose(res["dcent"], ct.grad.numpy(), rtol=0, atol=tol(ct.grad.numpy()))
    for e in range(cfg.E):
        grads = [w.grad.numpy() for w in rt[e]]
        if e in res["dw_routed"]:
            for got, ref in zip(res["dw_routed"][e], grads):
                np.testing.assert_allclose(got, ref, rtol=0, atol=tol(ref))
        else:                                   # an expert no token chose gets no gradient
            assert all(np.abs(g).max() == 0 for g in grads)
    for s in range(cfg.n_shared):
        for got, w in zip(res["dw_shared"][s], st[s]):
            np.testing.assert_allclose(got, w.grad.numpy(), rtol=0, atol=tol(w.grad.numpy()))


def _dense_numpy(u, c, routed, shared, idx):
    """The same layer in plain numpy fp64 with the selection fixed."""
    silu = lambda a: a / (1.0 + np.exp(-a))
    T = u.shape[0]
    s = 1.0 / (1.0 + np.exp(-np.einsum("td,tjd->tj", u, c[idx])))
    g = s / s.sum(1, keepdims=True)
    out = u.copy()
    for w1, w3, w2 in shared:
        out += (silu(u @ w1.T) * (u @ w3.T)) @ w2.T
    for t in range(T):
        for j, e in enumerate(idx[t]):
            w1, w3, w2 = routed[e]
            out[t] += g[t, j] * ((silu(u[t] @ w1.T) * (u[t] @ w3.T)) @ w2.T)
    return out


def test_backward_matches_central_differences():
    cfg, u, c, routed, shared, idx, G, res = _setup("tiny", seed=8)
    un, cn = u.double().numpy(), c.double().numpy()
    rn = [[w.double().numpy() for w in ws] for ws in routed]
    sn = [[w.double().numpy() for w in ws] for ws in shared]
    loss = lambda uu, cc, rr, ss: float((_dense_numpy(uu, cc, rr, ss, idx) * G).sum())
    rng = np.random.default_rng(9)
    eps = 1e-5
    e_used = sorted(res["dw_routed"])[0]
    checks = {
        "u": (lambda v: (un + eps * v, cn, rn, sn), lambda v: (un - eps * v, cn, rn, sn), un.shape, res["du"]),
        "centroids": (lambda v: (un, cn + eps * v, rn, sn), lambda v: (un, cn - eps * v, rn, sn), cn.shape,
                      res["dcent"]),
    }
    for m, name in ((0, "W1"), (1, "W3"), (2, "W2")):
        def plus(v, m=m):
            r2 = [list(ws) for ws in rn]
            r2[e_used][m] = rn[e_used][m] + eps * v
            return un, cn, r2, sn

        def minus(v, m=m):
            r2 = [list(ws) for ws in rn]
            r2[e_used][m] = rn[e_used][m] - eps * v
            return un, cn, r2, sn
        checks[f"routed {name}"] = (plus, minus, rn[e_used][m].shape, res["dw_routed"][e_used][m])

    def splus(v):
        return un, cn, rn, [[sn[0][0], sn[0][1], sn[0][2] + eps * v]]

    def sminus(v):
        return un, cn, rn, [[sn[0][0], sn[0][1], sn[0][2] - eps * v]]
    checks["shared W2"] = (splus, sminus, sn[0][2].shape, res["dw_shared"][0][2])
    for what, (plus, minus, shape, grad) in checks.items():
        v = rng.standard_normal(shape)
        fd = (loss(*plus(v)) - loss(*minus(v))) / (2 * eps)
        an = float((grad * v).sum())
        assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (what, fd, an)
