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


# ----------------------------------------------------------------------------
# The FP8 backward (ai.flicky.cc 3.3: forward, data-gradient and weight-gradient
# GEMMs in FP8, E4M3 everywhere, 1 x 128 activation tiles and 128 x 128 weight
# blocks, tiles along each GEMM's contraction axis).  The independent
# statement: torch autograd over the same layer, with every expert linear
# layer an autograd Function that quantises its operands (brute.quant_dequant,
# which shares no code with the oracle's C quantiser) and the rest (SwiGLU,
# gates, router, residual) differentiated by autograd itself.
from oracle import brute  # noqa: E402


def _q_row(m, pow2, recip=True):
    return brute.quant_dequant(m, 1, 128, pow2, recip)


def _q_tok(m, pow2):
    n, C = m.shape
    n_pad = -(-n // 128) * 128
    pad = np.zeros((n_pad, C))
    pad[:n] = m
    return brute.quant_dequant(pad, 128, 1, pow2, recip=True)[:n]


def _bf16_round(t):
    """torch's own fp64 -> fp32 -> bf16 rounding (the kernels' stored values)."""
    return t.float().to(torch.bfloat16).double()


class _RoundBoth(torch.autograd.Function):
    """A value the kernels store as bf16, and whose gradient they store as
    bf16 too: rounds in the forward and in the backward."""

    @staticmethod
    def forward(ctx, x):
        return _bf16_round(x)

    @staticmethod
    def backward(ctx, g):
        return _bf16_round(g)


def _fp8_linear(pow2, act_bf16=False, input_recip=True):
    """input_recip: the input's codes from x * (1/s) (an intermediate such as
    h), else from x / s (the layer input u)."""
    rnd = (lambda a: _bf16_round(torch.from_numpy(a)).numpy()) if act_bf16 else (lambda a: a)

    class Fp8Linear(torch.autograd.Function):
        """y = Q_row(x) Q_blk(W)^T; dx = Q_row(dy) Q_blk(W); dW = Q_tok(dy)^T Q_tok(x)
        (act_bf16: dx and the dequantised Q_tok operands rounded to bf16)."""

        @staticmethod
        def forward(ctx, x, w):
            ctx.save_for_backward(x, w)
            xn, wn = x.detach().numpy(), w.detach().numpy()
            return torch.from_numpy(_q_row(xn, pow2, input_recip) @ brute.quant_dequant(wn, 128, 128, pow2).T)

        @staticmethod
        def backward(ctx, gy):
            x, w = ctx.saved_tensors
            xn, wn, gn = x.numpy(), w.numpy(), gy.numpy()
            dx = rnd(_q_row(gn, pow2) @ brute.quant_dequant(wn, 128, 128, pow2))
            dw = rnd(_q_tok(gn, pow2)).T @ rnd(_q_tok(xn, pow2))
            return torch.from_numpy(dx), torch.from_numpy(dw)

    return Fp8Linear.apply


def _dense_fp8_grads(cfg, u, c, routed, shared, idx, G, pow2, act_bf16=False):
    """act_bf16: the kernels' bf16 intermediates -- [a b] and y rounded both
    ways (so da, db and dy are too), h in the forward; the linear layers
    round their data gradients (dh, dx) and weight-gradient operands."""
    lin_u = _fp8_linear(pow2, act_bf16, input_recip=False)   # gate/up: input u
    lin = _fp8_linear(pow2, act_bf16)                        # down: input h
    rb = _RoundBoth.apply if act_bf16 else (lambda t: t)
    rf = _bf16_round if act_bf16 else (lambda t: t)
    ut = u.double().requires_grad_()
    ct = c.double().requires_grad_()
    rt = [tuple(w.double().requires_grad_() for w in ws) for ws in routed]
    st = [tuple(w.double().requires_grad_() for w in ws) for ws in shared]

    def ffn(x, ws):
        w1, w3, w2 = ws
        ab = rb(lin_u(x, torch.cat([w1, w3])))        # gate and up: one GEMM, one bf16 output
        a, b = ab[:, :w1.shape[0]], ab[:, w1.shape[0]:]
        h = F.silu(a) * b
        h = h + (rf(h) - h).detach()                   # stored as bf16; its gradient is dh
        return rb(lin(h, w2))

    mask = torch.zeros((cfg.T, cfg.E), dtype=torch.float64)
    mask[torch.arange(cfg.T)[:, None], torch.from_numpy(idx.astype(np.int64))] = 1.0
    s = torch.sigmoid(ut @ ct.T) * mask
    g = s / s.sum(1, keepdim=True)
    out = ut
    for ws in st:
        out = out + ffn(ut, ws)
    for e in range(cfg.E):
        rows = torch.from_numpy(np.nonzero((idx == e).any(1))[0])   # token-ascending
        if rows.numel() == 0:
            continue
        out = out.index_add(0, rows, g[rows, e:e + 1] * ffn(ut[rows], rt[e]))
    (out * torch.from_numpy(G)).sum().backward()
    return ut.grad.numpy(), ct.grad.numpy(), [[w.grad for w in ws] for ws in rt], [[w.grad.numpy() for w in ws]
                                                                                       for ws in st]


def test_round_bf16_is_torch_rounding():
    """The oracle's bf16 rounding against torch's (fp64 -> fp32 -> bf16), on
    random values, exact halfway cases and values at the fp32 boundary."""
    rng = np.random.default_rng(5)
    x = np.concatenate([rng.standard_normal(20000) * 10.0 ** rng.integers(-8, 8, 20000),
                        (1.0 + np.arange(1, 256) / 256.0 + 2.0 ** -9) * 2.0 ** rng.integers(-20, 20, 255)])
    ref = torch.from_numpy(x).float().to(torch.bfloat16).double().numpy()
    np.testing.assert_array_equal(ob.round_bf16(x), ref)


def _fp8_setup(name, fp8, act_bf16=False):
    cfg = synth.get_config(name)
    u, c = synth.tokens(cfg), synth.centroids(cfg)
    b = np.asarray(synth.normal_f32(4245, (cfg.E,), 0.02))
    routed = [synth.expert_weights(cfg, e) for e in range(cfg.E)]
    shared = [synth.expert_weights(cfg, s, shared=True) for s in range(cfg.n_shared)]
    idx = oracle.route(synth.bf16_bits(u), synth.bf16_bits(c), b, cfg.k)["idx"]
    G = np.random.default_rng(11).standard_normal((cfg.T, cfg.d))
    bits = lambda ws: tuple(synth.bf16_bits(w) for w in ws)
    run = lambda: ob.layer_backward(synth.bf16_bits(u), synth.bf16_bits(c), idx, G, lambda e: bits(routed[e]),
                                    lambda s: bits(shared[s]), cfg.n_shared, cfg.E, fp8=fp8, act_bf16=act_bf16)
    return cfg, u, c, routed, shared, idx, G, run


def _max_rel(got, ref):
    return float(np.abs(got - ref).max() / max(np.abs(ref).max(), 1e-300))


def _compare_fp8(res, ref, cfg):
    du, dc, dr, dsh = ref
    errs = [_max_rel(res["du"], du), _max_rel(res["dcent"], dc)]
    for e in range(cfg.E):
        if e in res["dw_routed"]:
            errs += [_max_rel(got, w.numpy()) for got, w in zip(res["dw_routed"][e], dr[e])]
        else:
            assert all(w is None or float(w.abs().max()) == 0 for w in dr[e])
    for s in range(cfg.n_shared):
        errs += [_max_rel(got, w) for got, w in zip(res["dw_shared"][s], dsh[s])]
    return max(errs)


@pytest.mark.parametrize("name,fp8", [("tiny", True), ("ragged", True), ("tiny", "ue8m0"), ("ragged", "ue8m0")])
def test_fp8_backward_equals_autograd_with_fp8_linear_layers(name, fp8):
    cfg, u, c, routed, shared, idx, G, run = _fp8_setup(name, fp8)
    ref = _dense_fp8_grads(cfg, u, c, routed, shared, idx, G, fp8 == "ue8m0")
    assert _compare_fp8(run(), ref, cfg) <= 1e-10


@pytest.mark.parametrize("name,fp8", [("tiny", True), ("ragged", True), ("ragged", "ue8m0")])
def test_fp8_backward_with_bf16_intermediates_equals_autograd(name, fp8):
    """act_bf16: the same agreement with the bf16 roundings placed, in the
    autograd statement, on the values the kernels store."""
    cfg, u, c, routed, shared, idx, G, run = _fp8_setup(name, fp8, act_bf16=True)
    ref = _dense_fp8_grads(cfg, u, c, routed, shared, idx, G, fp8 == "ue8m0", act_bf16=True)
    assert _compare_fp8(run(), ref, cfg) <= 1e-10


def test_bf16_backward_with_bf16_intermediates_near_exact():
    """The bf16 backward with rounded intermediates stays within the bf16
    rounding of the exact one (a few 2^-9 in norm) and is not equal to it."""
    cfg, u, c, routed, shared, idx, G, res = _setup("ragged")
    bits = lambda ws: tuple(synth.bf16_bits(w) for w in ws)
    r = ob.layer_backward(synth.bf16_bits(u), synth.bf16_bits(c), idx, G, lambda e: bits(routed[e]),
                          lambda s: bits(shared[s]), cfg.n_shared, cfg.E, act_bf16=True)
    for key in ("du", "dcent"):
        err = float(np.linalg.norm(r[key] - res[key]) / np.linalg.norm(res[key]))
        assert 1e-5 < err < 2e-2, (key, err)


def test_fp8_backward_differs_from_bf16_by_the_quantisation():
    """The FP8 gradients are the bf16 ones up to E4M3's relative step (2^-4 per
    operand, a few operands per product): close, but not equal."""
    cfg, u, c, routed, shared, idx, G, run = _fp8_setup("ragged", True)
    f = run()
    ref = ob.layer_backward(synth.bf16_bits(u), synth.bf16_bits(c), idx, G,
                            lambda e: tuple(synth.bf16_bits(w) for w in routed[e]),
                            lambda s: tuple(synth.bf16_bits(w) for w in shared[s]), cfg.n_shared, cfg.E)
    for key in ("du", "dcent"):
        err = _max_rel(f[key], ref[key])
        assert 1e-4 < err < 0.2, (key, err)


@pytest.mark.parametrize("slip", ["wgrad_unquantised", "wgrad_tiles_along_features", "weights_unquantised"])
def test_fp8_backward_statement_catches_planted_slips(monkeypatch, slip):
    """Slips planted in the oracle's FP8 backward move it far from the autograd
    statement, so the agreement above is not vacuous."""
    cfg, u, c, routed, shared, idx, G, run = _fp8_setup("ragged", True)
    ref = _dense_fp8_grads(cfg, u, c, routed, shared, idx, G, False)
    if slip == "wgrad_unquantised":
        monkeypatch.setattr(ob, "_q_tok", lambda m, pow2: m)
    elif slip == "wgrad_tiles_along_features":
        monkeypatch.setattr(ob, "_q_tok", lambda m, pow2: oracle.fp8_roundtrip_1x128(m, pow2))
    else:
        monkeypatch.setattr(ob, "fp8_roundtrip_128x128", lambda w, pow2=False: w)
    assert _compare_fp8(run(), ref, cfg) > 1e-4


def test_one_expert_top1_is_the_gradient_of_a_dense_swiglu():
    """E = 1, k = 1, no shared expert: the layer is h' = u + W2 (SiLU(W1 u) * W3 u)
    (the single gate is s / s = 1), so its backward is autograd of that plain
    expression (torch F.silu), and the centroid gets exactly no gradient."""
    from dataclasses import replace
    cfg = replace(synth.get_config("tiny"), E=1, k=1, n_shared=0)
    u, c = synth.tokens(cfg), synth.centroids(cfg)
    w1, w3, w2 = synth.expert_weights(cfg, 0)
    idx = np.zeros((cfg.T, 1), np.int32)
    G = np.random.default_rng(11).standard_normal((cfg.T, cfg.d))
    bits = lambda ws: tuple(synth.bf16_bits(w) for w in ws)
    res = ob.layer_backward(synth.bf16_bits(u), synth.bf16_bits(c), idx, G, lambda e: bits((w1, w3, w2)),
                            lambda s: (), 0, 1)
    ut = u.double().requires_grad_()
    wt = [w.double().requires_grad_() for w in (w1, w3, w2)]
    out = ut + (F.silu(ut @ wt[0].T) * (ut @ wt[1].T)) @ wt[2].T
    (out * torch.from_numpy(G)).sum().backward()
    tol = lambda ref: 1e-10 * max(1.0, float(np.abs(ref).max()))
    np.testing.assert_allclose(res["du"], ut.grad.numpy(), rtol=0, atol=tol(ut.grad.numpy()))
    for got, w in zip(res["dw_routed"][0], wt):
        np.testing.assert_allclose(got, w.grad.numpy(), rtol=0, atol=tol(w.grad.numpy()))
    assert not np.any(res["dcent"])


def test_backward_of_an_empty_batch_is_zero():
    cfg = synth.get_config("tiny")
    c = synth.centroids(cfg)
    bits = lambda ws: tuple(synth.bf16_bits(w) for w in ws)
    res = ob.layer_backward(np.zeros((0, cfg.d), np.uint16), synth.bf16_bits(c), np.zeros((0, cfg.k), np.int32),
                            np.zeros((0, cfg.d)), lambda e: bits(synth.expert_weights(cfg, e)),
                            lambda s: bits(synth.expert_weights(cfg, s, shared=True)), cfg.n_shared, cfg.E)
    assert res["du"].shape == (0, cfg.d) and not np.any(res["dcent"])
    assert not res["dw_routed"]
    assert all(not np.any(g) for ws in res["dw_shared"] for g in ws)
