"""The backward pass on the GPU (moe_backward, bf16 and FP8) against the
backward oracle (oracle/backward.py, pinned to autograd statements and finite
differences), with the GPU's own selection held fixed on both sides.

Two oracle references per case:

1. The kernels' precision (act_bf16=True): the oracle rounds to bf16 every
   intermediate the kernels keep in bf16 (a, b, h, y, dy, dh, da/db, dx and
   the dequantised weight-gradient operands), so that every E4M3 code is
   decided from the same value on both sides.  What is left is the order of
   the fp32 sums against fp64 (~1e-6 relative), which moves a bf16 rounding
   in about one value in 4000 by one step (2^-8 of that value).  du sums k + 1
   bf16 dx rows whose elements reach a few times rms(du), so a moved rounding
   there is up to ~1.5e-2 of rms(du): data gradients max|err| / rms(ref) <=
   2e-2; weight gradients (fp32 sums of many such values, compared in norm)
   relative Frobenius norm <= 5e-3.  One exception, bf16 only: the kernels
   take the gates' gradient G . y as (dh . h) / g (equal in exact arithmetic,
   dh = g G W2), so it carries the bf16 roundings of dy, dh and h (three
   2^-9 steps) where the oracle's carries y's (one).  That ~2e-3 relative
   error of dg passes through the gates' Jacobian into dz, and dcentroids sums
   dz u over an expert's tokens, which point in similar directions (clustered
   tokens) while dz changes sign, so the sum cancels and its relative error
   grows several-fold: dcentroids <= 4e-2 there.
2. The exact arithmetic (fp64 intermediates).  bf16: every intermediate
   rounded to 8 significant bits (2^-9 relative), a gradient through up to
   four such roundings: data gradients max|err| / rms <= 5e-2 (a few roundings
   at the largest elements, max/rms ~ 5), weight gradients Frobenius <= 2e-2
   (their heavy-tailed elements make max/rms measure the tail).  FP8: on top
   of that, where a bf16 intermediate lies within its rounding of a midpoint
   between two E4M3 values its code differs from the exact one by a step
   (2^-3 to 2^-4 of the element): a few percent of the codes, in up to three
   quantised operands in series, about 2% rms each in a K-long product:
   data gradients max|err| / rms <= 1.5e-1, weight gradients Frobenius <= 5e-2.
   bf16 dcentroids carry both error sources, the (dh . h) / g form of the
   gates' gradient (4e-2, above) and the bf16 roundings of the intermediates
   (5e-2), so their exact bound is the sum, 9e-2.  With few tokens the second
   one alone reaches the 5e-2: an expert's row sums dz u over one or two
   tokens, so the cancellation in dz is not averaged out (the oracle in the
   kernels' precision is 2.2e-2 / 4.7e-2 / 3.1e-2 from the exact one at 1 / 2 /
   4 tokens of the tiny shape, 1.5e-2 at 64).

And the weight-gradient arithmetic itself: dW2 of the first experts against
the same product replayed from bf16-rounded a, b, h and dy (fp64; FP8: the
operands quantised along the tokens, each dequantised value rounded to bf16):
relative Frobenius norm <= 1e-3 (the GPU accumulates in fp32)."""
import numpy as np
import pytest
import torch

import oracle
import synth
from mixture_experts_layer_87_b300 import capi
from oracle import backward as ob
from parity import HostLayer, rel_err

pytestmark = pytest.mark.gpu
DEV = "cuda"
KP_TOL = 2e-2       # against the kernels' precision: data gradients, max|err| / rms(ref)
KP_DCENT_BF16 = 4e-2  # ... dcentroids of the bf16 path (the gates' gradient from dh . h, see above)
KP_WG_TOL = 5e-3    # against the kernels' precision: weight gradients, relative Frobenius norm
EXACT_TOL = {False: (5e-2, 2e-2), True: (1.5e-1, 5e-2)}   # against fp64 intermediates, bf16 / FP8
EXACT_DCENT_BF16 = KP_DCENT_BF16 + EXACT_TOL[False][0]   # ... dcentroids of the bf16 path: both sources add
REPLAY_TOL = 1e-3   # dW2 against the bf16-operand replay, relative Frobenius norm


def fro_err(got, ref):
    return float(np.linalg.norm(got - ref) / np.linalg.norm(ref))


def _bf16(a):
    return torch.from_numpy(np.asarray(a, np.float64)).float().to(torch.bfloat16).double().numpy()


def _interleave13(dw1, dw3, I, d):
    # w13 interleave: rows [256j, 256j+128) of W1 block j, [256j+128, 256j+256) of W3 block j
    return np.stack([dw1.reshape(I // 128, 128, d), dw3.reshape(I // 128, 128, d)], 1).reshape(2 * I, d)


def _errors(got, ref, cfg):
    errs = {"du": rel_err(got["du"], ref["du"])}
    if np.any(ref["dcent"]):
        errs["dcentroids"] = rel_err(got["dcentroids"], ref["dcent"])
    else:  # k = 1: every gate is s / s = 1, a constant, so the centroids get no gradient
        errs["dcentroids"] = float(np.abs(got["dcentroids"]).max() / np.sqrt((ref["du"] ** 2).mean()))
    werr = {}
    for e, (dw1, dw3, dw2) in ref["dw_routed"].items():
        werr[f"dw13[{e}]"] = fro_err(got["dw13"][e], _interleave13(dw1, dw3, cfg.inter, cfg.d))
        werr[f"dw2[{e}]"] = fro_err(got["dw2"][e], dw2)
    for s, (dw1, dw3, dw2) in enumerate(ref["dw_shared"]):
        werr[f"dws13[{s}]"] = fro_err(got["dws13"][s], _interleave13(dw1, dw3, cfg.inter, cfg.d))
        werr[f"dws2[{s}]"] = fro_err(got["dws2"][s], dw2)
    return errs, werr


def backward_parity(cfg, host_bias=None, exact_dcent=True):
    """One moe_backward of cfg's seeded layer against the oracle in the
    kernels' precision and in exact arithmetic (the bounds above;
    exact_dcent=False leaves dcentroids out of the exact comparison); experts
    that no token chose must get exactly zero weight gradients (the outputs
    start as NaN, so every checked element has been written).  host_bias
    replaces the seeded routing bias.  Returns the GPU's gradients, the
    selection and the kernel-precision reference."""
    fp8 = cfg.oracle_fp8
    host = HostLayer(cfg)
    if host_bias is not None:
        host.bias = host_bias
    layer = host.device_layer()
    u = synth.tokens(cfg)
    dout = synth.normal_bf16(synth.key(cfg.seed, "tokens", 999), (cfg.T, cfg.d), 1.0)
    g = {k: torch.full_like(v, float("nan")) for k, v in layer.grad_buffers().items()}  # all must be written
    layer.backward(u.to(DEV), host.bias.to(DEV), dout.to(DEV), grads=g)
    assert layer.backward_status() == 0
    # the selection the backward recomputed
    idx = torch.empty((cfg.T, cfg.k), dtype=torch.int32, device=DEV)
    gate = torch.empty((cfg.T, cfg.k), dtype=torch.float32, device=DEV)
    cnt = torch.empty(cfg.E, dtype=torch.int32, device=DEV)
    capi.moe_route(layer.dims, u.to(DEV), layer.centroids, host.bias.to(DEV), idx, gate, cnt, layer.ws)
    idx = idx.cpu().numpy()
    got = {k: v.cpu().numpy().astype(np.float64) for k, v in g.items()}
    oracle_of = lambda act_bf16: ob.layer_backward(
        synth.bf16_bits(u), synth.bf16_bits(host.cent), idx, oracle.bf16_to_f64(synth.bf16_bits(dout)),
        host.routed_bits, host.shared_bits, cfg.n_shared, cfg.E, fp8=fp8, act_bf16=act_bf16)
    refs = {}
    for act_bf16 in (True, False):
        ref = refs[act_bf16] = oracle_of(act_bf16)
        errs, werr = _errors(got, ref, cfg)
        data_tol, wg_tol = (KP_TOL, KP_WG_TOL) if act_bf16 else EXACT_TOL[bool(fp8)]
        dcent_tol = data_tol if fp8 else (KP_DCENT_BF16 if act_bf16 else EXACT_DCENT_BF16)
        worst = max(werr, key=werr.get)
        print(f"{cfg.name} vs {'kernel precision' if act_bf16 else 'exact'}: du {errs['du']:.3e}, "
              f"dcentroids {errs['dcentroids']:.3e} (max|err|/rms); weights worst {worst} {werr[worst]:.3e}")
        assert errs["du"] <= data_tol, errs
        assert errs["dcentroids"] <= dcent_tol or (not act_bf16 and not exact_dcent), errs
        assert all(v <= wg_tol for v in werr.values()), {k: v for k, v in werr.items() if v > wg_tol}
    for e in set(range(cfg.E)) - set(refs[True]["dw_routed"]):
        assert not got["dw13"][e].any() and not got["dw2"][e].any()
    return got, idx, gate.cpu().numpy().astype(np.float64), host, u, dout, refs[True]


@pytest.mark.parametrize("name", ["tiny", "ragged", "mid", "tiny_fp8", "ragged_fp8", "ragged_ue8m0", "mid_fp8"])
def test_backward_matches_oracle(name):
    cfg = synth.get_config("mid", prec="fp8") if name == "mid_fp8" else synth.get_config(name)
    fp8 = cfg.oracle_fp8
    got, idx, gate, host, u, dout, ref = backward_parity(cfg)
    # the weight-gradient GEMM's arithmetic: dW2 = dy^T h on the bf16-rounded operands
    x = oracle.bf16_to_f64(synth.bf16_bits(u))
    G = oracle.bf16_to_f64(synth.bf16_bits(dout))
    pow2 = fp8 == "ue8m0"
    for e in sorted(ref["dw_routed"])[:4]:
        w1, w3, _ = oracle.expert_operands(*host.routed_bits(e), fp8)
        rows, js = np.nonzero(idx == e)
        xr = oracle.fp8_roundtrip_1x128(x[rows], pow2) if fp8 else x[rows]
        a, b = _bf16(xr @ w1.T), _bf16(xr @ w3.T)
        h = _bf16(a / (1.0 + np.exp(-a)) * b)
        dy = _bf16(gate[rows, js][:, None] * G[rows])
        if fp8:  # quantised along the tokens, each dequantised value rounded to bf16
            dy, h = _bf16(ob._q_tok(dy, pow2)), _bf16(ob._q_tok(h, pow2))
        assert fro_err(got["dw2"][e], dy.T @ h) <= REPLAY_TOL, e


def test_transpose_expert_weights():
    E, I, d = 3, 256, 384
    w13 = torch.randn((E, 2 * I, d), device=DEV).to(torch.bfloat16)
    w2 = torch.randn((E, d, I), device=DEV).to(torch.bfloat16)
    w13t = torch.empty((E, d, 2 * I), dtype=torch.bfloat16, device=DEV)
    w2t = torch.empty((E, I, d), dtype=torch.bfloat16, device=DEV)
    capi.moe_transpose_expert_weights(E, I, d, w13, w2, w13t, w2t)
    assert torch.equal(w13t, w13.transpose(1, 2)) and torch.equal(w2t, w2.transpose(1, 2))


def test_transpose_expert_weights_fp8():
    """FP8 codes and block-scale grids transposed per expert equal the
    quantisation of the transposed bf16 weights (a 128 x 128 block keeps its
    codes and its scale when transposed)."""
    E, I, d = 3, 256, 384
    w13 = torch.randn((E, 2 * I, d), device=DEV).to(torch.bfloat16)
    w2 = torch.randn((E, d, I), device=DEV).to(torch.bfloat16)

    def quant(w):
        r, c = w.shape
        q = torch.empty((r, c), dtype=torch.uint8, device=DEV)
        s = torch.empty((r // 128, c // 128), dtype=torch.float32, device=DEV)
        capi.moe_quantize_fp8_blocks(w.contiguous(), r, c, q, s)
        return q, s

    w13q, w13s = (torch.stack(t) for t in zip(*[quant(w13[e]) for e in range(E)]))
    w2q, w2s = (torch.stack(t) for t in zip(*[quant(w2[e]) for e in range(E)]))
    w13t = torch.empty((E, d, 2 * I), dtype=torch.uint8, device=DEV)
    w2t = torch.empty((E, I, d), dtype=torch.uint8, device=DEV)
    w13ts = torch.empty((E, d // 128, 2 * I // 128), device=DEV)
    w2ts = torch.empty((E, I // 128, d // 128), device=DEV)
    capi.moe_transpose_expert_weights_fp8(E, I, d, w13q, w13s, w2q, w2s, w13t, w13ts, w2t, w2ts)
    assert torch.equal(w13t, w13q.transpose(1, 2)) and torch.equal(w2t, w2q.transpose(1, 2))
    assert torch.equal(w13ts, w13s.transpose(1, 2)) and torch.equal(w2ts, w2s.transpose(1, 2))
    for e in range(E):  # the same as quantising the transposed bf16 weights
        tq, ts = quant(w13[e].t())
        assert torch.equal(tq, w13t[e]) and torch.equal(ts, w13ts[e])
