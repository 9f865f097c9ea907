"""The backward pass on the GPU (moe_backward, bf16) against the fp64 backward
oracle (oracle/backward.py, itself pinned to autograd and finite differences),
with the GPU's own selection held fixed on both sides.

Tolerances.  The pass keeps its activations in bf16 as the forward does (a,
b, h, y, dy, dh, da/db, dx: each rounded to 8 significant bits, 2^-9
relative), and a gradient goes through up to four of those roundings:
  * data gradients (du, dcentroids): max|err| / rms(ref) <= 5e-2 -- a few
    roundings at the largest elements (max/rms ~ 5);
  * weight gradients: ||err|| / ||ref|| (Frobenius) <= 2e-2.  Their elements
    are sums over an expert's few tokens of products of two activations, so
    their distribution is heavy-tailed and max|err|/rms measures the tail, not
    the arithmetic; four roundings of 2^-9/sqrt(3) rms each give ~0.5% in norm.
  * and the arithmetic itself: dW2 of the first experts against the same
    product replayed from the bf16-rounded a, b, h and dy (fp64):
    ||err|| / ||ref|| <= 1e-3 (the GPU accumulates in fp32)."""
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
BWD_TOL = 5e-2      # data gradients, max|err| / rms(ref)
WG_TOL = 2e-2       # weight gradients, relative Frobenius norm
REPLAY_TOL = 1e-3   # dW2 against the bf16-operand replay, relative Frobenius norm


def fro_err(got, ref):
    return float(np.linalg.norm(got - ref) / np.linalg.norm(ref))


def _bf16(a):
    return torch.from_numpy(np.asarray(a, np.float64)).float().to(torch.bfloat16).double().numpy()


@pytest.mark.parametrize("name", ["tiny", "ragged", "mid"])
def test_backward_matches_oracle(name):
    cfg = synth.get_config(name)
    host = HostLayer(cfg)
    layer = host.device_layer()
    u = synth.tokens(cfg)
    dout = synth.normal_bf16(synth.key(cfg.seed, "tokens", 999), (cfg.T, cfg.d), 1.0)
    g = layer.backward(u.to(DEV), host.bias.to(DEV), dout.to(DEV))
    assert layer.backward_status() == 0
    # the selection the backward recomputed
    idx = torch.empty((cfg.T, cfg.k), dtype=torch.int32, device=DEV)
    gate = torch.empty((cfg.T, cfg.k), dtype=torch.float32, device=DEV)
    cnt = torch.empty(cfg.E, dtype=torch.int32, device=DEV)
    capi.moe_route(layer.dims, u.to(DEV), layer.centroids, host.bias.to(DEV), idx, gate, cnt, layer.ws)
    idx = idx.cpu().numpy()
    ref = ob.layer_backward(synth.bf16_bits(u), synth.bf16_bits(host.cent), idx,
                            oracle.bf16_to_f64(synth.bf16_bits(dout)), host.routed_bits, host.shared_bits,
                            cfg.n_shared, cfg.E)
    got = {k: v.cpu().numpy().astype(np.float64) for k, v in g.items()}
    errs = {"du": rel_err(got["du"], ref["du"]), "dcentroids": rel_err(got["dcentroids"], ref["dcent"])}
    print(f"{name}: du {errs['du']:.3e}, dcentroids {errs['dcentroids']:.3e} (max|err|/rms)")
    assert all(v <= BWD_TOL for v in errs.values()), errs
    I = cfg.inter
    werr = {}
    for e, (dw1, dw3, dw2) in ref["dw_routed"].items():
        # w13 interleave: rows [256j, 256j+128) of W1 block j, [256j+128, 256j+256) of W3 block j
        ref13 = np.stack([dw1.reshape(I // 128, 128, cfg.d), dw3.reshape(I // 128, 128, cfg.d)], 1).reshape(2 * I, cfg.d)
        werr[f"dw13[{e}]"] = fro_err(got["dw13"][e], ref13)
        werr[f"dw2[{e}]"] = fro_err(got["dw2"][e], dw2)
    for e in set(range(cfg.E)) - set(ref["dw_routed"]):
        assert not got["dw13"][e].any() and not got["dw2"][e].any()
    for s, (dw1, dw3, dw2) in enumerate(ref["dw_shared"]):
        ref13 = np.stack([dw1.reshape(I // 128, 128, cfg.d), dw3.reshape(I // 128, 128, cfg.d)], 1).reshape(2 * I, cfg.d)
        werr[f"dws13[{s}]"] = fro_err(got["dws13"][s], ref13)
        werr[f"dws2[{s}]"] = fro_err(got["dws2"][s], dw2)
    worst = max(werr, key=werr.get)
    print(f"{name}: weight gradients, worst {worst} {werr[worst]:.3e} (relative Frobenius)")
    assert all(v <= WG_TOL for v in werr.values()), {k: v for k, v in werr.items() if v > WG_TOL}
    # the weight-gradient GEMM's arithmetic: dW2 = dy^T h on the bf16-rounded operands
    x = oracle.bf16_to_f64(synth.bf16_bits(u))
    G = oracle.bf16_to_f64(synth.bf16_bits(dout))
    gate = gate.cpu().numpy().astype(np.float64)
    for e in sorted(ref["dw_routed"])[:4]:
        w1, w3, _ = (oracle.bf16_to_f64(w) for w in host.routed_bits(e))
        rows, js = np.nonzero(idx == e)
        a, b = _bf16(x[rows] @ w1.T), _bf16(x[rows] @ w3.T)
        h = _bf16(a / (1.0 + np.exp(-a)) * b)
        dy = _bf16(gate[rows, js][:, None] * G[rows])
        assert fro_err(got["dw2"][e], dy.T @ h) <= REPLAY_TOL, e


def test_transpose_expert_weights():
    E, I, d = 3, 256, 384
    w13 = torch.randn((E, 2 * I, d), device=DEV).to(torch.bfloat16)
    w2 = torch.randn((E, d, I), device=DEV).to(torch.bfloat16)
    w13t = torch.empty((E, d, 2 * I), dtype=torch.bfloat16, device=DEV)
    w2t = torch.empty((E, I, d), dtype=torch.bfloat16, device=DEV)
    capi.moe_transpose_expert_weights(E, I, d, w13, w2, w13t, w2t)
    assert torch.equal(w13t, w13.transpose(1, 2)) and torch.equal(w2t, w2.transpose(1, 2))
