"""The backward pass on the GPU (moe_backward, bf16) against the fp64 backward
oracle (oracle/backward.py, itself pinned to autograd and finite differences),
with the GPU's own selection held fixed on both sides.

Tolerance: max|err| / rms(ref) <= 5e-2 on every gradient.  The pass keeps its
activations in bf16 as the forward does (a, b, h, y, dy, dh, da/db, dx: each
rounded to 8 significant bits, 2^-9 relative), and a data gradient goes
through up to four of those roundings; at the largest elements (max/rms ~ 5)
that is a few percent.  Weight gradients sum over tokens in fp32."""
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
BWD_TOL = 5e-2


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
    I = cfg.inter
    for e, (dw1, dw3, dw2) in ref["dw_routed"].items():
        # w13 interleave: rows [256j, 256j+128) of W1 block j, [256j+128, 256j+256) of W3 block j
        ref13 = np.stack([dw1.reshape(I // 128, 128, cfg.d), dw3.reshape(I // 128, 128, cfg.d)], 1).reshape(2 * I, cfg.d)
        errs[f"dw13[{e}]"] = rel_err(got["dw13"][e], ref13)
        errs[f"dw2[{e}]"] = rel_err(got["dw2"][e], dw2)
    for e in set(range(cfg.E)) - set(ref["dw_routed"]):
        assert not got["dw13"][e].any() and not got["dw2"][e].any()
    for s, (dw1, dw3, dw2) in enumerate(ref["dw_shared"]):
        ref13 = np.stack([dw1.reshape(I // 128, 128, cfg.d), dw3.reshape(I // 128, 128, cfg.d)], 1).reshape(2 * I, cfg.d)
        errs[f"dws13[{s}]"] = rel_err(got["dws13"][s], ref13)
        errs[f"dws2[{s}]"] = rel_err(got["dws2"][s], dw2)
    worst = max(errs, key=errs.get)
    print(f"{name}: du {errs['du']:.3e}, dcentroids {errs['dcentroids']:.3e}, worst {worst} {errs[worst]:.3e}")
    assert all(v <= BWD_TOL for v in errs.values()), {k: v for k, v in errs.items() if v > BWD_TOL}


def test_transpose_expert_weights():
    E, I, d = 3, 256, 384
    w13 = torch.randn((E, 2 * I, d), device=DEV).to(torch.bfloat16)
    w2 = torch.randn((E, d, I), device=DEV).to(torch.bfloat16)
    w13t = torch.empty((E, d, 2 * I), dtype=torch.bfloat16, device=DEV)
    w2t = torch.empty((E, I, d), dtype=torch.bfloat16, device=DEV)
    capi.moe_transpose_expert_weights(E, I, d, w13, w2, w13t, w2t)
    assert torch.equal(w13t, w13.transpose(1, 2)) and torch.equal(w2t, w2.transpose(1, 2))
