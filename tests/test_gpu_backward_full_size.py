"""The backward pass at the full size the bench times (T=8192, d=7168, 256
routed experts top-8 + 1 shared, I=2048; bf16 and FP8) against the oracle in
the kernels' precision (act_bf16; the bounds and their derivation are those of
test_gpu_backward.py).

The oracle cannot take the whole V3 backward in fp64 in a test's time, but
the parts it checks are exact on a subset: du_t depends on token t alone (its
experts' data gradients, the residual, the router's share), and an expert's
weight gradients and centroid gradient on that expert's tokens alone.  So the
oracle runs the layer's backward on the union of
  * a strided token sample (every 256th token): du of those rows, and
  * every token of the three least-loaded experts that hold at least 32
    tokens: those experts' dW13, dW2 and dcentroids rows, whole;
which is the same function as the full backward restricted to those outputs.
The shared expert's weight gradient sums over all 8192 tokens and is checked
at the mid size instead."""
import numpy as np
import pytest
import torch

import oracle
import synth
from mixture_experts_layer_87_b300 import capi
from oracle import backward as ob
from parity import HostLayer, rel_err
from test_gpu_backward import KP_DCENT_BF16, KP_TOL, KP_WG_TOL, _interleave13, fro_err

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.mark.parametrize("name", ["v3", "v3_fp8"])
def test_v3_backward_sampled_tokens_and_whole_experts(name):
    cfg = synth.get_config(name)
    fp8 = cfg.oracle_fp8
    host = HostLayer(cfg, keep_weights=False)
    layer = host.device_layer()
    layer.release_staging()
    u = synth.tokens(cfg)
    dout = synth.normal_bf16(synth.key(cfg.seed, "tokens", 999), (cfg.T, cfg.d), 1.0)
    g = layer.backward(u.to(DEV), host.bias.to(DEV), dout.to(DEV))
    torch.cuda.synchronize()
    assert layer.backward_status() == 0
    idx = torch.empty((cfg.T, cfg.k), dtype=torch.int32, device=DEV)
    gate = torch.empty((cfg.T, cfg.k), dtype=torch.float32, device=DEV)
    cnt = torch.empty(cfg.E, dtype=torch.int32, device=DEV)
    capi.moe_route(layer.dims, u.to(DEV), layer.centroids, host.bias.to(DEV), idx, gate, cnt, layer.ws)
    idx, cnt = idx.cpu().numpy(), cnt.cpu().numpy()
    sample = np.arange(0, cfg.T, 256)
    eligible = np.nonzero(cnt >= 32)[0]
    experts = eligible[np.argsort(cnt[eligible], kind="stable")[:3]]
    whole = np.nonzero(np.isin(idx, experts).any(1))[0]
    tokens = np.union1d(sample, whole)
    got_du = g["du"][torch.from_numpy(tokens).to(DEV)].cpu().numpy().astype(np.float64)
    got = {k: g[k][torch.from_numpy(experts.astype(np.int64)).to(DEV)].cpu().numpy().astype(np.float64)
           for k in ("dw13", "dw2", "dcentroids")}
    del g, layer
    torch.cuda.empty_cache()

    ref = ob.layer_backward(synth.bf16_bits(u)[tokens], synth.bf16_bits(host.cent), idx[tokens],
                            oracle.bf16_to_f64(synth.bf16_bits(dout))[tokens], host.routed_bits, host.shared_bits,
                            cfg.n_shared, cfg.E, fp8=fp8, act_bf16=True, keep_dw={int(e) for e in experts})
    e_du = rel_err(got_du, ref["du"])
    e_dc = rel_err(got["dcentroids"], ref["dcent"][experts])
    werr = {}
    for i, e in enumerate(experts):
        dw1, dw3, dw2 = ref["dw_routed"][int(e)]
        werr[f"dw13[{e}]"] = fro_err(got["dw13"][i], _interleave13(dw1, dw3, cfg.inter, cfg.d))
        werr[f"dw2[{e}]"] = fro_err(got["dw2"][i], dw2)
    worst = max(werr, key=werr.get)
    print(f"{name}: du of {len(tokens)} tokens {e_du:.3e}, dcentroids of experts {experts.tolist()} "
          f"({cnt[experts].tolist()} tokens) {e_dc:.3e} (max|err|/rms); weights worst {worst} {werr[worst]:.3e}")
    assert e_du <= KP_TOL
    assert e_dc <= (KP_TOL if fp8 else KP_DCENT_BF16)
    assert all(v <= KP_WG_TOL for v in werr.values()), werr
