"""GPU parity at the edges of the layer's shape space, through the C ABI,
against the CPU oracle:
  * an empty batch (T = 0): nothing is enqueued but the loads are zeroed;
  * one token;
  * one routed expert with k = 1 and no shared expert: the layer reduces to
    u + SwiGLU(u) (ai.flicky.cc 2.1.2 with N_r = K_r = 1, N_s = 0);
  * no shared expert at all (N_s = 0), bf16 and FP8;
  * the largest routing the library accepts: E = 1024 experts, k = 32, which
    runs the widest top-k variant (32 experts per lane);
  * every token routed to the same k experts (a fully skewed load: the other
    experts are empty groups).
The backward pass (moe_backward) is held to the same edges: an empty batch
(every gradient zero), one token, the one-expert top-1 layer (a dense SwiGLU,
whose centroids get no gradient since the one gate is s / s = 1), no shared
expert, and the fully skewed load (the empty experts' weight gradients exactly
zero), each against the backward oracle with the bounds of the backward tests.
"""
from dataclasses import replace

import numpy as np
import pytest
import torch

import synth
from mixture_experts_layer_87_b300 import MoELayer, capi
from parity import TOL, Y_TOL
from test_gpu_backward import backward_parity
from test_gpu_parity import _forward_parity

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _cfg(name, **kw):
    return replace(synth.get_config(name), name=f"{name}_edge", **kw)


@pytest.mark.parametrize("prec", ["bf16", "fp8"])
def test_empty_batch(prec):
    layer = MoELayer(0, 256, 16, 4, 1, 128, prec)
    for e in range(16):
        layer.load_expert(e, *synth.expert_weights(synth.get_config("tiny"), e))
    layer.load_expert(0, *synth.expert_weights(synth.get_config("tiny"), 0, shared=True), shared=True)
    layer.set_centroids(synth.centroids(synth.get_config("tiny")))
    u = torch.empty((0, 256), dtype=torch.bfloat16, device=DEV)
    counts = torch.full((16,), 7, dtype=torch.int32, device=DEV)
    out = layer.forward(u, torch.zeros(16, device=DEV), counts=counts)
    assert out.shape == (0, 256)
    assert layer.status() == 0
    assert int(counts.abs().sum()) == 0


@pytest.mark.parametrize("name", ["tiny", "tiny_fp8"])
def test_single_token(name):
    cfg = _cfg(name, T=1)
    err, err_y = _forward_parity(cfg)
    assert err <= TOL[cfg.prec] and err_y <= Y_TOL[cfg.prec]


@pytest.mark.parametrize("prec", ["bf16", "fp8"])
def test_one_expert_top1_no_shared_is_a_dense_swiglu(prec):
    cfg = _cfg("tiny", E=1, k=1, n_shared=0, prec=prec)
    err, err_y = _forward_parity(cfg)
    assert err <= TOL[cfg.prec] and err_y <= Y_TOL[cfg.prec]


@pytest.mark.parametrize("name", ["ragged", "ragged_fp8"])
def test_no_shared_expert(name):
    cfg = _cfg(name, n_shared=0)
    err, err_y = _forward_parity(cfg)
    assert err <= TOL[cfg.prec] and err_y <= Y_TOL[cfg.prec]


def test_largest_routing_1024_experts_top32():
    cfg = _cfg("tiny", T=96, d=128, E=1024, k=32, n_shared=1, inter=128, bias="normal")
    err, err_y = _forward_parity(cfg)
    assert err <= TOL[cfg.prec] and err_y <= Y_TOL[cfg.prec]


@pytest.mark.parametrize("prec", ["bf16", "fp8"])
def test_all_tokens_on_the_same_experts(prec):
    # a bias of +10 on experts 3, 5, 11, 12 wins every token's top-4 (sigmoid
    # scores are in (0, 1)); gates still come from the unbiased affinities
    cfg = _cfg("tiny", prec=prec, bias="zero")
    host_bias = torch.zeros(cfg.E)
    host_bias[[3, 5, 11, 12]] = 10.0

    import test_gpu_parity as tp
    orig = synth.bias
    try:
        synth.bias = lambda c: host_bias.clone() if c.name == cfg.name else orig(c)
        err, err_y = tp._forward_parity(cfg)
    finally:
        synth.bias = orig
    assert err <= TOL[cfg.prec] and err_y <= Y_TOL[cfg.prec]


@pytest.mark.parametrize("d,k", [(128, 32), (384, 31), (256, 16)])
def test_permute_copies_every_row(d, k):
    """x_perm[r] == u[perm[r]] for every permuted row, bit for bit, also when
    a row is not a whole number of 512-byte warp strides (d = 128, 384)."""
    cfg = _cfg("tiny", T=96, d=d, E=64, k=k, inter=128, bias="normal")
    u = synth.tokens(cfg).to(DEV)
    dm = capi.dims(cfg.T, d, cfg.E, k, 1, cfg.inter, "bf16")
    ws = torch.empty(capi.moe_workspace_size(dm), dtype=torch.uint8, device=DEV)
    idx = torch.empty((cfg.T, k), dtype=torch.int32, device=DEV)
    gate = torch.empty((cfg.T, k), device=DEV)
    cnt = torch.empty(cfg.E, dtype=torch.int32, device=DEV)
    capi.moe_route(dm, u, synth.centroids(cfg).to(DEV), synth.bias(cfg).to(DEV), idx, gate, cnt, ws)
    R = cfg.T * k
    offs = torch.empty(cfg.E + 1, dtype=torch.int32, device=DEV)
    perm = torch.empty(R, dtype=torch.int32, device=DEV)
    slot = torch.empty((cfg.T, k), dtype=torch.int32, device=DEV)
    x = torch.full((R, d), float("nan"), dtype=torch.bfloat16, device=DEV)
    capi.moe_permute(dm, idx, u, offs, perm, slot, x, None, ws)
    assert capi.moe_read_device_status(ws) == 0
    p = perm.long()
    assert torch.equal(x.view(torch.int16), u[p].view(torch.int16))


def test_gates_when_every_selected_affinity_underflows():
    """Logits near -150: every sigmoid affinity underflows to 0 in fp32, yet the
    gates s_j / sum s (well defined in fp64) must come out finite, summing to
    1, and equal to the oracle's for the GPU's (near-tie) selection."""
    import oracle
    from parity import check_selection
    T, d, E, k = 8, 256, 16, 4
    u = (1.0 + torch.arange(T, dtype=torch.float32)[:, None] / 16).expand(T, d).to(torch.bfloat16).contiguous()
    c = (-(150.0 + 0.5 * torch.arange(E, dtype=torch.float32)[:, None]) / d).expand(E, d)
    cent = c.to(torch.bfloat16).contiguous()
    bias = torch.zeros(E, dtype=torch.float32)
    dm = capi.dims(T, d, E, k, 0, 128, "bf16")
    ws = torch.empty(capi.moe_workspace_size(dm), dtype=torch.uint8, device=DEV)
    idx = torch.empty((T, k), dtype=torch.int32, device=DEV)
    gate = torch.empty((T, k), dtype=torch.float32, device=DEV)
    cnt = torch.empty(E, dtype=torch.int32, device=DEV)
    capi.moe_route(dm, u.to(DEV), cent.to(DEV), bias.to(DEV), idx, gate, cnt, ws)
    assert capi.moe_read_device_status(ws) == 0
    idx, gate = idx.cpu().numpy(), gate.cpu().numpy()
    r = oracle.route(synth.bf16_bits(u), synth.bf16_bits(cent), bias.numpy(), k, want_all=True)
    assert (r["s_all"] < 1e-60).all() and (r["s_all"] > 0).all()     # underflows fp32, not fp64
    check_selection(idx, r, bias.numpy(), k)
    assert np.isfinite(gate).all()
    np.testing.assert_allclose(gate.sum(1), 1.0, atol=1e-6)
    np.testing.assert_allclose(gate, oracle.gates_for(r["s_all"], idx), rtol=0, atol=2e-6)


@pytest.mark.parametrize("prec", ["bf16", "fp8"])
def test_backward_empty_batch(prec):
    cfg = synth.get_config("tiny")
    layer = MoELayer(0, 256, 16, 4, 1, 128, prec)
    for e in range(16):
        layer.load_expert(e, *synth.expert_weights(cfg, e))
    layer.load_expert(0, *synth.expert_weights(cfg, 0, shared=True), shared=True)
    layer.set_centroids(synth.centroids(cfg))
    u = torch.empty((0, 256), dtype=torch.bfloat16, device=DEV)
    g = {k: torch.full_like(v, float("nan")) for k, v in layer.grad_buffers().items()}
    layer.backward(u, torch.zeros(16, device=DEV), u, grads=g)
    torch.cuda.synchronize()
    assert layer.backward_status() == 0
    assert g["du"].shape == (0, 256)
    for k in ("dcentroids", "dw13", "dw2", "dws13", "dws2"):
        assert not g[k].any(), k


@pytest.mark.parametrize("name", ["tiny", "tiny_fp8"])
def test_backward_single_token(name):
    # dcentroids only against the oracle in the kernels' precision: with one
    # token an expert's row is dz u, and dz = (dg_j - sum_i g_i dg_i) terms can
    # cancel, so the bf16 / E4M3 roundings of the intermediates move it by an
    # unbounded relative amount (the two oracle modes alone are 2.2e-2 apart in
    # bf16 and 6.2e-1 in FP8 at this token, 1.5e-2 and 9.2e-2 at 64 tokens).
    backward_parity(_cfg(name, T=1), exact_dcent=False)


@pytest.mark.parametrize("prec", ["bf16", "fp8"])
def test_backward_one_expert_top1_no_shared(prec):
    got, *_ = backward_parity(_cfg("tiny", E=1, k=1, n_shared=0, prec=prec))
    assert not got["dcentroids"].any()


@pytest.mark.parametrize("name", ["ragged", "ragged_fp8"])
def test_backward_no_shared_expert(name):
    backward_parity(_cfg(name, n_shared=0))


@pytest.mark.parametrize("prec", ["bf16", "fp8"])
def test_backward_all_tokens_on_the_same_experts(prec):
    cfg = _cfg("tiny", prec=prec, bias="zero")
    host_bias = torch.zeros(cfg.E)
    host_bias[[3, 5, 11, 12]] = 10.0
    got, idx, *_ = backward_parity(cfg, host_bias)
    assert (np.sort(idx, 1) == [3, 5, 11, 12]).all()
