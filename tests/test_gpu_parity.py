"""GPU parity: every C-ABI call of the CUDA path against the CPU oracle on the
same seeded inputs.  Integer work (selection, counts, permutation, FP8 codes)
is compared bit for bit; floating point within the stated tolerances."""
import numpy as np
import pytest
import torch

import oracle
import synth
from mixture_experts_layer_87_b300 import capi
from parity import (NEAR_TIE, TOL, Y_TOL, HostLayer, bf16_to_np, check_routing_and_dispatch, check_selection,
                    chunk_covering_tokens, gpu_layer_pass, gpu_rows, oracle_rows, rel_err)

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _ws(cfg, T=None):
    dm = capi.dims(cfg.T if T is None else T, cfg.d, cfg.E, cfg.k, cfg.n_shared, cfg.inter, cfg.prec,
                   cfg.route_groups, cfg.route_group_limit)
    return dm, torch.empty(capi.moe_workspace_size(dm), dtype=torch.uint8, device=DEV)


def _route_gpu(cfg, u, cent, bias):
    dm, ws = _ws(cfg)
    idx = torch.empty((cfg.T, cfg.k), dtype=torch.int32, device=DEV)
    gate = torch.empty((cfg.T, cfg.k), dtype=torch.float32, device=DEV)
    counts = torch.empty(cfg.E, dtype=torch.int32, device=DEV)
    capi.moe_route(dm, u.to(DEV), cent.to(DEV), bias.to(DEV), idx, gate, counts, ws)
    assert capi.moe_read_device_status(ws) == 0
    return idx.cpu().numpy(), gate.cpu().numpy(), counts.cpu().numpy()


# ----------------------------------------------------------------------------
def test_bounded_wait_times_out_and_context_survives():
    ws = torch.zeros(1 << 12, dtype=torch.uint8, device=DEV)
    capi.moe_selftest_wait_timeout(ws, 20000)          # 20 ms, nothing ever arrives
    assert capi.moe_read_device_status(ws) == 5        # MOE_ERR_TIMEOUT
    x = torch.ones(4, device=DEV)
    assert float((x * 2).sum()) == 8.0                 # the context is still usable


ROUTE_CASES = {"tiny": {}, "ragged": {}, "mid": {},
               # node-limited routing: experts on nodes, a token on at most `limit` of them
               "ragged_nodes": dict(route_groups=5, route_group_limit=2),
               "mid_nodes": dict(route_groups=8, route_group_limit=3)}


@pytest.mark.parametrize("name", list(ROUTE_CASES))
def test_route_parity(name):
    cfg = synth.get_config(name.replace("_nodes", ""), **ROUTE_CASES[name])
    u, cent, bias = synth.tokens(cfg), synth.centroids(cfg), synth.bias(cfg)
    idx, gate, counts = _route_gpu(cfg, u, cent, bias)
    r = oracle.route(synth.bf16_bits(u), synth.bf16_bits(cent), np.asarray(bias), cfg.k, want_all=True,
                     groups=cfg.route_groups, group_limit=cfg.route_group_limit)
    ties = check_selection(idx, r, np.asarray(bias), cfg.k, cfg.route_groups, cfg.route_group_limit)
    # counts are the histogram of the GPU's own selection, bit for bit
    np.testing.assert_array_equal(counts, np.bincount(idx.ravel(), minlength=cfg.E))
    if not ties:
        np.testing.assert_array_equal(counts, np.bincount(r["idx"].ravel(), minlength=cfg.E))
    # gates: fp32 on the GPU vs fp64, for the GPU's selection
    ref_gate = oracle.gates_for(r["s_all"], idx)
    np.testing.assert_allclose(gate, ref_gate, rtol=0, atol=2e-6)
    np.testing.assert_allclose(gate.sum(1), 1.0, atol=1e-6)
    # order: by biased score descending where the scores are clearly apart
    score = r["s_all"] + np.asarray(bias, np.float64)[None, :]
    s_sel = np.take_along_axis(score, idx.astype(np.int64), 1)
    d = np.diff(s_sel, axis=1)
    assert (d[np.abs(d) > NEAR_TIE] < 0).all()


@pytest.mark.parametrize("name", ["tiny", "ragged", "mid", "tiny_fp8", "ragged_fp8", "ragged_ue8m0"])
def test_permute_parity(name):
    cfg = synth.get_config(name)
    u, cent, bias = synth.tokens(cfg), synth.centroids(cfg), synth.bias(cfg)
    idx, _, _ = _route_gpu(cfg, u, cent, bias)
    dm, ws = _ws(cfg)
    R = cfg.T * cfg.k
    fp8 = cfg.is_fp8
    offsets = torch.empty(cfg.E + 1, dtype=torch.int32, device=DEV)
    perm = torch.empty(R, dtype=torch.int32, device=DEV)
    slot = torch.empty((cfg.T, cfg.k), dtype=torch.int32, device=DEV)
    x = torch.empty((R, cfg.d), dtype=torch.uint8 if fp8 else torch.bfloat16, device=DEV)
    xs = torch.empty((cfg.d // 128, R), dtype=torch.float32, device=DEV) if fp8 else None
    capi.moe_permute(dm, torch.from_numpy(idx).to(DEV), u.to(DEV), offsets, perm, slot, x, xs, ws)
    assert capi.moe_read_device_status(ws) == 0
    lay = oracle.dispatch_layout(idx, cfg.E)
    np.testing.assert_array_equal(offsets.cpu().numpy(), lay["offsets"])
    np.testing.assert_array_equal(perm.cpu().numpy(), lay["perm"])
    np.testing.assert_array_equal(slot.cpu().numpy(), lay["slot"])
    ub = synth.bf16_bits(u)
    if not fp8:
        np.testing.assert_array_equal(x.view(torch.int16).cpu().numpy().view(np.uint16), ub[lay["perm"]])
    else:
        q, s = oracle.quant_1x128(oracle.bf16_to_f64(ub), pow2=cfg.prec == "fp8_ue8m0")
        np.testing.assert_array_equal(x.cpu().numpy(), q[lay["perm"]])
        np.testing.assert_array_equal(xs.cpu().numpy().T, s[lay["perm"]])


@pytest.mark.parametrize("pow2", [False, True])
def test_quantize_blocks_bit_exact(pow2):
    w = synth.normal_bf16(synth.key(5, "w1", 3), (384, 512), 0.05)
    w[:128, :128] = 0                                      # all-zero block -> scale 1
    q = torch.empty((384, 512), dtype=torch.uint8, device=DEV)
    s = torch.empty((3, 4), dtype=torch.float32, device=DEV)
    capi.moe_quantize_fp8_blocks(w.to(DEV), 384, 512, q, s, pow2_scales=pow2)
    torch.cuda.synchronize()
    rq, rs = oracle.quant_128x128(oracle.bf16_to_f64(synth.bf16_bits(w)), pow2=pow2)
    np.testing.assert_array_equal(q.cpu().numpy(), rq)
    np.testing.assert_array_equal(s.cpu().numpy(), rs)
    assert s[0, 0].item() == 1.0


def test_pack_gate_up_layout():
    E, I, d = 3, 256, 128
    w1 = torch.arange(E * I * d, dtype=torch.float32).reshape(E, I, d).to(torch.bfloat16).to(DEV)
    w3 = (-torch.arange(E * I * d, dtype=torch.float32)).reshape(E, I, d).to(torch.bfloat16).to(DEV)
    out = torch.empty((E, 2 * I, d), dtype=torch.bfloat16, device=DEV)
    capi.moe_pack_gate_up(w1, w3, E, I, d, out)
    ref = torch.stack([w1.view(E, I // 128, 128, d), w3.view(E, I // 128, 128, d)], dim=2).reshape(E, 2 * I, d)
    assert torch.equal(out, ref)


def test_bias_update_bit_exact_trajectory():
    E, T, k = 64, 256, 6
    rng = np.random.default_rng(0)
    b = np.zeros(E, np.float32)
    bd = torch.zeros(E, dtype=torch.float32, device=DEV)
    for step in range(50):
        counts = rng.multinomial(T * k, rng.dirichlet(np.ones(E) * 0.5)).astype(np.int32)
        counts[step % E] = T * k // E                    # exactly at the mean somewhere
        capi.moe_bias_update(E, T, k, torch.from_numpy(counts).to(DEV), 0.001, bd)
        b = oracle.bias_update(counts, b, T, k, 0.001)
    np.testing.assert_array_equal(bd.cpu().numpy(), b)


# ----------------------------------------------------------------------------
def _forward_parity(cfg, sample=None, extra_chunks=True):
    """moe_forward against the oracle: routing and dispatch of the whole batch
    bit for bit (near-ties excepted), h' on the sampled tokens (all by
    default; with a sample, the tokens that cover every expert chunk of the
    grouped GEMMs are added) and the routed expert outputs y_perm of the same
    tokens row by row.  Returns (max|err|/rms on h', the same on y)."""
    host = HostLayer(cfg)
    layer = host.device_layer()
    u = synth.tokens(cfg)
    bias = np.asarray(host.bias)
    res = gpu_layer_pass(layer, u.to(DEV), host.bias.to(DEV))
    ub = synth.bf16_bits(u)
    r = oracle.route(ub, synth.bf16_bits(host.cent), bias, cfg.k, want_all=True, groups=cfg.route_groups,
                     group_limit=cfg.route_group_limit)
    check_routing_and_dispatch(res, r, bias, cfg.E, cfg.k, cfg.route_groups, cfg.route_group_limit)
    if sample is None:
        tokens = np.arange(cfg.T)
    else:
        tokens = chunk_covering_tokens(res["idx"], cfg.E, base=sample) if extra_chunks else np.asarray(sample)
    idx = res["idx"][tokens]
    h_ref, y_ref = oracle_rows(host, ub[tokens], idx, oracle.gates_for(r["s_all"][tokens], idx))
    h, y = gpu_rows(res, tokens)
    return rel_err(h, h_ref), rel_err(y, y_ref)


@pytest.mark.parametrize("name", ["tiny", "ragged", "tiny_fp8", "ragged_fp8", "tiny_ue8m0", "ragged_ue8m0"])
def test_forward_parity_full(name):
    cfg = synth.get_config(name)
    err, err_y = _forward_parity(cfg)
    print(f"{name}: max|err|/rms h' = {err:.3e}, routed y = {err_y:.3e}")
    assert err <= TOL[cfg.prec]
    assert err_y <= Y_TOL[cfg.prec]


@pytest.mark.parametrize("name", ["mid", "mid_fp8", "mid_nodes", "mid_ue8m0"])
def test_forward_parity_mid_sampled(name):
    extra = {"mid": {}, "mid_fp8": dict(prec="fp8"), "mid_nodes": dict(route_groups=8, route_group_limit=3),
             "mid_ue8m0": dict(prec="fp8_ue8m0")}
    cfg = synth.get_config("mid", **extra[name])
    sample = np.arange(0, cfg.T, 29)           # 142 tokens from every part of the batch, plus chunk cover
    err, err_y = _forward_parity(cfg, sample)
    print(f"{name}: max|err|/rms h' = {err:.3e}, routed y = {err_y:.3e}")
    assert err <= TOL[cfg.prec]
    assert err_y <= Y_TOL[cfg.prec]


def test_forward_is_deterministic():
    cfg = synth.get_config("ragged")
    host = HostLayer(cfg)
    layer = host.device_layer()
    u = synth.tokens(cfg).to(DEV)
    b = host.bias.to(DEV)
    o1 = layer.forward(u, b).clone()
    o2 = layer.forward(u, b).clone()
    assert torch.equal(o1, o2)


def test_grouped_ffn_and_combine_calls():
    """moe_grouped_ffn on caller offsets (with empty groups) and moe_combine,
    against the oracle expert and combine."""
    cfg = synth.get_config("ragged")
    host = HostLayer(cfg)
    layer = host.device_layer()
    dm, ws = _ws(cfg)
    G = 5
    sizes = np.array([0, 37, 130, 0, 200], np.int32)
    offs = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    rows = int(offs[-1])
    x = synth.normal_bf16(77, (rows, cfg.d), 1.0)
    y = torch.empty((rows, cfg.d), dtype=torch.bfloat16, device=DEV)
    capi.moe_grouped_ffn(dm, G, rows, torch.from_numpy(offs).to(DEV), x.to(DEV), None, layer.w13, None,
                         layer.w2, None, y, ws)
    assert capi.moe_read_device_status(ws) == 0
    xb = oracle.bf16_to_f64(synth.bf16_bits(x))
    ref = np.zeros((rows, cfg.d))
    for g in range(G):
        sl = slice(offs[g], offs[g + 1])
        ref[sl] = oracle.swiglu(xb[sl], *oracle.expert_operands(*host.routed_bits(g), fp8=False))
    # y is bf16: its own rounding reaches 2^-9 |y| ~ 1% of rms(y) at the largest
    # outputs, plus the bf16 rounding of h carried through the down product
    assert rel_err(bf16_to_np(y), ref) <= 3e-2
    # combine: random slots / gates over these rows
    T, k = 50, 3
    rng = np.random.default_rng(1)
    slot = np.stack([rng.choice(T * k, k, replace=False) for _ in range(T)]).astype(np.int32)  # y_perm = y[:T*k]
    gate = rng.dirichlet(np.ones(k), size=T).astype(np.float32)
    u = synth.normal_bf16(78, (T, cfg.d), 1.0)
    ysh = synth.normal_bf16(79, (1, T, cfg.d), 0.5)
    dmc = capi.dims(T, cfg.d, cfg.E, k, 1, cfg.inter, "bf16")
    out = torch.empty((T, cfg.d), dtype=torch.bfloat16, device=DEV)
    capi.moe_combine(dmc, u.to(DEV), ysh.to(DEV), y, torch.from_numpy(slot).to(DEV),
                     torch.from_numpy(gate).to(DEV), out)
    refc = oracle.combine(synth.bf16_bits(u), bf16_to_np(ysh.to(DEV)), bf16_to_np(y)[:T * k], slot, gate)
    assert np.abs(bf16_to_np(out) - refc).max() <= 2 ** -7 * np.abs(refc).max()
