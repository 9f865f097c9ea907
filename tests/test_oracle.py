"""Pins of the CPU oracle against what the pages and the mathematics fix (no GPU).

Each test checks the oracle against something other than itself: a closed
form, a value the pages print (tests/golden/), a library routine for a
special case, the dense brute force, or an invariant the method states.
"""
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
import synth
from oracle import brute

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bf16_bits_from_f64(a: np.ndarray) -> np.ndarray:
    return synth.bf16_bits(torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(torch.bfloat16))


def _tiny_layer(cfg, seed_bias=None):
    u = synth.tokens(cfg)
    c = synth.centroids(cfg)
    b = synth.bias(cfg) if seed_bias is None else seed_bias
    routed = [synth.expert_weights(cfg, e) for e in range(cfg.E)]
    shared = [synth.expert_weights(cfg, s, shared=True) for s in range(cfg.n_shared)]
    return u, c, b, routed, shared


def _bits(ws):
    return tuple(synth.bf16_bits(w) for w in ws)


# ----------------------------------------------------------------------------
# router
def test_affinity_matches_library_sigmoid():
    """s_{i,t} = sigmoid(u_t^T e_i): against torch.sigmoid of a float64 matmul."""
    cfg = synth.get_config("ragged")
    u, c = synth.tokens(cfg), synth.centroids(cfg)
    r = oracle.route(synth.bf16_bits(u), synth.bf16_bits(c), np.zeros(cfg.E, np.float32), cfg.k, want_all=True)
    ref = torch.sigmoid(u.double() @ c.double().T).numpy()
    np.testing.assert_allclose(r["s_all"], ref, rtol=0, atol=1e-12)


def test_gates_sum_to_one_and_use_unbiased_affinity():
    cfg = synth.get_config("ragged")
    u, c = synth.tokens(cfg), synth.centroids(cfg)
    b = np.asarray(synth.normal_f32(12345, (cfg.E,), 0.05))
    r = oracle.route(synth.bf16_bits(u), synth.bf16_bits(c), b, cfg.k, want_all=True)
    np.testing.assert_allclose(r["gate"].sum(1), 1.0, rtol=0, atol=1e-12)
    s = torch.sigmoid(u.double() @ c.double().T).numpy()
    sel = np.take_along_axis(s, r["idx"].astype(np.int64), 1)
    np.testing.assert_allclose(r["gate"], sel / sel.sum(1, keepdims=True), rtol=0, atol=1e-12)
    # the bias changed the selection somewhere (else the test says nothing) ...
    r0 = oracle.route(synth.bf16_bits(u), synth.bf16_bits(c), np.zeros(cfg.E, np.float32), cfg.k)
    assert (np.sort(r0["idx"], 1) != np.sort(r["idx"], 1)).any()
    # ... yet a token that keeps its selection keeps its gates (up to the
    # summation order of the normaliser, which follows the biased ranking)
    same = (np.sort(r0["idx"], 1) == np.sort(r["idx"], 1)).all(1)
    assert same.any()
    g0 = {(t, int(e)): g for t in np.nonzero(same)[0] for e, g in zip(r0["idx"][t], r0["gate"][t])}
    for t in np.nonzero(same)[0]:
        for e, g in zip(r["idx"][t], r["gate"][t]):
            assert abs(g - g0[(t, int(e))]) <= 4e-16


def test_selection_is_topk_of_biased_scores():
    """Selected = K_r largest s+b (checked with numpy's argsort); order score desc."""
    cfg = synth.get_config("ragged")
    u, c = synth.tokens(cfg), synth.centroids(cfg)
    b = np.asarray(synth.normal_f32(777, (cfg.E,), 0.02))
    r = oracle.route(synth.bf16_bits(u), synth.bf16_bits(c), b, cfg.k, want_all=True)
    score = r["s_all"] + b.astype(np.float64)
    ref = np.argsort(-score, axis=1, kind="stable")[:, :cfg.k]
    np.testing.assert_array_equal(r["idx"], ref)
    kth = np.take_along_axis(score, ref[:, -1:], 1)[:, 0]
    nxt = np.take_along_axis(score, np.argsort(-score, axis=1, kind="stable")[:, cfg.k:cfg.k + 1], 1)[:, 0]
    np.testing.assert_allclose(r["gap"], kth - nxt, rtol=0, atol=0)


def test_bias_shift_invariance():
    """Adding a constant to every bias changes nothing (selection is by rank)."""
    cfg = synth.get_config("ragged")
    u, c = synth.tokens(cfg), synth.centroids(cfg)
    b = np.asarray(synth.normal_f32(99, (cfg.E,), 0.01))
    r0 = oracle.route(synth.bf16_bits(u), synth.bf16_bits(c), b, cfg.k)
    for shift in (-0.3, 0.05, 1.0):
        r1 = oracle.route(synth.bf16_bits(u), synth.bf16_bits(c), (b + np.float32(shift)).astype(np.float32), cfg.k)
        safe = r0["gap"] > 1e-6       # rounding of b+shift cannot reorder these
        np.testing.assert_array_equal(r0["idx"][safe], r1["idx"][safe])
        np.testing.assert_array_equal(r0["gate"][safe], r1["gate"][safe])


def test_zero_bias_selection_equals_topk_logits():
    """sigmoid is monotone: with b = 0, top-k on s is top-k on the logits."""
    cfg = synth.get_config("tiny")
    u, c = synth.tokens(cfg), synth.centroids(cfg)
    r = oracle.route(synth.bf16_bits(u), synth.bf16_bits(c), np.zeros(cfg.E, np.float32), cfg.k)
    logits = (u.double() @ c.double().T).numpy()
    ref = np.argsort(-logits, axis=1, kind="stable")[:, :cfg.k]
    np.testing.assert_array_equal(np.sort(r["idx"], 1), np.sort(ref, 1))


def test_zero_input_closed_form():
    """u = 0: every s is exactly 1/2, all scores tie, the lowest indices win,
    every gate is 1/k and every FFN(0) = 0, so h' = 0.  With a bias, the
    selection is the top-k of b but the gates stay 1/k (bias not in gates)."""
    T, d, E, k = 5, 128, 8, 3
    u = np.zeros((T, d), np.uint16)
    c = _bf16_bits_from_f64(np.random.default_rng(0).standard_normal((E, d)))
    r = oracle.route(u, c, np.zeros(E, np.float32), k)
    np.testing.assert_array_equal(r["idx"], np.tile(np.arange(k), (T, 1)))
    np.testing.assert_array_equal(r["gate"], np.full((T, k), 1.0 / k))
    b = np.array([0.0, 0.3, -0.1, 0.2, 0.5, 0.0, 0.1, -0.2], np.float32)
    r = oracle.route(u, c, b, k)
    np.testing.assert_array_equal(r["idx"], np.tile([4, 1, 3], (T, 1)))
    np.testing.assert_array_equal(r["gate"], np.full((T, k), 1.0 / k))
    w = [tuple(_bf16_bits_from_f64(np.ones(s)) for s in ((64, d), (64, d), (d, 64)))]
    out = oracle.layer_output(u, np.arange(T), r["idx"], r["gate"], lambda e: w[0], lambda s: w[0], 1, E)
    np.testing.assert_array_equal(out, 0.0)


def test_exact_ties_go_to_lower_index():
    T, d, E, k = 4, 128, 6, 2
    rng = np.random.default_rng(1)
    base = rng.standard_normal((3, d))
    cent = np.concatenate([base, base])          # experts i and i+3 identical
    u = _bf16_bits_from_f64(rng.standard_normal((T, d)))
    r = oracle.route(u, _bf16_bits_from_f64(cent), np.zeros(E, np.float32), k)
    # the best expert's twin has the same score, so the pair (i, i+3) is chosen
    assert (r["idx"][:, 1] == r["idx"][:, 0] + 3).all()
    assert (r["gap"] >= 0).all()


# ----------------------------------------------------------------------------
# dispatch layout (dropless, canonical order)
def test_dispatch_layout_invariants_and_sorted_reference():
    cfg = synth.get_config("ragged")
    u, c, b = synth.tokens(cfg), synth.centroids(cfg), synth.bias(cfg)
    r = oracle.route(synth.bf16_bits(u), synth.bf16_bits(c), np.asarray(b), cfg.k)
    for t in range(cfg.T):
        assert len(set(r["idx"][t].tolist())) == cfg.k          # k distinct experts
    lay = oracle.dispatch_layout(r["idx"], cfg.E)
    assert lay["counts"].sum() == cfg.T * cfg.k                 # dropless
    np.testing.assert_array_equal(np.bincount(r["idx"].ravel(), minlength=cfg.E), lay["counts"])
    assert sorted(lay["slot"].ravel().tolist()) == list(range(cfg.T * cfg.k))   # bijection
    pairs = sorted((int(r["idx"][t, j]), t) for t in range(cfg.T) for j in range(cfg.k))
    np.testing.assert_array_equal(lay["perm"], [t for _, t in pairs])
    for t in range(cfg.T):
        for j in range(cfg.k):
            assert lay["perm"][lay["slot"][t, j]] == t
            s = lay["slot"][t, j]
            e = r["idx"][t, j]
            assert lay["offsets"][e] <= s < lay["offsets"][e + 1]


# ----------------------------------------------------------------------------
# the layer
@pytest.mark.parametrize("name", ["tiny", "ragged"])
def test_sparse_equals_dense_bruteforce(name):
    cfg = synth.get_config(name)
    b = np.asarray(synth.normal_f32(4242, (cfg.E,), 0.02))
    u, c, _, routed, shared = _tiny_layer(cfg)
    r = oracle.route(synth.bf16_bits(u), synth.bf16_bits(c), b, cfg.k)
    out = oracle.layer_output(synth.bf16_bits(u), np.arange(cfg.T), r["idx"], r["gate"],
                              lambda e: _bits(routed[e]), lambda s: _bits(shared[s]), cfg.n_shared, cfg.E)
    f = lambda ws: tuple(w.double().numpy() for w in ws)
    dense = brute.dense_layer(u.double().numpy(), c.double().numpy(), b, cfg.k,
                              [f(w) for w in routed], [f(w) for w in shared])
    for t in range(cfg.T):
        assert set(r["idx"][t].tolist()) == dense["sel"][t]
    scale = np.abs(dense["out"]).max()
    np.testing.assert_allclose(out, dense["out"], rtol=0, atol=1e-12 * scale)


def test_single_expert_reduces_to_dense_swiglu():
    """E=1, k=1: g = 1 and h' = u + SwiGLU(u) (torch F.silu, float64 matmuls);
    with one shared expert the shared SwiGLU adds on top."""
    T, d, I = 7, 256, 128
    rng = np.random.default_rng(5)
    u = torch.from_numpy(rng.standard_normal((T, d))).to(torch.bfloat16)
    ws = [torch.from_numpy(rng.standard_normal(s) / math.sqrt(s[1])).to(torch.bfloat16)
          for s in ((I, d), (I, d), (d, I), (I, d), (I, d), (d, I))]
    cent = torch.from_numpy(rng.standard_normal((1, d))).to(torch.bfloat16)
    r = oracle.route(synth.bf16_bits(u), synth.bf16_bits(cent), np.zeros(1, np.float32), 1)
    np.testing.assert_array_equal(r["gate"], 1.0)
    ud = u.double()

    def ref_ffn(w1, w3, w2):
        return (F.silu(ud @ w1.double().T) * (ud @ w3.double().T)) @ w2.double().T

    routed = lambda e: _bits(ws[:3])
    out0 = oracle.layer_output(synth.bf16_bits(u), np.arange(T), r["idx"], r["gate"], routed, None, 0, 1)
    np.testing.assert_allclose(out0, (ud + ref_ffn(*ws[:3])).numpy(), rtol=0, atol=1e-11)
    out1 = oracle.layer_output(synth.bf16_bits(u), np.arange(T), r["idx"], r["gate"], routed,
                               lambda s: _bits(ws[3:]), 1, 1)
    np.testing.assert_allclose(out1, (ud + ref_ffn(*ws[:3]) + ref_ffn(*ws[3:])).numpy(), rtol=0, atol=1e-11)


# ----------------------------------------------------------------------------
# FP8 E4M3 codec and quantisers
def test_e4m3_code_table_and_roundtrip():
    """All 254 non-NaN codes (+-0 included) decode to the enumerated format
    values and re-encode to themselves; max finite is the printed 448."""
    gold = json.load(open(os.path.join(GOLDEN, "e4m3_format.json")))
    table = brute.e4m3_value_table()
    assert len(table) == 254
    codes = np.array(sorted(table), np.uint8)
    vals = oracle.e4m3_decode(codes)
    np.testing.assert_array_equal(vals, [table[int(cd)] for cd in codes])
    np.testing.assert_array_equal(oracle.e4m3_encode(vals), codes)
    assert max(table.values()) == gold["e4m3_max"]
    assert np.isnan(oracle.e4m3_decode(np.array([0x7F, 0xFF], np.uint8))).all()


def test_e4m3_encode_matches_library_and_bruteforce():
    rng = np.random.default_rng(3)
    x = np.concatenate([rng.standard_normal(4000) * 50, rng.standard_normal(2000) * 0.01,
                        rng.uniform(-447, 447, 2000)])
    got = oracle.e4m3_decode(oracle.e4m3_encode(x))
    lib = torch.from_numpy(x).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    np.testing.assert_array_equal(got, lib)
    for v in x[:300]:
        assert oracle.e4m3_decode(oracle.e4m3_encode(np.array([v])))[0] == brute.nearest_e4m3(float(v))


def test_e4m3_saturation_and_halfway_cases():
    enc = lambda v: int(oracle.e4m3_encode(np.array([v]))[0])
    assert enc(448.0) == 0x7E and enc(1e6) == 0x7E and enc(-500.0) == 0xFE and enc(460.0) == 0x7E
    assert enc(1.0625) == enc(1.0)        # halfway 1.0 | 1.125 -> even mantissa 0
    assert enc(1.1875) == enc(1.25)       # halfway 1.125 | 1.25 -> even mantissa 2
    assert enc(2.0 ** -10) == 0x00        # halfway 0 | 2^-9 -> 0
    assert enc(3 * 2.0 ** -10) == 0x02    # halfway 2^-9 | 2^-8 -> code 2
    assert enc(float("nan")) == 0x7F


def test_quantisers_scale_rule_and_error_bound():
    rng = np.random.default_rng(11)
    x = rng.standard_normal((6, 384)) * np.exp(rng.standard_normal((6, 1)))
    x[2, 128:256] = 0.0
    q, s = oracle.quant_1x128(x)
    for r in range(6):
        for g in range(3):
            amax = np.abs(x[r, 128 * g:128 * g + 128]).max()
            expect = np.float32(1.0) if amax == 0 else np.float32(np.float32(amax) / np.float32(448.0))
            assert s[r, g] == expect
    assert (q[2, 128:256] == 0).all()
    deq = oracle.dequant_1x128(q, s)
    sc = np.repeat(s.astype(np.float64), 128, 1)
    normal = np.abs(x) / sc >= 2.0 ** -6
    assert (np.abs(x - deq)[normal] <= 2.0 ** -4 * np.abs(x)[normal] * (1 + 1e-6)).all()
    assert (np.abs(x - deq)[~normal] <= 2.0 ** -10 * sc[~normal] * (1 + 1e-6)).all()
    w = rng.standard_normal((256, 384))
    qw, sw = oracle.quant_128x128(w)
    assert sw.shape == (2, 3)
    assert sw[1, 2] == np.float32(np.float32(np.abs(w[128:, 256:]).max()) / np.float32(448))


def test_quantisers_exact_on_representable_values():
    """x = (E4M3 value) * 2^j with a group maximum of exactly 448 * 2^j: the
    scale is 2^j and the codes come back unchanged."""
    rng = np.random.default_rng(7)
    codes = rng.integers(0, 0x7E + 1, size=(4, 256)).astype(np.uint8)
    codes[:, 0] = 0x7E
    codes[:, 128] = 0xFE
    sign = rng.integers(0, 2, size=codes.shape).astype(np.uint8) << 7
    codes = codes | sign
    pw = 2.0 ** rng.integers(-8, 8, size=(4, 1))
    x = oracle.e4m3_decode(codes) * pw
    q, s = oracle.quant_1x128(x)
    np.testing.assert_array_equal(q, codes)
    np.testing.assert_array_equal(s, np.repeat(pw, 2, 1).astype(np.float32))
    w = oracle.e4m3_decode(np.tile(codes, (32, 1))) * 0.25
    qw, sw = oracle.quant_128x128(w)
    np.testing.assert_array_equal(qw, np.tile(codes, (32, 1)))
    np.testing.assert_array_equal(sw, 0.25)


def test_fp8_ffn_is_exact_product_of_dequantised_operands():
    """The FP8 oracle's expert equals fp64 matmuls of the dequantised operands
    (the limit the FP32 promotion every 128 of K approaches)."""
    rng = np.random.default_rng(8)
    n, d, I = 5, 256, 256
    x = rng.standard_normal((n, d))
    w1, w3 = rng.standard_normal((I, d)) / 16, rng.standard_normal((I, d)) / 16
    w2 = rng.standard_normal((d, I)) / 16
    xq = oracle.fp8_roundtrip_1x128(x)
    w1q, w3q, w2q = (oracle.fp8_roundtrip_128x128(w) for w in (w1, w3, w2))
    y = oracle.swiglu(xq, w1q, w3q, w2q, h_quant=True)
    g = xq @ w1q.T
    h = g / (1 + np.exp(-g)) * (xq @ w3q.T)
    hq = oracle.fp8_roundtrip_1x128(h)
    np.testing.assert_allclose(y, hq @ w2q.T, rtol=1e-12, atol=1e-12)
    # and the quantised expert stays close to the unquantised one (rms error
    # of a few percent: 3 mantissa bits on every operand)
    y0 = oracle.swiglu(x, w1, w3, w2)
    assert np.sqrt(((y - y0) ** 2).mean() / (y0 ** 2).mean()) < 0.1


# ----------------------------------------------------------------------------
# bias update
def test_bias_update_sign_rule_fp32():
    """Overloaded experts drop by gamma, underloaded rise by gamma, an expert
    at the mean load keeps its bias; arithmetic in fp32."""
    counts = np.array([10, 2, 6, 6, 0], np.int32)    # T*k = 24, mean 24/5 = 4.8
    b = np.array([0.1, -0.2, 0.0, 1e-8, 3.0], np.float32)
    out = oracle.bias_update(counts, b, T=8, k=3, gamma=0.001)
    g = np.float32(0.001)
    np.testing.assert_array_equal(out, np.array([b[0] - g, b[1] + g, b[2] - g, b[3] - g, b[4] + g], np.float32))
    counts = np.array([4, 4, 4, 4], np.int32)        # every expert exactly at the mean
    np.testing.assert_array_equal(oracle.bias_update(counts, b[:4], T=4, k=4, gamma=0.001), b[:4])


def test_bias_update_lowers_imbalance_on_a_skewed_stream():
    """Applied step after step on a skewed synthetic stream, the update lowers
    the max/mean expert load (its purpose in ai.flicky.cc 2.1.2)."""
    cfg = synth.get_config("ragged", T=512, alpha=2.0, rho=0.6)
    c = synth.bf16_bits(synth.centroids(cfg))
    b = np.zeros(cfg.E, np.float32)
    ratios = []
    for step in range(40):
        u = synth.bf16_bits(synth.tokens(cfg, step=step))
        r = oracle.route(u, c, b, cfg.k)
        counts = np.bincount(r["idx"].ravel(), minlength=cfg.E).astype(np.int32)
        ratios.append(counts.max() / (cfg.T * cfg.k / cfg.E))
        b = oracle.bias_update(counts, b, cfg.T, cfg.k, gamma=0.01)
    assert np.mean(ratios[-5:]) < 0.8 * ratios[0]


# ----------------------------------------------------------------------------
# closed forms printed on the pages
def test_param_count_closed_forms():
    gold = json.load(open(os.path.join(GOLDEN, "v3_param_counts.json")))
    per = oracle.expert_param_count(gold["d"], gold["d_expert"])
    assert per == 44_040_192
    total = gold["moe_layers"] * gold["experts_per_layer"] * per
    assert abs(total / 1e9 - gold["expert_params_total_billions_printed"]) < gold["printed_rounding_billions"]
    active = gold["moe_layers"] * gold["active_experts_per_layer"] * per
    assert abs(active / 1e9 - gold["active_expert_params_billions_printed"]) < gold["active_rounding_billions"]
    # 256 routed experts of one layer in bf16
    assert 256 * per * 2 == 22_548_578_304


def test_combine_matches_layer_assembly():
    """The combine over per-expert outputs equals the expert-major layer sum
    (itself pinned to the dense brute force above)."""
    cfg = synth.get_config("ragged")
    u, c, b, routed, shared = _tiny_layer(cfg)
    ub = synth.bf16_bits(u)
    r = oracle.route(ub, synth.bf16_bits(c), np.asarray(b), cfg.k)
    lay = oracle.dispatch_layout(r["idx"], cfg.E)
    x = oracle.bf16_to_f64(ub)
    y_perm = np.zeros((cfg.T * cfg.k, cfg.d))
    for e in range(cfg.E):
        rows = np.arange(lay["offsets"][e], lay["offsets"][e + 1])
        w1, w3, w2 = oracle.expert_operands(*_bits(routed[e]), fp8=False)
        y_perm[rows] = oracle.swiglu(x[lay["perm"][rows]], w1, w3, w2)
    ysh = np.stack([oracle.swiglu(x, *oracle.expert_operands(*_bits(w), fp8=False)) for w in shared])
    got = oracle.combine(ub, ysh, y_perm, lay["slot"], r["gate"])
    ref = oracle.layer_output(ub, np.arange(cfg.T), r["idx"], r["gate"], lambda e: _bits(routed[e]),
                              lambda s: _bits(shared[s]), cfg.n_shared, cfg.E)
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12 * np.abs(ref).max())


# ----------------------------------------------------------------------------
# the FP8 layer against its own dense statement
def test_e4m3_round_matches_exhaustive_search():
    """The dense FP8 statement's vectorised rounding equals the exhaustive
    nearest-value search, halfway cases and saturation included."""
    rng = np.random.default_rng(21)
    table = brute.e4m3_value_table()
    pos = sorted(v for c, v in table.items() if c < 0x80)
    mids = [(a + b) / 2 for a, b in zip(pos[:-1], pos[1:])]           # every halfway point
    x = np.concatenate([rng.standard_normal(1500) * 40, rng.standard_normal(500) * 1e-3,
                        np.array(mids), -np.array(mids[::7]), [448.0, 460.0, 1e6, -1e6, 0.0]])
    got = brute.e4m3_round(x)
    ref = np.array([brute.nearest_e4m3(float(v)) for v in x])
    np.testing.assert_array_equal(got, ref)


@pytest.mark.parametrize("name", ["tiny_fp8", "ragged_fp8"])
def test_fp8_layer_equals_dense_fp8_statement(name):
    """layer_output(fp8=True) -- which operands are quantised, the residual,
    the gates -- against the dense all-experts-then-mask FP8 statement."""
    cfg = synth.get_config(name)
    b = np.asarray(synth.normal_f32(4243, (cfg.E,), 0.02))
    u, c, _, routed, shared = _tiny_layer(cfg)
    r = oracle.route(synth.bf16_bits(u), synth.bf16_bits(c), b, cfg.k)
    out = oracle.layer_output(synth.bf16_bits(u), np.arange(cfg.T), r["idx"], r["gate"],
                              lambda e: _bits(routed[e]), lambda s: _bits(shared[s]), cfg.n_shared, cfg.E, fp8=True)
    f = lambda ws: tuple(w.double().numpy() for w in ws)
    dense = brute.dense_layer_fp8(u.double().numpy(), c.double().numpy(), b, cfg.k,
                                  [f(w) for w in routed], [f(w) for w in shared])
    np.testing.assert_allclose(r["gate"], np.take_along_axis(dense["g"], r["idx"].astype(np.int64), 1),
                               rtol=0, atol=1e-15)
    scale = np.abs(dense["out"]).max()
    np.testing.assert_allclose(out, dense["out"], rtol=0, atol=1e-12 * scale)


def test_fp8_dense_statement_catches_planted_assembly_slips(monkeypatch):
    """Slips planted in the oracle's FP8 assembly move it far from the dense
    statement, so the comparison above would catch them: a quantised residual,
    shared experts on the unquantised u, h left unquantised, weights left
    unquantised."""
    cfg = synth.get_config("ragged_fp8")
    b = np.asarray(synth.normal_f32(4243, (cfg.E,), 0.02))
    u, c, _, routed, shared = _tiny_layer(cfg)
    ub = synth.bf16_bits(u)
    r = oracle.route(ub, synth.bf16_bits(c), b, cfg.k)
    f = lambda ws: tuple(w.double().numpy() for w in ws)
    dense = brute.dense_layer_fp8(u.double().numpy(), c.double().numpy(), b, cfg.k,
                                  [f(w) for w in routed], [f(w) for w in shared])["out"]
    scale = np.abs(dense).max()
    args = (ub, np.arange(cfg.T), r["idx"], r["gate"], lambda e: _bits(routed[e]), lambda s: _bits(shared[s]),
            cfg.n_shared, cfg.E)
    good = oracle.layer_output(*args, fp8=True)
    assert np.abs(good - dense).max() <= 1e-12 * scale
    x = oracle.bf16_to_f64(ub)
    slips = {"quantised residual": good - x + oracle.fp8_roundtrip_1x128(x)}
    w_sh = oracle.expert_operands(*_bits(shared[0]), fp8=True)
    slips["shared on unquantised u"] = (good - oracle.swiglu(oracle.fp8_roundtrip_1x128(x), *w_sh, h_quant=True)
                                        + oracle.swiglu(x, *w_sh, h_quant=True))
    real_swiglu, real_ops = oracle.swiglu, oracle.expert_operands
    monkeypatch.setattr(oracle, "swiglu", lambda *a, h_quant=False: real_swiglu(*a, h_quant=False))
    slips["h unquantised"] = oracle.layer_output(*args, fp8=True)
    monkeypatch.setattr(oracle, "swiglu", real_swiglu)
    monkeypatch.setattr(oracle, "expert_operands", lambda w1, w3, w2, fp8: real_ops(w1, w3, w2, False))
    slips["weights unquantised"] = oracle.layer_output(*args, fp8=True)
    for what, bad in slips.items():
        assert np.abs(bad - dense).max() > 1e-4 * scale, what


@pytest.mark.parametrize("name", ["tiny", "ragged", "tiny_fp8", "ragged_fp8"])
def test_expert_rows_assemble_to_layer_output(name):
    """expert_rows keeps the expert outputs apart; combined with the gates
    they give layer_output (itself pinned to the dense statements)."""
    cfg = synth.get_config(name)
    u, c, b, routed, shared = _tiny_layer(cfg)
    ub = synth.bf16_bits(u)
    r = oracle.route(ub, synth.bf16_bits(c), np.asarray(b), cfg.k)
    fp8 = cfg.prec == "fp8"
    tokens = np.arange(0, cfg.T, 3)
    args = (ub, tokens, r["idx"][tokens], r["gate"][tokens], lambda e: _bits(routed[e]),
            lambda s: _bits(shared[s]), cfg.n_shared, cfg.E)
    y, ysh = oracle.expert_rows(*args[:3], *args[4:], fp8=fp8)
    n, k = len(tokens), cfg.k
    got = oracle.combine(ub[tokens], ysh, y.reshape(n * k, cfg.d), np.arange(n * k).reshape(n, k),
                         r["gate"][tokens])
    ref = oracle.layer_output(*args, fp8=fp8)
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12 * np.abs(ref).max())


# ----------------------------------------------------------------------------
# node-limited routing (ai.flicky.cc 2.1.2: a token goes to at most 4 nodes)
@pytest.mark.parametrize("groups,limit,k", [(8, 2, 4), (8, 3, 6), (4, 1, 3), (10, 4, 8)])
def test_node_limited_selection_matches_node_ranking_statement(groups, limit, k):
    """The oracle's greedy selection under a node budget equals the statement
    'keep the `limit` nodes with the best experts, then top-k inside them',
    every token spans at most `limit` nodes, and the gates stay normalised
    over the selected unbiased affinities."""
    E = 40 if groups == 10 else 32
    cfg = synth.get_config("ragged", E=E, k=k)
    u, c = synth.tokens(cfg), synth.centroids(cfg)
    b = np.asarray(synth.normal_f32(99, (E,), 0.03))
    r = oracle.route(synth.bf16_bits(u), synth.bf16_bits(c), b, k, want_all=True, groups=groups, group_limit=limit)
    score = r["s_all"] + b.astype(np.float64)
    gs = E // groups
    for t in range(cfg.T):
        assert r["idx"][t].tolist() == brute.node_limited_topk(score[t], k, groups, limit)
        assert len({int(e) // gs for e in r["idx"][t]}) <= limit
    sel = np.take_along_axis(r["s_all"], r["idx"].astype(np.int64), 1)
    np.testing.assert_allclose(r["gate"], sel / sel.sum(1, keepdims=True), rtol=0, atol=1e-12)
    # the limit binds somewhere (else this test says nothing about it)
    free = oracle.route(synth.bf16_bits(u), synth.bf16_bits(c), b, k)
    assert (np.sort(free["idx"], 1) != np.sort(r["idx"], 1)).any()


def test_node_limit_that_cannot_bind_changes_nothing():
    """limit = groups, or a limit of at least k nodes: the plain top-k."""
    cfg = synth.get_config("ragged")
    u, c = synth.bf16_bits(synth.tokens(cfg)), synth.bf16_bits(synth.centroids(cfg))
    b = np.asarray(synth.bias(cfg))
    free = oracle.route(u, c, b, cfg.k)
    for groups, limit in ((5, 5), (20, cfg.k), (10, cfg.k + 1)):
        r = oracle.route(u, c, b, cfg.k, groups=groups, group_limit=limit)
        np.testing.assert_array_equal(r["idx"], free["idx"])
        np.testing.assert_array_equal(r["gate"], free["gate"])


# ----------------------------------------------------------------------------
# UE8M0 scales (ai.flicky.cc, continuation of 3.5: DeepSeek-V3.1's FP8 with
# UE8M0 scales -- a scale is a bare power of two)
def test_ue8m0_scales_are_the_next_power_of_two():
    rng = np.random.default_rng(31)
    x = rng.standard_normal((8, 512)) * np.exp2(rng.integers(-12, 12, (8, 1)))
    x[3, :128] = 0.0
    x[5, 128:256] = 0.0
    x[5, 130] = 448.0 * 2.0 ** -3          # amax exactly 448 * 2^-3: the scale is 2^-3 itself
    q, s = oracle.quant_1x128(x, pow2=True)
    _, s_amax = oracle.quant_1x128(x)
    m, e = np.frexp(s.astype(np.float64))
    assert (m == 0.5).all()                                  # every scale a power of two
    assert (s >= s_amax).all() and (s < 2 * s_amax).all()    # the smallest one >= amax/448
    assert s[3, 0] == 1.0 and s[5, 1] == np.float32(2.0 ** -3)
    assert (np.abs(oracle.e4m3_decode(q)) <= 448).all()
    deq = oracle.dequant_1x128(q, s)
    sc = np.repeat(s.astype(np.float64), 128, 1)
    normal = np.abs(x) / sc >= 2.0 ** -6
    assert (np.abs(x - deq)[normal] <= 2.0 ** -4 * np.abs(x)[normal] * (1 + 1e-6)).all()
    w = rng.standard_normal((256, 384)) / 20
    _, sw = oracle.quant_128x128(w, pow2=True)
    assert (np.frexp(sw.astype(np.float64))[0] == 0.5).all()


def test_ue8m0_quantisers_match_the_dense_statement():
    rng = np.random.default_rng(32)
    x = rng.standard_normal((6, 384)) * np.exp2(rng.integers(-8, 8, (6, 1)))
    np.testing.assert_array_equal(oracle.fp8_roundtrip_1x128(x, pow2=True), brute.quant_dequant(x, 1, 128, True))
    w = rng.standard_normal((256, 256)) * 0.03
    np.testing.assert_array_equal(oracle.fp8_roundtrip_128x128(w, pow2=True), brute.quant_dequant(w, 128, 128, True))
    # and the pow2 rule of the dense statement itself, on hand-picked values
    np.testing.assert_array_equal(brute.pow2_at_least(np.array([1.0, 1.5, 0.25, 0.3, 3.0], np.float32)),
                                  np.array([1.0, 2.0, 0.25, 0.5, 4.0], np.float32))


@pytest.mark.parametrize("name", ["tiny_fp8", "ragged_fp8"])
def test_ue8m0_layer_equals_dense_statement(name):
    cfg = synth.get_config(name)
    b = np.asarray(synth.normal_f32(4244, (cfg.E,), 0.02))
    u, c, _, routed, shared = _tiny_layer(cfg)
    r = oracle.route(synth.bf16_bits(u), synth.bf16_bits(c), b, cfg.k)
    out = oracle.layer_output(synth.bf16_bits(u), np.arange(cfg.T), r["idx"], r["gate"],
                              lambda e: _bits(routed[e]), lambda s: _bits(shared[s]), cfg.n_shared, cfg.E,
                              fp8="ue8m0")
    f = lambda ws: tuple(w.double().numpy() for w in ws)
    dense = brute.dense_layer_fp8(u.double().numpy(), c.double().numpy(), b, cfg.k,
                                  [f(w) for w in routed], [f(w) for w in shared], pow2=True)
    scale = np.abs(dense["out"]).max()
    np.testing.assert_allclose(out, dense["out"], rtol=0, atol=1e-12 * scale)
    # a different quantisation from the amax/448 one (else the test says nothing)
    other = oracle.layer_output(synth.bf16_bits(u), np.arange(cfg.T), r["idx"], r["gate"],
                                lambda e: _bits(routed[e]), lambda s: _bits(shared[s]), cfg.n_shared, cfg.E, fp8=True)
    assert np.abs(other - out).max() > 1e-6 * scale


def test_reciprocal_codes_reading():
    """quant_1x128(recip=True) takes the codes from x * (1/s): with UE8M0
    scales 1/s is exact and the codes are those of x / s; with amax/448 scales
    they agree except where the two fp32 values straddle an E4M3 rounding
    boundary, and there by one code step."""
    rng = np.random.default_rng(17)
    x = rng.standard_normal((64, 1024)) * np.exp(rng.standard_normal((64, 1)))
    q_p, s_p = oracle.quant_1x128(x, pow2=True)
    q_pr, s_pr = oracle.quant_1x128(x, pow2=True, recip=True)
    assert np.array_equal(q_p, q_pr) and np.array_equal(s_p, s_pr)
    q, s = oracle.quant_1x128(x)
    q_r, s_r = oracle.quant_1x128(x, recip=True)
    assert np.array_equal(s, s_r)
    diff = q != q_r
    assert diff.mean() < 1e-3
    v, v_r = oracle.e4m3_decode(q[diff]), oracle.e4m3_decode(q_r[diff])
    # adjacent codes of the same sign: their magnitudes differ by one step
    assert np.all(np.sign(v) == np.sign(v_r))
    assert np.all(np.abs(q[diff].astype(int) - q_r[diff].astype(int)) == 1)
    # and brute's statement of the same reading agrees with the oracle's codes
    np.testing.assert_array_equal(brute.quant_dequant(x, 1, 128, recip=True), oracle.dequant_1x128(q_r, s_r))
