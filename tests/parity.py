"""Shared helpers of the GPU parity tests: build a layer from seeded inputs,
run the CUDA path through the C ABI, and compare with the CPU oracle."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import synth
from mixture_experts_layer_87_b300 import MoELayer

NEAR_TIE = 1e-4          # oracle gap between the k-th and (k+1)-th biased score
TOL = {"bf16": 2e-2, "fp8": 6e-2, "fp8_ue8m0": 6e-2}   # max|err| / rms(ref) on h'
# max|err| / rms(ref) on the routed expert outputs y = FFN_e(x), compared row
# by row with the oracle's expert.  y has no residual to hide behind, and it is
# stored as bf16: that rounding alone is up to 2^-9 |y|, about 1% of rms(y) at
# the largest elements (max/rms ~ 5 over the ~10^6 outputs of a check), and
# the bf16 rounding of h before the down product adds ~0.5% more there -- so
# bf16 is held to 3e-2.  FP8 (h quantised to E4M3 on both sides, codes that may
# differ by one step where the fp32 and fp64 h straddle a rounding boundary)
# keeps the layer's 6e-2.
Y_TOL = {"bf16": 3e-2, "fp8": 6e-2, "fp8_ue8m0": 6e-2}


class HostLayer:
    """Seeded inputs of one config, kept on the host as bf16 bit patterns."""

    def __init__(self, cfg, keep_weights=True):
        self.cfg = cfg
        self.cent = synth.centroids(cfg)
        self.bias = synth.bias(cfg)
        self.keep = keep_weights
        self._routed = {}
        self._shared = {}

    def routed(self, e):
        if e in self._routed:
            return self._routed[e]
        w = synth.expert_weights(self.cfg, e)
        if self.keep:
            self._routed[e] = w
        return w

    def shared(self, s):
        if s in self._shared:
            return self._shared[s]
        w = synth.expert_weights(self.cfg, s, shared=True)
        if self.keep:
            self._shared[s] = w
        return w

    def routed_bits(self, e):
        return tuple(synth.bf16_bits(w) for w in self.routed(e))

    def shared_bits(self, s):
        return tuple(synth.bf16_bits(w) for w in self.shared(s))

    def device_layer(self, T=None) -> MoELayer:
        c = self.cfg
        layer = MoELayer(c.T if T is None else T, c.d, c.E, c.k, c.n_shared, c.inter, c.prec,
                         route_groups=c.route_groups, route_group_limit=c.route_group_limit)
        layer.set_centroids(self.cent)
        for e in range(c.E):
            layer.load_expert(e, *self.routed(e))
        for s in range(c.n_shared):
            layer.load_expert(s, *self.shared(s), shared=True)
        return layer


def check_selection(idx_gpu: np.ndarray, r: dict, bias: np.ndarray, k: int, groups: int = 0, limit: int = 0):
    """GPU selection vs oracle: identical sets except on near-tie tokens, where
    the GPU may pick any experts within NEAR_TIE of the k-th score (and must
    keep every expert clearly above it).  With node-limited routing (groups >
    0) every selection spans at most `limit` nodes, and a near-tie selection
    must score within k * NEAR_TIE of the oracle's in total (a tie between two
    nodes can swap every expert of one for the other's).  Returns the near-tie
    token list."""
    T = idx_gpu.shape[0]
    score = r["s_all"] + bias.astype(np.float64)[None, :]
    gs = score.shape[1] // groups if groups else 0
    ties = []
    for t in range(T):
        g = sorted(idx_gpu[t].tolist())
        o = sorted(r["idx"][t].tolist())
        assert len(set(g)) == k, f"token {t}: duplicate experts {g}"
        if groups:
            assert len({e // gs for e in g}) <= limit, f"token {t}: experts {g} on more than {limit} nodes"
        if r["gap"][t] >= NEAR_TIE:
            assert g == o, f"token {t}: gpu {g} oracle {o} gap {r['gap'][t]}"
        elif groups:
            ties.append(t)
            assert score[t, g].sum() >= score[t, o].sum() - k * NEAR_TIE, f"token {t}: gpu pick far from the best"
        else:
            ties.append(t)
            kth = score[t, r["idx"][t, -1]]
            assert all(score[t, e] >= kth - NEAR_TIE for e in g), f"token {t}: gpu pick outside near-tie set"
            must = [e for e in range(score.shape[1]) if score[t, e] > kth + NEAR_TIE]
            assert set(must) <= set(g), f"token {t}: clear winner dropped"
    return ties


def rel_err(got: np.ndarray, ref: np.ndarray) -> float:
    return float(np.abs(got - ref).max() / np.sqrt((ref ** 2).mean()))


def bf16_to_np(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def chunk_covering_tokens(idx: np.ndarray, E: int, chunk: int = 128, base=()) -> np.ndarray:
    """Tokens such that every (expert, chunk of `chunk` permuted rows) of the
    grouped GEMMs holds at least one of their rows -- every expert's last,
    ragged chunk included -- picked greedily (most uncovered chunks first),
    starting from the tokens in `base`.  The expert GEMMs hand out work items
    (expert, weight block, token chunk); a checked row of a chunk checks every
    weight block of that chunk, so this sample reaches every item."""
    T, k = idx.shape
    lay = oracle.dispatch_layout(idx, E)
    rank = lay["slot"] - lay["offsets"][idx]                   # row of (t, j) inside its expert
    n_ch = (lay["counts"] + chunk - 1) // chunk
    first = np.concatenate([[0], np.cumsum(n_ch)])
    item = first[idx] + rank // chunk                          # [T, k] chunk id of every pair
    covered = np.zeros(int(first[-1]), bool)
    chosen = list(dict.fromkeys(int(t) for t in base))
    for t in chosen:
        covered[item[t]] = True
    while not covered.all():
        gain = (~covered[item]).sum(1)
        t = int(np.argmax(gain))
        chosen.append(t)
        covered[item[t]] = True
    return np.array(sorted(chosen), np.int64)


def gpu_layer_pass(layer: MoELayer, u_dev: torch.Tensor, bias_dev: torch.Tensor) -> dict:
    """One moe_forward (with the loads), then the routing, dispatch and routed
    experts again through their own C-ABI calls (moe_route, moe_permute,
    moe_grouped_ffn over the experts' offsets), which run the same kernels and
    expose what the forward keeps inside its workspace: the selection, the
    permutation and the expert outputs y_perm.  Small results come back as
    numpy arrays; out and y_perm stay on the device."""
    from mixture_experts_layer_87_b300 import capi
    dev = u_dev.device
    T, E, k, d = layer.T, layer.E, layer.k, layer.d
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    out = layer.forward(u_dev, bias_dev, counts=counts)
    assert layer.status() == 0
    dm = layer.dims
    idx = torch.empty((T, k), dtype=torch.int32, device=dev)
    gate = torch.empty((T, k), dtype=torch.float32, device=dev)
    cnt = torch.empty(E, dtype=torch.int32, device=dev)
    capi.moe_route(dm, u_dev, layer.centroids, bias_dev, idx, gate, cnt, layer.ws)
    R = T * k
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    perm = torch.empty(R, dtype=torch.int32, device=dev)
    slot = torch.empty((T, k), dtype=torch.int32, device=dev)
    x = torch.empty((R, d), dtype=torch.uint8 if layer.fp8 else torch.bfloat16, device=dev)
    xs = torch.empty((d // 128, R), dtype=torch.float32, device=dev) if layer.fp8 else None
    capi.moe_permute(dm, idx, u_dev, offsets, perm, slot, x, xs, layer.ws)
    y = torch.empty((R, d), dtype=torch.bfloat16, device=dev)
    capi.moe_grouped_ffn(dm, E, R, offsets, x, xs, layer.w13, layer.w13_scale, layer.w2, layer.w2_scale, y,
                         layer.ws)
    assert capi.moe_read_device_status(layer.ws) == 0
    return dict(out=out, y=y, counts_dev=counts, counts=counts.cpu().numpy(), cnt=cnt.cpu().numpy(), idx=idx.cpu().numpy(),
                gate=gate.cpu().numpy(), offsets=offsets.cpu().numpy(), perm=perm.cpu().numpy(),
                slot=slot.cpu().numpy())


def check_routing_and_dispatch(res: dict, r: dict, bias: np.ndarray, E: int, k: int, groups: int = 0,
                               limit: int = 0) -> list:
    """Selection against the oracle (near-ties excepted), and the loads,
    offsets, permutation and slots of the GPU's own selection bit for bit
    against the oracle's canonical dropless layout.  Returns the near-ties."""
    ties = check_selection(res["idx"], r, bias, k, groups, limit)
    np.testing.assert_array_equal(res["counts"], res["cnt"])
    lay = oracle.dispatch_layout(res["idx"], E)
    np.testing.assert_array_equal(res["counts"], lay["counts"])
    np.testing.assert_array_equal(res["offsets"], lay["offsets"])
    np.testing.assert_array_equal(res["perm"], lay["perm"])
    np.testing.assert_array_equal(res["slot"], lay["slot"])
    if not ties:
        np.testing.assert_array_equal(res["counts"], np.bincount(r["idx"].ravel(), minlength=E))
    return ties


def oracle_rows(host: HostLayer, ub_rows: np.ndarray, idx_rows: np.ndarray, gate_rows: np.ndarray):
    """The oracle's h' and routed expert outputs y [n, k, d] of the given rows
    of u (bf16 bits) with the given selection and gates, one pass over the
    experts."""
    c = host.cfg
    n, k = idx_rows.shape
    y, ysh = oracle.expert_rows(ub_rows, np.arange(n), idx_rows, host.routed_bits, host.shared_bits, c.n_shared,
                                c.E, fp8=c.oracle_fp8)
    h = oracle.combine(ub_rows, ysh, y.reshape(n * k, -1), np.arange(n * k).reshape(n, k), gate_rows)
    return h, y


def gpu_rows(res: dict, tokens: np.ndarray):
    """h' and y_perm rows [n, k, d] of the given tokens from a gpu_layer_pass."""
    t = torch.from_numpy(np.asarray(tokens, np.int64)).to(res["out"].device)
    h = bf16_to_np(res["out"][t])
    s = torch.from_numpy(res["slot"][tokens].astype(np.int64).ravel()).to(res["y"].device)
    y = bf16_to_np(res["y"][s]).reshape(len(tokens), res["slot"].shape[1], -1)
    return h, y
