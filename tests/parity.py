"""Shared helpers of the GPU parity tests: build a layer from seeded inputs,
run the CUDA path through the C ABI, and compare with the CPU oracle."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import synth
from mixture_experts_layer_87_b300 import MoELayer

NEAR_TIE = 1e-4          # oracle gap between the k-th and (k+1)-th biased score
TOL = {"bf16": 2e-2, "fp8": 6e-2}   # max|err| / rms(ref) on h'


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
        layer = MoELayer(c.T if T is None else T, c.d, c.E, c.k, c.n_shared, c.inter, c.prec)
        layer.set_centroids(self.cent)
        for e in range(c.E):
            layer.load_expert(e, *self.routed(e))
        for s in range(c.n_shared):
            layer.load_expert(s, *self.shared(s), shared=True)
        return layer


def check_selection(idx_gpu: np.ndarray, r: dict, bias: np.ndarray, k: int):
    """GPU selection vs oracle: identical sets except on near-tie tokens, where
    the GPU may pick any experts within NEAR_TIE of the k-th score (and must
    keep every expert clearly above it).  Returns the near-tie token list."""
    T = idx_gpu.shape[0]
    score = r["s_all"] + bias.astype(np.float64)[None, :]
    ties = []
    for t in range(T):
        g = sorted(idx_gpu[t].tolist())
        o = sorted(r["idx"][t].tolist())
        assert len(set(g)) == k, f"token {t}: duplicate experts {g}"
        if r["gap"][t] >= NEAR_TIE:
            assert g == o, f"token {t}: gpu {g} oracle {o} gap {r['gap'][t]}"
        else:
            ties.append(t)
            kth = score[t, r["idx"][t, -1]]
            assert all(score[t, e] >= kth - NEAR_TIE for e in g), f"token {t}: gpu pick outside near-tie set"
            must = [e for e in range(score.shape[1]) if score[t, e] > kth + NEAR_TIE]
            assert set(must) <= set(g), f"token {t}: clear winner dropped"
    return ties


def rel_err(got: np.ndarray, ref: np.ndarray) -> float:
    return float(np.abs(got - ref).max() / np.sqrt((ref ** 2).mean()))


def ffn_rel_err(got: np.ndarray, ref: np.ndarray, u: np.ndarray) -> float:
    """max|err|/rms on the FFN part h' - u, with the unavoidable rounding of
    the bf16 output taken out.  h' is stored as bf16 and dominated by u, so
    half a bf16 ulp of h' can be a large share of the (much smaller) FFN part;
    that rounding is the output format, not an error of the computation."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    mag = np.maximum(np.abs(ref), 2.0 ** -126)
    half_ulp = np.exp2(np.floor(np.log2(mag)) - 8)       # bf16: 8 significant bits
    excess = np.maximum(np.abs(got - ref) - half_ulp, 0.0)
    return float(excess.max() / np.sqrt(np.mean((ref - np.asarray(u, np.float64)) ** 2)))


def bf16_to_np(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)
