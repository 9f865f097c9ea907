"""Seeded synthetic inputs for the DeepSeekMoE layer.

This module draws inputs and nothing else: it holds none of the layer's
arithmetic.  The CPU oracle and the CUDA library both receive byte-identical
copies of what it returns, so a parity test compares two implementations of
the layer on the same bytes.

Workload recipe (the pages name no dataset, so every input is synthetic):
  * expert weights W1, W3 ~ N(0, std 1/sqrt(d)); W2 ~ N(0, std 1/sqrt(I));
    centroids e_i ~ N(0, std 1/sqrt(d)); all rounded to bf16 (RNE);
  * bias b_i ~ N(0, std 0.01) in fp32, or zero where the config says so;
  * tokens either u ~ N(0, 1) or "clustered": 32 centres c_j ~ N(0, I_d),
    a cluster z_t drawn with weights p_j proportional to j^-alpha, and
    u_t = sqrt(rho) c_{z_t} + sqrt(1-rho) eps_t, so every coordinate stays
    close to N(0, 1) while tokens of one cluster prefer the same experts.
Every tensor has its own 64-bit key derived from (config seed, tensor tag,
expert / step index), so any one expert can be regenerated on its own.
"""
from __future__ import annotations

import ctypes
import json
import math
import os
import subprocess
from dataclasses import dataclass, field, replace

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "libsynth.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile gen.c into libsynth.so (host code, gcc + OpenMP)."""
    src = os.path.join(_HERE, "gen.c")
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(src):
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", src, "-o", _SO, "-lm"])
    return _SO


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_SO)
        u64, i64, f32, vp = ctypes.c_uint64, ctypes.c_int64, ctypes.c_float, ctypes.c_void_p
        lib.synth_key.argtypes = [u64, u64]
        lib.synth_key.restype = u64
        lib.synth_normal_bf16.argtypes = [u64, i64, f32, vp]
        lib.synth_normal_f32.argtypes = [u64, i64, f32, vp]
        lib.synth_uniform_f64.argtypes = [u64, i64, vp]
        lib.synth_clustered_bf16.argtypes = [u64, i64, i64, vp, vp, f32, vp]
        _lib = lib
    return _lib


# ----------------------------------------------------------------------------
# keys
_TAGS = {"centroids": 1, "bias": 2, "w1": 3, "w3": 4, "w2": 5, "ws1": 6, "ws3": 7, "ws2": 8,
         "tokens": 9, "centres": 10, "cluster": 11}


def key(seed: int, tag: str, index: int = 0) -> int:
    lib = _load()
    k = lib.synth_key(seed & 0xFFFFFFFFFFFFFFFF, _TAGS[tag])
    return lib.synth_key(k, index & 0xFFFFFFFFFFFFFFFF)


def normal_bf16(k: int, shape, std: float) -> torch.Tensor:
    out = torch.empty(shape, dtype=torch.bfloat16)
    _load().synth_normal_bf16(k, out.numel(), std, out.data_ptr())
    return out


def normal_f32(k: int, shape, std: float) -> torch.Tensor:
    out = torch.empty(shape, dtype=torch.float32)
    _load().synth_normal_f32(k, out.numel(), std, out.data_ptr())
    return out


def uniform_f64(k: int, n: int) -> np.ndarray:
    out = np.empty(n, dtype=np.float64)
    _load().synth_uniform_f64(k, n, out.ctypes.data)
    return out


# ----------------------------------------------------------------------------
# configurations
@dataclass(frozen=True)
class LayerConfig:
    name: str
    T: int            # tokens per step
    d: int            # hidden size
    E: int            # routed experts
    k: int            # routed experts per token
    n_shared: int     # shared experts
    inter: int        # SwiGLU intermediate size of every expert
    prec: str = "bf16"         # "bf16" | "fp8"
    bias: str = "normal"       # "zero" | "normal" (std 0.01)
    tokens: str = "clustered"  # "normal" | "clustered"
    rho: float = 0.0           # clustered tokens: share of the centre
    alpha: float = 1.0         # clustered tokens: Zipf exponent of cluster weights
    n_clusters: int = 32
    steps: int = 1             # >1: decode loop with the bias update between steps
    gamma: float = 0.001       # bias update speed
    seed: int = 0
    route_groups: int = 0      # >0: experts on this many nodes of E/route_groups consecutive experts ...
    route_group_limit: int = 0 # ... and a token's experts on at most this many of them

    @property
    def rows(self) -> int:
        return self.T * self.k

    @property
    def is_fp8(self) -> bool:
        """E4M3 expert GEMMs (amax/448 scales, or UE8M0 power-of-two scales)."""
        return self.prec in ("fp8", "fp8_ue8m0")

    @property
    def oracle_fp8(self):
        """The oracle's fp8 argument for this precision: False, True or "ue8m0"."""
        return {"bf16": False, "fp8": True, "fp8_ue8m0": "ue8m0"}[self.prec]


# (rho, alpha) of the clustered stream, chosen once with the oracle router so
# that the 8192-token V3 batch has a max/mean expert load close to 4
# (oracle/calibrate.py writes calibration.json; this module only reads it).
with open(os.path.join(_HERE, "calibration.json")) as _f:
    CALIBRATION = json.load(_f)
V3_RHO, V3_ALPHA = float(CALIBRATION["rho"]), float(CALIBRATION["alpha"])
DECODE_ALPHA = float(CALIBRATION["decode_alpha"])

CONFIGS = {
    "tiny": LayerConfig("tiny", T=64, d=256, E=16, k=4, n_shared=1, inter=128,
                        bias="zero", tokens="normal"),
    "mid": LayerConfig("mid", T=4096, d=2048, E=64, k=6, n_shared=2, inter=1408,
                       rho=V3_RHO, alpha=V3_ALPHA),
    "v3": LayerConfig("v3", T=8192, d=7168, E=256, k=8, n_shared=1, inter=2048,
                      rho=V3_RHO, alpha=V3_ALPHA),
    "v3_fp8": LayerConfig("v3_fp8", T=8192, d=7168, E=256, k=8, n_shared=1, inter=2048,
                          prec="fp8", rho=V3_RHO, alpha=V3_ALPHA),
    "decode": LayerConfig("decode", T=256, d=7168, E=256, k=8, n_shared=1, inter=2048,
                          prec="fp8", bias="zero", rho=V3_RHO, alpha=DECODE_ALPHA, steps=50),
    # V3 expert shapes with 32 experts (mean 256 rows per expert, as at V3):
    # the workload ncu captures, small enough to hold on the device many times.
    "v3_slice": LayerConfig("v3_slice", T=1024, d=7168, E=32, k=8, n_shared=1, inter=2048,
                            rho=V3_RHO, alpha=V3_ALPHA),
    "v3_slice_fp8": LayerConfig("v3_slice_fp8", T=1024, d=7168, E=32, k=8, n_shared=1, inter=2048,
                                prec="fp8", rho=V3_RHO, alpha=V3_ALPHA),
    # V3 token shapes (router, dispatch and combine are V3-sized: T, d, E and k
    # are V3's) with tiny experts, so the whole layer fits a few GB: the
    # workload ncu captures the bandwidth-bound kernels on.
    "v3_tokens": LayerConfig("v3_tokens", T=8192, d=7168, E=256, k=8, n_shared=1, inter=128,
                             rho=V3_RHO, alpha=V3_ALPHA),
    "v3_tokens_fp8": LayerConfig("v3_tokens_fp8", T=8192, d=7168, E=256, k=8, n_shared=1, inter=128,
                                 prec="fp8", rho=V3_RHO, alpha=V3_ALPHA),
    # Decode-shaped slice: 8 tokens per expert on average (as a V3 decode step
    # of 256 tokens over 256 experts) with 32 experts, for profiling.
    "decode_slice": LayerConfig("decode_slice", T=32, d=7168, E=32, k=8, n_shared=1, inter=2048,
                                prec="fp8", bias="zero", rho=V3_RHO, alpha=DECODE_ALPHA),
    # V3 expert shapes, 8 experts each chosen by all 256 tokens (256 rows per
    # expert, V3's mean): the backward's kernels at V3 shape on a few GB, for
    # profiling.
    "bwd_slice": LayerConfig("bwd_slice", T=256, d=7168, E=8, k=8, n_shared=1, inter=2048,
                             rho=V3_RHO, alpha=V3_ALPHA),
    # V3 with node-limited routing: 256 experts on 8 nodes of 32, a token's 8
    # experts on at most 4 nodes.
    "v3_nodes": LayerConfig("v3_nodes", T=8192, d=7168, E=256, k=8, n_shared=1, inter=2048,
                            rho=V3_RHO, alpha=V3_ALPHA, route_groups=8, route_group_limit=4),
    # Small parity shapes: several M/N/K tiles, ragged tails, odd expert counts.
    "ragged": LayerConfig("ragged", T=300, d=384, E=20, k=3, n_shared=1, inter=256,
                          rho=0.3, alpha=1.0),
    "ragged_fp8": LayerConfig("ragged_fp8", T=300, d=384, E=20, k=3, n_shared=1, inter=256,
                              prec="fp8", rho=0.3, alpha=1.0),
    "tiny_fp8": LayerConfig("tiny_fp8", T=64, d=256, E=16, k=4, n_shared=1, inter=128,
                            prec="fp8", bias="zero", tokens="normal"),
    # The FP8 scheme with UE8M0 (power-of-two) scales.
    "tiny_ue8m0": LayerConfig("tiny_ue8m0", T=64, d=256, E=16, k=4, n_shared=1, inter=128,
                              prec="fp8_ue8m0", bias="zero", tokens="normal"),
    "ragged_ue8m0": LayerConfig("ragged_ue8m0", T=300, d=384, E=20, k=3, n_shared=1, inter=256,
                                prec="fp8_ue8m0", rho=0.3, alpha=1.0),
    "v3_ue8m0": LayerConfig("v3_ue8m0", T=8192, d=7168, E=256, k=8, n_shared=1, inter=2048,
                            prec="fp8_ue8m0", rho=V3_RHO, alpha=V3_ALPHA),
}


def get_config(name: str, **overrides) -> LayerConfig:
    cfg = CONFIGS[name]
    return replace(cfg, **overrides) if overrides else cfg


# ----------------------------------------------------------------------------
# tensors of one layer instance
def centroids(cfg: LayerConfig) -> torch.Tensor:
    """Router centroids e_i, [E, d] bf16, std 1/sqrt(d)."""
    return normal_bf16(key(cfg.seed, "centroids"), (cfg.E, cfg.d), 1.0 / math.sqrt(cfg.d))


def bias(cfg: LayerConfig) -> torch.Tensor:
    """Per-expert selection bias b, [E] fp32."""
    if cfg.bias == "zero":
        return torch.zeros(cfg.E, dtype=torch.float32)
    return normal_f32(key(cfg.seed, "bias"), (cfg.E,), 0.01)


def expert_weights(cfg: LayerConfig, e: int, shared: bool = False):
    """(W1 [I,d], W3 [I,d], W2 [d,I]) bf16 of routed expert e (or shared expert e)."""
    t1, t3, t2 = ("ws1", "ws3", "ws2") if shared else ("w1", "w3", "w2")
    I, d = cfg.inter, cfg.d
    w1 = normal_bf16(key(cfg.seed, t1, e), (I, d), 1.0 / math.sqrt(d))
    w3 = normal_bf16(key(cfg.seed, t3, e), (I, d), 1.0 / math.sqrt(d))
    w2 = normal_bf16(key(cfg.seed, t2, e), (d, I), 1.0 / math.sqrt(I))
    return w1, w3, w2


def cluster_weights(n: int, alpha: float) -> np.ndarray:
    p = np.arange(1, n + 1, dtype=np.float64) ** (-alpha)
    return p / p.sum()


def tokens(cfg: LayerConfig, step: int = 0, T: int | None = None) -> torch.Tensor:
    """Layer input u, [T, d] bf16, for decode step `step` (0 for one-shot configs)."""
    T = cfg.T if T is None else T
    if cfg.tokens == "normal":
        return normal_bf16(key(cfg.seed, "tokens", step), (T, cfg.d), 1.0)
    centres = normal_f32(key(cfg.seed, "centres"), (cfg.n_clusters, cfg.d), 1.0)
    cdf = np.cumsum(cluster_weights(cfg.n_clusters, cfg.alpha))
    uz = uniform_f64(key(cfg.seed, "cluster", step), T)
    z = np.minimum(np.searchsorted(cdf, uz, side="right"), cfg.n_clusters - 1).astype(np.int32)
    out = torch.empty((T, cfg.d), dtype=torch.bfloat16)
    _load().synth_clustered_bf16(key(cfg.seed, "tokens", step), T, cfg.d, centres.data_ptr(),
                                 z.ctypes.data, float(cfg.rho), out.data_ptr())
    return out


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """Zero-copy uint16 view of a contiguous CPU bf16 tensor."""
    assert t.dtype == torch.bfloat16 and t.is_contiguous() and not t.is_cuda
    return t.view(torch.int16).numpy().view(np.uint16)
