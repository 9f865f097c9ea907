"""CPU oracle of the DeepSeekMoE layer forward -- TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` import this package.  It shares no code with the CUDA library
and never receives anything the CUDA library computed.  Its arithmetic lives
in ``moe_oracle.c`` (plain C, fp64 loops, OpenMP over rows); this file only
marshals arrays and writes out the parts of the method that are bookkeeping
(the canonical permutation, the expert-major assembly of h'_t).

Sources (the DeepSeek-V3 technical report as read on two web pages):
  * ai.flicky.cc "06 - DeepSeek-V3 reading", section 2.1.2 (layer equation,
    sigmoid affinity, bias-in-selection-only rule, gates normalised among the
    selected experts, bias update, dropless routing), section 3.3 (FP8 scheme:
    1x128 activation tiles, 128x128 weight blocks, E4M3, router kept in high
    precision), and the practice exercise (SwiGLU expert of three matrices);
  * xyznot.com "DeepSeek-V3 technical report", Method 2 (the same equations,
    with g' normalised into g).

Parity status: every function here is pinned by the CPU tests (closed forms,
a dense all-experts-then-mask brute force, library routines for the special
cases, the exhaustive FP8 code table).  The pages print no worked numerical
example, so absolute output values are pinned only through those checks.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile moe_oracle.c with gcc (-O2, OpenMP, no fast-math: IEEE semantics kept)."""
    src = os.path.join(_HERE, "moe_oracle.c")
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(src):
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", src, "-o", _SO, "-lm"])
    return _SO


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_SO)
        i64, i32, vp, f32 = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_float
        lib.oracle_bf16_to_f64.argtypes = [i64, vp, vp]
        lib.oracle_route.argtypes = [i64, i32, i32, i32, vp, vp, vp, vp, vp, vp, vp, vp]
        lib.oracle_route_limited.argtypes = [i64, i32, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, vp, vp]
        lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_decode.restype = ctypes.c_double
        lib.oracle_e4m3_encode.argtypes = [ctypes.c_double]
        lib.oracle_e4m3_encode.restype = ctypes.c_uint8
        lib.oracle_quant_1x128.argtypes = [i64, i32, vp, vp, vp, i32, i32]
        lib.oracle_quant_128x128.argtypes = [i64, i32, vp, vp, vp, i32]
        lib.oracle_dequant.argtypes = [i64, i32, vp, vp, i32, vp]
        lib.oracle_swiglu.argtypes = [i64, i32, i32, vp, vp, vp, vp, i32, vp]
        lib.oracle_bias_update.argtypes = [i32, i64, i32, vp, f32, vp]
        _lib = lib
    return _lib


def _c(a: np.ndarray, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


# ----------------------------------------------------------------------------
# conversions
def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns (uint16) to fp64."""
    bits = _c(bits, np.uint16)
    out = np.empty(bits.shape, np.float64)
    _load().oracle_bf16_to_f64(bits.size, bits.ctypes.data, out.ctypes.data)
    return out


# ----------------------------------------------------------------------------
# router
def route(u_bits: np.ndarray, cent_bits: np.ndarray, bias: np.ndarray, k: int, want_all: bool = False,
          groups: int = 0, group_limit: int = 0):
    """Sigmoid affinities, biased top-k, normalised gates (ai.flicky.cc 2.1.2).

    u_bits [T, d] and cent_bits [E, d] are bf16 bit patterns, bias [E] fp32.
    groups > 0: the experts sit on `groups` nodes of E/groups consecutive
    experts and a token's k experts may span at most `group_limit` of them
    (the same section: a token is sent to at most 4 nodes).
    Returns dict(idx [T,k] int32, s_sel [T,k], gate [T,k], gap [T], s_all [T,E]|None).
    """
    u_bits, cent_bits, bias = _c(u_bits, np.uint16), _c(cent_bits, np.uint16), _c(bias, np.float32)
    T, d = u_bits.shape
    E = cent_bits.shape[0]
    assert cent_bits.shape[1] == d and bias.shape == (E,) and 1 <= k <= E
    if groups:
        assert E % groups == 0 and 1 <= group_limit <= groups and group_limit * (E // groups) >= k
    idx = np.empty((T, k), np.int32)
    s_sel = np.empty((T, k), np.float64)
    gate = np.empty((T, k), np.float64)
    gap = np.empty(T, np.float64)
    s_all = np.empty((T, E), np.float64) if want_all else None
    _load().oracle_route_limited(T, d, E, k, int(groups), int(group_limit), u_bits.ctypes.data,
                                 cent_bits.ctypes.data, bias.ctypes.data, idx.ctypes.data, s_sel.ctypes.data,
                                 gate.ctypes.data, gap.ctypes.data, None if s_all is None else s_all.ctypes.data)
    return dict(idx=idx, s_sel=s_sel, gate=gate, gap=gap, s_all=s_all)


def gates_for(s_all: np.ndarray, idx: np.ndarray) -> np.ndarray:
    """g_{i,t} = s_{i,t} / sum over the given selection (xyznot.com Method 2)."""
    s = np.take_along_axis(s_all, idx.astype(np.int64), axis=1)
    return s / s.sum(axis=1, keepdims=True)


def dispatch_layout(idx: np.ndarray, E: int):
    """Counts, offsets and the canonical dropless permutation of a selection.

    Every (token, expert) pair gets one row (no token is dropped: ai.flicky.cc
    2.1.2).  Rows are grouped by expert ascending and, within an expert, by
    token ascending.  Returns counts [E], offsets [E+1], perm [T*k] (token of
    each permuted row) and slot [T,k] (permuted row of pair (t, j)).
    """
    T, k = idx.shape
    buckets = [[] for _ in range(E)]
    for t in range(T):
        for j in range(k):
            buckets[int(idx[t, j])].append((t, j))
    counts = np.array([len(b) for b in buckets], np.int32)
    offsets = np.zeros(E + 1, np.int32)
    offsets[1:] = np.cumsum(counts)
    perm = np.empty(T * k, np.int32)
    slot = np.empty((T, k), np.int32)
    r = 0
    for e in range(E):
        for (t, j) in buckets[e]:
            perm[r] = t
            slot[t, j] = r
            r += 1
    return dict(counts=counts, offsets=offsets, perm=perm, slot=slot)


# ----------------------------------------------------------------------------
# FP8 E4M3 (ai.flicky.cc 3.3)
def e4m3_encode(x: np.ndarray) -> np.ndarray:
    lib = _load()
    flat = np.asarray(x, np.float64).ravel()
    return np.array([lib.oracle_e4m3_encode(float(v)) for v in flat], np.uint8).reshape(np.shape(x))


def e4m3_decode(q: np.ndarray) -> np.ndarray:
    lib = _load()
    flat = np.asarray(q, np.uint8).ravel()
    table = np.array([lib.oracle_e4m3_decode(c) for c in range(256)], np.float64)
    return table[flat].reshape(np.shape(q))


def quant_1x128(x: np.ndarray, pow2: bool = False, recip: bool = False):
    """1 x 128 activation tiles along the last axis: (codes uint8, scales fp32 [rows, cols/128]).
    pow2: UE8M0 scales (amax/448 rounded up to a power of two).  recip: codes
    from x * (1/scale) in fp32 (one correctly rounded reciprocal per tile)
    instead of x / scale."""
    x = _c(x, np.float64)
    rows, cols = x.shape
    assert cols % 128 == 0
    q = np.empty((rows, cols), np.uint8)
    s = np.empty((rows, cols // 128), np.float32)
    _load().oracle_quant_1x128(rows, cols, x.ctypes.data, q.ctypes.data, s.ctypes.data, int(pow2), int(recip))
    return q, s


def quant_128x128(w: np.ndarray, pow2: bool = False):
    """128 x 128 weight blocks: (codes uint8, scales fp32 [rows/128, cols/128]).
    pow2: UE8M0 scales (amax/448 rounded up to a power of two)."""
    w = _c(w, np.float64)
    rows, cols = w.shape
    assert rows % 128 == 0 and cols % 128 == 0
    q = np.empty((rows, cols), np.uint8)
    s = np.empty((rows // 128, cols // 128), np.float32)
    _load().oracle_quant_128x128(rows, cols, w.ctypes.data, q.ctypes.data, s.ctypes.data, int(pow2))
    return q, s


def _dequant(q: np.ndarray, s: np.ndarray, block_rows: int) -> np.ndarray:
    q, s = _c(q, np.uint8), _c(s, np.float32)
    rows, cols = q.shape
    out = np.empty((rows, cols), np.float64)
    _load().oracle_dequant(rows, cols, q.ctypes.data, s.ctypes.data, block_rows, out.ctypes.data)
    return out


def dequant_1x128(q: np.ndarray, s: np.ndarray) -> np.ndarray:
    """E4M3 value of every code times its 1 x 128 tile's scale (fp64)."""
    return _dequant(q, s, 1)


def dequant_128x128(q: np.ndarray, s: np.ndarray) -> np.ndarray:
    """E4M3 value of every code times its 128 x 128 block's scale (fp64)."""
    return _dequant(q, s, 128)


def fp8_roundtrip_1x128(x: np.ndarray, pow2: bool = False, recip: bool = False) -> np.ndarray:
    return dequant_1x128(*quant_1x128(x, pow2, recip))


def fp8_roundtrip_128x128(w: np.ndarray, pow2: bool = False) -> np.ndarray:
    return dequant_128x128(*quant_128x128(w, pow2))


# ----------------------------------------------------------------------------
# expert FFN and the layer
def swiglu(x: np.ndarray, w1: np.ndarray, w3: np.ndarray, w2: np.ndarray, h_quant=False) -> np.ndarray:
    """y = W2 (SiLU(W1 x) * (W3 x)) per row, fp64 (three d x I matrices: ai.flicky.cc exercise).
    h_quant: False, True (h quantised per 1 x 128 tile, amax/448 scales) or "ue8m0" (UE8M0 scales)."""
    x, w1, w3, w2 = (_c(a, np.float64) for a in (x, w1, w3, w2))
    n, d = x.shape
    I = w1.shape[0]
    assert w1.shape == (I, d) and w3.shape == (I, d) and w2.shape == (d, I)
    y = np.empty((n, d), np.float64)
    if n:
        _load().oracle_swiglu(n, d, I, x.ctypes.data, w1.ctypes.data, w3.ctypes.data, w2.ctypes.data,
                              2 if h_quant == "ue8m0" else int(bool(h_quant)), y.ctypes.data)
    return y


def expert_operands(w1_bits, w3_bits, w2_bits, fp8):
    """fp64 operands of one expert: the bf16 weights, or their 128x128-block FP8
    round trip (fp8 = True: amax/448 scales; fp8 = "ue8m0": UE8M0 scales)."""
    ws = [bf16_to_f64(w) for w in (w1_bits, w3_bits, w2_bits)]
    if fp8:
        ws = [fp8_roundtrip_128x128(w, pow2=fp8 == "ue8m0") for w in ws]
    return ws


def layer_output(u_bits: np.ndarray, tokens: np.ndarray, idx: np.ndarray, gate: np.ndarray,
                 routed_weights, shared_weights, n_shared: int, E: int, fp8=False) -> np.ndarray:
    """h'_t = u_t + sum_s FFN_s(u_t) + sum_j g_{t,j} FFN_{S_j}(u_t) for the given tokens, fp64.

    The layer equation of ai.flicky.cc 2.1.2 / xyznot.com Method 2.  idx and
    gate are [len(tokens), k].  routed_weights(e) and shared_weights(s) return
    the bf16 bit patterns (W1, W3, W2) of one expert; experts are visited one
    at a time (expert-major), so only one expert's fp64 copy is alive.
    fp8=True: every main-GEMM input is its FP8 round trip (weights 128x128
    blocks, u and h 1x128 tiles; the router stays high precision, 3.3 item 1);
    the residual u is the layer input itself.  fp8="ue8m0": the same with
    UE8M0 scales (powers of two) in every quantisation.
    """
    tokens = np.asarray(tokens, np.int64)
    u_rows = bf16_to_f64(u_bits[tokens])
    x = fp8_roundtrip_1x128(u_rows, pow2=fp8 == "ue8m0") if fp8 else u_rows
    out = u_rows.copy()
    for s in range(n_shared):
        w1, w3, w2 = expert_operands(*shared_weights(s), fp8)
        out += swiglu(x, w1, w3, w2, h_quant=fp8)
    for e in range(E):
        rows, js = np.nonzero(idx == e)
        if rows.size == 0:
            continue
        w1, w3, w2 = expert_operands(*routed_weights(e), fp8)
        y = swiglu(x[rows], w1, w3, w2, h_quant=fp8)
        out[rows] += gate[rows, js][:, None] * y
    return out


def expert_rows(u_bits: np.ndarray, tokens: np.ndarray, idx: np.ndarray, routed_weights, shared_weights,
                n_shared: int, E: int, fp8=False):
    """The expert outputs layer_output sums, kept apart, fp64.

    Returns (y [n, k, d], ysh [N_s, n, d]) for the n given tokens:
    y[t, j] = FFN_{idx[t, j]}(x_t) and ysh[s, t] = FFN_s(x_t), with the same
    operands as layer_output (fp8=True: u quantised per 1x128 tile, weights
    per 128x128 block, h per 1x128 tile; ai.flicky.cc 3.3 items 1-2).
    combine(u, ysh, y.reshape(n*k, d), slot=arange, gate) then assembles
    h'_t of the layer equation (ai.flicky.cc 2.1.2).
    """
    tokens = np.asarray(tokens, np.int64)
    u_rows = bf16_to_f64(u_bits[tokens])
    x = fp8_roundtrip_1x128(u_rows, pow2=fp8 == "ue8m0") if fp8 else u_rows
    n, k = idx.shape
    d = u_rows.shape[1]
    y = np.zeros((n, k, d))
    ysh = np.zeros((n_shared, n, d))
    for s in range(n_shared):
        w1, w3, w2 = expert_operands(*shared_weights(s), fp8)
        ysh[s] = swiglu(x, w1, w3, w2, h_quant=fp8)
    for e in range(E):
        rows, js = np.nonzero(idx == e)
        if rows.size == 0:
            continue
        w1, w3, w2 = expert_operands(*routed_weights(e), fp8)
        y[rows, js] = swiglu(x[rows], w1, w3, w2, h_quant=fp8)
    return y, ysh


def combine(u_bits: np.ndarray, shared_y: np.ndarray, y_perm: np.ndarray, slot: np.ndarray,
            gate: np.ndarray) -> np.ndarray:
    """out_t = u_t + sum_s shared_y[s, t] + sum_j gate[t, j] y_perm[slot[t, j]], fp64.

    The layer equation of ai.flicky.cc 2.1.2 written over already computed
    expert outputs: shared_y [N_s, T, d] and y_perm [T*k, d] (any float
    arrays, widened exactly), slot [T, k], gate [T, k].
    """
    out = bf16_to_f64(u_bits)
    for s in range(shared_y.shape[0]):
        out = out + np.asarray(shared_y[s], np.float64)
    T, k = slot.shape
    yp = np.asarray(y_perm, np.float64)
    for j in range(k):
        out = out + np.asarray(gate[:, j], np.float64)[:, None] * yp[slot[:, j]]
    return out


def bias_update(counts: np.ndarray, bias: np.ndarray, T: int, k: int, gamma: float) -> np.ndarray:
    """One auxiliary-loss-free bias step in fp32 (ai.flicky.cc 2.1.2; xyznot.com Method 2)."""
    counts = _c(counts, np.int32)
    b = _c(bias, np.float32).copy()
    _load().oracle_bias_update(b.size, T, k, counts.ctypes.data, ctypes.c_float(gamma), b.ctypes.data)
    return b


def expert_param_count(d: int, inter: int) -> int:
    """Parameters of one SwiGLU expert: three d x I matrices (ai.flicky.cc exercise)."""
    return 3 * d * inter
