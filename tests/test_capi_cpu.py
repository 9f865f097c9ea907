"""The C-ABI library loads without a GPU, exports every symbol include/moe.h
declares, and rejects bad arguments before touching the device."""
import ctypes
import os
import re

import pytest

from mixture_experts_layer_87_b300 import build, capi

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return capi.lib()


def _declared():
    text = open(os.path.join(ROOT, "include", "moe.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert set(names) == set(capi.EXPORTS)
    for n in names:
        assert hasattr(lib, n), n


def test_library_is_sm103a_only(lib):
    assert "arch=compute_103a,code=sm_103a" in " ".join(build.NVCC_FLAGS)


def test_status_strings(lib):
    assert capi.status_string(0) == "ok"
    assert "workspace" in capi.status_string(3)
    assert capi.status_string(99) == "unknown status"


def _dims(**kw):
    base = dict(T=64, d=256, E=16, k=4, n_shared=1, inter=128, prec="bf16")
    base.update(kw)
    return capi.dims(**base)


@pytest.mark.parametrize("kw,code", [
    (dict(k=17), 1),           # k > E
    (dict(E=40, k=33), 1),     # k > 32
    (dict(E=2000), 2),         # E > 1024
    (dict(d=200), 2),          # d % 128
    (dict(inter=100), 2),      # I % 128
    (dict(T=-1), 1),
    (dict(prec=7), 1),
    (dict(route_groups=3, route_group_limit=1), 1),    # E % groups
    (dict(route_groups=4, route_group_limit=0), 1),    # limit < 1
    (dict(route_groups=4, route_group_limit=5), 1),    # limit > groups
    (dict(route_groups=8, route_group_limit=1), 1),    # 1 node of 2 experts < k = 4
    (dict(E=64, route_groups=64, route_group_limit=4), 2),  # more than 32 nodes
    (dict(route_groups=-1), 1),
])
def test_workspace_size_rejects_bad_dims(lib, kw, code):
    n = ctypes.c_size_t(0)
    dm = _dims(**kw)
    assert lib.moe_workspace_size(ctypes.byref(dm), ctypes.byref(n)) == code


def test_workspace_size_grows_with_shape(lib):
    small = capi.moe_workspace_size(_dims())
    big = capi.moe_workspace_size(_dims(T=8192, d=7168, E=256, k=8, inter=2048))
    fp8 = capi.moe_workspace_size(_dims(T=8192, d=7168, E=256, k=8, inter=2048, prec="fp8"))
    assert 0 < small < fp8 < big


def test_calls_reject_null_and_small_workspace_without_a_gpu(lib):
    dm = _dims()
    need = capi.moe_workspace_size(dm)
    fake = 1 << 20   # never dereferenced: validation fails first
    w = capi.moe_weights()
    # null weights
    assert lib.moe_forward(ctypes.byref(dm), ctypes.byref(w), fake, fake, fake, None, fake, need, None) == 1
    # workspace too small
    assert lib.moe_route(ctypes.byref(dm), fake, fake, fake, fake, fake, fake, fake, need - 256, None) == 3
    # misaligned workspace
    assert lib.moe_route(ctypes.byref(dm), fake, fake, fake, fake, fake, fake, fake + 8, need, None) == 1
    # null u
    assert lib.moe_route(ctypes.byref(dm), None, fake, fake, fake, fake, fake, fake, need, None) == 1
    # FP8 permute without scales
    d8 = _dims(prec="fp8")
    n8 = capi.moe_workspace_size(d8)
    assert lib.moe_permute(ctypes.byref(d8), fake, fake, fake, fake, fake, fake, None, fake, n8, None) == 1
    # grouped ffn: more rows than the workspace was sized for
    assert lib.moe_grouped_ffn(ctypes.byref(dm), 2, 64 * 4 + 1, fake, None, 0, fake, None, fake, None, fake, None,
                               fake, fake, need, None) == 3
    # grouped ffn: a group -> expert table without the number of experts it indexes
    assert lib.moe_grouped_ffn(ctypes.byref(dm), 2, 64, fake, fake, 0, fake, None, fake, None, fake, None,
                               fake, fake, need, None) == 1
    # bias update: k > E
    assert lib.moe_bias_update(4, 10, 5, fake, ctypes.c_float(0.001), fake, None) == 1
    # block quantiser: shape not a multiple of 128
    assert lib.moe_quantize_fp8_blocks(fake, 100, 128, fake, fake, 0, None) == 1
    # misaligned bf16 input
    assert lib.moe_combine(ctypes.byref(dm), fake + 2, fake, fake, fake, fake, fake, None) == 1


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(capi, "_lib", None)
    monkeypatch.setattr(capi, "LIB_PATH", str(tmp_path / "absent.so"))
    with pytest.raises(RuntimeError, match="not built"):
        capi.lib()


def test_range_checked_build_exports_the_same_symbols():
    """The -DMOE_CHECK variant (every computed global index range-checked
    into the status word) builds and exports the same C ABI."""
    so = build.build(check=True)
    L = ctypes.CDLL(so)
    for n in capi.EXPORTS:
        assert hasattr(L, n), n
    L.moe_status_string.restype = ctypes.c_char_p
    assert b"range-checked" in L.moe_status_string(7)


def test_backward_workspace_and_argument_errors(lib):
    dm, d8 = _dims(), _dims(prec="fp8")
    need = capi.moe_backward_workspace_size(dm)
    assert need > capi.moe_workspace_size(dm)
    # FP8: the E4M3 operands of the data-gradient GEMMs on top of the bf16 activations
    assert capi.moe_backward_workspace_size(d8) > capi.moe_workspace_size(d8)
    fake = 1 << 20
    w, wt, gr = capi.moe_weights(), capi.moe_weights_t(), capi.moe_grads()
    assert lib.moe_backward(ctypes.byref(dm), ctypes.byref(w), ctypes.byref(wt), fake, fake, fake, ctypes.byref(gr),
                            fake, need, None) == 1
    # FP8 without the transposed weights' block scales
    w8 = capi.moe_weights(fake, fake, fake, fake, fake, fake, fake, fake, fake)
    wt8 = capi.moe_weights_t(fake, fake, fake, fake, None, None, None, None)
    gr8 = capi.moe_grads(fake, fake, fake, fake, fake, fake)
    assert lib.moe_backward(ctypes.byref(d8), ctypes.byref(w8), ctypes.byref(wt8), fake, fake, fake, ctypes.byref(gr8),
                            fake, capi.moe_backward_workspace_size(d8), None) == 1
    assert lib.moe_transpose_expert_weights_fp8(2, 100, 128, fake, fake, fake, fake, fake, fake, fake, fake,
                                                None) == 1                                  # I % 128
    assert lib.moe_transpose_expert_weights_fp8(2, 128, 128, fake, None, fake, fake, fake, fake, fake, fake,
                                                None) == 1                                  # no scales
    assert lib.moe_transpose_expert_weights(2, 100, 128, fake, fake, fake, fake, None) == 1       # I % 128


def test_backward_rejects_bad_gradient_pointers_and_small_workspace(lib):
    """moe_backward validates before it enqueues anything: with tokens, du must
    be given; every gradient must be 16-byte aligned (vector and TMA stores);
    the workspace must be at least moe_backward_workspace_size."""
    dm = _dims()
    need = capi.moe_backward_workspace_size(dm)
    fake = 1 << 20
    w = capi.moe_weights(fake, None, fake, None, fake, None, fake, None, fake)
    wt = capi.moe_weights_t(fake, fake, fake, fake, None, None, None, None)
    call = lambda gr, ws_bytes=need: lib.moe_backward(ctypes.byref(dm), ctypes.byref(w), ctypes.byref(wt), fake, fake,
                                                      fake, ctypes.byref(gr), fake, ws_bytes, None)
    assert call(capi.moe_grads(None, fake, fake, fake, fake, fake)) == 1            # du missing, T > 0
    assert call(capi.moe_grads(fake + 8, fake, fake, fake, fake, fake)) == 1        # du misaligned
    assert call(capi.moe_grads(fake, fake, fake + 4, fake, fake, fake)) == 1        # dw13 misaligned
    assert call(capi.moe_grads(fake, fake, fake, fake, fake, fake), need - 256) == 3  # workspace too small
