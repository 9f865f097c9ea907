"""moe_route_noalloc: the router entry point for callers that cannot allocate
device memory (an engine that owns every byte through its own pool, or a
serving path where cudaMalloc is forbidden because it can stall the device or
fail under memory pressure).  Its logits scratch is a fixed array inside the
library instead of a caller workspace.

The test compares it, through the C ABI, with moe_route (which takes a
workspace) on two calls in a row with different shapes, so the second call
runs on an array that still holds the first call's logits.  This file is
collected last on purpose: a run that stops at the first failure has run every
other test before it gets here."""
import numpy as np
import pytest
import torch

import synth
from mixture_experts_layer_87_b300 import capi

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _route_both(name):
    cfg = synth.get_config(name)
    u = synth.tokens(cfg).to(DEV)
    cent = synth.centroids(cfg).to(DEV)
    bias = synth.bias(cfg).to(DEV)
    dm = capi.dims(cfg.T, cfg.d, cfg.E, cfg.k, cfg.n_shared, cfg.inter, cfg.prec)

    def outputs():
        return (torch.empty((cfg.T, cfg.k), dtype=torch.int32, device=DEV),
                torch.empty((cfg.T, cfg.k), dtype=torch.float32, device=DEV),
                torch.empty(cfg.E, dtype=torch.int32, device=DEV))

    ws = torch.empty(capi.moe_workspace_size(dm), dtype=torch.uint8, device=DEV)
    idx_ref, gate_ref, cnt_ref = outputs()
    capi.moe_route(dm, u, cent, bias, idx_ref, gate_ref, cnt_ref, ws)
    assert capi.moe_read_device_status(ws) == 0

    idx, gate, cnt = outputs()
    status = torch.full((1,), -1, dtype=torch.int32, device=DEV)
    capi.moe_route_noalloc(dm, u, cent, bias, idx, gate, cnt, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return (idx_ref.cpu().numpy(), gate_ref.cpu().numpy(), cnt_ref.cpu().numpy()), \
           (idx.cpu().numpy(), gate.cpu().numpy(), cnt.cpu().numpy())


def test_noalloc_route_matches_workspace_route_on_two_calls():
    # first call: mid layer (T*E = 262144 logits); second call: a ragged shape
    # (T=300, E=20) that reuses the array left dirty by the first.
    for name in ("mid", "ragged"):
        (idx_ref, gate_ref, cnt_ref), (idx, gate, cnt) = _route_both(name)
        # selection and loads are integer results: bit for bit
        np.testing.assert_array_equal(idx, idx_ref)
        np.testing.assert_array_equal(cnt, cnt_ref)
        # gates: the tolerance the router parity tests use against the oracle
        np.testing.assert_allclose(gate, gate_ref, rtol=0, atol=2e-6)


def test_noalloc_route_rejects_shapes_beyond_its_scratch():
    T, E = capi.MOE_ROUTE_NOALLOC_MAX_LOGITS // 256 + 32, 256
    dm = capi.dims(T, 256, E, 8, 0, 128, "bf16")
    dummy = torch.zeros(16, dtype=torch.int32, device=DEV)
    with pytest.raises(capi.MoEError) as err:
        capi.moe_route_noalloc(dm, dummy, dummy, dummy, dummy, dummy, dummy)
    assert err.value.status == 2   # MOE_ERR_UNSUPPORTED: nothing was enqueued
