"""Redundant (duplicated) hot experts on the GPU (ai.flicky.cc 3.5): with a
plan from the step's own loads, moe_forward_replicated splits each hot
expert's tokens between its copies (one grouped-GEMM group per copy, on the
shared weights).  The layer output and the experts' loads must be those of
moe_forward, bit for bit: a token's rows go through the same arithmetic, only
in other groups."""
import numpy as np
import pytest
import torch

import synth
from mixture_experts_layer_87_b300 import ReplicatedExperts
from parity import HostLayer

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.mark.parametrize("name,n_extra", [("tiny", 4), ("ragged", 7), ("mid", 16), ("tiny_fp8", 4),
                                          ("ragged_fp8", 7), ("mid_fp8", 16)])
def test_replicated_forward_equals_forward(name, n_extra):
    cfg = synth.get_config(name) if name != "mid_fp8" else synth.get_config("mid", prec="fp8")
    host = HostLayer(cfg)
    layer = host.device_layer()
    u = synth.tokens(cfg).to(DEV)
    b = host.bias.to(DEV)
    counts = torch.empty(cfg.E, dtype=torch.int32, device=DEV)
    out = layer.forward(u, b, counts=counts).clone()
    assert layer.status() == 0
    rep = ReplicatedExperts(layer, counts, n_extra)
    counts_r = torch.full_like(counts, -1)
    out_r = rep.forward(u, b, counts=counts_r)
    assert rep.status() == 0
    assert torch.equal(counts_r, counts)
    assert torch.equal(out_r.view(torch.int16), out.view(torch.int16))
    # the copies went to the most loaded experts
    c = counts.cpu().numpy()
    copies = rep.replica_count_host.numpy()
    assert copies.sum() == cfg.E + n_extra
    assert c[copies > 1].min() >= np.sort(c)[-(copies > 1).sum()]
