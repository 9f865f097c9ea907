"""The forward captured in a CUDA graph (CapturedForward): replays give the
eager forward's output and loads bit for bit, on new inputs copied into the
graph's buffer, and read the bias tensor's current contents (a bias update
between replays is seen by the next one)."""
import pytest
import torch

import synth
from mixture_experts_layer_87_b300 import CapturedForward, capi
from parity import HostLayer

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.mark.parametrize("name", ["ragged", "ragged_fp8"])
def test_graph_replay_equals_eager(name):
    cfg = synth.get_config(name)
    host = HostLayer(cfg)
    layer = host.device_layer()
    bias = host.bias.to(DEV).clone()
    cap = CapturedForward(layer, bias)
    for step in range(3):
        u = synth.tokens(cfg, step=step).to(DEV)
        got = cap(u).clone()
        got_counts = cap.counts.clone()
        out = torch.empty_like(got)
        counts = torch.zeros(cfg.E, dtype=torch.int32, device=DEV)
        layer.forward(u, bias, out, counts=counts)
        torch.cuda.synchronize()
        assert layer.status() == 0
        assert torch.equal(got.view(torch.int16), out.view(torch.int16)), step
        assert torch.equal(got_counts, counts), step
        # the bias update between steps changes the next replay's selection input
        capi.moe_bias_update(cfg.E, cfg.T, cfg.k, counts, 0.05, bias)
