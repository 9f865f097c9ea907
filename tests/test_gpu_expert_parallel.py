"""Expert parallelism through the CUDA library on one GPU: W ranks emulated in
one process (mixture_experts_layer_87_b300.expert_parallel.loopback_forward,
phase by phase, so no kernel waits on another rank).  Rank r owns experts
[r E/W, (r+1) E/W) and its own batch; its rows travel to the experts' ranks,
run there in (sender, local expert) groups on the local weights, and come
back.  Every rank's h' must equal moe_forward of the whole layer on the same
batch with the same node-limited routing, bit for bit (a row meets the same
arithmetic in either grouping)."""
import numpy as np
import pytest
import torch

import synth
from mixture_experts_layer_87_b300 import expert_parallel as ep
from parity import HostLayer

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.mark.parametrize("name,world,node_limit", [("tiny", 2, 0), ("tiny", 4, 2), ("ragged", 4, 2),
                                                   ("mid", 8, 3), ("tiny_fp8", 4, 2), ("ragged_fp8", 2, 1)])
def test_expert_parallel_ranks_match_the_whole_layer(name, world, node_limit):
    base = synth.get_config(name)
    cfg = synth.get_config(name, route_groups=world if node_limit else 0, route_group_limit=node_limit)
    host = HostLayer(cfg)
    ranks = [ep.ExpertParallelRank(cfg.T, cfg.d, cfg.E, cfg.k, cfg.n_shared, cfg.inter, cfg.prec, r, world,
                                   host.cent, host.routed, host.shared, node_limit=node_limit) for r in range(world)]
    bias = host.bias.to(DEV)
    us = [synth.tokens(base, step=r).to(DEV) for r in range(world)]
    outs = ep.loopback_forward(ranks, us, bias)
    assert all(r.status() == 0 for r in ranks)
    whole = host.device_layer()
    gs = cfg.E // world
    for r in range(world):
        ref = whole.forward(us[r], bias)
        assert whole.status() == 0
        assert torch.equal(outs[r].view(torch.int16), ref.view(torch.int16)), f"rank {r}"
        if node_limit:
            nodes = [len({int(e) // gs for e in row}) for row in ranks[r].idx.cpu().numpy()]
            assert max(nodes) <= node_limit
