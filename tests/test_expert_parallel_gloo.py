"""The expert-parallel exchange (ai.flicky.cc 3.4: experts spread over ranks,
tokens sent to them and back with all-to-all; 2.1.2: a token on at most 4
nodes), tested as two gloo ranks on the CPU.

Each rank owns half of the routed experts and its own tokens.  The exchange
code of mixture_experts_layer_87_b300.expert_parallel (split sizes, the
all-to-all of counts and rows, the layout of what arrives) runs as it does on
GPUs; the CPU oracle stands in for the CUDA kernels on either side of it
(router, dispatch, the experts, the combine).  Every rank's h' must equal the
oracle's single-process layer output for its tokens, and with the node limit
no token may send rows to more ranks than the limit."""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir, name, node_limit):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import oracle
        import synth
        from mixture_experts_layer_87_b300 import expert_parallel as ep

        cfg = synth.get_config(name)
        el = cfg.E // world
        groups = world if node_limit else 0
        cent = synth.bf16_bits(synth.centroids(cfg))
        bias = np.asarray(synth.bias(cfg), np.float32)
        u = synth.bf16_bits(synth.tokens(cfg, step=rank))              # this rank's tokens
        routed = lambda e: tuple(synth.bf16_bits(w) for w in synth.expert_weights(cfg, e))
        shared = lambda s: tuple(synth.bf16_bits(w) for w in synth.expert_weights(cfg, s, shared=True))
        ex = ep.DistExchange()
        # phase 1 (oracle stand-in for moe_route + moe_permute)
        r = oracle.route(u, cent, bias, cfg.k, groups=groups, group_limit=node_limit)
        lay = oracle.dispatch_layout(r["idx"], cfg.E)
        x = torch.from_numpy(u[lay["perm"]].view(np.int16).copy())
        split = ep.send_splits(lay["offsets"], world)
        dests = [{int(e) // el for e in row} for row in r["idx"]]
        # phase 2: the exchange under test
        send_counts = torch.from_numpy(np.diff(lay["offsets"]).astype(np.int32).reshape(world, el))
        recv_counts = ex.counts(send_counts)
        recv_split = [int(v) for v in recv_counts.sum(1)]
        x_recv = ex.rows(x, split, recv_split).numpy().view(np.uint16)
        # phase 3 (oracle stand-in for moe_grouped_ffn over (sender, local expert) groups)
        offs, gexp = ep.receive_layout(recv_counts.numpy())
        xf = oracle.bf16_to_f64(x_recv)
        y = np.zeros((len(xf), cfg.d))
        for g, e_loc in enumerate(gexp):
            if offs[g + 1] > offs[g]:
                w = oracle.expert_operands(*routed(rank * el + int(e_loc)), fp8=False)
                y[offs[g]:offs[g + 1]] = oracle.swiglu(xf[offs[g]:offs[g + 1]], *w)
        # phase 4: results back to their senders
        y_back = ex.rows(torch.from_numpy(y), recv_split, split).numpy()
        # phase 5 (oracle stand-in for the shared experts and moe_combine)
        uf = oracle.bf16_to_f64(u)
        ysh = np.stack([oracle.swiglu(uf, *oracle.expert_operands(*shared(s), fp8=False))
                        for s in range(cfg.n_shared)])
        out = oracle.combine(u, ysh, y_back, lay["slot"], r["gate"])
        ref = oracle.layer_output(u, np.arange(cfg.T), r["idx"], r["gate"], routed, shared, cfg.n_shared, cfg.E)
        np.save(os.path.join(out_dir, f"err_{rank}.npy"), np.array([np.abs(out - ref).max() / np.abs(ref).max()]))
        np.save(os.path.join(out_dir, f"dests_{rank}.npy"), np.array([len(d) for d in dests]))
        np.save(os.path.join(out_dir, f"rows_{rank}.npy"), np.array([sum(split), sum(recv_split)]))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("name,node_limit", [("tiny", 0), ("tiny", 1), ("ragged", 1)])
def test_expert_parallel_exchange_two_ranks(tmp_path, name, node_limit):
    world = 2
    mp.spawn(_worker, args=(world, _free_port(), str(tmp_path), name, node_limit), nprocs=world, join=True)
    for rank in range(world):
        assert np.load(tmp_path / f"err_{rank}.npy")[0] <= 1e-12
        if node_limit:
            assert np.load(tmp_path / f"dests_{rank}.npy").max() <= node_limit
    rows = [np.load(tmp_path / f"rows_{rank}.npy") for rank in range(world)]
    assert sum(r[0] for r in rows) == sum(r[1] for r in rows)        # every row sent was received
