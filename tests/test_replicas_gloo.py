"""The multi-GPU path, tested as two gloo ranks on the CPU.

Token-sharded replicas run the whole layer on their own share of the tokens.
The only exchange is the all-reduce of the per-expert loads before the bias
update (the update compares each expert's load over the step's batch with
the mean T*k/E).  The CPU oracle stands in for each replica's router here.
The test checks four things:
  * the shards partition the batch;
  * the all-reduced loads equal the loads of the whole batch, bit for bit;
  * both replicas end a multi-step loop with identical biases, equal to a
    single process stepping over the whole batch;
  * max over ranks and the aggregate throughput value behave as bench.py uses them.
"""
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


def _worker(rank: int, world: int, port: int, out_dir: str) -> None:
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import oracle
        import synth
        from mixture_experts_layer_87_b300 import replicas

        cfg = synth.get_config("ragged")          # T=300, E=20, k=3: T not a multiple of the world
        cent = synth.bf16_bits(synth.centroids(cfg))
        bias = np.asarray(synth.bias(cfg), np.float32)
        assert replicas.world_and_rank() == (world, rank)
        sl = replicas.shard(cfg.T, world, rank)
        steps = 3
        for step in range(steps):
            u = synth.bf16_bits(synth.tokens(cfg, step=step))      # the step's whole batch
            local = oracle.route(u[sl], cent, bias, cfg.k)["idx"]
            counts = torch.from_numpy(np.bincount(local.ravel(), minlength=cfg.E).astype(np.int32))
            replicas.global_counts(counts)
            bias = oracle.bias_update(counts.numpy(), bias, cfg.T, cfg.k, cfg.gamma)
            np.save(os.path.join(out_dir, f"counts_{rank}_{step}.npy"), counts.numpy())
        np.save(os.path.join(out_dir, f"bias_{rank}.npy"), bias)
        # timing reduction and the aggregate value bench.py reports
        ms = float(rank + 1)
        slowest = replicas.max_over_ranks(ms)
        tokens_local = sl.stop - sl.start
        tot = torch.tensor([tokens_local], dtype=torch.int64)
        dist.all_reduce(tot)
        np.save(os.path.join(out_dir, f"timing_{rank}.npy"), np.array([slowest, float(tot.item())]))
        replicas.barrier()
    finally:
        dist.destroy_process_group()


def test_shards_partition_the_batch():
    from mixture_experts_layer_87_b300 import replicas
    for total, world in ((300, 2), (7, 3), (8, 4), (1, 2), (0, 2)):
        covered = []
        for r in range(world):
            s = replicas.shard(total, world, r)
            covered.extend(range(s.start, s.stop))
        assert covered == list(range(total))


def test_two_gloo_replicas_share_loads_and_biases(tmp_path):
    world = 2
    mp.start_processes(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    sys.path.insert(0, ROOT)
    import oracle
    import synth
    cfg = synth.get_config("ragged")
    cent = synth.bf16_bits(synth.centroids(cfg))
    bias = np.asarray(synth.bias(cfg), np.float32)
    for step in range(3):
        u = synth.bf16_bits(synth.tokens(cfg, step=step))
        full = np.bincount(oracle.route(u, cent, bias, cfg.k)["idx"].ravel(), minlength=cfg.E).astype(np.int32)
        for r in range(world):
            np.testing.assert_array_equal(np.load(tmp_path / f"counts_{r}_{step}.npy"), full)
        bias = oracle.bias_update(full, bias, cfg.T, cfg.k, cfg.gamma)
    for r in range(world):
        np.testing.assert_array_equal(np.load(tmp_path / f"bias_{r}.npy"), bias)
        slowest, tokens = np.load(tmp_path / f"timing_{r}.npy")
        assert slowest == float(world) and tokens == cfg.T
