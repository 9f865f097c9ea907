"""Token-sharded replicas of the layer on several GPUs (host-side plumbing).

The forward pass has no cross-token exchange: every token's output depends
only on its own routing and the shared expert weights (ai.flicky.cc 2.1.2, the
h'_t equation).  So each GPU holds all experts and runs the whole layer on its
own share of the tokens, with no collective on the data path.

The one real exchange is the auxiliary-loss-free bias update between steps.
It compares every expert's load over the step's batch with the mean load
T*k/E.  With the batch split over replicas, the loads must be summed over
the replicas (one all-reduce of E int32) before moe_bias_update, so every
replica applies the same update and the biases stay identical.

These helpers take any torch.distributed process group (NCCL on GPUs, gloo
in the CPU tests); with a world of one they are no-ops.
"""
from __future__ import annotations

import torch


def _dist():
    import torch.distributed as dist
    return dist if dist.is_available() and dist.is_initialized() else None


def world_and_rank(group=None) -> tuple[int, int]:
    dist = _dist()
    if dist is None:
        return 1, 0
    return dist.get_world_size(group), dist.get_rank(group)


def shard(total: int, world: int, rank: int) -> slice:
    """Contiguous share of `total` tokens for `rank`; the first total % world
    ranks take one extra token."""
    base, extra = divmod(total, world)
    start = rank * base + min(rank, extra)
    return slice(start, start + base + (1 if rank < extra else 0))


def global_counts(counts: torch.Tensor, group=None) -> torch.Tensor:
    """Sum the per-expert loads of all replicas in place (int32, exact)."""
    dist = _dist()
    if dist is not None and dist.get_world_size(group) > 1:
        dist.all_reduce(counts, op=dist.ReduceOp.SUM, group=group)
    return counts


def max_over_ranks(x: float, device="cpu", group=None) -> float:
    """The largest of the ranks' values (e.g. their step times)."""
    dist = _dist()
    if dist is None or dist.get_world_size(group) == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX, group=group)
    return float(t.item())


def barrier(group=None) -> None:
    dist = _dist()
    if dist is not None and dist.get_world_size(group) > 1:
        dist.barrier(group=group)
