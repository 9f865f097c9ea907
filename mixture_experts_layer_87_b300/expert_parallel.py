"""Expert parallelism: the routed experts of a layer spread over W ranks.

The deployment of the DeepSeek-V3 report as ai.flicky.cc reads it: 64-way
expert parallelism over 8 nodes, tokens sent to their experts and back with
all-to-all exchanges (section 3.4), and no token sent to more than 4 nodes
(section 2.1.2) -- with one rank per node here, the node-limited routing of
moe_dims (route_groups = W, route_group_limit = M) bounds every token's
destinations to M ranks.

Rank r holds the routed experts [r E/W, (r+1) E/W) and every shared expert,
and owns a batch of T tokens.  One forward is five phases:
  1. route + dispatch (moe_route, moe_permute): rows grouped expert-major, so
     the rows bound for rank r are one contiguous segment;
  2. exchange: every rank sends each destination its segment (and the
     per-expert row counts); what a rank receives is grouped by (sender,
     local expert);
  3. experts: moe_grouped_ffn over the received rows with one group per
     (sender, local expert), mapped onto the local expert's weights by the
     group -> expert table;
  4. exchange back: each result segment returns to its sender, where it lands
     in the sender's expert-major order again;
  5. shared experts on the rank's own tokens and moe_combine.
Every arithmetic step runs in the CUDA library; this module moves rows
between ranks (torch.distributed all_to_all_single, NCCL on GPUs) and keeps
the bookkeeping.  The exchange functions take any `exchange` object with the
all_to_all_single signature, so the same code runs under torch.distributed or
with all ranks emulated in one process (LoopbackExchange: phase by phase, no
kernel ever waits on another rank).
"""
from __future__ import annotations

import numpy as np
import torch

from . import capi
from .layer import MoELayer


# ----------------------------------------------------------------------------
# exchange plumbing
def send_splits(offsets_host: np.ndarray, world: int) -> list:
    """Rows bound for every rank: expert-major offsets [E+1] cut at the ranks'
    expert boundaries."""
    E = len(offsets_host) - 1
    el = E // world
    cut = offsets_host[::el]
    return [int(cut[r + 1] - cut[r]) for r in range(world)]


def receive_layout(recv_counts: np.ndarray):
    """Groups of the received rows, in arrival order (sender-major, then local
    expert): offsets [W*E_loc + 1] and the local expert of every group."""
    W, el = recv_counts.shape
    offsets = np.zeros(W * el + 1, np.int32)
    offsets[1:] = np.cumsum(recv_counts.ravel())
    group_expert = np.tile(np.arange(el, dtype=np.int32), W)
    return offsets, group_expert


class DistExchange:
    """all_to_all_single over a torch.distributed process group."""

    def __init__(self, group=None):
        import torch.distributed as dist
        self.dist, self.group = dist, group
        self.world = dist.get_world_size(group)

    def counts(self, send: torch.Tensor) -> torch.Tensor:
        """send [W, n] int32 (row w goes to rank w) -> recv [W, n] (row w came from rank w)."""
        recv = torch.empty_like(send)
        self.dist.all_to_all_single(recv, send, group=self.group)
        return recv

    def rows(self, send: torch.Tensor, send_split: list, recv_split: list) -> torch.Tensor:
        """Rows [n, ...] of any dtype, moved as 32-bit words (every backend
        carries int32; a row here is always a multiple of 4 bytes)."""
        send = send.contiguous()
        words = send.view(send.shape[0], -1).view(torch.uint8).view(torch.int32)
        recv = torch.empty((sum(recv_split), words.shape[1]), dtype=torch.int32, device=send.device)
        self.dist.all_to_all_single(recv, words, output_split_sizes=recv_split, input_split_sizes=send_split,
                                    group=self.group)
        return recv.view(torch.uint8).view(send.dtype).view((sum(recv_split),) + tuple(send.shape[1:]))


class LoopbackExchange:
    """W ranks in one process: each collective is called by every virtual
    rank in turn (rank 0 first) with its send buffer and completes when the
    last one has called; results come back from `collect`."""

    def __init__(self, world: int):
        self.world = world

    def counts_all(self, sends: list) -> list:
        return [torch.stack([sends[src][dst] for src in range(self.world)]) for dst in range(self.world)]

    def rows_all(self, sends: list, send_splits_all: list) -> list:
        out = []
        for dst in range(self.world):
            parts = []
            for src in range(self.world):
                start = sum(send_splits_all[src][:dst])
                parts.append(sends[src][start:start + send_splits_all[src][dst]])
            out.append(torch.cat(parts))
        return out


# ----------------------------------------------------------------------------
class ExpertParallelRank:
    """One rank of an expert-parallel layer on this process's GPU.

    centroids [E, d] bf16 (every rank routes over all experts); routed(e)
    gives the bf16 (W1, W3, W2) of global expert e, shared(s) those of shared
    expert s.  node_limit > 0: a token's experts on at most node_limit ranks.
    """

    def __init__(self, T, d, E, k, n_shared, inter, prec, rank, world, centroids, routed, shared, node_limit=0,
                 device="cuda"):
        assert E % world == 0, "the experts must split evenly over the ranks"
        self.T, self.d, self.E, self.k, self.n_shared, self.inter, self.prec = T, d, E, k, n_shared, inter, prec
        self.rank, self.world = rank, world
        self.el = E // world
        self.fp8 = prec == "fp8"
        dev = self.device = torch.device(device)
        groups = world if node_limit else 0
        self.route_dims = capi.dims(T, d, E, k, n_shared, inter, prec, groups, node_limit)
        self.ws = torch.empty(capi.moe_workspace_size(self.route_dims), dtype=torch.uint8, device=dev)
        # receiver: up to every rank's T*k rows, one group per (sender, local expert)
        self.ffn_dims = capi.dims(world * T, d, E, k, 0, inter, prec)
        self.ws_ffn = torch.empty(capi.moe_workspace_size(self.ffn_dims), dtype=torch.uint8, device=dev)
        # weights: the local routed experts, and the shared experts
        self.weights = MoELayer(T, d, self.el, min(k, self.el), n_shared, inter, prec, device=dev)
        for j in range(self.el):
            self.weights.load_expert(j, *routed(rank * self.el + j))
        for s in range(n_shared):
            self.weights.load_expert(s, *shared(s), shared=True)
        self.weights.release_staging()
        self.centroids = centroids.to(dev)
        if n_shared:
            self.sh_dims = capi.dims(T, d, 1, 1, 0, inter, prec)
            self.ws_sh = torch.empty(capi.moe_workspace_size(self.sh_dims), dtype=torch.uint8, device=dev)

    # phase 1
    def dispatch(self, u: torch.Tensor, bias: torch.Tensor):
        T, k, d, dev = self.T, self.k, self.d, self.device
        R = T * k
        self.u = u
        self.idx = torch.empty((T, k), dtype=torch.int32, device=dev)
        self.gate = torch.empty((T, k), dtype=torch.float32, device=dev)
        self.counts = torch.empty(self.E, dtype=torch.int32, device=dev)
        capi.moe_route(self.route_dims, u, self.centroids, bias, self.idx, self.gate, self.counts, self.ws)
        offsets = torch.empty(self.E + 1, dtype=torch.int32, device=dev)
        perm = torch.empty(R, dtype=torch.int32, device=dev)
        self.slot = torch.empty((T, k), dtype=torch.int32, device=dev)
        x = torch.empty((R, d), dtype=torch.uint8 if self.fp8 else torch.bfloat16, device=dev)
        xs = torch.empty((d // 128, R), dtype=torch.float32, device=dev) if self.fp8 else None
        capi.moe_permute(self.route_dims, self.idx, u, offsets, perm, self.slot, x, xs, self.ws)
        offs = offsets.cpu().numpy()          # the exchange needs its sizes on the host
        self.send_split = send_splits(offs, self.world)
        send_counts = torch.from_numpy(np.diff(offs).astype(np.int32).reshape(self.world, self.el)).to(dev)
        # rows, and for FP8 their 1 x 128 tile scales as rows [R, d/128]
        return x, (xs.t().contiguous() if self.fp8 else None), send_counts

    # phase 3
    def experts(self, x_recv: torch.Tensor, xs_recv_rows, recv_counts: torch.Tensor) -> torch.Tensor:
        rc = recv_counts.cpu().numpy()
        self.recv_split = [int(v) for v in rc.sum(1)]
        rows = int(rc.sum())
        y = torch.empty((rows, self.d), dtype=torch.bfloat16, device=self.device)
        if rows == 0:
            return y
        offsets, group_expert = receive_layout(rc)
        W = self.weights
        xs = xs_recv_rows.t().contiguous() if self.fp8 else None
        capi.moe_grouped_ffn(self.ffn_dims, len(group_expert), rows, torch.from_numpy(offsets).to(self.device),
                             x_recv, xs, W.w13, W.w13_scale, W.w2, W.w2_scale, y, self.ws_ffn,
                             group_expert=torch.from_numpy(group_expert).to(self.device), n_weight_experts=self.el)
        return y

    # phase 5
    def combine(self, y_back: torch.Tensor) -> torch.Tensor:
        T, d, dev = self.T, self.d, self.device
        ysh = None
        if self.n_shared:
            ysh = torch.empty((self.n_shared, T, d), dtype=torch.bfloat16, device=dev)
            x, xs = self.u, None
            if self.fp8:     # the 1 x 128 codes of u in token order: a dispatch to one expert
                zero = torch.zeros((T, 1), dtype=torch.int32, device=dev)
                offs = torch.empty(2, dtype=torch.int32, device=dev)
                perm = torch.empty(T, dtype=torch.int32, device=dev)
                slot = torch.empty((T, 1), dtype=torch.int32, device=dev)
                x = torch.empty((T, d), dtype=torch.uint8, device=dev)
                xs = torch.empty((d // 128, T), dtype=torch.float32, device=dev)
                capi.moe_permute(self.sh_dims, zero, self.u, offs, perm, slot, x, xs, self.ws_sh)
            offs = torch.tensor([0, T], dtype=torch.int32, device=dev)
            W = self.weights
            for s in range(self.n_shared):
                sc = (lambda t: t[s:s + 1] if t is not None else None)
                capi.moe_grouped_ffn(self.sh_dims, 1, T, offs, x, xs, W.ws13[s:s + 1], sc(W.ws13_scale),
                                     W.ws2[s:s + 1], sc(W.ws2_scale), ysh[s], self.ws_sh)
        out = torch.empty((T, d), dtype=torch.bfloat16, device=dev)
        capi.moe_combine(self.route_dims, self.u, ysh, y_back, self.slot, self.gate, out)
        return out

    def status(self) -> int:
        codes = [capi.moe_read_device_status(w) for w in (self.ws, self.ws_ffn) + ((self.ws_sh,) if self.n_shared else ())]
        return next((c for c in codes if c), 0)

    # all five phases under torch.distributed
    def forward(self, u: torch.Tensor, bias: torch.Tensor, ex: DistExchange) -> torch.Tensor:
        x, xs, send_counts = self.dispatch(u, bias)
        recv_counts = ex.counts(send_counts)
        recv_split = [int(v) for v in recv_counts.sum(1).cpu()]
        x_recv = ex.rows(x, self.send_split, recv_split)
        xs_recv = ex.rows(xs, self.send_split, recv_split) if self.fp8 else None
        y_recv = self.experts(x_recv, xs_recv, recv_counts)
        y_back = ex.rows(y_recv, self.recv_split, self.send_split)
        return self.combine(y_back)


def loopback_forward(ranks: list, us: list, bias: torch.Tensor) -> list:
    """The forward of W ranks emulated in one process, phase by phase."""
    ex = LoopbackExchange(len(ranks))
    sent = [r.dispatch(u, bias) for r, u in zip(ranks, us)]
    recv_counts = ex.counts_all([s[2] for s in sent])
    splits = [r.send_split for r in ranks]
    x_recv = ex.rows_all([s[0] for s in sent], splits)
    xs_recv = ex.rows_all([s[1] for s in sent], splits) if ranks[0].fp8 else [None] * len(ranks)
    y_recv = [r.experts(x, xs, c) for r, x, xs, c in zip(ranks, x_recv, xs_recv, recv_counts)]
    y_back = ex.rows_all(y_recv, [r.recv_split for r in ranks])
    return [r.combine(y) for r, y in zip(ranks, y_back)]
