"""MoELayer: device-resident weights + workspace of one DeepSeekMoE layer.

Plumbing around the C ABI: torch provides the device memory, the library
does every step of the layer.  Weights are loaded one expert at a time from
host tensors (nn.Linear layout: W1, W3 [I, d], W2 [d, I], bf16); the
gate/up pair is interleaved on the device by moe_pack_gate_up and, for FP8,
quantised per 128 x 128 block by moe_quantize_fp8_blocks, so a V3-sized
layer never needs a second full bf16 copy on the device.
"""
from __future__ import annotations

import torch

from . import capi


class MoELayer:
    def __init__(self, T: int, d: int, E: int, k: int, n_shared: int, inter: int, prec: str = "bf16",
                 device: str | torch.device = "cuda", route_groups: int = 0, route_group_limit: int = 0):
        """route_groups, route_group_limit: node-limited routing (moe_dims)."""
        self.T, self.d, self.E, self.k, self.n_shared, self.inter, self.prec = T, d, E, k, n_shared, inter, prec
        self.route_groups, self.route_group_limit = route_groups, route_group_limit
        self.device = torch.device(device)
        self.fp8 = prec in ("fp8", "fp8_ue8m0")
        self.pow2 = prec == "fp8_ue8m0"   # UE8M0 (power-of-two) scales
        self.dims = capi.dims(T, d, E, k, n_shared, inter, prec, route_groups, route_group_limit)
        self.ws = torch.empty(capi.moe_workspace_size(self.dims), dtype=torch.uint8, device=self.device)
        wt = torch.uint8 if self.fp8 else torch.bfloat16
        dev = self.device
        self.w13 = torch.empty((E, 2 * inter, d), dtype=wt, device=dev)
        self.w2 = torch.empty((E, d, inter), dtype=wt, device=dev)
        self.ws13 = torch.empty((max(n_shared, 1), 2 * inter, d), dtype=wt, device=dev)
        self.ws2 = torch.empty((max(n_shared, 1), d, inter), dtype=wt, device=dev)
        if self.fp8:
            f = torch.float32
            self.w13_scale = torch.empty((E, 2 * inter // 128, d // 128), dtype=f, device=dev)
            self.w2_scale = torch.empty((E, d // 128, inter // 128), dtype=f, device=dev)
            self.ws13_scale = torch.empty((max(n_shared, 1), 2 * inter // 128, d // 128), dtype=f, device=dev)
            self.ws2_scale = torch.empty((max(n_shared, 1), d // 128, inter // 128), dtype=f, device=dev)
        else:
            self.w13_scale = self.w2_scale = self.ws13_scale = self.ws2_scale = None
        self.centroids = torch.empty((E, d), dtype=torch.bfloat16, device=dev)
        self._stage13 = torch.empty((2, inter, d), dtype=torch.bfloat16, device=dev)
        self._stage_pack = torch.empty((2 * inter, d), dtype=torch.bfloat16, device=dev)
        self._stage2 = torch.empty((d, inter), dtype=torch.bfloat16, device=dev)

    # ------------------------------------------------------------ weights
    def set_centroids(self, c: torch.Tensor) -> None:
        self.centroids.copy_(c)

    def load_expert(self, e: int, w1: torch.Tensor, w3: torch.Tensor, w2: torch.Tensor, shared: bool = False):
        """Upload one expert's bf16 W1, W3 [I, d] and W2 [d, I]."""
        I, d = self.inter, self.d
        w13 = (self.ws13 if shared else self.w13)[e]
        w2d = (self.ws2 if shared else self.w2)[e]
        self._stage13[0].copy_(w1)
        self._stage13[1].copy_(w3)
        if not self.fp8:
            capi.moe_pack_gate_up(self._stage13[0], self._stage13[1], 1, I, d, w13)
            w2d.copy_(w2)
            return
        capi.moe_pack_gate_up(self._stage13[0], self._stage13[1], 1, I, d, self._stage_pack)
        s13 = (self.ws13_scale if shared else self.w13_scale)[e]
        s2 = (self.ws2_scale if shared else self.w2_scale)[e]
        capi.moe_quantize_fp8_blocks(self._stage_pack, 2 * I, d, w13, s13, pow2_scales=self.pow2)
        self._stage2.copy_(w2)
        capi.moe_quantize_fp8_blocks(self._stage2, d, I, w2d, s2, pow2_scales=self.pow2)

    def release_staging(self) -> None:
        torch.cuda.current_stream().synchronize()
        self._stage13 = self._stage_pack = self._stage2 = None

    def weights(self) -> capi.moe_weights:
        return capi.weights_struct(self.w13, self.w13_scale, self.w2, self.w2_scale,
                                   self.ws13 if self.n_shared else None,
                                   self.ws13_scale if self.n_shared else None,
                                   self.ws2 if self.n_shared else None,
                                   self.ws2_scale if self.n_shared else None, self.centroids)

    # ------------------------------------------------------------ forward
    def forward(self, u: torch.Tensor, bias: torch.Tensor, out: torch.Tensor | None = None,
                counts: torch.Tensor | None = None, stream=None) -> torch.Tensor:
        if out is None:
            out = torch.empty((self.T, self.d), dtype=torch.bfloat16, device=self.device)
        capi.moe_forward(self.dims, self.weights(), u, bias, out, counts, self.ws, stream)
        return out

    def with_tokens(self, T: int) -> "MoELayer":
        """A layer of the same weights (shared, not copied) for batches of T
        tokens, with its own workspace: e.g. the decode-shaped T=256 steps of a
        layer loaded for 8192-token batches."""
        view = MoELayer.__new__(MoELayer)
        view.__dict__.update(self.__dict__)
        view.T = T
        view.dims = capi.dims(T, self.d, self.E, self.k, self.n_shared, self.inter, self.prec, self.route_groups,
                              self.route_group_limit)
        view.ws = torch.empty(capi.moe_workspace_size(view.dims), dtype=torch.uint8, device=self.device)
        return view

    def status(self) -> int:
        return capi.moe_read_device_status(self.ws)

    # ------------------------------------------------------------ backward
    def prepare_backward(self) -> None:
        """Transposed copies of the expert weights (FP8: their codes and block
        scales) and the backward workspace."""
        dev, I, d = self.device, self.inter, self.d
        ns = max(self.n_shared, 1)
        wt = torch.uint8 if self.fp8 else torch.bfloat16
        self.w13t = torch.empty((self.E, d, 2 * I), dtype=wt, device=dev)
        self.w2t = torch.empty((self.E, I, d), dtype=wt, device=dev)
        self.ws13t = torch.empty((ns, d, 2 * I), dtype=wt, device=dev)
        self.ws2t = torch.empty((ns, I, d), dtype=wt, device=dev)
        if self.fp8:
            f = torch.float32
            self.w13t_scale = torch.empty((self.E, d // 128, 2 * I // 128), dtype=f, device=dev)
            self.w2t_scale = torch.empty((self.E, I // 128, d // 128), dtype=f, device=dev)
            self.ws13t_scale = torch.empty((ns, d // 128, 2 * I // 128), dtype=f, device=dev)
            self.ws2t_scale = torch.empty((ns, I // 128, d // 128), dtype=f, device=dev)
            capi.moe_transpose_expert_weights_fp8(self.E, I, d, self.w13, self.w13_scale, self.w2, self.w2_scale,
                                                  self.w13t, self.w13t_scale, self.w2t, self.w2t_scale)
            if self.n_shared:
                capi.moe_transpose_expert_weights_fp8(self.n_shared, I, d, self.ws13, self.ws13_scale, self.ws2,
                                                      self.ws2_scale, self.ws13t, self.ws13t_scale, self.ws2t,
                                                      self.ws2t_scale)
        else:
            self.w13t_scale = self.w2t_scale = self.ws13t_scale = self.ws2t_scale = None
            capi.moe_transpose_expert_weights(self.E, I, d, self.w13, self.w2, self.w13t, self.w2t)
            if self.n_shared:
                capi.moe_transpose_expert_weights(self.n_shared, I, d, self.ws13, self.ws2, self.ws13t, self.ws2t)
        self.ws_bwd = torch.empty(capi.moe_backward_workspace_size(self.dims), dtype=torch.uint8, device=dev)

    def grad_buffers(self) -> dict:
        """Uninitialised fp32 gradient tensors in the shapes backward() writes."""
        dev, I, d, f = self.device, self.inter, self.d, torch.float32
        ns = max(self.n_shared, 1)
        return dict(du=torch.empty((self.T, d), dtype=f, device=dev),
                    dcentroids=torch.empty((self.E, d), dtype=f, device=dev),
                    dw13=torch.empty((self.E, 2 * I, d), dtype=f, device=dev),
                    dw2=torch.empty((self.E, d, I), dtype=f, device=dev),
                    dws13=torch.empty((ns, 2 * I, d), dtype=f, device=dev),
                    dws2=torch.empty((ns, d, I), dtype=f, device=dev))

    def backward(self, u: torch.Tensor, bias: torch.Tensor, dout: torch.Tensor, stream=None,
                 grads: dict | None = None) -> dict:
        """Gradients (fp32) of the layer for dL/dh' = dout: du, dcentroids,
        dw13/dw2 (routed, in the w13/w2 layouts) and dws13/dws2 (shared); for
        an FP8 layer in the FP8 scheme of moe_backward.  grads: tensors from
        grad_buffers() to overwrite (every element is written), else new ones."""
        if not hasattr(self, "ws_bwd"):
            self.prepare_backward()
        g = self.grad_buffers() if grads is None else grads
        ptr = lambda t: t.data_ptr() if t is not None else None
        wt = capi.moe_weights_t(ptr(self.w13t), ptr(self.w2t), ptr(self.ws13t), ptr(self.ws2t), ptr(self.w13t_scale),
                                ptr(self.w2t_scale), ptr(self.ws13t_scale), ptr(self.ws2t_scale))
        gr = capi.moe_grads(*(g[k].data_ptr() for k in ("du", "dcentroids", "dw13", "dw2", "dws13", "dws2")))
        capi.moe_backward(self.dims, self.weights(), wt, u, bias, dout, gr, self.ws_bwd, stream)
        return g

    def backward_status(self) -> int:
        return capi.moe_read_device_status(self.ws_bwd)


class CapturedForward:
    """The layer's forward recorded once in a CUDA graph and replayed.

    A forward enqueues ~10 kernels and two small memsets and never waits on
    the device or allocates, so the whole call captures into one graph; a
    replay then costs one launch from the host.  The graph reads its own
    input buffer (u is copied in), the bias tensor given here (its current
    contents at each replay, so moe_bias_update may change it in place) and
    writes its own output and counts buffers."""

    def __init__(self, layer: MoELayer, bias: torch.Tensor):
        dev = layer.device
        self.layer, self.bias = layer, bias
        self.u = torch.zeros((layer.T, layer.d), dtype=torch.bfloat16, device=dev)
        self.out = torch.empty((layer.T, layer.d), dtype=torch.bfloat16, device=dev)
        self.counts = torch.zeros(layer.E, dtype=torch.int32, device=dev)
        side = torch.cuda.Stream(device=dev)          # warm-up off the capturing stream, as torch requires
        side.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(side):
            layer.forward(self.u, bias, self.out, counts=self.counts)
        torch.cuda.current_stream(dev).wait_stream(side)
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            layer.forward(self.u, bias, self.out, counts=self.counts)

    def __call__(self, u: torch.Tensor) -> torch.Tensor:
        self.u.copy_(u)
        self.graph.replay()
        return self.out


class HostPipeline:
    """The layer over batches that live in pinned host memory.

    Batch i's copy to the device, batch i's forward and batch i's result copy
    back run on three streams, with two device buffers each way, so the copy of
    batch i+1 in and of batch i-1 out overlap the forward of batch i.  Every
    batch still makes the whole round trip: u from host to device, h' from
    device to host.  Batches run one forward at a time (the forwards share the
    layer's workspace).
    """

    DEPTH = 2

    def __init__(self, layer: MoELayer):
        self.layer = layer
        dev = layer.device
        self.u = [torch.empty((layer.T, layer.d), dtype=torch.bfloat16, device=dev) for _ in range(self.DEPTH)]
        self.out = [torch.empty((layer.T, layer.d), dtype=torch.bfloat16, device=dev) for _ in range(self.DEPTH)]
        self.s_in, self.s_run, self.s_out = (torch.cuda.Stream(dev) for _ in range(3))
        ev = lambda: [torch.cuda.Event() for _ in range(self.DEPTH)]
        self.copied_in, self.computed, self.copied_out = ev(), ev(), ev()
        self.used = [False] * self.DEPTH

    def run(self, u_host, bias: torch.Tensor, out_host, after: torch.cuda.Stream | None = None) -> None:
        """u_host, out_host: sequences of pinned [T, d] bf16 host tensors (the
        same tensor may repeat).  The calling stream (or `after`) waits for the
        last copy back before it continues."""
        start = torch.cuda.current_stream() if after is None else after
        self.s_in.wait_stream(start)
        for i, (uh, oh) in enumerate(zip(u_host, out_host)):
            b = i % self.DEPTH
            if self.used[b]:
                self.s_in.wait_event(self.computed[b])        # the forward that read u[b] is done
            with torch.cuda.stream(self.s_in):
                self.u[b].copy_(uh, non_blocking=True)
                self.copied_in[b].record(self.s_in)
            self.s_run.wait_event(self.copied_in[b])
            if self.used[b]:
                self.s_run.wait_event(self.copied_out[b])     # out[b] of two batches ago is on the host
            self.layer.forward(self.u[b], bias, self.out[b], stream=self.s_run)
            self.computed[b].record(self.s_run)
            self.s_out.wait_event(self.computed[b])
            with torch.cuda.stream(self.s_out):
                oh.copy_(self.out[b], non_blocking=True)
                self.copied_out[b].record(self.s_out)
            self.used[b] = True
        start.wait_stream(self.s_out)


class ReplicatedExperts:
    """Copies of the most loaded experts of a layer (moe_plan_replicas), run
    by moe_forward_replicated: the copies share the layer's weights, and the
    plan tables live on the device with a workspace sized for the slots."""

    def __init__(self, layer: MoELayer, counts: torch.Tensor, n_extra: int):
        first, copies, slot_expert = capi.moe_plan_replicas(counts.detach().cpu(), n_extra)
        self.layer = layer
        self.replica_count_host = copies
        self.slot_expert_host = slot_expert
        dev = layer.device
        self.replica_first = first.to(dev)
        self.replica_count = copies.to(dev)
        self.slot_expert = slot_expert.to(dev)
        wd = capi.dims(layer.T, layer.d, layer.E + n_extra, layer.k, layer.n_shared, layer.inter, layer.prec)
        self.ws = torch.empty(capi.moe_workspace_size(wd), dtype=torch.uint8, device=dev)

    def forward(self, u: torch.Tensor, bias: torch.Tensor, out: torch.Tensor | None = None,
                counts: torch.Tensor | None = None, stream=None) -> torch.Tensor:
        L = self.layer
        if out is None:
            out = torch.empty((L.T, L.d), dtype=torch.bfloat16, device=L.device)
        capi.moe_forward_replicated(L.dims, L.weights(), u, bias, self.replica_first, self.replica_count,
                                    self.slot_expert, out, counts, self.ws, stream)
        return out

    def status(self) -> int:
        return capi.moe_read_device_status(self.ws)
