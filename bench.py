"""Benchmark of the B300 DeepSeekMoE layer forward.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload v3|v3_fp8|mid|decode] [--no-variants]

One step = one moe_forward over the workload's T tokens (V3 shape by default:
T=8192, d=7168, 256 routed experts top-8 + 1 shared, I=2048, bf16), inputs
resident in HBM.  Prints one JSON line (rank 0).  With torchrun (N > 1) every
rank runs an independent replica of the layer on its own GPU and its own
tokens (the forward has no cross-token exchange), value = all ranks' tokens /
the slowest rank's time ("scaling": "weak").

The reference arm (--impl reference) times the CPU oracle, as it stands, on a
bounded sample of the same workload on this host's cores.
"""
from __future__ import annotations

import argparse
import csv
import hashlib
import io
import json
import os
import statistics
import subprocess
import sys
import time
from dataclasses import replace

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "MoE layer tokens/s at V3 shape (bf16, FP8); % of tensor/HBM roofline"
UNIT = "tokens/s"
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "traffic.json")
# the sources of the expert GEMM kernels: a recorded DRAM-traffic figure is
# reported only while these are unchanged since its ncu capture
KERNEL_SOURCES = [os.path.join(ROOT, "mixture_experts_layer_87_b300", "csrc", f)
                  for f in ("gemm.cuh", "expert_gemm.cuh", "fp8_gemm.cuh", "ptx.cuh")]


# ----------------------------------------------------------------------------
# distributed plumbing
def dist_init():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    from mixture_experts_layer_87_b300 import replicas
    replicas.barrier()


def max_over_ranks(x: float, world: int) -> float:
    from mixture_experts_layer_87_b300 import replicas
    return replicas.max_over_ranks(x, device="cuda")


# ----------------------------------------------------------------------------
# peaks and clocks
FALLBACK_PEAKS = dict(hbm=6400.0, bf16=1800.0, bf16_sus=1400.0)
# B300 HBM3e nominal bandwidth, reported beside the measured copy bandwidth
NOMINAL_HBM_GBS = 7700.0


def _peak_number(v):
    """A peak given as a number, or as an object holding one (value / median / mean)."""
    if isinstance(v, (int, float)) and not isinstance(v, bool):
        return float(v)
    if isinstance(v, str):
        return float(v)
    if isinstance(v, dict):
        for key in ("value", "median", "mean", "gbs", "tflops"):
            if key in v:
                return _peak_number(v[key])
    raise ValueError(f"no number in {v!r}")


def peaks(path=None):
    """Roofline denominators: the peaks measured on this machine when MEASURED_PEAKS.json
    is present and readable, else the fallback figures (source says which).
    bf16 is the burst figure (cuBLAS timed alone, at full clocks): the expert
    GEMMs are timed one forward at a time, a few milliseconds each, not in a
    seconds-long loop at the power cap.  bf16_sus is reported beside it."""
    path = path or os.path.join(ROOT, "MEASURED_PEAKS.json")
    if not os.path.exists(path):
        return dict(FALLBACK_PEAKS, source="fallback")
    try:
        p = json.load(open(path))
        bf16 = _peak_number(p["bf16_tflops"])
        sus = _peak_number(p["bf16_tflops_sustained"]) if "bf16_tflops_sustained" in p else bf16
        return dict(hbm=_peak_number(p["hbm_gbs"]), bf16=bf16, bf16_sus=sus, source="measured")
    except (OSError, ValueError, KeyError, TypeError) as e:
        return dict(FALLBACK_PEAKS, source=f"fallback (MEASURED_PEAKS.json unreadable: {type(e).__name__})")


def _best_ms(fn, reps: int = 10, warm: int = 5) -> float:
    for _ in range(warm):
        fn()
    best = float("inf")
    for _ in range(reps):
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        fn()
        e.record()
        torch.cuda.synchronize()
        best = min(best, s.elapsed_time(e))
    return best


def measure_fp8_peak(bf16_burst: float):
    """Dense FP8 (E4M3 x E4M3 -> bf16, fp32 accumulation) tensor peak of this
    GPU, stated on the same footing as the bf16 burst peak: cuBLASLt through
    torch._scaled_mm and cuBLAS through torch.matmul at 8192^3 (2 N^3 flops),
    timed back to back in this process (best of 10 after 5 warm-up calls,
    CUDA events); the FP8:bf16 ratio measured here times the bf16 burst.  A
    GPU that is warm or power-capped at this moment slows both GEMMs alike,
    so the ratio, unlike a raw FP8 figure, does not depend on when the
    measurement ran.  Returns (peak, raw fp8, raw bf16) in TFLOP/s, or None if
    the FP8 call is not available here."""
    try:
        n = 8192
        g = torch.Generator(device="cuda").manual_seed(0)
        a = torch.randn((n, n), device="cuda", generator=g)
        b = torch.randn((n, n), device="cuda", generator=g)
        a8, b8 = a.to(torch.float8_e4m3fn), b.to(torch.float8_e4m3fn).t()   # column-major second operand
        a16, b16 = a.to(torch.bfloat16), b.to(torch.bfloat16)
        del a, b
        one = torch.ones((), device="cuda", dtype=torch.float32)
        flop = 2.0 * n ** 3
        t8 = _best_ms(lambda: torch._scaled_mm(a8, b8, scale_a=one, scale_b=one, out_dtype=torch.bfloat16))
        t16 = _best_ms(lambda: torch.matmul(a16, b16))
        del a8, b8, a16, b16
        torch.cuda.empty_cache()
        fp8, bf16 = flop / (t8 * 1e-3) / 1e12, flop / (t16 * 1e-3) / 1e12
        return fp8 / bf16 * bf16_burst, fp8, bf16
    except Exception:  # pragma: no cover - depends on the torch build
        return None


def tensor_peak(cfg, pk):
    """(TFLOP/s, description) the expert GEMMs of this precision are measured against."""
    if cfg.prec == "bf16":
        return pk["bf16"], f"bf16 burst ({pk['source']})"
    if pk.get("fp8"):
        return pk["fp8"], ("fp8: bf16 burst x the FP8:bf16 ratio measured here (cuBLASLt E4M3 / cuBLAS bf16, "
                           "8192^3, best of 10 each, back to back)")
    return 2 * pk["bf16"], f"2 x bf16 burst ({pk['source']}; nominal fp8:bf16 ratio, fp8 not measurable here)"


class ClockSampler:
    """nvidia-smi sampling of this GPU's clocks during the timed region."""

    FIELDS = ("uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self):
        self.proc = None
        try:
            self.uuid = str(torch.cuda.get_device_properties(torch.cuda.current_device()).uuid)
        except Exception:
            self.uuid = None

    def start(self):
        if not self.uuid:
            return                      # without this GPU's id, other GPUs' clocks could be reported
        gid = self.uuid if self.uuid.startswith("GPU-") else "GPU-" + self.uuid
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", gid, f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            why = "nvidia-smi unavailable" if self.uuid else "GPU uuid unknown: not sampled"
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [why]}
        time.sleep(0.25)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        rows = [r for r in csv.reader(io.StringIO(out)) if len(r) >= 9]
        rows = [r for r in rows if self.uuid.replace("GPU-", "") in r[0]]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no sample of this GPU's uuid"], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].strip().replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].strip().replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if "Active" in v and "Not" not in v})
        load = [s for s in sm if s > 0.5 * max(sm)] if sm else []
        return {"sm_mhz": statistics.median(load) if load else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(rows)}


# ----------------------------------------------------------------------------
# workload
def build_layer(cfg, T=None):
    from mixture_experts_layer_87_b300 import MoELayer
    layer = MoELayer(cfg.T if T is None else T, cfg.d, cfg.E, cfg.k, cfg.n_shared, cfg.inter, cfg.prec)
    layer.set_centroids(synth.centroids(cfg))
    for e in range(cfg.E):
        layer.load_expert(e, *synth.expert_weights(cfg, e))
    for s in range(cfg.n_shared):
        layer.load_expert(s, *synth.expert_weights(cfg, s, shared=True), shared=True)
    layer.release_staging()
    return layer


def stage_work(cfg, counts: np.ndarray):
    """Algorithmic FLOPs and bytes of every stage of one forward (padding and
    repeated reads excluded)."""
    T, d, E, k, Ns, I = cfg.T, cfg.d, cfg.E, cfg.k, cfg.n_shared, cfg.inter
    fp8 = cfg.is_fp8
    wb, xb = (1, 1) if fp8 else (2, 2)
    R = T * k
    active = int((counts > 0).sum())
    s13 = (2 * I // 128) * (d // 128) * 4 if fp8 else 0
    s2 = (d // 128) * (I // 128) * 4 if fp8 else 0
    xs = R * (d // 128) * 4 if fp8 else 0
    hs = R * (I // 128) * 4 if fp8 else 0
    w = {
        "router_gemm": (2 * T * d * E, T * d * 2 + E * d * 2 + T * E * 4),
        "topk": (0, T * E * 4 + R * 8),
        "scan_plan": (0, 0),
        # FP8 with shared experts: the gather also writes u's own codes and scales once per token
        "gather": (0, T * d * 2 + R * d * xb + xs + (T * d + T * (d // 128) * 4 if fp8 and Ns else 0)),
        "routed_gate_up": (2 * R * d * 2 * I, active * (2 * I * d * wb + s13) + R * d * xb + xs + R * I * xb + hs),
        "routed_down": (2 * R * I * d, active * (d * I * wb + s2) + R * I * xb + hs + R * d * 2),
        "shared_gate_up": (2 * Ns * T * d * 2 * I,
                           Ns * (2 * I * d * wb + s13) + T * d * xb + Ns * T * I * xb),
        "shared_down": (2 * Ns * T * I * d, Ns * (d * I * wb + s2) + Ns * T * I * xb + Ns * T * d * 2),
        "combine": (0, (1 + Ns + k) * T * d * 2 + T * d * 2 + R * 8),
    }
    return w


def layer_work(cfg, counts):
    """The layer's algorithmic FLOPs and bytes (weights of the experts used, u in, h' out)."""
    T, d, E, k, Ns, I = cfg.T, cfg.d, cfg.E, cfg.k, cfg.n_shared, cfg.inter
    fp8 = cfg.is_fp8
    wb = 1 if fp8 else 2
    active = int((counts > 0).sum())
    F = 2 * T * d * E + 2 * T * (k + Ns) * 3 * d * I
    scales = ((2 * I // 128) * (d // 128) + (d // 128) * (I // 128)) * 4 if fp8 else 0
    B = (active + Ns) * (3 * d * I * wb + scales) + E * d * 2 + T * d * 2 * 2
    return F, B


def kernel_traffic(kernel: str, workload: str):
    """dram bytes per launch from the committed ncu summary, if the kernel
    sources still match the ones that were profiled."""
    if not os.path.exists(PROFILE_TRAFFIC):
        return None
    rec = json.load(open(PROFILE_TRAFFIC)).get(f"{workload}/{kernel}")
    if not rec:
        return None
    h = hashlib.sha256()
    for p in KERNEL_SOURCES:
        h.update(open(p, "rb").read())
    if rec.get("sources_sha256") != h.hexdigest():
        return None
    return rec.get("dram_bytes_per_launch")


def sources_hash() -> str:
    h = hashlib.sha256()
    for p in KERNEL_SOURCES:
        h.update(open(p, "rb").read())
    return h.hexdigest()


def roofline(cfg, stage_ms: dict, counts, pk, kernel="routed_gate_up"):
    """The kernel against its roofline: the slower of its algorithmic flops at
    the tensor peak and its algorithmic bytes at the HBM copy bandwidth.
    tensor_frac and hbm_frac give both sides; frac is the bound's."""
    F, B = stage_work(cfg, counts)[kernel]
    t = stage_ms[kernel] * 1e-3
    peak_tf, peak_what = tensor_peak(cfg, pk)
    t_f, t_b = F / (peak_tf * 1e12), B / (pk["hbm"] * 1e9)
    if t_f >= t_b:
        ach, peak, unit, bound = F / t / 1e12, peak_tf, "TFLOP/s", "tensor"
    else:
        ach, peak, unit, bound = B / t / 1e9, pk["hbm"], "GB/s", "hbm"
    return {"kernel": kernel, "bound": bound, "achieved": round(ach, 2), "peak": round(peak, 1), "unit": unit,
            "frac": round(ach / peak, 4), "traffic": kernel_traffic(kernel, cfg.name),
            "tensor_frac": round(t_f / t, 4), "hbm_frac": round(t_b / t, 4),
            "hbm_frac_of_nominal": round(B / t / 1e9 / NOMINAL_HBM_GBS, 4),
            "tflops": round(F / t / 1e12, 1), "gbs": round(B / t / 1e9, 1),
            "algorithmic_bytes": int(B), "algorithmic_flops": int(F), "ms": round(stage_ms[kernel], 4),
            "peak_source": f"tensor: {peak_what}; HBM: copy bandwidth ({pk['source']})",
            "frac_of_sustained_bf16": round(F / t / 1e12 / (pk["bf16_sus"] * (1 if cfg.prec == "bf16" else 2)), 4)}


# ----------------------------------------------------------------------------
# timing
def time_forward(layer, u, bias, out, steps, warmup, world):
    for _ in range(warmup):
        layer.forward(u, bias, out)
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record()
    for _ in range(steps):
        layer.forward(u, bias, out)
    e.record()
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    return s.elapsed_time(e) / steps


def time_stages(layer, u, bias, out, steps):
    from mixture_experts_layer_87_b300 import capi
    stages = capi.PROFILE_STAGES
    acc = {s: 0.0 for s in stages}
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(capi.MOE_PROFILE_EVENTS)]
    for e in evs:
        e.record()          # creates the underlying events
    torch.cuda.synchronize()
    for _ in range(steps):
        capi.moe_forward_profiled(layer.dims, layer.weights(), u, bias, out, None, layer.ws, evs)
        torch.cuda.synchronize()
        for i, st in enumerate(stages):
            acc[st] += evs[i].elapsed_time(evs[i + 1])
    return {s: v / steps for s, v in acc.items()}


def time_e2e(layer, u_host, bias, steps, warmup, world):
    """Same metric through the public call with host buffers: every step copies
    its u from pinned host memory to the device and its h' back, inside the
    timed region; the copies of neighbouring steps overlap the forward
    (layer.HostPipeline)."""
    from mixture_experts_layer_87_b300 import HostPipeline
    pipe = HostPipeline(layer)
    out_host = [torch.empty((layer.T, layer.d), dtype=torch.bfloat16, pin_memory=True)
                for _ in range(HostPipeline.DEPTH)]
    outs = lambda n: [out_host[i % len(out_host)] for i in range(n)]
    pipe.run([u_host] * warmup, bias, outs(warmup))
    torch.cuda.synchronize()
    barrier(world)
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record()
    pipe.run([u_host] * steps, bias, outs(steps))
    e.record()
    torch.cuda.synchronize()
    barrier(world)
    ms = s.elapsed_time(e) / steps
    return ms, u_host.numel() * 2, out_host[0].numel() * 2


# ----------------------------------------------------------------------------
# CPU oracle (baseline leg and reference arm)
def oracle_sample(cfg, u_host, sample, cache=None):
    """Time the oracle on tokens `sample` of the batch: routing + the full
    layer output of those tokens.  Input generation is excluded (timed and
    subtracted); with a cache dict the generated expert weights are kept for
    the next call."""
    import oracle
    ub = synth.bf16_bits(u_host)[sample]
    cent = synth.bf16_bits(synth.centroids(cfg))
    bias = np.asarray(synth.bias(cfg))
    gen = [0.0]

    def getter(shared):
        def f(e):
            key = (shared, e)
            if cache is not None and key in cache:
                return cache[key]
            t0 = time.perf_counter()
            w = tuple(synth.bf16_bits(w).copy() for w in synth.expert_weights(cfg, e, shared=shared))
            gen[0] += time.perf_counter() - t0
            if cache is not None:
                cache[key] = w
            return w
        return f

    t0 = time.perf_counter()
    r = oracle.route(ub, cent, bias, cfg.k)
    oracle.layer_output(ub, np.arange(len(sample)), r["idx"], r["gate"], getter(False), getter(True),
                        cfg.n_shared, cfg.E, fp8=cfg.oracle_fp8)
    return time.perf_counter() - t0 - gen[0]


def oracle_route_all(cfg, u_host):
    """Seconds the oracle takes to route the whole batch."""
    import oracle
    ub = synth.bf16_bits(u_host)
    cent = synth.bf16_bits(synth.centroids(cfg))
    t0 = time.perf_counter()
    oracle.route(ub, cent, np.asarray(synth.bias(cfg)), cfg.k)
    return time.perf_counter() - t0


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def host_cpu_model() -> str:
    try:
        for line in open("/proc/cpuinfo"):
            if line.startswith("model name"):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def workload_config(cfg, world=1):
    """The `config` object of the bench line; the reference arm prints the same."""
    wbytes = (cfg.E + cfg.n_shared) * 3 * cfg.d * cfg.inter * (2 if cfg.prec == "bf16" else 1)
    shape = "DeepSeek-V3-shaped" if cfg.d == 7168 else "mid-sized"
    return {"workload": f"{shape} MoE layer forward ({cfg.name}): T={cfg.T}, d={cfg.d}, {cfg.E} routed experts "
                        f"top-{cfg.k} + {cfg.n_shared} shared, I={cfg.inter}, {cfg.prec}, clustered tokens",
            "T": cfg.T, "d": cfg.d, "E": cfg.E, "k": cfg.k, "n_shared": cfg.n_shared, "inter": cfg.inter,
            "prec": cfg.prec, "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
            "l2": f"inputs larger than L2: every step streams the expert weights ({wbytes / 1e9:.1f} GB)"}


# ----------------------------------------------------------------------------
def run_reference(args, world, rank):
    """The CPU oracle on this host's cores, on bounded samples of the workload:
    each step takes the routing and the full layer output of a strided token
    sample, sized so that all warm-up and timed steps take a few minutes."""
    if rank != 0:
        return
    cfg = synth.get_config(args.workload)
    u = synth.tokens(cfg)
    # ~0.25 s of oracle work per sampled token when the sample is small (few
    # rows per expert to spread over the cores): ~150 s for the whole run
    per_step = args.ref_tokens or int(min(512, max(4, 150.0 / (args.steps + args.warmup) / 0.25)))
    stride = max(1, cfg.T // per_step)
    sample = np.arange(0, cfg.T, stride)[:per_step]
    cache = {}
    for _ in range(args.warmup):
        oracle_sample(cfg, u, sample, cache)
    secs = [oracle_sample(cfg, u, sample, cache) for _ in range(args.steps)]
    total = sum(secs)
    value = per_step * args.steps / total
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * total / args.steps, 2),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(cfg, args.gpus),
            "cpu_baseline": {"value": round(value, 3), "unit": UNIT, "cores": host_cores(), "kind": "oracle",
                             "cpu": host_cpu_model(),
                             "sample": f"{per_step} tokens (every {stride}th) of the {cfg.T}-token batch per step: "
                                       f"routing + full layer output in the fp64 C oracle (OpenMP over rows), "
                                       f"input generation excluded"},
            "e2e": {"value": round(value, 3), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def measure(cfg, args, world, pk):
    layer = build_layer(cfg)
    # every replica runs the layer on its own batch of T tokens (weak scaling)
    rank = int(os.environ.get("RANK", "0"))
    u_host = synth.tokens(cfg, step=rank)
    u = u_host.cuda()
    bias = synth.bias(cfg).cuda()
    out = torch.empty((cfg.T, cfg.d), dtype=torch.bfloat16, device="cuda")
    counts = torch.zeros(cfg.E, dtype=torch.int32, device="cuda")
    layer.forward(u, bias, out, counts=counts)
    if layer.status() != 0:
        raise RuntimeError(f"device status {layer.status()}")
    counts_np = counts.cpu().numpy()
    ms = time_forward(layer, u, bias, out, args.steps, args.warmup, world)
    ms = max_over_ranks(ms, world)
    stage_ms = time_stages(layer, u, bias, out, max(3, args.steps // 2))
    F, B = layer_work(cfg, counts_np)
    peak_tf, _ = tensor_peak(cfg, pk)
    t_f, t_b = F / (peak_tf * 1e12), B / (pk["hbm"] * 1e9)
    res = {"ms_per_step": ms, "value": world * cfg.T / (ms * 1e-3), "stage_ms": stage_ms,
           "roofline": roofline(cfg, stage_ms, counts_np, pk),
           "layer_roofline_frac": max(t_f, t_b) / (ms * 1e-3),
           "layer_bound": "tensor" if t_f >= t_b else "hbm",
           "layer_tflops": F / (ms * 1e-3) / 1e12, "layer_gbs": B / (ms * 1e-3) / 1e9,
           "max_over_mean_load": float(counts_np.max() / (cfg.T * cfg.k / cfg.E)),
           "layer": layer, "u_host": u_host, "bias": bias, "counts": counts_np}
    return res


def variant_summary(r):
    return {"value": round(r["value"], 1), "ms_per_step": round(r["ms_per_step"], 4), "roofline": r["roofline"],
            "layer_roofline_frac": round(r["layer_roofline_frac"], 4), "layer_bound": r["layer_bound"],
            "layer_tflops": round(r["layer_tflops"], 1), "max_over_mean_load": round(r["max_over_mean_load"], 3),
            "stage_ms": {k: round(v, 4) for k, v in r["stage_ms"].items()}}


def measure_decode(args, world, pk, layer=None):
    """50 steps of 256 fresh tokens with the bias update between steps."""
    from mixture_experts_layer_87_b300 import capi
    cfg = synth.get_config("decode")
    if layer is None:
        layer = build_layer(cfg)
    # replica r draws its tokens of step s from the stream position r * steps + s;
    # the bias update sees the loads of all replicas (one all-reduce of E int32)
    from mixture_experts_layer_87_b300 import replicas
    rank = int(os.environ.get("RANK", "0"))
    us = [synth.tokens(cfg, step=rank * cfg.steps + s).cuda() for s in range(cfg.steps)]
    bias = torch.zeros(cfg.E, dtype=torch.float32, device="cuda")
    out = torch.empty((cfg.T, cfg.d), dtype=torch.bfloat16, device="cuda")
    counts = torch.zeros((cfg.steps, cfg.E), dtype=torch.int32, device="cuda")

    def loop(b):
        for s in range(cfg.steps):
            layer.forward(us[s], b, out, counts=counts[s])
            replicas.global_counts(counts[s])
            capi.moe_bias_update(cfg.E, world * cfg.T, cfg.k, counts[s], cfg.gamma, b)

    loop(torch.zeros_like(bias))           # warm-up pass
    torch.cuda.synchronize()
    barrier(world)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(cfg.steps + 1)]
    ev[0].record()
    for s in range(cfg.steps):
        layer.forward(us[s], bias, out, counts=counts[s])
        replicas.global_counts(counts[s])
        capi.moe_bias_update(cfg.E, world * cfg.T, cfg.k, counts[s], cfg.gamma, bias)
        ev[s + 1].record()
    torch.cuda.synchronize()
    barrier(world)
    step_ms = [ev[s].elapsed_time(ev[s + 1]) for s in range(cfg.steps)]
    total = max_over_ranks(sum(step_ms), world)
    stage_ms = time_stages(layer, us[0], bias, out, 5)
    c = counts.cpu().numpy()
    mean = world * cfg.T * cfg.k / cfg.E
    gbs = [layer_work(cfg, c[s])[1] / (step_ms[s] * 1e-3) / 1e9 for s in range(cfg.steps)]
    return {"value": world * cfg.T * cfg.steps / (total * 1e-3), "ms_per_step": total / cfg.steps,
            "hbm_gbs_mean": round(float(np.mean(gbs)), 1),
            "hbm_frac_of_measured": round(float(np.mean(gbs)) / pk["hbm"], 4),
            "hbm_frac_of_nominal": round(float(np.mean(gbs)) / NOMINAL_HBM_GBS, 4),
            "max_over_mean_load_first": round(float(c[0].max() / mean), 3),
            "max_over_mean_load_last": round(float(c[-1].max() / mean), 3),
            "stage_ms": {k: round(v, 4) for k, v in stage_ms.items()},
            "per_step": [{"ms": round(m, 4), "hbm_gbs": round(g, 1), "max_over_mean": round(float(x.max() / mean), 3)}
                         for m, g, x in zip(step_ms, gbs, c)]}


def measure_replicated(layer, cfg, res, args, world, n_extra=32):
    """moe_forward_replicated on the same batch: n_extra copies of the most
    loaded experts, planned from this batch's loads (the copies share the
    weights on one GPU; the output is moe_forward's)."""
    from mixture_experts_layer_87_b300 import ReplicatedExperts
    rep = ReplicatedExperts(layer, torch.from_numpy(res["counts"]), n_extra)
    u = res["u_host"].cuda()
    out = torch.empty((cfg.T, cfg.d), dtype=torch.bfloat16, device="cuda")
    ms = time_forward(rep, u, res["bias"], out, args.steps, args.warmup, world)
    if rep.status() != 0:
        raise RuntimeError(f"replicated forward device status {rep.status()}")
    copies = rep.replica_count_host.numpy()
    per_copy = res["counts"] / copies
    return {"value": round(world * cfg.T / (ms * 1e-3), 1), "unit": UNIT, "ms_per_step": round(ms, 4),
            "n_extra": n_extra, "max_over_mean_load_per_copy": round(float(per_copy.max() / per_copy.mean()), 3),
            "note": "moe_forward_replicated, the extra copies planned from this batch's loads"}


def measure_backward(layer, cfg, u, bias, pk, steps=5, warmup=3):
    """The layer's backward pass on the same batch (bf16, or the FP8 scheme for
    an FP8 layer): dL/dh' a seeded Gaussian, all gradients (du, dcentroids,
    every expert's dW in fp32)."""
    layer.prepare_backward()
    g = torch.Generator(device="cuda").manual_seed(1)
    dout = torch.randn((cfg.T, cfg.d), device="cuda", generator=g).to(torch.bfloat16)
    for _ in range(warmup):
        grads = layer.backward(u, bias, dout)
    torch.cuda.synchronize()
    if layer.backward_status() != 0:
        raise RuntimeError(f"backward device status {layer.backward_status()}")
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record()
    for _ in range(steps):
        grads = layer.backward(u, bias, dout)
    e.record()
    torch.cuda.synchronize()
    ms = s.elapsed_time(e) / steps
    del grads
    T, d, E, k, Ns, I = cfg.T, cfg.d, cfg.E, cfg.k, cfg.n_shared, cfg.inter
    # algorithmic work: the forward's expert GEMMs recomputed, two data-gradient
    # and two weight-gradient products per expert; weights read twice (w and
    # its transpose; 1 byte each in FP8), fp32 weight gradients written.  In
    # the FP8 scheme the recompute and the data gradients run on the FP8
    # tensor path and the weight gradients on the bf16 one.
    wb = 1 if cfg.is_fp8 else 2
    f_ffn = 2 * T * (k + Ns) * 3 * d * I
    F = 3 * f_ffn + 2 * T * d * E
    B = (E + Ns) * 3 * d * I * (wb + wb + 4) + E * d * (2 + 4) + T * d * (2 + 2 + 4)
    if cfg.is_fp8 and pk.get("fp8"):
        t_f = 2 * f_ffn / (pk["fp8"] * 1e12) + (f_ffn + 2 * T * d * E) / (pk["bf16"] * 1e12)
    else:
        t_f = F / (pk["bf16"] * 1e12)
    t_b = B / (pk["hbm"] * 1e9)
    return {"value": round(T / (ms * 1e-3), 1), "unit": "tokens/s", "ms_per_step": round(ms, 3),
            "tflops": round(F / (ms * 1e-3) / 1e12, 1), "gbs": round(B / (ms * 1e-3) / 1e9, 1),
            "roofline_frac": round(max(t_f, t_b) / (ms * 1e-3), 4), "bound": "tensor" if t_f >= t_b else "hbm",
            "algorithmic_flops": int(F), "algorithmic_bytes": int(B)}


def cpu_baseline_leg(cfg, u_host, n_sample):
    """The oracle beside the GPU: routing of the whole batch, and the routing +
    full layer output of a strided sample of n_sample tokens (tokens are
    independent, so the sample's tokens/s is the layer's)."""
    stride = max(1, cfg.T // n_sample)
    sample = np.arange(0, cfg.T, stride)[:n_sample]
    secs = oracle_sample(cfg, u_host, sample)
    route_s = oracle_route_all(cfg, u_host)
    return {"value": round(len(sample) / secs, 3), "unit": UNIT, "cores": host_cores(), "kind": "oracle",
            "cpu": host_cpu_model(), "seconds": round(secs, 2),
            "route_all_tokens_per_s": round(cfg.T / route_s, 1),
            "sample": f"{len(sample)} tokens (every {stride}th) of the {cfg.T}-token batch: routing + full layer "
                      f"output in the fp64 C oracle (OpenMP over rows), input generation excluded; the routing "
                      f"of all {cfg.T} tokens is timed apart (route_all_tokens_per_s)"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="v3", choices=["v3", "v3_fp8", "v3_ue8m0", "v3_nodes", "mid", "decode",
                                                            "v3_slice", "v3_slice_fp8", "decode_slice", "v3_tokens",
                                                            "v3_tokens_fp8", "bwd_slice"])
    ap.add_argument("--no-variants", action="store_true", help="skip the mid, FP8 and decode measurements")
    ap.add_argument("--prec", default=None, choices=["bf16", "fp8", "fp8_ue8m0"],
                    help="override the workload's precision")
    ap.add_argument("--tokens", type=int, default=0,
                    help="override the workload's token count T (its name gets a _T<n> suffix; no variants)")
    ap.add_argument("--cpu-tokens", type=int, default=512, help="tokens in the CPU-oracle baseline sample")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU-oracle baseline leg")
    ap.add_argument("--ref-tokens", type=int, default=0,
                    help="tokens per step of the reference arm (0: sized so the run takes a few minutes)")
    ap.add_argument("--backward", action="store_true", help="with --profile-case: backward passes")
    ap.add_argument("--profile-case", action="store_true",
                    help="only build the layer and run warmup+steps forwards (the command ncu wraps)")
    ap.add_argument("--write-traffic", nargs=3, metavar=("KEY", "BYTES", "SOURCE"),
                    help="record measured DRAM bytes per launch of KEY (workload/stage) in profiles/traffic.json, "
                         "stamped with the hash of the current kernel sources; SOURCE says where the figure comes from")
    args = ap.parse_args()
    if args.write_traffic:
        key, nbytes, source = args.write_traffic
        rec = json.load(open(PROFILE_TRAFFIC)) if os.path.exists(PROFILE_TRAFFIC) else {}
        rec[key] = {"dram_bytes_per_launch": int(float(nbytes)), "sources_sha256": sources_hash(), "source": source}
        with open(PROFILE_TRAFFIC, "w") as f:
            json.dump(rec, f, indent=1, sort_keys=True)
            f.write("\n")
        return
    if args.profile_case:
        profile_case(args)
        return
    args.warmup = max(args.warmup, 3)

    if args.impl == "reference":
        # CPU only: rank 0 times the oracle, other ranks exit without work
        run_reference(args, int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")))
        return
    world, rank, _ = dist_init()

    from mixture_experts_layer_87_b300 import capi
    capi.lib()
    pk = peaks()
    if rank == 0 or world > 1:
        m = measure_fp8_peak(pk["bf16"])
        if m:
            pk["fp8"], pk["fp8_raw"], pk["bf16_raw"] = m
    clocks = ClockSampler()
    if args.workload == "decode":
        clocks.start()
        dec = measure_decode(args, world, pk)
        clk = clocks.stop()
        if rank == 0:
            print(json.dumps({"metric": METRIC, "value": round(dec["value"], 1), "unit": UNIT, "n_gpus": world,
                              "steps": 50, "warmup": 1, "ms_per_step": round(dec["ms_per_step"], 4),
                              "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "fp8-e4m3",
                              "data": "synthetic", "config": {"workload": "decode"}, "clocks": clk, "decode": dec}))
        return

    cfg = layer_config(args)
    clocks.start()
    res = measure(cfg, args, world, pk)
    clk = clocks.stop()
    layer = res["layer"]
    e2e_ms, h2d, d2h = time_e2e(layer, res["u_host"].pin_memory(), res["bias"], args.steps, args.warmup, world)
    e2e_ms = max_over_ranks(e2e_ms, world)
    launches_per_step = 8 + (2 if cfg.n_shared else 0)

    variants = {}
    if not args.no_variants and args.workload == "v3" and not args.tokens:
        variants["v3_replicated"] = measure_replicated(layer, cfg, res, args, world)
        variants["v3_backward"] = measure_backward(layer, cfg, res["u_host"].cuda(), res["bias"], pk)
        del layer, res["layer"]
        torch.cuda.empty_cache()
        rm = measure(synth.get_config("mid"), args, world, pk)
        variants["mid"] = variant_summary(rm)
        del rm
        torch.cuda.empty_cache()
        r8 = measure(synth.get_config("v3_fp8"), args, world, pk)
        variants["v3_fp8"] = variant_summary(r8)
        variants["v3_fp8_backward"] = measure_backward(r8["layer"], synth.get_config("v3_fp8"), r8["u_host"].cuda(),
                                                       r8["bias"], pk)
        dec_layer = r8["layer"]
        dec_layer.__dict__.pop("ws_bwd", None)   # the backward's workspace and transposed weights are not needed
        for name in ("w13t", "w2t", "ws13t", "ws2t", "w13t_scale", "w2t_scale", "ws13t_scale", "ws2t_scale"):
            dec_layer.__dict__.pop(name, None)
        del r8
        torch.cuda.empty_cache()
        dec = measure_decode(args, world, pk, dec_layer.with_tokens(synth.get_config("decode").T))
        variants["decode_fp8"] = {k: v for k, v in dec.items() if k != "per_step"}
        del dec_layer
        torch.cuda.empty_cache()
        ru = measure(synth.get_config("v3_ue8m0"), args, world, pk)
        variants["v3_fp8_ue8m0"] = variant_summary(ru)
        del ru
        torch.cuda.empty_cache()

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        cpu = cpu_baseline_leg(cfg, res["u_host"], args.cpu_tokens)

    if rank == 0:
        conf = workload_config(cfg, world)
        conf["max_over_mean_load"] = round(res["max_over_mean_load"], 3)
        line = {
            "metric": METRIC, "value": round(res["value"], 1), "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(res["ms_per_step"], 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": cfg.prec, "data": "synthetic",
            "config": conf,
            "roofline": res["roofline"],
            "layer_roofline_frac": round(res["layer_roofline_frac"], 4),
            "layer_bound": res["layer_bound"],
            "layer_tflops": round(res["layer_tflops"], 1),
            "peaks": {"bf16_burst_tflops": pk["bf16"], "bf16_sustained_tflops": pk["bf16_sus"],
                      "fp8_tflops": round(pk["fp8"], 1) if pk.get("fp8") else None,
                      "fp8_raw_tflops_here": round(pk["fp8_raw"], 1) if pk.get("fp8_raw") else None,
                      "bf16_raw_tflops_here": round(pk["bf16_raw"], 1) if pk.get("bf16_raw") else None,
                      "hbm_gbs": pk["hbm"], "source": pk["source"]},
            "stage_ms": {k: round(v, 4) for k, v in res["stage_ms"].items()},
            "cpu_baseline": cpu,
            "e2e": {"value": round(world * cfg.T / (e2e_ms * 1e-3), 1), "unit": UNIT, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h,
                    "note": "copies of neighbouring steps overlap the forward on separate streams"},
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clk,
            "variants": variants,
        }
        print(json.dumps(line), flush=True)


def layer_config(args):
    """The workload's config with the --prec / --tokens overrides; a token
    override renames it, so no figure recorded for the named size (profiled
    DRAM traffic) is applied to another size."""
    over = {}
    if args.prec:
        over["prec"] = args.prec
    if args.tokens:
        over["T"] = args.tokens
    cfg = synth.get_config(args.workload, **over)
    return replace(cfg, name=f"{cfg.name}_T{args.tokens}") if args.tokens else cfg


def profile_case(args):
    """The program ncu wraps: build the workload's layer, run warmup + steps
    forwards (launch order per forward: router GEMM, top-k, scan, plan,
    gather, routed gate/up GEMM, routed down GEMM, shared gate/up GEMM, shared
    down GEMM, combine) -- or, with --backward, backward passes (after the
    untimed weight transposes) --, check the device status, exit."""
    torch.cuda.set_device(0)
    cfg = layer_config(args)
    layer = build_layer(cfg)
    u = synth.tokens(cfg).cuda()
    bias = synth.bias(cfg).cuda()
    if args.backward:
        layer.prepare_backward()
        g = torch.Generator(device="cuda").manual_seed(1)
        dout = torch.randn((cfg.T, cfg.d), device="cuda", generator=g).to(torch.bfloat16)
        for _ in range(args.warmup + args.steps):
            grads = layer.backward(u, bias, dout)
            del grads
        torch.cuda.synchronize()
        st = layer.backward_status()
    else:
        out = torch.empty((cfg.T, cfg.d), dtype=torch.bfloat16, device="cuda")
        for _ in range(args.warmup + args.steps):
            layer.forward(u, bias, out)
        torch.cuda.synchronize()
        st = layer.status()
    print(json.dumps({"profile_case": cfg.name, "prec": cfg.prec, "passes": args.warmup + args.steps,
                      "backward": bool(args.backward), "status": st}))
    if st != 0:
        sys.exit(1)


if __name__ == "__main__":
    main()
