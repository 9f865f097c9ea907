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
    """Roofline denominators: the measured peaks when MEASURED_PEAKS.json
    is present and readable, else the fallback figures (source says which)."""
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
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        rows = [r for r in csv.reader(io.StringIO(out)) if len(r) >= 9]
        if self.uuid:
            mine = [r for r in rows if self.uuid.replace("GPU-", "") in r[0]]
            rows = mine or rows
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
    fp8 = cfg.prec == "fp8"
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
        "gather": (0, T * d * 2 + R * d * xb + xs),
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
    fp8 = cfg.prec == "fp8"
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
    F, B = stage_work(cfg, counts)[kernel]
    t = stage_ms[kernel] * 1e-3
    tens_peak = (pk["bf16_sus"] if cfg.prec == "bf16" else 2 * pk["bf16_sus"]) * 1e12
    t_f, t_b = F / tens_peak, B / (pk["hbm"] * 1e9)
    if t_f >= t_b:
        ach, peak, unit, bound = F / t / 1e12, tens_peak / 1e12, "TFLOP/s", "tensor"
    else:
        ach, peak, unit, bound = B / t / 1e9, pk["hbm"], "GB/s", "hbm"
    return {"kernel": kernel, "bound": bound, "achieved": round(ach, 2), "peak": round(peak, 1), "unit": unit,
            "frac": round(ach / peak, 4), "traffic": kernel_traffic(kernel, cfg.name),
            "algorithmic_bytes": int(B), "algorithmic_flops": int(F), "ms": round(stage_ms[kernel], 4),
            "peak_source": f"{pk['source']} ({'bf16 sustained' if cfg.prec == 'bf16' else '2 x bf16 sustained (nominal fp8:bf16 ratio)'}; HBM copy)"}


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
    """Same metric through the public call with host buffers: H2D of u and
    D2H of h' inside the timed region, every step."""
    u_dev = torch.empty_like(u_host, device="cuda")
    out_dev = torch.empty((layer.T, layer.d), dtype=torch.bfloat16, device="cuda")
    out_host = torch.empty((layer.T, layer.d), dtype=torch.bfloat16, pin_memory=True)

    def step():
        u_dev.copy_(u_host, non_blocking=True)
        layer.forward(u_dev, bias, out_dev)
        out_host.copy_(out_dev, non_blocking=True)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    barrier(world)
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record()
    for _ in range(steps):
        step()
    e.record()
    torch.cuda.synchronize()
    barrier(world)
    ms = s.elapsed_time(e) / steps
    return ms, u_host.numel() * 2, out_host.numel() * 2


# ----------------------------------------------------------------------------
# CPU oracle (baseline leg and reference arm)
def oracle_sample(cfg, u_host, sample, cache=None):
    """Time the oracle on tokens `sample` of the batch: routing + the full
    layer output of those tokens.  Input generation is excluded."""
    import oracle
    ub = synth.bf16_bits(u_host)[sample]
    cent = synth.bf16_bits(synth.centroids(cfg))
    bias = np.asarray(synth.bias(cfg))
    gen = [0.0]
    cache = {} if cache is None else cache

    def getter(shared):
        def f(e):
            key = (shared, e)
            if key not in cache:
                t0 = time.perf_counter()
                cache[key] = tuple(synth.bf16_bits(w).copy() for w in synth.expert_weights(cfg, e, shared=shared))
                gen[0] += time.perf_counter() - t0
            return cache[key]
        return f

    t0 = time.perf_counter()
    r = oracle.route(ub, cent, bias, cfg.k)
    oracle.layer_output(ub, np.arange(len(sample)), r["idx"], r["gate"], getter(False), getter(True),
                        cfg.n_shared, cfg.E, fp8=cfg.prec == "fp8")
    return time.perf_counter() - t0 - gen[0]


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


# ----------------------------------------------------------------------------
def run_reference(args, world, rank):
    if rank != 0:
        return
    cfg = synth.get_config(args.workload)
    u = synth.tokens(cfg)
    per_step = max(1, args.ref_tokens)
    sample = np.arange(0, cfg.T, cfg.T // per_step)[:per_step]
    cache = {}
    for _ in range(args.warmup):
        oracle_sample(cfg, u, sample, cache)
    secs = [oracle_sample(cfg, u, sample, cache) for _ in range(args.steps)]
    total = sum(secs)
    value = per_step * args.steps / total
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * total / args.steps, 2),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": cfg.name, "T": cfg.T, "d": cfg.d, "E": cfg.E, "k": cfg.k,
                       "n_shared": cfg.n_shared, "inter": cfg.inter, "prec": cfg.prec},
            "cpu_baseline": {"value": round(value, 3), "unit": UNIT, "cores": host_cores(), "kind": "oracle",
                             "sample": f"{per_step} tokens of the {cfg.T}-token batch per step (routing + full "
                                       f"layer output), fp64 C oracle, input generation excluded"},
            "e2e": {"value": round(value, 3), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def measure(cfg, args, world, pk, variants_only=False):
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
    tens_peak = (pk["bf16_sus"] if cfg.prec == "bf16" else 2 * pk["bf16_sus"]) * 1e12
    t_roof = max(F / tens_peak, B / (pk["hbm"] * 1e9))
    res = {"ms_per_step": ms, "value": world * cfg.T / (ms * 1e-3), "stage_ms": stage_ms,
           "roofline": roofline(cfg, stage_ms, counts_np, pk),
           "layer_roofline_frac": t_roof / (ms * 1e-3),
           "max_over_mean_load": float(counts_np.max() / (cfg.T * cfg.k / cfg.E)),
           "layer": layer, "u_host": u_host, "bias": bias, "counts": counts_np}
    return res


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
            "max_over_mean_load_first": round(float(c[0].max() / mean), 3),
            "max_over_mean_load_last": round(float(c[-1].max() / mean), 3),
            "stage_ms": {k: round(v, 4) for k, v in stage_ms.items()},
            "per_step": [{"ms": round(m, 4), "hbm_gbs": round(g, 1), "max_over_mean": round(float(x.max() / mean), 3)}
                         for m, g, x in zip(step_ms, gbs, c)]}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="v3", choices=["v3", "v3_fp8", "mid", "decode", "v3_slice", "v3_slice_fp8",
                                                            "decode_slice", "v3_tokens", "v3_tokens_fp8"])
    ap.add_argument("--no-variants", action="store_true", help="skip the FP8 and decode measurements")
    ap.add_argument("--prec", default=None, choices=["bf16", "fp8"], help="override the workload's precision")
    ap.add_argument("--cpu-tokens", type=int, default=32, help="tokens in the CPU-oracle baseline sample")
    ap.add_argument("--ref-tokens", type=int, default=4, help="tokens per step of the reference arm")
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

    cfg = synth.get_config(args.workload)
    clocks.start()
    res = measure(cfg, args, world, pk)
    clk = clocks.stop()
    layer = res["layer"]
    e2e_ms, h2d, d2h = time_e2e(layer, res["u_host"].pin_memory(), res["bias"], args.steps, args.warmup, world)
    e2e_ms = max_over_ranks(e2e_ms, world)
    launches_per_step = 8 + (2 if cfg.n_shared else 0)

    variants = {}
    if not args.no_variants and args.workload == "v3":
        del layer, res["layer"]
        torch.cuda.empty_cache()
        r8 = measure(synth.get_config("v3_fp8"), args, world, pk)
        variants["v3_fp8"] = {"value": round(r8["value"], 1), "ms_per_step": round(r8["ms_per_step"], 4),
                              "roofline": r8["roofline"], "layer_roofline_frac": round(r8["layer_roofline_frac"], 4),
                              "stage_ms": {k: round(v, 4) for k, v in r8["stage_ms"].items()}}
        dec_layer = r8["layer"]
        del r8
        dl = _retarget(dec_layer, synth.get_config("decode"))
        dec = measure_decode(args, world, pk, dl)
        variants["decode_fp8"] = {k: v for k, v in dec.items() if k != "per_step"}
        del dec_layer, dl
        torch.cuda.empty_cache()

    cpu = None
    if rank == 0 and world == 1:
        sample = np.arange(0, cfg.T, cfg.T // args.cpu_tokens)[:args.cpu_tokens]
        secs = oracle_sample(cfg, res["u_host"], sample)
        cpu = {"value": round(len(sample) / secs, 3), "unit": UNIT, "cores": host_cores(), "kind": "oracle",
               "sample": f"{len(sample)} tokens (every {cfg.T // args.cpu_tokens}th) of the {cfg.T}-token batch: "
                         f"routing + full layer output in the fp64 C oracle, input generation excluded"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(res["value"], 1), "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(res["ms_per_step"], 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": cfg.prec, "data": "synthetic",
            "config": {"workload": f"DeepSeek-V3-shaped MoE layer forward ({cfg.name}): T={cfg.T}, d={cfg.d}, "
                                   f"{cfg.E} routed experts top-{cfg.k} + {cfg.n_shared} shared, I={cfg.inter}, "
                                   f"{cfg.prec}, clustered tokens (max/mean load "
                                   f"{res['max_over_mean_load']:.2f})",
                       "T": cfg.T, "d": cfg.d, "E": cfg.E, "k": cfg.k, "n_shared": cfg.n_shared, "inter": cfg.inter,
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                       "l2": "inputs larger than L2: every step streams the expert weights "
                             f"({(cfg.E + cfg.n_shared) * 3 * cfg.d * cfg.inter * (2 if cfg.prec == 'bf16' else 1) / 1e9:.1f} GB)"},
            "roofline": res["roofline"],
            "layer_roofline_frac": round(res["layer_roofline_frac"], 4),
            "stage_ms": {k: round(v, 4) for k, v in res["stage_ms"].items()},
            "cpu_baseline": cpu,
            "e2e": {"value": round(world * cfg.T / (e2e_ms * 1e-3), 1), "unit": UNIT, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h},
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clk,
            "variants": variants,
        }
        print(json.dumps(line), flush=True)


def profile_case(args):
    """The program ncu wraps: build the workload's layer, run warmup + steps
    forwards (launch order per forward: router GEMM, top-k, scan, plan,
    gather, routed gate/up GEMM, routed down GEMM, shared gate/up GEMM, shared
    down GEMM, combine), check the device status, exit."""
    torch.cuda.set_device(0)
    cfg = synth.get_config(args.workload, **({"prec": args.prec} if args.prec else {}))
    layer = build_layer(cfg)
    u = synth.tokens(cfg).cuda()
    bias = synth.bias(cfg).cuda()
    out = torch.empty((cfg.T, cfg.d), dtype=torch.bfloat16, device="cuda")
    for _ in range(args.warmup + args.steps):
        layer.forward(u, bias, out)
    torch.cuda.synchronize()
    st = layer.status()
    print(json.dumps({"profile_case": cfg.name, "prec": cfg.prec, "forwards": args.warmup + args.steps,
                      "status": st}))
    if st != 0:
        sys.exit(1)


def _retarget(layer, cfg):
    """A decode-shaped view of an already loaded FP8 layer: same weights, T=256."""
    from mixture_experts_layer_87_b300 import MoELayer, capi
    view = MoELayer.__new__(MoELayer)
    view.__dict__.update(layer.__dict__)
    view.T = cfg.T
    view.dims = capi.dims(cfg.T, cfg.d, cfg.E, cfg.k, cfg.n_shared, cfg.inter, cfg.prec)
    view.ws = torch.empty(capi.moe_workspace_size(view.dims), dtype=torch.uint8, device="cuda")
    return view


if __name__ == "__main__":
    main()
