"""Choose the clustered-token mix so the V3-shaped batch is skewed as specified.

TEST INFRASTRUCTURE: run by hand, never by the library.  It bisects the
centre share rho of the clustered token stream (Zipf exponent alpha fixed)
until the oracle router, at the V3 shape and the layer's seeded bias, gives a
max/mean expert load inside [3.8, 4.2] on the 8192-token batch, then writes
the result to synth/calibration.json, which the input generator reads.

    python -m oracle.calibrate
"""
import json
import os
import sys
from dataclasses import replace

import numpy as np

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import oracle  # noqa: E402
import synth   # noqa: E402

TARGET = (3.8, 4.2)


def max_over_mean(cfg) -> float:
    u = synth.bf16_bits(synth.tokens(cfg))
    r = oracle.route(u, synth.bf16_bits(synth.centroids(cfg)), np.asarray(synth.bias(cfg)), cfg.k)
    counts = np.bincount(r["idx"].ravel(), minlength=cfg.E)
    return counts.max() / (cfg.T * cfg.k / cfg.E)


def main():
    base = synth.get_config("v3")
    lo, hi = 0.0, base.rho
    while max_over_mean(replace(base, rho=hi)) < TARGET[1]:
        hi = min(0.95, hi * 1.5)
    rho, ratio = hi, None
    for _ in range(30):
        rho = 0.5 * (lo + hi)
        ratio = max_over_mean(replace(base, rho=rho))
        print(f"rho={rho:.5f} max/mean={ratio:.3f}", flush=True)
        if TARGET[0] <= ratio <= TARGET[1]:
            break
        if ratio > TARGET[1]:
            hi = rho
        else:
            lo = rho
    mid = max_over_mean(replace(synth.get_config("mid"), rho=rho))
    dec = synth.get_config("decode")
    dec_ratio = max_over_mean(replace(dec, rho=rho))
    out = {"rho": round(rho, 6), "alpha": base.alpha, "decode_alpha": dec.alpha,
           "v3_max_over_mean": round(float(ratio), 4), "mid_max_over_mean": round(float(mid), 4),
           "decode_step0_max_over_mean": round(float(dec_ratio), 4)}
    path = os.path.join(os.path.dirname(synth.__file__), "calibration.json")
    with open(path, "w") as f:
        json.dump(out, f, indent=1)
    print(out)


if __name__ == "__main__":
    main()
