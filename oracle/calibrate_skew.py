"""Choose the selection-bias amplitude beta of the skewed 48-row MXFP8 workload.

The workload adds beta * r_e^-1.2 (a Zipf(s=1.2) profile over a seeded permutation of
the ranks) to each expert's selection bias, so that hot experts are chosen by more
than 8 rows and about 40% of the experts stay idle. This script bisects beta with the
oracle's router over 16 seeded batches and prints the value stored as
``synth.SKEW_BETA``. It calls only the oracle and the input generators.

    python -m oracle.calibrate_skew
"""
import numpy as np
import torch

import oracle
from moe_decode_step_router_gb300 import synth


def idle_fraction(beta, batches, cfg, L):
    idle = []
    for x16, li, base, z in batches:
        bias = (base + beta * z).astype(np.float32)
        _, _, idx, _, _ = oracle.router(L, x16, np.zeros((cfg["E"], cfg["H"]), np.uint16), bias=bias,
                                        logits_in=li)
        idle.append(1.0 - len(np.unique(idx)) / cfg["E"])
    return float(np.mean(idle))


def main(target=0.40, n_batches=16):
    cfg = synth.config("mxfp8_skew_48rows")
    L = oracle.make_layer(cfg)
    batches = []
    for seed in range(n_batches):
        d = synth.make_inputs(dict(cfg, skew=False), seed, weights=False)
        x16 = d["x"].view(torch.int16).numpy().astype(np.uint16)
        wg = d["wg"].view(torch.int16).numpy().astype(np.uint16)
        li, _, _, _, _ = oracle.router(L, x16, wg, bias=d["bias"].numpy())
        z = synth.skew_bias(cfg["E"], synth._gen(seed + 7919, "cpu"), "cpu", beta=1.0).numpy().astype(np.float64)
        batches.append((x16, li, d["bias"].numpy().astype(np.float64), z))
    lo, hi = 0.0, 4.0
    for _ in range(30):
        mid = 0.5 * (lo + hi)
        if idle_fraction(mid, batches, cfg, L) < target:
            lo = mid
        else:
            hi = mid
    beta = round(0.5 * (lo + hi), 4)
    print("beta = %.4f  idle fraction = %.4f" % (beta, idle_fraction(beta, batches, cfg, L)))
    return beta


if __name__ == "__main__":
    main()
