"""Calibrate the Zipf strength of the capacity-limited workload (writes a golden file).

The capacity-limited layer (Mixtral-like shapes, T = 8192, top-2, capacity
factor 1.0) gets a Zipf(s = 1.2) expert skew through the router bias
b_e = -beta * 1.2 * ln(e + 1), expert 0 hottest.  beta is chosen by bisection
so that the CPU oracle's routing drops 15 % (+-0.5 %) of the routes at seed 0.
Only the oracle is called; the result goes to tests/golden/cap_bias.json.

    python -m oracle.calibrate_cap_bias
"""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import oracle  # noqa: E402
from synth import workloads as W  # noqa: E402

OUT = os.path.join(ROOT, "tests", "golden", "cap_bias.json")


def drop_fraction(beta: float, h, wg, wl, T) -> float:
    _, bias = W.make_router(wl, beta=beta)
    l = oracle.router_logits(h, wg, bias)
    idx, _ = oracle.select_topk(l, wl.top_k)
    cap = oracle.capacity(T, wl.num_experts, wl.top_k, wl.capacity_factor)
    d = oracle.dispatch(idx, wl.num_experts, wl.block_size, cap)
    return d["num_dropped"] / (T * wl.top_k)


def main():
    wl = W.WORKLOADS["cap"]
    T = wl.tokens[0]
    h = W.make_h(wl, T, seed=0)
    wg, _ = W.make_router(wl, beta=0.0)
    lo, hi = 0.0, 4.0
    f_lo, f_hi = drop_fraction(lo, h, wg, wl, T), drop_fraction(hi, h, wg, wl, T)
    assert f_lo < 0.15 < f_hi, (f_lo, f_hi)
    beta, f = hi, f_hi
    for _ in range(40):
        mid = 0.5 * (lo + hi)
        f = drop_fraction(mid, h, wg, wl, T)
        beta = mid
        if abs(f - 0.15) <= 0.002:
            break
        if f < 0.15:
            lo = mid
        else:
            hi = mid
    assert abs(f - 0.15) <= 0.005, f
    beta = float(np.float32(beta))
    f = drop_fraction(beta, h, wg, wl, T)
    rec = {"beta": beta, "drop_fraction_seed0": f, "T": T, "seed": 0,
           "recipe": "router bias b_e = -beta * 1.2 * ln(e + 1) computed in float64, stored as float32",
           "written_by": "python -m oracle.calibrate_cap_bias (calls only the CPU oracle)"}
    with open(OUT, "w") as fh:
        json.dump(rec, fh, indent=1)
    print(json.dumps(rec))


if __name__ == "__main__":
    main()
