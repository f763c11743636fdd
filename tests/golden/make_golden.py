"""Writes tests/golden/tiny_oracle.json from the CPU oracle (and nothing else).

Workload: T=16 tokens, A=2 active experts, H=256, F=128, E=8, x and W ~ N(0, 1) in
bfloat16, idx uniform in [0, 8), seeds x=1, W=2, idx=3 -- the small correctness case the
issue's microbenchmark shape is scaled down to.  The fixture is a regression pin: a later
change to the oracle's arithmetic that moves any of these numbers must say which passage
of the pages (or which reading of it) justifies the change.

Run:  python tests/golden/make_golden.py
"""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
import workloads as wl  # noqa: E402


def main():
    w = wl.workloads()["tiny"]
    inp = wl.make_inputs(w)
    wq, sc, bs = oracle.quantize(inp["w"])
    perm, offsets, _ = oracle.route_sort(inp["idx"], w.E)
    y = oracle.gather_qmm(inp["x"], wq, sc, bs, inp["idx"], w.E)
    out = {
        "workload": "T=16, A=2, H=256, F=128, E=8; seeds x=1, W=2, idx=3",
        "wq_sum": int(wq.astype(np.uint64).sum()),
        "scales_head": [int(v) for v in sc.reshape(-1)[:8]],
        "biases_head": [int(v) for v in bs.reshape(-1)[:8]],
        "offsets": [int(v) for v in offsets],
        "y_row0_head": [float(v) for v in y[0, :8]],
        "y_abs_sum": float(np.abs(y).sum()),
    }
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_oracle.json")
    with open(path, "w") as fh:
        json.dump(out, fh, indent=1)
        fh.write("\n")
    print("wrote", path)


if __name__ == "__main__":
    main()
