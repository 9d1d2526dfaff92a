"""Writes the stored oracle fixtures under tests/golden/. Calls only the oracle and the
seeded input generators; nothing here comes from the CUDA path.

Usage: python tests/golden/make_golden.py
"""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import oracle  # noqa: E402
from workloads import workload  # noqa: E402

SAMPLE = [0, 1, 2, 63, 64, 127, 128, 255, 256, 300, 383, 384, 447, 500, 510, 511]


def main():
    pr = workload(1)
    f, g, loss = oracle.solve(pr.X, pr.Y, pr.a, pr.b, pr.eps_schedule, pr.iters_per_stage)
    out = {
        "what": "fp64 oracle on the 512x512 d=3 point-cloud workload (Uniform[0,1]^3, "
                "uniform weights, eps=0.05, 100 alternating iterations from g=0)",
        "source": "oracle/sinkhorn_oracle.c via tests/golden/make_golden.py",
        "method": "FlashSinkhorn: IO-Aware Entropic Optimal Transport on GPU, abstract "
                  "(stabilized log-domain Sinkhorn, squared Euclidean cost)",
        "input_checksums": {"X_sum": float(pr.X.astype(np.float64).sum()),
                            "Y_sum": float(pr.Y.astype(np.float64).sum())},
        "loss": loss,
        "sample_index": SAMPLE,
        "f": [float(f[i]) for i in SAMPLE],
        "g": [float(g[i]) for i in SAMPLE],
    }
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "pc512_d3_oracle.json")
    with open(path, "w") as fh:
        json.dump(out, fh, indent=1)
        fh.write("\n")
    print("wrote", path)


if __name__ == "__main__":
    main()
