"""Writes the stored oracle fixtures under tests/golden/. Calls only the oracle and the
seeded input generators; nothing here comes from the CUDA path.

Usage:
  python tests/golden/make_golden.py                  # the 512-point d=3 fixture (seconds)
  python tests/golden/make_golden.py --workload 2 5 4 3
      # full-size solves of the 10k^2 d=64, 20k^2 d=1024, 20k x 80k d=16 annealed and
      # 50k^2 d=512 workloads: full fp64 potentials f, g and the loss. They use the
      # dense-cost solve (bitwise the streaming oracle solve; 8nm bytes of host memory:
      # 0.8 / 3.2 / 12.8 / 20 GB) and take minutes to tens of minutes on a few cores.
"""
import argparse
import json
import os
import sys
import time

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import oracle  # noqa: E402
from workloads import WORKLOADS, workload  # noqa: E402

HERE = os.path.dirname(os.path.abspath(__file__))
SAMPLE = [0, 1, 2, 63, 64, 127, 128, 255, 256, 300, 383, 384, 447, 500, 510, 511]
METHOD = ("FlashSinkhorn: IO-Aware Entropic Optimal Transport on GPU, abstract "
          "(stabilized log-domain Sinkhorn, squared Euclidean cost)")


def checksums(pr):
    return {"X_sum": float(pr.X.astype(np.float64).sum()),
            "Y_sum": float(pr.Y.astype(np.float64).sum()),
            "a_sum": float(pr.a.astype(np.float64).sum()),
            "b_sum": float(pr.b.astype(np.float64).sum())}


def write_small():
    pr = workload(1)
    f, g, loss = oracle.solve(pr.X, pr.Y, pr.a, pr.b, pr.eps_schedule, pr.iters_per_stage)
    out = {
        "what": "fp64 oracle on the 512x512 d=3 point-cloud workload (Uniform[0,1]^3, "
                "uniform weights, eps=0.05, 100 alternating iterations from g=0)",
        "source": "oracle/sinkhorn_oracle.c via tests/golden/make_golden.py",
        "method": METHOD,
        "input_checksums": {"X_sum": float(pr.X.astype(np.float64).sum()),
                            "Y_sum": float(pr.Y.astype(np.float64).sum())},
        "loss": loss,
        "sample_index": SAMPLE,
        "f": [float(f[i]) for i in SAMPLE],
        "g": [float(g[i]) for i in SAMPLE],
    }
    path = os.path.join(HERE, "pc512_d3_oracle.json")
    with open(path, "w") as fh:
        json.dump(out, fh, indent=1)
        fh.write("\n")
    print("wrote", path)


def full_size_paths(idx):
    name = WORKLOADS[idx]["name"]
    return (os.path.join(HERE, f"{name}_oracle.json"),
            os.path.join(HERE, f"{name}_oracle_fg.npz"))


def write_full(idx):
    pr = workload(idx)
    t0 = time.time()
    f, g, loss = oracle.solve_dense(pr.X, pr.Y, pr.a, pr.b, pr.eps_schedule,
                                    pr.iters_per_stage)
    secs = time.time() - t0
    jpath, npath = full_size_paths(idx)
    meta = {
        "what": f"fp64 oracle, full-size {pr.name} workload: n={pr.n}, m={pr.m}, d={pr.d}, "
                f"{len(pr.eps_schedule)} eps stage(s) x {pr.iters_per_stage} alternating "
                "iterations from g=0; full potentials f, g in the .npz beside this file",
        "source": "oracle.solve_dense (oracle/sinkhorn_oracle.c, oracle_solve_dense: bitwise "
                  "oracle_solve) via tests/golden/make_golden.py",
        "method": METHOD,
        "workload": idx,
        "seed": 1000 + idx,
        "n": pr.n, "m": pr.m, "d": pr.d,
        "eps_schedule": [float(e) for e in pr.eps_schedule],
        "iters_per_stage": pr.iters_per_stage,
        "input_checksums": checksums(pr),
        "loss": loss,
        "max_abs_f": float(np.abs(f).max()),
        "max_abs_g": float(np.abs(g).max()),
        "oracle_seconds": round(secs, 1),
        "oracle_threads": oracle.num_threads(),
    }
    np.savez_compressed(npath, f=f, g=g)
    with open(jpath, "w") as fh:
        json.dump(meta, fh, indent=1)
        fh.write("\n")
    print(f"wrote {jpath} and {npath} ({secs:.0f} s, loss {loss!r})", flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", type=int, nargs="*", default=None,
                    help="full-size workloads to solve (2..5); none = the 512-point fixture")
    args = ap.parse_args()
    if not args.workload:
        write_small()
        return
    for idx in args.workload:
        if idx not in (2, 3, 4, 5):
            raise SystemExit(f"no full-size fixture for workload {idx}")
        write_full(idx)


if __name__ == "__main__":
    main()
