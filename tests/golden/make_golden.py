"""Writes tests/golden/tiny_layer_out.txt from the oracle alone.

Run from the repository root:  python tests/golden/make_golden.py
The values are the fp64 oracle's bf16-boundary layer output for the tiny
workload (seed 0), sampled at fixed (row, column) pairs and stored as exact
hexadecimal floats; they pin the oracle against accidental change.
"""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
import workload as wl  # noqa: E402


def main():
    w = wl.WORKLOADS["tiny"]
    b = wl.make_batch(w, 0)
    x = oracle.to_f64(wl.make_x(w, b, 0))
    W = oracle.LayerWeights64.from_torch(wl.make_weights(w, 0))
    kp, vp = wl.make_pools(w, b, 0)
    out = oracle.layer_step(x, W, w.shape, b, oracle.to_f64(kp), oracle.to_f64(vp))["out"]
    picks = [(r, c) for r in (0, 1, 17, 63, 64, 65, 66, 67) for c in (0, 1, 127, 128, 255)]
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_layer_out.txt")
    with open(path, "w") as f:
        f.write("# oracle layer output, tiny workload, seed 0: row col value(hex)\n")
        f.write("# written by tests/golden/make_golden.py (calls only oracle/ and workload/)\n")
        for r, c in picks:
            f.write(f"{r} {c} {float(out[r, c]).hex()}\n")


if __name__ == "__main__":
    main()
