"""Write tests/golden/tiny_oracle_rows.txt.

Regression fixture for the FP64 oracle on the tiny workload (B=1, H=2, L=64,
d=64, fp16, RoPE base 10000 at positions 0..63, full non-causal attention).
It calls only the oracle and the seeded input generator.  Each line: the
flattened row id (h*L + i) followed by the 64 output values.
"""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
import synth  # noqa: E402


def main():
    w = synth.WORKLOADS["tiny"]
    x = synth.make_inputs(w)
    rows = np.array([0, 1, 31, 63, 64, 100, 127], dtype=np.int64)
    out = oracle.rope_attn_workload(x, rows=rows)
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_oracle_rows.txt")
    with open(path, "w") as f:
        f.write("# oracle rows of the tiny workload (B=1 H=2 L=64 d=64 fp16), written by make_golden.py\n")
        for r, o in zip(rows, out):
            f.write(str(int(r)) + " " + " ".join(repr(float(v)) for v in o) + "\n")


if __name__ == "__main__":
    main()
