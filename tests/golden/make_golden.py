"""Writes the oracle regression fixture for the tiny fp32 workload.

Calls only the oracle and the seeded input generator; nothing here touches the
CUDA library. Each line: token, head, then the dv output values (fp64, %.17g).
Run from the repository root: python tests/golden/make_golden.py
"""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

from oracle import oracle as orc  # noqa: E402
from differential_attention_diffattn_gb300 import workloads as W  # noqa: E402


def main():
    inp = W.generate(W.WORKLOADS["tiny_f32"], seed=0)
    out = orc.forward(inp)
    rows = [(t, h) for t in (0, 1, 2, 31, 62, 63) for h in range(inp.wl.num_heads)]
    lines = ["# oracle output of the tiny fp32 workload (seed 0): token head y[0..dv)"]
    for t, h in rows:
        lines.append(" ".join([str(t), str(h)] + ["%.17g" % x for x in out[t, h]]))
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "oracle_tiny_f32_seed0.txt")
    with open(path, "w") as f:
        f.write("\n".join(lines) + "\n")


if __name__ == "__main__":
    main()
