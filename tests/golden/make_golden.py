"""Write tests/golden/tiny_oracle_samples.txt from the CPU oracle only.

The samples are regression values for the oracle on the tiny fp32 workload
(batch 1, L 64, H 2, P 16, N 16, R 1, seed 0); they detect drift in the
oracle, they are not a pin by themselves. Run: python tests/golden/make_golden.py
"""
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import m3synth  # noqa: E402
from oracle import oracle  # noqa: E402


def main():
    inp = m3synth.scan_inputs(m3synth.TINY, seed=0)
    y, st = oracle.scan_seq(inp["x"], inp["dt"], inp["A"], inp["lam"], inp["B"], inp["C"],
                            inp["theta"], inp["B_bias"], inp["C_bias"])
    rng = np.random.default_rng(1234)
    lines = ["# oracle samples on the tiny workload (seed 0); written by make_golden.py",
             "# kind index value"]
    for _ in range(24):
        ix = tuple(int(rng.integers(0, s)) for s in y.shape)
        lines.append("y %s %.17g" % (",".join(map(str, ix)), y[ix]))
    for _ in range(8):
        ix = tuple(int(rng.integers(0, s)) for s in st.shape)
        lines.append("state %s %.17g" % (",".join(map(str, ix)), st[ix]))
    with open(os.path.join(HERE, "tiny_oracle_samples.txt"), "w") as f:
        f.write("\n".join(lines) + "\n")


if __name__ == "__main__":
    main()
