"""Writes the stored expected values under tests/golden/ from the CPU oracle only.

    python tests/golden/make_golden.py

tiny_m1_k256_n128.txt: y[0][n] for the seeded tiny problem (M=1, K=256, N=128,
group 128, seed 0) of w4a16_inputs, as fp64 hex floats.
"""
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
import w4a16_inputs as wi  # noqa: E402


def main():
    p = wi.generate_named("tiny", 1, 0)
    y = oracle.gemm(p.x, p.qweight, p.scales, p.qzeros)
    with open(os.path.join(HERE, "tiny_m1_k256_n128.txt"), "w") as f:
        f.write("# y[0][n], n = 0..127, fp64 hex floats, written by tests/golden/make_golden.py\n")
        f.write("# problem: w4a16_inputs.generate_named('tiny', M=1, seed=0): K=256, N=128, group 128\n")
        for v in y[0]:
            f.write(float(v).hex() + "\n")


if __name__ == "__main__":
    main()
