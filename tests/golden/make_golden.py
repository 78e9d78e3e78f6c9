"""Writes the stored expected values of tests/golden from the CPU oracle.

Calls only the oracle and the seeded input generators. Run from the
repository root:  python tests/golden/make_golden.py

pr1_*.txt: the smallest workload (X bf16 [16, 256] ~ N(0, 1), W [320, 256]
~ N(0, 0.02) quantised per 128x128 block, last row block 64 rows; seed 0):
act_quant scales, the bf16 product, and SHA-256 digests of the code bytes.
"""
import hashlib
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import numpy as np  # noqa: E402

import oracle  # noqa: E402
import synthetic  # noqa: E402


def pr1():
    x = synthetic.activations(16, 256, synthetic.SEED_PR1)
    w = synthetic.weights(320, 256, synthetic.SEED_PR1)
    xq, xs = oracle.act_quant(x)
    wq, ws = oracle.weight_quant(w)
    ref = oracle.gemm(xq, xs, wq, ws)
    return x, xq, xs, wq, ws, ref


def main():
    x, xq, xs, wq, ws, ref = pr1()
    with open(os.path.join(HERE, "pr1_digests.txt"), "w") as f:
        f.write("# SHA-256 of oracle outputs for the 16x320x256 workload (seed 0)\n")
        for name, a in (("x_bf16", x), ("xq_e4m3", xq), ("xs_f32", xs), ("wq_e4m3", wq), ("ws_f32", ws)):
            f.write(f"{name} {hashlib.sha256(np.ascontiguousarray(a).tobytes()).hexdigest()}\n")
    with open(os.path.join(HERE, "pr1_out_bf16.txt"), "w") as f:
        f.write("# bf16 bits of the oracle product C[16, 320], one row per line\n")
        for row in oracle.bf16_round(ref):
            f.write(" ".join(f"{v:04x}" for v in row) + "\n")


if __name__ == "__main__":
    main()
