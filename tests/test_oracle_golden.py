"""The oracle against its stored values for the 16x320x256 workload
(written by tests/golden/make_golden.py, which calls only the oracle):
a guard against silent drift in the oracle or the input generators."""
import hashlib
import os

import numpy as np

import oracle
import synthetic

HERE = os.path.join(os.path.dirname(__file__), "golden")


def load_pr1_out():
    rows = []
    with open(os.path.join(HERE, "pr1_out_bf16.txt")) as f:
        for line in f:
            if not line.startswith("#"):
                rows.append([int(v, 16) for v in line.split()])
    return np.array(rows, np.uint16)


def test_pr1_digests_and_product():
    x = synthetic.activations(16, 256, synthetic.SEED_PR1)
    w = synthetic.weights(320, 256, synthetic.SEED_PR1)
    xq, xs = oracle.act_quant(x)
    wq, ws = oracle.weight_quant(w)
    want = {}
    with open(os.path.join(HERE, "pr1_digests.txt")) as f:
        for line in f:
            if not line.startswith("#"):
                k, v = line.split()
                want[k] = v
    for name, a in (("x_bf16", x), ("xq_e4m3", xq), ("xs_f32", xs), ("wq_e4m3", wq), ("ws_f32", ws)):
        assert hashlib.sha256(np.ascontiguousarray(a).tobytes()).hexdigest() == want[name], name
    out = oracle.bf16_round(oracle.gemm(xq, xs, wq, ws))
    assert np.array_equal(out, load_pr1_out())
