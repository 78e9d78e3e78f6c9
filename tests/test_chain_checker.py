"""The chain checker (tests/helpers.py: admissible intermediates of the
SwiGLU FFN and the expert chain) against the oracle itself, on the CPU.

The GPU tests accept a re-quantised intermediate and a chain output only
inside intervals computed from the oracle's fp64 h1, h3. Here the oracle's
own results must pass, and mistakes planted in a copy of them must fail: a
code moved by one e4m3 step where the admissible interval holds one code, a
block scale off by a factor the interval excludes, a code rounded away from
the amax element's +-448, and an output moved past its allowance."""
import numpy as np
import pytest

import oracle
import synthetic
from helpers import (admissible_quant, admissible_u, assert_chain_close, assert_quant_admissible, dequant_weight,
                     ffn_chain_allowance)


def problem(M, dim, inter, seed, ue8m0):
    x = synthetic.activations(M, dim, seed, outlier_frac=0.02)
    xq, xs = oracle.act_quant(x, ue8m0)
    w1q, w1s = oracle.weight_quant(synthetic.weights(inter, dim, seed + 1), ue8m0)
    w3q, w3s = oracle.weight_quant(synthetic.weights(inter, dim, seed + 2), ue8m0)
    w2q, w2s = oracle.weight_quant(synthetic.weights(dim, inter, seed + 3), ue8m0)
    return xq, xs, w1q, w1s, w3q, w3s, w2q, w2s


def intermediate(p, ue8m0):
    xq, xs, w1q, w1s, w3q, w3s, w2q, w2s = p
    H1, H3 = oracle.gemm(xq, xs, w1q, w1s), oracle.gemm(xq, xs, w3q, w3s)
    y, uq, us = oracle.ffn_rows(xq, xs, w1q, w1s, w3q, w3s, w2q, w2s, range(xq.shape[0]), ue8m0=ue8m0,
                                return_u=True)
    return H1, H3, y, uq, us


@pytest.mark.parametrize("ue8m0", [False, True])
def test_oracle_intermediate_is_admissible(ue8m0):
    p = problem(24, 256, 384, 70, ue8m0)
    H1, H3, y, uq, us = intermediate(p, ue8m0)
    u_lo, u_hi = admissible_u(H1, H3)
    assert np.all(u_lo <= u_hi)
    adm = admissible_quant(u_lo, u_hi, ue8m0)
    assert_quant_admissible(uq, us, adm, ue8m0, what="oracle")
    # the intervals are narrow: most elements admit a single code, most blocks a narrow scale range
    s_lo, s_hi, c_lo, c_hi = adm
    assert np.mean(c_lo == c_hi) > 0.9
    assert np.all(s_hi <= s_lo * 2.0 ** (1 if ue8m0 else 2.0 ** -5))


def test_planted_intermediate_errors_fail():
    p = problem(24, 256, 384, 71, False)
    H1, H3, y, uq, us = intermediate(p, False)
    adm = admissible_quant(*admissible_u(H1, H3), False)
    s_lo, s_hi, c_lo, c_hi = adm
    code = oracle.e4m3_decode_array(uq)
    # a code one step off where only one code is admissible (away from zero and from +-448)
    single = np.argwhere((c_lo == c_hi) & (np.abs(code) > 1) & (np.abs(code) < 400))
    r, c = single[len(single) // 2]
    bad = uq.copy()
    bad[r, c] = uq[r, c] + 1                  # the next code of the same sign
    with pytest.raises(AssertionError):
        assert_quant_admissible(bad, us, adm, False)
    # a block scale twice its value
    bad_s = us.copy()
    bad_s[3, 1] *= 2
    with pytest.raises(AssertionError):
        assert_quant_admissible(uq, bad_s, adm, False)
    # the amax element of a block not coded +-448 (one step down: 416)
    blk = np.abs(code[5, 128:256])
    i = 128 + int(np.argmax(blk))
    bad = uq.copy()
    bad[5, i] = uq[5, i] - 1
    with pytest.raises(AssertionError):
        assert_quant_admissible(bad, us, adm, False)


@pytest.mark.parametrize("ue8m0", [False, True])
def test_chain_allowance_bounds_admissible_outputs(ue8m0):
    """The oracle's output passes with zero slack beyond the allowance; an
    output recomputed from another admissible intermediate (every code that can
    move moved to the far end of its interval, at the scales the oracle chose)
    stays inside it; a planted error past it fails."""
    p = problem(16, 256, 384, 72, ue8m0)
    xq, xs, w1q, w1s, w3q, w3s, w2q, w2s = p
    H1, H3, y, uq, us = intermediate(p, ue8m0)
    w2d = dequant_weight(w2q, w2s)
    allow = ffn_chain_allowance(xq, xs, w1q, w1s, w3q, w3s, w2d, uq, us, ue8m0)
    assert np.all(allow >= 0)
    ref_bits = oracle.bf16_round(y)
    ref = synthetic.bf16_bits_to_f32(ref_bits).astype(np.float64)
    assert_chain_close(ref_bits, y, allow, what="oracle")
    # another admissible intermediate: codes at the far end of their intervals
    s_lo, s_hi, c_lo, c_hi = admissible_quant(*admissible_u(H1, H3), ue8m0)
    code = oracle.e4m3_decode_array(uq)
    alt = np.where(c_hi - code > code - c_lo, c_hi, c_lo)
    y_alt = (alt * np.repeat(us.astype(np.float64), 128, axis=1)) @ w2d.T
    assert np.all(np.abs(y_alt - y) <= allow + 1e-12)
    # a planted output error: past tolerance + allowance at one element
    tol = 2.0 ** -7 * np.abs(y) + 1e-3 * np.sqrt(np.mean(y ** 2)) + allow
    bad = ref.copy()
    bad[2, 7] = y[2, 7] + 2 * tol[2, 7]
    with pytest.raises(AssertionError):
        assert_chain_close(oracle.bf16_round(bad), y, allow)
