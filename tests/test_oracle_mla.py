"""Pins of the oracle's MLA absorb projections (no GPU).

"Administrator & Developer Guide" 8.3, steps 5 and 7 (attn_impl "absorb"):
q_nope folded through wkv_b's no-positional rows, einsum("bshd,hdc->bshc"),
and the attention output projected to V through its v rows,
einsum("bshc,hdc->bshd"), with the FP8 wkv_b used as weight_dequant gives it.
Checked against a composition of pinned and library parts: the oracle's
weight_dequant (pinned against torch in test_oracle_quant), numpy's fp64
einsum, and the oracle's bf16 encoder (pinned against torch)."""
import numpy as np
import pytest

import oracle
import synthetic


def problem(T, H, dn, dv, C, seed):
    wq, ws = oracle.weight_quant(synthetic.weights(H * (dn + dv), C, seed))
    wdq = synthetic.bf16_bits_to_f32(oracle.weight_dequant(wq, ws)).astype(np.float64)
    return wq, ws, wdq.reshape(H, dn + dv, C)


@pytest.mark.parametrize("T,H,C", [(5, 3, 256), (1, 2, 512)])
def test_qk_is_dequant_then_einsum(T, H, C):
    dn = dv = 128
    wq, ws, w = problem(T, H, dn, dv, C, 70 + T)
    q = synthetic.activations(T, H * dn, 71 + T)
    got = oracle.mla_absorb(q, wq, ws, H, dn, dv, "qk")
    qf = synthetic.bf16_bits_to_f32(q).astype(np.float64).reshape(T, H, dn)
    ref = np.einsum("thd,hdc->thc", qf, w[:, :dn, :])
    assert np.array_equal(got, oracle.bf16_round(ref))


@pytest.mark.parametrize("T,H,C", [(5, 3, 256), (2, 2, 512)])
def test_v_is_dequant_then_einsum(T, H, C):
    dn = dv = 128
    wq, ws, w = problem(T, H, dn, dv, C, 80 + T)
    x = synthetic.activations(T, H * C, 81 + T)
    got = oracle.mla_absorb(x, wq, ws, H, dn, dv, "v")
    xf = synthetic.bf16_bits_to_f32(x).astype(np.float64).reshape(T, H, C)
    ref = np.einsum("thc,hdc->thd", xf, w[:, dn:, :])
    assert np.array_equal(got, oracle.bf16_round(ref))


def test_heads_are_independent():
    """Changing head 1's weights leaves head 0's outputs unchanged."""
    T, H, dn, dv, C = 3, 2, 128, 128, 256
    wq, ws, _ = problem(T, H, dn, dv, C, 90)
    q = synthetic.activations(T, H * dn, 91)
    a = oracle.mla_absorb(q, wq, ws, H, dn, dv, "qk")
    wq2 = wq.copy()
    wq2[dn + dv:] ^= 0x11
    b = oracle.mla_absorb(q, wq2, ws, H, dn, dv, "qk")
    assert np.array_equal(a[:, 0], b[:, 0]) and not np.array_equal(a[:, 1], b[:, 1])
