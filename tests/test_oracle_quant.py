"""Pins for the oracle's act_quant, weight quantisation and weight_dequant.

The pins are the invariants the pages fix ("Administrator & Developer Guide",
8.5.1 act_quant_kernel and 8.5.2 weight_dequant_kernel; "Algolia docsearch"
README section 3 on weight_scale_inv and zero padding), closed forms, and
torch's CPU casts as library routines."""
import numpy as np
import pytest
import torch

import oracle
import synthetic


def f32(bits):
    return synthetic.bf16_bits_to_f32(bits)


def blocks(a, M, K):
    return a.reshape(M, K // 128, 128)


@pytest.mark.parametrize("ue8m0", [False, True])
def test_act_quant_error_bound_and_range(ue8m0):
    """|x - s*decode(q)| is at most half an e4m3 step: 2^-4 |x| for normals,
    2^-10 s for subnormals (plus fp32 division rounding), and |q| <= 448."""
    x = synthetic.activations(64, 1024, 11, outlier_frac=0.01)
    q, s = oracle.act_quant(x, ue8m0)
    xv = blocks(f32(x).astype(np.float64), 64, 1024)
    deq = blocks(oracle.e4m3_decode_array(q), 64, 1024)
    sv = s.astype(np.float64)[:, :, None]
    err = np.abs(xv - sv * deq)
    bound = np.maximum(2.0 ** -4 * np.abs(xv), 2.0 ** -10 * sv) * (1 + 2.0 ** -20)
    assert np.all(err <= bound)
    assert np.all(np.abs(deq) <= 448.0)


def test_act_quant_amax_element_maps_to_448():
    x = synthetic.activations(32, 2048, 12, outlier_frac=0.01)
    q, s = oracle.act_quant(x, False)
    xv = blocks(f32(x), 32, 2048)
    qb = blocks(q, 32, 2048)
    arg = np.abs(xv).argmax(axis=2)
    picked = np.take_along_axis(qb, arg[:, :, None], axis=2)[:, :, 0]
    sign = np.take_along_axis(xv, arg[:, :, None], axis=2)[:, :, 0] < 0
    assert np.all(picked == np.where(sign, 0xFE, 0x7E))
    # and the scale is amax/448 in fp32
    amax = np.abs(xv).max(axis=2).astype(np.float32)
    assert np.array_equal(s, (np.maximum(amax, np.float32(1e-4)) / np.float32(448.0)).astype(np.float32))


def test_act_quant_zero_block():
    x = np.zeros((3, 256), np.uint16)
    x[1, :128] = 0x8000           # negative zeros
    q, s = oracle.act_quant(x, False)
    assert np.all(s == np.float32(np.float32(1e-4) / np.float32(448.0)))
    assert np.all(q[1, :128] == 0x80) and np.all(q[0] == 0) and np.all(q[1, 128:] == 0)
    _, su = oracle.act_quant(x, True)
    assert np.all(su == np.float32(2.0 ** -22))


def test_act_quant_ue8m0_power_of_two_and_upper_bound():
    x = synthetic.activations(16, 1024, 13)
    q, s = oracle.act_quant(x, True)
    m, e = np.frexp(s.astype(np.float64))
    assert np.all(m == 0.5)                                  # powers of two
    amax = np.abs(blocks(f32(x), 16, 1024)).max(axis=2)
    assert np.all(s.astype(np.float64) >= amax / 448.0)      # rounded up
    assert np.all(s.astype(np.float64) < 2 * np.maximum(amax, 1e-4) / 448.0 * (1 + 1e-6))


@pytest.mark.parametrize("ue8m0", [False, True])
def test_act_quant_power_of_two_scaling(ue8m0):
    """Multiplying a block by 2^j scales s by exactly 2^j and keeps the codes,
    as long as amax >= 1e-4 before and after (the clamp is not active)."""
    x = synthetic.activations(8, 512, 14)
    q0, s0 = oracle.act_quant(x, ue8m0)
    for j in (-3, 2, 5):
        xs = synthetic.to_bf16_bits(f32(x) * np.float32(2.0 ** j))   # exact
        q1, s1 = oracle.act_quant(xs, ue8m0)
        assert np.array_equal(q1, q0)
        assert np.array_equal(s1, (s0 * np.float32(2.0 ** j)).astype(np.float32))


@pytest.mark.parametrize("ue8m0", [False, True])
def test_act_quant_matches_library_casts(ue8m0):
    """Same result from torch's CPU ops: amax, fp32 division, and torch's
    float8_e4m3fn cast (a library routine that rounds to nearest even)."""
    x = synthetic.activations(16, 768, 15, outlier_frac=0.02)
    q, s = oracle.act_quant(x, ue8m0)
    xt = torch.from_numpy(f32(x)).view(16, 6, 128)
    amax = xt.abs().amax(dim=2, keepdim=True).clamp(min=1e-4)
    st = amax / 448.0
    if ue8m0:
        st = torch.pow(2.0, torch.ceil(torch.log2(st)))
    qt = (xt / st).to(torch.float8_e4m3fn).view(torch.uint8).view(16, 768)
    assert np.array_equal(qt.numpy(), q)
    assert np.array_equal(st.view(16, 6).numpy(), s)


def test_act_quant_rejects_unaligned_k():
    with pytest.raises(ValueError):
        oracle.act_quant(np.zeros((2, 100), np.uint16))


@pytest.mark.parametrize("ue8m0", [False, True])
def test_weight_quant_padding_rule(ue8m0):
    """Zero padding a non-aligned weight to a multiple of 128 changes neither
    the scales nor the real elements' codes."""
    w = synthetic.weights(320, 200, 21)
    q, s = oracle.weight_quant(w, ue8m0)
    assert s.shape == (3, 2)
    wp = np.zeros((384, 256), np.float32)
    wp[:320, :200] = w
    qp, sp = oracle.weight_quant(wp, ue8m0)
    assert np.array_equal(sp, s)
    assert np.array_equal(qp[:320, :200], q)
    assert np.all(qp[320:] == 0) and np.all(qp[:, 200:] == 0)


def test_weight_quant_block_invariants():
    w = synthetic.weights(256, 384, 22)
    q, s = oracle.weight_quant(w, False)
    wb = w.reshape(2, 128, 3, 128).transpose(0, 2, 1, 3)
    qb = q.reshape(2, 128, 3, 128).transpose(0, 2, 1, 3)
    amax = np.abs(wb).max(axis=(2, 3))
    assert np.array_equal(s, (amax / np.float32(448.0)).astype(np.float32))
    flat_w = wb.reshape(2, 3, -1)
    flat_q = qb.reshape(2, 3, -1)
    arg = np.abs(flat_w).argmax(axis=2)
    picked = np.take_along_axis(flat_q, arg[:, :, None], axis=2)[:, :, 0]
    assert np.all((picked & 0x7F) == 0x7E)
    # each block: codes equal torch's cast of w / s
    st = torch.from_numpy(np.repeat(np.repeat(s, 128, 0), 128, 1))
    qt = (torch.from_numpy(w) / st).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(qt, q)


def test_weight_dequant_scale_one_is_decode():
    """With unit scales the output is the e4m3 value itself (every e4m3 value
    is a bf16 value)."""
    g = np.random.Generator(np.random.PCG64(31))
    q = g.integers(0, 256, (130, 260), dtype=np.uint8)
    q[(q & 0x7F) == 0x7F] = 0
    s = np.ones((2, 3), np.float32)
    out = oracle.weight_dequant(q, s)
    ref = torch.from_numpy(q).view(torch.float8_e4m3fn).to(torch.bfloat16)
    assert np.array_equal(out, ref.view(torch.int16).numpy().view(np.uint16))


def test_weight_dequant_power_of_two_scale_is_exact():
    g = np.random.Generator(np.random.PCG64(32))
    q = g.integers(0, 256, (256, 128), dtype=np.uint8)
    q[(q & 0x7F) == 0x7F] = 0
    s = np.array([[2.0 ** -7], [2.0 ** 3]], np.float32)
    out = f32(oracle.weight_dequant(q, s)).astype(np.float64)
    dec = oracle.e4m3_decode_array(q)
    assert np.array_equal(out[:128], dec[:128] * 2.0 ** -7)
    assert np.array_equal(out[128:], dec[128:] * 2.0 ** 3)


def test_weight_dequant_matches_library_ops():
    """bf16(fp32(q) * s): torch's fp32 multiply and bf16 cast."""
    w = synthetic.weights(320, 256, 33)
    q, s = oracle.weight_quant(w)
    out = oracle.weight_dequant(q, s)
    st = torch.from_numpy(np.repeat(np.repeat(s, 128, 0), 128, 1))[:320, :256]
    ref = (torch.from_numpy(q).view(torch.float8_e4m3fn).to(torch.float32) * st).to(torch.bfloat16)
    assert np.array_equal(out, ref.view(torch.int16).numpy().view(np.uint16))


def test_weight_dequant_padding_rule():
    """Dequant of [320, 200] equals the real part of the dequant of the
    zero-padded [384, 256]; the padded part contributes zeros."""
    w = synthetic.weights(320, 200, 34)
    q, s = oracle.weight_quant(w)
    qp = np.zeros((384, 256), np.uint8)
    qp[:320, :200] = q
    out = oracle.weight_dequant(q, s)
    outp = oracle.weight_dequant(qp, s)
    assert np.array_equal(outp[:320, :200], out)
    assert np.all(outp[320:] == 0) and np.all(outp[:, 200:] == 0)


def test_dequant_quant_roundtrip_within_half_step():
    w = synthetic.weights(256, 256, 35)
    q, s = oracle.weight_quant(w)
    back = f32(oracle.weight_dequant(q, s)).astype(np.float64)
    sv = np.repeat(np.repeat(s.astype(np.float64), 128, 0), 128, 1)
    err = np.abs(back - w)
    # e4m3 half step (2^-4 relative, 2^-10 s absolute) plus the bf16 rounding (2^-9 relative)
    bound = np.maximum(2.0 ** -4 * np.abs(w), 2.0 ** -10 * sv) + 2.0 ** -8 * np.abs(w) + 1e-30
    assert np.all(err <= bound)
