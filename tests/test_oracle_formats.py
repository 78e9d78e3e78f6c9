"""Pins for the oracle's number formats: the e4m3fn encoder/decoder and the
bf16 rounding. Each check is against something other than the oracle itself:
torch's CPU float8_e4m3fn / bf16 casts (library routines that round to nearest
even), the bit layout of the formats, and closed-form special values."""
import numpy as np
import pytest
import torch

import oracle
import synthetic

GOLDEN = __import__("os").path.join(__import__("os").path.dirname(__file__), "golden")


def torch_e4m3(v: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(v, np.float32)).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy()


def test_decode_matches_torch_for_every_code():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = oracle.e4m3_decode_array(codes)
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert set(np.flatnonzero(nan)) == {0x7F, 0xFF}
    assert np.array_equal(ref[~nan], got[~nan])
    # -0 decodes to a negative zero
    assert np.signbit(got[0x80]) and got[0x80] == 0.0


def test_encode_decode_identity_on_finite_codes():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    vals = oracle.e4m3_decode_array(codes).astype(np.float32)
    assert np.array_equal(oracle.e4m3_encode_array(vals), codes)


def test_encode_special_values_golden():
    """Closed-form codes, listed with their derivation in tests/golden."""
    rows = []
    with open(f"{GOLDEN}/e4m3_special.txt") as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                v, c = line.split()
                rows.append((float.fromhex(v) if "p" in v else float(v), int(c, 16)))
    assert len(rows) >= 10
    for v, c in rows:
        assert oracle.e4m3_encode(v) == c, (v, hex(c))


def test_encode_matches_torch_on_all_bf16_inputs_and_scales():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    x = synthetic.bf16_bits_to_f32(bits)
    finite = np.isfinite(x)
    for s in (1.0, 3.0e-3, 0.00390625, 1e-4 / 448.0, 7.1e-2, 2.2321428e-07):
        with np.errstate(over="ignore"):
            y = (x[finite] / np.float32(s)).astype(np.float32)
        y = y[np.abs(y) < 464.0]          # torch's cast is not saturating beyond
        assert np.array_equal(oracle.e4m3_encode_array(y), torch_e4m3(y)), s


def test_encode_matches_torch_at_midpoints():
    """Every midpoint between adjacent finite codes, and one fp32 ulp either
    side: the ties must go to the even code."""
    pos = np.array(sorted(set(oracle.e4m3_decode_array(np.arange(0, 0x7F, dtype=np.uint8)))))
    mids = ((pos[:-1] + pos[1:]) / 2).astype(np.float32)
    cand = np.concatenate([mids, np.nextafter(mids, np.float32(np.inf)),
                           np.nextafter(mids, np.float32(0))]).astype(np.float32)
    cand = np.concatenate([cand, -cand])
    assert np.array_equal(oracle.e4m3_encode_array(cand), torch_e4m3(cand))
    # at a tie the code is even (mantissa lsb 0)
    tie_codes = oracle.e4m3_encode_array(mids)
    assert np.all(tie_codes % 2 == 0)


def test_encode_matches_torch_on_random_fp32():
    g = np.random.Generator(np.random.PCG64(1234))
    y = np.concatenate([
        g.uniform(-464, 464, 1_000_000),
        g.standard_normal(500_000) * 1e-2,
        np.exp(g.uniform(-25, 6.1, 500_000)) * g.choice([-1, 1], 500_000),
    ]).astype(np.float32)
    y = y[np.abs(y) < 464.0]
    assert np.array_equal(oracle.e4m3_encode_array(y), torch_e4m3(y))


def test_encode_saturates_beyond_range():
    big = np.array([448.0, 463.99, 464.0, 479.0, 480.0, 1e4, 3e38], np.float32)
    assert np.all(oracle.e4m3_encode_array(big) == 0x7E)
    assert np.all(oracle.e4m3_encode_array(-big) == 0xFE)


def test_encode_keeps_sign_of_zero_and_underflow():
    assert oracle.e4m3_encode(0.0) == 0x00
    assert oracle.e4m3_encode(-0.0) == 0x80
    assert oracle.e4m3_encode(-1e-30) == 0x80
    assert oracle.e4m3_encode(2.0 ** -11) == 0x00
    assert oracle.e4m3_encode(-(2.0 ** -10)) == 0x80   # tie to the even code 0


def test_bf16_encode_matches_torch_on_fp32_inputs():
    g = np.random.Generator(np.random.PCG64(7))
    x = np.concatenate([g.standard_normal(200_000) * 10.0 ** g.integers(-30, 30, 200_000),
                        g.uniform(-1, 1, 100_000)]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle.bf16_round(x.astype(np.float64)), ref)


def test_bf16_encode_rounds_doubles_once():
    # 1 + 2^-8 + 2^-40 lies just above the midpoint of 1 and 1 + 2^-7.
    # One rounding gives 1 + 2^-7 (0x3F81); rounding through fp32 first would
    # land on the midpoint and tie to 1.0 (0x3F80).
    assert oracle.bf16_encode(1.0 + 2.0 ** -8 + 2.0 ** -40) == 0x3F81
    assert oracle.bf16_encode(1.0 + 2.0 ** -8) == 0x3F80        # tie -> even
    assert oracle.bf16_encode(1.0 + 3 * 2.0 ** -8) == 0x3F82    # tie -> even
    assert oracle.bf16_encode(-2.5) == 0xC020
    assert oracle.bf16_encode(0.0) == 0x0000


@pytest.mark.parametrize("amax,ue8m0,expect", [
    (448.0, False, 1.0),
    (0.0, False, np.float32(1e-4) / np.float32(448.0)),
    (5e-5, False, np.float32(1e-4) / np.float32(448.0)),
    (448.0, True, 1.0),              # already a power of two
    (449.0, True, 2.0),              # rounded up
    (224.0, True, 0.5),
    (1.0, True, 2.0 ** -8),          # 1/448 in (2^-9, 2^-8]
    (0.0, True, 2.0 ** -22),         # 1e-4/448 = 2.23e-7 in (2^-23, 2^-22]
])
def test_block_scale_closed_forms(amax, ue8m0, expect):
    assert oracle.block_scale(amax, ue8m0) == np.float32(expect)
