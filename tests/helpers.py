"""Shared helpers for the GPU parity tests: moving seeded inputs between host
and device, and the GEMM tolerance.

GEMM tolerance, per element, against the oracle's fp64 value ref:
    |gpu - ref| <= 2^-7 * |ref| + 1e-3 * rms(ref over the whole output)
(2^-7 is two bf16 rounding steps: the output's own rounding, 2^-9 relative,
leaves ample room for fp32 accumulation of the per-block partials)."""
import numpy as np
import torch

import synthetic


def bits_to_dev_bf16(bits: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(bits.view(np.int16).copy()).to(device).view(torch.bfloat16)


def dev_to_bits(t: torch.Tensor) -> np.ndarray:
    """Raw bytes of a device tensor as a numpy array (uint8 for fp8, uint16 for bf16)."""
    if t.dtype == torch.float8_e4m3fn:
        return t.view(torch.uint8).cpu().numpy()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


def bf16_bits_to_f64(b: np.ndarray) -> np.ndarray:
    return synthetic.bf16_bits_to_f32(b).astype(np.float64)


def gemm_tol(ref: np.ndarray, rms: float | None = None) -> np.ndarray:
    if rms is None:
        rms = float(np.sqrt(np.mean(np.square(ref))))
    return 2.0 ** -7 * np.abs(ref) + 1e-3 * rms


def assert_gemm_close(got_bits: np.ndarray, ref: np.ndarray, rms: float | None = None, what: str = ""):
    got = bf16_bits_to_f64(got_bits)
    tol = gemm_tol(ref, rms)
    err = np.abs(got - ref)
    bad = err > tol
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} outside tolerance; first {idx.tolist()}: "
                             f"got {got[bad][:5]}, ref {ref[bad][:5]}")


# ---- the FFN / MoE chains: admissible intermediates ------------------------------
#
# The chains (SwiGLU FFN, routed experts) re-quantise their intermediate
# u = bf16(bf16(silu(h1)) * h3) to e4m3 before the w2 GEMM ("Administrator &
# Developer Guide" 1.2 MLP / Expert; 6.3: every Linear quantises its input).
# h1 and h3 are GEMM outputs, fixed only up to fp32 summation order, so the
# GPU's u may legitimately differ from the oracle's by a bf16 step, which can
# move an e4m3 code (u near a rounding midpoint) or a block scale (the block's
# amax element). Instead of counting such differences, the tests bound them:
#
#   1. h = bf16(fp32 GEMM value) with the fp32 value within
#      2^-12 |H| + 2^-13 rms(H) of the oracle's fp64 H (fp32 accumulation of
#      the per-block partials; far inside the GEMM tolerance);
#   2. silu in fp32 within 2^-19 relative of the exact value, rounded to bf16;
#   3. u = bf16(g * h3) (the product of two bf16 numbers is exact in fp32);
#   4. the block scale s = scale(amax) is monotone in amax, and each code
#      e4m3(u / s) (fp32 division, round to nearest even) is monotone in u / s.
#
# Every admissible (scale, code) pair then lies in intervals computed from
# the oracle's H alone. The intermediate test requires the GPU's scales and
# codes to lie in them; the chain tests allow, on top of the GEMM tolerance,
# exactly the output change those intervals permit:
#   |y' - y| <= sum_i |c'_i - c_i| s_hi |w2_i| + sum_b |s'_b - s_b| / s_b |Y_b|,
# with Y_b the oracle's contribution of block b. Elements whose code and
# block scale are unique contribute nothing.

def dequant_weight(q: np.ndarray, s: np.ndarray) -> np.ndarray:
    import oracle

    N, K = q.shape
    return oracle.e4m3_decode_array(q) * np.repeat(np.repeat(s.astype(np.float64), 128, 0), 128, 1)[:N, :K]


def bf16_rn(v: np.ndarray) -> np.ndarray:
    """fp64 values of the oracle's bf16 rounding (nearest even) of v."""
    import oracle

    return synthetic.bf16_bits_to_f32(oracle.bf16_round(np.asarray(v, np.float64))).astype(np.float64)


def _silu(v):
    with np.errstate(over="ignore"):
        return v / (1.0 + np.exp(-v))


def _silu_minimum():
    """(argmin, min) of v / (1 + e^-v): where 1 + v (1 - sigmoid(v)) = 0, by bisection."""
    lo, hi = -2.0, -1.0
    for _ in range(200):
        mid = 0.5 * (lo + hi)
        sg = 1.0 / (1.0 + np.exp(-mid))
        if 1.0 + mid * (1.0 - sg) > 0.0:
            hi = mid
        else:
            lo = mid
    return lo, float(_silu(lo))


SILU_ARGMIN, SILU_MIN = _silu_minimum()


def admissible_u(H1: np.ndarray, H3: np.ndarray):
    """[u_lo, u_hi] (fp64 values of bf16 numbers, elementwise) holding every u
    a chain may compute from GEMM values within rule 1 of the oracle's H1, H3."""
    def h_range(H):
        e = 2.0 ** -12 * np.abs(H) + 2.0 ** -13 * float(np.sqrt(np.mean(np.square(H))))
        return bf16_rn(H - e), bf16_rn(H + e)

    h1_lo, h1_hi = h_range(H1)
    h3_lo, h3_hi = h_range(H3)
    f_a, f_b = _silu(h1_lo), _silu(h1_hi)
    f_min = np.where((h1_lo <= SILU_ARGMIN) & (SILU_ARGMIN <= h1_hi), SILU_MIN, np.minimum(f_a, f_b))
    f_max = np.maximum(f_a, f_b)
    d = 2.0 ** -19
    g_lo = bf16_rn(f_min - d * np.abs(f_min))
    g_hi = bf16_rn(f_max + d * np.abs(f_max))
    corners = np.stack([g_lo * h3_lo, g_lo * h3_hi, g_hi * h3_lo, g_hi * h3_hi])
    return bf16_rn(corners.min(0)), bf16_rn(corners.max(0))


def admissible_quant(u_lo: np.ndarray, u_hi: np.ndarray, ue8m0: bool = False):
    """Bounds of act_quant over every u in [u_lo, u_hi]: block scales
    s_lo <= s <= s_hi (fp32 [rows, cols/128]) and decoded code values
    c_lo <= c <= c_hi (fp64 [rows, cols])."""
    import oracle

    rows, cols = u_lo.shape
    nb = cols // 128
    a_lo = np.where((u_lo <= 0) & (u_hi >= 0), 0.0, np.minimum(np.abs(u_lo), np.abs(u_hi)))
    a_hi = np.maximum(np.abs(u_lo), np.abs(u_hi))
    amax_lo = a_lo.reshape(rows, nb, 128).max(-1).astype(np.float32)
    amax_hi = a_hi.reshape(rows, nb, 128).max(-1).astype(np.float32)
    scale = np.vectorize(lambda a: oracle.block_scale(float(a), int(ue8m0)), otypes=[np.float32])
    s_lo, s_hi = scale(amax_lo), scale(amax_hi)
    sl, sh = np.repeat(s_lo, 128, axis=1), np.repeat(s_hi, 128, axis=1)
    q = np.stack([u.astype(np.float32) / s for u in (u_lo, u_hi) for s in (sl, sh)])   # IEEE fp32 divisions
    c_lo = oracle.e4m3_decode_array(oracle.e4m3_encode_array(q.min(0)))
    c_hi = oracle.e4m3_decode_array(oracle.e4m3_encode_array(q.max(0)))
    return s_lo, s_hi, c_lo, c_hi


def assert_quant_admissible(got_q: np.ndarray, got_s: np.ndarray, adm, ue8m0: bool, what: str = ""):
    """Every GPU scale and code of the re-quantised intermediate lies in the
    admissible intervals, and each block is consistent with its own scale: its
    largest code is +-448 (fp32 scales) or in [224, 448] (UE8M0), unless the
    block's amax was below the 1e-4 clamp."""
    import oracle

    s_lo, s_hi, c_lo, c_hi = adm
    assert np.all((got_s >= s_lo) & (got_s <= s_hi)), f"{what}: a block scale outside its admissible interval"
    c = oracle.e4m3_decode_array(got_q)
    bad = ~((c >= c_lo) & (c <= c_hi))
    assert not bad.any(), f"{what}: {bad.sum()} codes outside their admissible interval, first {np.argwhere(bad)[:3]}"
    rows, cols = c.shape
    top = np.abs(c).reshape(rows, cols // 128, 128).max(-1)
    live = got_s > np.float32(1e-4) / np.float32(448.0)
    if ue8m0:
        assert np.all((top[live] >= 224) & (top[live] <= 448)), f"{what}: block maximum code off its UE8M0 scale"
    else:
        assert np.all(top[live] == 448), f"{what}: a block's amax element is not coded +-448"


def chain_allowance(uq: np.ndarray, us: np.ndarray, adm, w2_deq: np.ndarray) -> np.ndarray:
    """[rows, dim]: the most any admissible re-quantised intermediate can move
    the chain's output from the oracle's (its own uq, us), by the bound above."""
    import oracle

    s_lo, s_hi, c_lo, c_hi = adm
    rows, cols = uq.shape
    nb = cols // 128
    c = oracle.e4m3_decode_array(uq)
    s = us.astype(np.float64)
    dc = np.maximum(c_hi - c, c - c_lo) * np.repeat(s_hi.astype(np.float64), 128, axis=1)
    out = dc @ np.abs(w2_deq).T
    ds = np.maximum(s_hi.astype(np.float64) - s, s - s_lo.astype(np.float64)) / s
    for b in range(nb):
        if not ds[:, b].any():
            continue
        yb = (c[:, b * 128:(b + 1) * 128] * s[:, b:b + 1]) @ w2_deq[:, b * 128:(b + 1) * 128].T
        out += ds[:, b:b + 1] * np.abs(yb)
    return out * (1.0 + 2.0 ** -7)


def assert_chain_close(got_bits: np.ndarray, ref: np.ndarray, allowance: np.ndarray, rms: float | None = None,
                       what: str = ""):
    """Every element within the GEMM tolerance of the oracle's output plus the
    chain allowance (no fraction of elements is exempt)."""
    got = bf16_bits_to_f64(got_bits)
    tol = gemm_tol(ref, rms) + allowance
    err = np.abs(got - ref)
    bad = err > tol
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} elements beyond tolerance + chain allowance; first "
                             f"{idx.tolist()}: got {got[bad][:5]}, ref {ref[bad][:5]}, tol {tol[bad][:5]}")


def ffn_chain_allowance(xq, xs, w1q, w1s, w3q, w3s, w2_deq, uq, us, ue8m0=False) -> np.ndarray:
    """chain_allowance for the FFN rows xq (their oracle intermediates uq, us),
    from the oracle's fp64 h1 and h3 of those rows."""
    import oracle

    H1 = oracle.gemm(xq, xs, w1q, w1s)
    H3 = oracle.gemm(xq, xs, w3q, w3s)
    return chain_allowance(uq, us, admissible_quant(*admissible_u(H1, H3), ue8m0), w2_deq)
