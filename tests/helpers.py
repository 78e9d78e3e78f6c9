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


# ---- tolerance of the FFN / MoE chains ------------------------------------------
#
# The chains (SwiGLU FFN, routed experts) re-quantise their intermediate
# u = bf16(bf16(silu(h1)) * h3) to e4m3 before the w2 GEMM. A legitimate fp32
# summation order can move h1 or h3 (or silu in fp32) by one bf16 step from the
# fp64 oracle's, and when u/s then sits at an e4m3 rounding midpoint its code
# moves by one step. Such a flip shifts output element n of that row by
# step_i * |w2[n, i]|, which the plain GEMM tolerance does not cover for small
# outputs. The chain criterion is therefore:
#   (1) at least 99.5 % of the elements meet the plain GEMM tolerance, and
#   (2) every element meets it plus the effect of up to two one-step flips in
#       its row, 2 * max_i step_i * |w2[n, i]|, with step_i the e4m3 step at
#       the oracle's own u (at most 2^-3 |u_i| for normal codes, 2^-9 s for
#       subnormal ones).

def dequant_weight(q: np.ndarray, s: np.ndarray) -> np.ndarray:
    import oracle

    N, K = q.shape
    return oracle.e4m3_decode_array(q) * np.repeat(np.repeat(s.astype(np.float64), 128, 0), 128, 1)[:N, :K]


def flip_allowance(uq: np.ndarray, us: np.ndarray, w2_deq: np.ndarray, flips: int = 2) -> np.ndarray:
    """[rows, dim]: flips * max_i step_i * |w2[n, i]| for each row of the
    oracle's quantised intermediate (uq [rows, inter], us [rows, inter/128])."""
    import oracle

    sc = np.repeat(us.astype(np.float64), 128, axis=1)
    dq = oracle.e4m3_decode_array(uq) * sc
    step = np.maximum(2.0 ** -3 * np.abs(dq), 2.0 ** -9 * sc)
    aw = np.abs(w2_deq)
    out = np.empty((uq.shape[0], w2_deq.shape[0]))
    for r in range(uq.shape[0]):
        out[r] = flips * np.max(aw * step[r][None, :], axis=1)
    return out


def assert_chain_close(got_bits: np.ndarray, ref: np.ndarray, allowance: np.ndarray, rms: float | None = None,
                       frac: float = 0.995, what: str = ""):
    got = bf16_bits_to_f64(got_bits)
    tol = gemm_tol(ref, rms)
    err = np.abs(got - ref)
    within = err <= tol
    assert within.mean() >= frac, f"{what}: only {within.mean():.4%} within the GEMM tolerance"
    bad = err > tol + allowance
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(f"{what}: {bad.sum()} elements beyond tolerance + flip allowance; first "
                             f"{idx.tolist()}: got {got[bad][:5]}, ref {ref[bad][:5]}")
