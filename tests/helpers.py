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
