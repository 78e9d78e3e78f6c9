"""The C-ABI library loads without a GPU and exports every function that
include/fp8blk.h declares; argument checks that need no device return their
status codes (no kernel is launched)."""
import ctypes
import os
import subprocess

import pytest

import fp8_block_scaled_quant_gb300 as fb


@pytest.fixture(scope="module")
def L():
    if not os.path.exists(fb.lib_path()):
        from fp8_block_scaled_quant_gb300 import _build
        _build.build()
    return fb.lib()


def test_header_declares_the_api():
    names = fb.header_functions()
    for n in ("fp8blk_act_quant", "fp8blk_weight_dequant", "fp8blk_gemm", "fp8blk_linear",
              "fp8blk_linear_host", "fp8blk_weight_quant", "fp8blk_last_device_error"):
        assert n in names


def test_every_declared_symbol_is_exported(L):
    raw = ctypes.CDLL(fb.lib_path())
    for name in fb.header_functions():
        assert hasattr(raw, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", fb.lib_path()], capture_output=True, text=True).stdout
    exported = {ln.split()[-1] for ln in out.splitlines() if " T " in ln}
    assert set(fb.header_functions()) <= exported
    # nothing else leaks out of the library under the fp8blk_ prefix
    assert {n for n in exported if n.startswith("fp8blk_")} == set(fb.header_functions())


def test_no_gpu_runtime_needed_to_load():
    out = subprocess.run(["ldd", fb.lib_path()], capture_output=True, text=True).stdout
    assert "libcuda.so" not in out and "libcudart" not in out


def test_status_strings_and_version(L):
    assert L.fp8blk_status_string(0) == b"ok"
    assert b"128" in L.fp8blk_status_string(2)
    assert L.fp8blk_status_string(12345) == b"unknown status"
    assert L.fp8blk_version() >= 100


def test_host_side_argument_checks_without_gpu(L):
    # shape / enum / null errors are decided before any device query
    assert L.fp8blk_act_quant(None, 4, 100, None, None, 0, None) == 2      # K % 128
    assert L.fp8blk_act_quant(None, 4, 128, None, None, 3, None) == 8      # scale format
    assert L.fp8blk_act_quant(None, 4, 128, None, None, 0, None) == 1      # null
    assert L.fp8blk_act_quant(None, 0, 128, None, None, 0, None) == 0      # empty: no-op
    assert L.fp8blk_act_quant(None, -1, 128, None, None, 0, None) == 2
    assert L.fp8blk_weight_dequant(None, None, 0, 5, None, None) == 0
    assert L.fp8blk_weight_dequant(None, None, 3, 5, None, None) == 1
    assert L.fp8blk_gemm(None, None, None, None, None, 2, 2, 100, 0, None, 0, None) == 2
    n = ctypes.c_int(-1)
    assert L.fp8blk_linear_kernels(4, 8, 100, ctypes.byref(n)) == 2       # K % 128
    assert L.fp8blk_linear_kernels(4, 8, 128, None) == 1                  # null
    assert L.fp8blk_linear_kernels(0, 8, 128, ctypes.byref(n)) == 0 and n.value == 0   # empty
    assert L.fp8blk_gemm(None, None, None, None, None, 0, 2, 128, 0, None, 0, None) == 0
    assert L.fp8blk_linear(None, None, None, None, 2, 2, 100, 0, None, 0, None) == 2
    assert L.fp8blk_linear_host(None, None, None, None, 2, 2, 128, 0, None, 0, None) == 1
    assert L.fp8blk_gemm_workspace_bytes(8, 10944, 2048) > 0
