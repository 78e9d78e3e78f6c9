"""fp8blk_gemm_noalloc: the GEMM for callers that cannot allocate device
memory (an engine plugin that must not allocate while it runs, a loop that
must never reach cudaMalloc/cudaFree, a caller holding only device pointers).
Its scratch is a buffer the library keeps in device memory, shared by every
call on the device.

Checked through the C ABI against fp8blk_gemm (the entry point that takes a
workspace), within the GEMM tolerance the other tests use, on two calls in a
row with different problems -- the second call must not see the first call's
leftovers in the shared buffer -- and on a repeat of the first problem.
Problems that need more scratch than the buffer holds are refused on the
host. This file is collected last; it passes alone and after the others."""
import ctypes

import numpy as np
import pytest
import torch

import fp8_block_scaled_quant_gb300 as fb
import synthetic
from helpers import gemm_tol

pytestmark = pytest.mark.gpu

ERR_TOO_LARGE = 9


def noalloc_fn():
    f = fb.lib().fp8blk_gemm_noalloc
    f.argtypes = [ctypes.c_void_p] * 5 + [ctypes.c_int64] * 3 + [ctypes.c_int, ctypes.c_void_p]
    f.restype = ctypes.c_int
    return f


def problem(M, N, K, seed):
    dev = torch.device("cuda")
    x = synthetic.device_activations(M, K, seed, dev, outlier_frac=0.01)
    w = synthetic.device_normal((N, K), seed + 1, 0.02, dev)
    a, a_s = fb.act_quant(x)
    q, s = fb.weight_quant(w)
    return a, a_s, q, s


def call_noalloc(f, a, a_s, q, s, out):
    M, K = a.shape
    N = q.shape[0]
    stream = torch.cuda.current_stream().cuda_stream
    return f(a.data_ptr(), a_s.data_ptr(), q.data_ptr(), s.data_ptr(), out.data_ptr(), M, N, K, 0, stream)


def assert_close(got, ref):
    g = got.float().cpu().numpy().astype(np.float64)
    r = ref.float().cpu().numpy().astype(np.float64)
    assert np.all(np.abs(g - r) <= gemm_tol(r))


def test_noalloc_matches_gemm_on_two_calls_in_a_row():
    f = noalloc_fn()
    p1 = problem(8, 10944, 2048, 31)      # decode-shaped: stream-K partials in the scratch
    p2 = problem(16, 320, 256, 32)        # another plan on the same scratch
    ref1 = fb.fp8_gemm(*p1)
    ref2 = fb.fp8_gemm(*p2)
    out1 = torch.empty((8, 10944), dtype=torch.bfloat16, device="cuda")
    out2 = torch.empty((16, 320), dtype=torch.bfloat16, device="cuda")
    assert call_noalloc(f, *p1, out1) == 0
    assert call_noalloc(f, *p2, out2) == 0
    torch.cuda.synchronize()
    assert_close(out1, ref1)
    assert_close(out2, ref2)
    out3 = torch.empty_like(out1)
    assert call_noalloc(f, *p1, out3) == 0
    torch.cuda.synchronize()
    assert_close(out3, ref1)
    assert fb.last_device_error() == 0


def test_noalloc_refuses_problems_beyond_its_scratch():
    f = noalloc_fn()
    M, N, K = 4096, 18432, 7168
    assert fb.gemm_workspace_bytes(M, N, K) > (8 << 20)
    # refused on the host before any pointer is read or kernel launched
    assert f(None, None, None, None, None, M, N, K, 0, None) == ERR_TOO_LARGE
    assert b"fp8blk_gemm" in fb.lib().fp8blk_status_string(ERR_TOO_LARGE)
