"""fp8blk_gemm_noalloc: the GEMM for callers that cannot allocate device
memory (an engine plugin that must not allocate while it runs, a loop that
must never reach cudaMalloc/cudaFree, a caller holding only device pointers).
Its scratch is a buffer the library keeps in device memory, shared by every
call on the device.

Checked through the C ABI against fp8blk_gemm (the entry point that takes a
workspace). Both run the same plan and the same kernels, whose partial sums
are added in a fixed order, so the outputs must be bit-identical. The calls
come in a row on the shared buffer: a problem whose plan splits tiles
stream-K (partial sums written to the buffer's slots, tile counters
incremented and reset), then problems with other plans, then the first
problem again -- no call may see another's leftovers. Problems that need
more scratch than the buffer holds are refused on the host, after the same
argument checks as fp8blk_gemm. This file is collected last; it passes alone
and after the others."""
import ctypes

import numpy as np
import pytest
import torch

import fp8_block_scaled_quant_gb300 as fb
import synthetic
from test_gemm_schedule import decode_plan, make_plan, units

pytestmark = pytest.mark.gpu

ERR_NULL = 1
ERR_ARG = 8
ERR_TOO_LARGE = 9
SCRATCH = 8 << 20


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


def assert_same_bits(got, ref):
    assert torch.equal(got.view(torch.int16), ref.view(torch.int16))


def test_stream_k_shape_writes_partials():
    """The first problem below really runs stream-K with split tiles (plan
    mirror at this GPU's SM count), within the scratch."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for M, N, K in ((24, 320, 256), (20, 640, 384)):
        assert decode_plan(M, N, K, sms) is None   # more than 16 tokens: the tcgen05 swapped kernel
        p = make_plan(M, N, K, sms)
        assert p["swap"] and p["ksplit"] == 1 and not p.get("whole") and p["sk_tiles"] > 0
        assert any(u[4] > 1 for c in range(p["grid"]) for u in units(p, c)), "no tile is split"
        assert fb.gemm_workspace_bytes(M, N, K) <= SCRATCH


def test_noalloc_matches_gemm_on_calls_in_a_row():
    f = noalloc_fn()
    # stream-K with split tiles; whole tiles round-robin past one per SM; the
    # slice-per-SM decode kernel; one CTA per whole tile (BN 64); stream-K
    # again with another split.
    shapes = [(24, 320, 256), (8, 24576, 1536), (8, 10944, 2048), (64, 10944, 2048), (20, 640, 384)]
    probs = [problem(M, N, K, 31 + i) for i, (M, N, K) in enumerate(shapes)]
    refs = [fb.fp8_gemm(*p) for p in probs]
    outs = [torch.empty_like(r) for r in refs]
    for p, o in zip(probs, outs):
        assert call_noalloc(f, *p, o) == 0
    again = torch.empty_like(refs[0])
    assert call_noalloc(f, *probs[0], again) == 0
    torch.cuda.synchronize()
    for o, r in zip(outs, refs):
        assert_same_bits(o, r)
    assert_same_bits(again, refs[0])
    assert fb.last_device_error() == 0


def test_noalloc_checks_arguments_then_size():
    f = noalloc_fn()
    M, N, K = 4096, 18432, 7168
    assert fb.gemm_workspace_bytes(M, N, K) > SCRATCH
    buf = torch.zeros(256, dtype=torch.uint8, device="cuda")   # aligned, never read: the call is refused
    p = buf.data_ptr()
    stream = torch.cuda.current_stream().cuda_stream
    # argument errors come first, as in fp8blk_gemm
    assert f(None, None, None, None, None, M, N, K, 0, stream) == ERR_NULL
    assert f(p, p, p, p, p, M, N, K, 7, stream) == ERR_ARG
    # then the size: refused on the host, nothing launched or cleared
    assert f(p, p, p, p, p, M, N, K, 0, stream) == ERR_TOO_LARGE
    torch.cuda.synchronize()
    assert int(buf.sum()) == 0
    assert b"fp8blk_gemm" in fb.lib().fp8blk_status_string(ERR_TOO_LARGE)
