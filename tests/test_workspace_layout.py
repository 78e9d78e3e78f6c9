"""Host-side check of the workspace sizes the library reports (no GPU).

Without a device the library plans for 256 SMs, no cluster pairs and no
split-K clusters. Every GEMM workspace is then the fixed 64 KB counter region,
followed, for plans that cut tiles stream-K, by two partial slots (BN x 128
fp32) per CTA of the plan, the CTA count coming from the same schedule rule
the kernels walk (mirrored in test_gemm_schedule); plans of whole tiles or
weight slices need the counter region only. The composite layouts put that GEMM workspace first,
then their own parts, each 256-byte aligned: the sizes must be exactly those
sums, so that the GEMM's counters sit at offset 0 whatever the shape."""
import ctypes

import pytest

import fp8_block_scaled_quant_gb300 as fb
from test_gemm_schedule import make_plan

COUNTERS = 64 * 1024


def a256(v):
    return (v + 255) // 256 * 256


def lib_size(name, *args):
    f = getattr(fb.lib(), name)
    f.argtypes = [ctypes.c_int64] * len(args)
    f.restype = ctypes.c_size_t
    return int(f(*args))


def gemm_ws(M, N, K):
    p = make_plan(M, N, K, 256, pairs=0, split_k=False)
    slots = 2 * p["grid"] * p["cluster"] * p["bn"] * 128 * 4 if p["sk_tiles"] > 0 else 0
    return COUNTERS + slots


def swiglu_ws(M, inter, dim):
    """The fused w1/w3 GEMM: 128 x 256 tiles (128 output columns), no pairs;
    whole tiles (more tiles than counters, or stream-K saving the busiest CTA
    at most 32 K blocks: no slots) or data-parallel waves use every SM,
    stream-K at most one CTA per (tile, K block)."""
    tiles = -(-M // 128) * (inter // 128)
    if tiles > COUNTERS // 4:
        return COUNTERS
    Kb = dim // 128
    if -(-tiles // 256) * Kb * 256 - tiles * Kb <= 32 * 256:
        return COUNTERS
    grid = 256 if tiles >= 2 * 256 else min(256, tiles * (dim // 128))
    return COUNTERS + 2 * grid * 256 * 128 * 4


SHAPES = [(16, 320, 256), (8, 10944, 2048), (64, 10944, 2048), (8, 65536, 1024), (32, 40960, 1536),
          (100, 24576, 1536), (300, 576, 1024), (1300, 7000, 640),
          (4096, 18432, 7168), (4096, 7168, 18432), (2048, 32768, 512), (129, 130, 128), (40000, 60000, 256)]


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_gemm_workspace_is_counters_then_slots(M, N, K):
    assert lib_size("fp8blk_gemm_workspace_bytes", M, N, K) == gemm_ws(M, N, K)


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_linear_workspaces_start_with_the_gemm_workspace(M, N, K):
    g = lib_size("fp8blk_gemm_workspace_bytes", M, N, K)
    lin = lib_size("fp8blk_linear_workspace_bytes", M, N, K)
    assert lin == a256(g) + a256(M * K) + a256(M * (K // 128) * 4)
    host = lib_size("fp8blk_linear_host_workspace_bytes", M, N, K)
    assert host == a256(lin) + a256(M * K * 2) + a256(M * N * 2)


@pytest.mark.parametrize("M,dim,inter", [(5, 256, 384), (300, 256, 1024), (1300, 512, 1024),
                                         (4096, 7168, 18432)])
def test_ffn_workspace_shares_one_gemm_region(M, dim, inter):
    sw = lib_size("fp8blk_swiglu_workspace_bytes", M, inter, dim)
    assert sw == swiglu_ws(M, inter, dim)
    g2 = lib_size("fp8blk_gemm_workspace_bytes", M, dim, inter)
    ffn = lib_size("fp8blk_ffn_workspace_bytes", M, dim, inter)
    assert ffn == a256(max(sw, g2)) + a256(M * dim) + a256(M * (dim // 128) * 4) + a256(M * inter) + \
        a256(M * (inter // 128) * 4)
