"""GPU parity of fp8_gemm (and the FP8 linear layer) against the CPU oracle.

Small and medium shapes compare every output element; the full-size
workloads compare sampled elements (all edge tiles plus random ones) that the
oracle computes one by one. The oracle always quantises its inputs itself
from the same seeded bf16 / fp32 data; the GPU codes are checked bit-exact
against it on the way."""
import numpy as np
import pytest
import torch

import fp8_block_scaled_quant_gb300 as fb
import oracle
import synthetic
from helpers import assert_gemm_close, bits_to_dev_bf16, dev_to_bits, gemm_tol

pytestmark = pytest.mark.gpu


def host_problem(M, N, K, seed, frac=0.0, ue8m0=False):
    x = synthetic.activations(M, K, seed, outlier_frac=frac)
    w = synthetic.weights(N, K, seed)
    xq, xs = oracle.act_quant(x, ue8m0)
    wq, ws = oracle.weight_quant(w, ue8m0)
    return x, w, xq, xs, wq, ws


def gpu_quantised(x, w, fmt):
    a, a_s = fb.act_quant(bits_to_dev_bf16(x), fmt)
    q, s = fb.weight_quant(torch.from_numpy(w).cuda(), fmt)
    return a, a_s, q, s


SHAPES = [
    (16, 320, 256, 0.0),      # the smallest workload: last weight block 64 rows
    (1, 10944, 2048, 0.01),   # decode
    (8, 10944, 2048, 0.01),
    (64, 10944, 2048, 0.01),
    (5, 2999, 1024, 0.0),     # swapped, ragged last weight tile (N % 128 = 55)
    (24, 4000, 1024, 0.0),    # swapped, BN 32
    (40, 9000, 2048, 0.01),   # swapped, BN 64, ragged last weight tile
    (8, 1000, 8192, 0.0),     # swapped, 64 K blocks through the stage and TMEM rings
    (17, 576, 7168, 0.0),     # swapped, BN 32, N not 128-aligned
    (100, 1536, 512, 0.0),    # swapped, BN 128
    (128, 260, 384, 0.0),
    (129, 320, 256, 0.0),     # first non-swapped size, ragged M tail
    (300, 576, 1024, 0.02),   # N = 576: last block partial, 128-column tiles (few tiles)
    (1300, 7000, 640, 0.0),   # 128 x 256 cluster pairs: odd row-tile count, ragged N
    (257, 128, 2048, 0.0),    # BN 128 path
    (1000, 1000, 128, 0.0),   # single K block, N % 8 == 0
    (80, 20000, 128, 0.0),    # swapped BN 128, 157 whole weight tiles round-robin (more than SMs), ragged N
    (512, 2304, 1536, 0.0),   # several data-parallel waves
    (64, 1536, 7168, 0.0),    # few weight tiles: split-K clusters (8 CTAs per tile)
    (8, 1536, 7168, 0.01),
    (50, 300, 1024, 0.0),     # split-K clusters of 4, ragged M and N
    (1, 640, 4096, 0.01),     # split-K, one token
    (24, 7300, 512, 0.0),     # weight slices of 56 rows (BN 32): ragged last slice, slices across scale blocks
    (3, 12160, 1024, 0.01),   # weight slices of exactly 80 rows
    (16, 11000, 384, 0.0),    # slices of 80 rows, the last one 40
    (33, 10944, 1024, 0.0),   # slices of 72 rows with BN 64
    # The slice-per-SM decode kernel (M <= 16, a CTA's weight slice in shared memory):
    (9, 10944, 2048, 0.01),   # two token fragments, seven of them padding; 72-row slices (a half row group)
    (16, 38912, 256, 0.0),    # 256-row slices: 16 row groups, one K slice each, one K block per box
    (4, 7, 128, 0.0),         # one CTA, one K block, weight rows past N read as zeros
    (1, 1217, 640, 0.01),     # 16-row slices, the last one a single row; 5 K blocks in boxes of 3 (one past K)
    (7, 3600, 384, 0.0),      # 24-row slices, some across 128-row scale blocks; 3 K slices of one K block
    (12, 640, 7168, 0.0),     # 8-row slices, 20 K slices of 2-3 K blocks
    # M <= 16 where the slice does not fit: the tcgen05 swapped kernel
    (8, 24576, 1536, 0.0),
    (16, 10944, 7168, 0.01),
]


@pytest.mark.parametrize("M,N,K,frac", SHAPES)
def test_gemm_full_compare(M, N, K, frac):
    x, w, xq, xs, wq, ws = host_problem(M, N, K, 1000 + M + N, frac)
    a, a_s, q, s = gpu_quantised(x, w, fb.SCALE_FP32)
    assert np.array_equal(dev_to_bits(a), xq) and np.array_equal(dev_to_bits(q), wq)
    c = fb.fp8_gemm(a, a_s, q, s)
    ref = oracle.gemm(xq, xs, wq, ws)
    assert_gemm_close(dev_to_bits(c), ref, what=f"{M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K", [(8, 1000, 1024), (300, 700, 512)])
def test_gemm_ue8m0_scales(M, N, K):
    x, w, xq, xs, wq, ws = host_problem(M, N, K, 77, 0.01, ue8m0=True)
    a, a_s, q, s = gpu_quantised(x, w, fb.SCALE_UE8M0)
    assert np.array_equal(dev_to_bits(a), xq) and np.array_equal(dev_to_bits(q), wq)
    c = fb.fp8_gemm(a, a_s, q, s, scale_fmt=fb.SCALE_UE8M0)
    assert_gemm_close(dev_to_bits(c), oracle.gemm(xq, xs, wq, ws))


def test_gemm_pr1_golden():
    """The 16x320x256 workload against the stored oracle output (bf16 of the
    fp64 product), within the GEMM tolerance plus one bf16 step."""
    import test_oracle_golden as g
    x = synthetic.activations(16, 256, synthetic.SEED_PR1)
    w = synthetic.weights(320, 256, synthetic.SEED_PR1)
    a, a_s, q, s = gpu_quantised(x, w, fb.SCALE_FP32)
    c = dev_to_bits(fb.fp8_gemm(a, a_s, q, s))
    want = synthetic.bf16_bits_to_f32(g.load_pr1_out()).astype(np.float64)
    got = synthetic.bf16_bits_to_f32(c).astype(np.float64)
    assert np.all(np.abs(got - want) <= gemm_tol(want) + 2.0 ** -8 * np.abs(want))


def test_gemm_deterministic_and_workspace_restored():
    x, w, xq, xs, wq, ws = host_problem(8, 10944, 2048, 5, 0.01)
    a, a_s, q, s = gpu_quantised(x, w, fb.SCALE_FP32)
    nbytes = fb.gemm_workspace_bytes(8, 10944, 2048)
    wsb = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    c1 = fb.fp8_gemm(a, a_s, q, s, ws=wsb)
    tiles = (10944 + 127) // 128
    assert torch.count_nonzero(wsb[: tiles * 4]) == 0      # counters back at zero
    c2 = fb.fp8_gemm(a, a_s, q, s, ws=wsb)
    assert torch.equal(c1.view(torch.int16), c2.view(torch.int16))


def test_gemm_workspace_shared_by_plans_of_different_shapes():
    """One workspace serves GEMMs of different shapes. A small stream-K GEMM
    (15 tiles, each cut into parts) fills its partial slots; a larger one
    (cluster-pair tiles with a stream-K tail) then counts part arrivals in the
    same buffer. Its output must equal, bit for bit, the output on a fresh
    workspace, and the counters must end at zero."""
    dev = torch.device("cuda")
    small, big = (300, 576, 1024), (1300, 7000, 640)
    ops = []
    for i, (M, N, K) in enumerate((small, big)):
        a, a_s = fb.act_quant(synthetic.device_activations(M, K, 61 + i, dev))
        q, s = fb.weight_quant(synthetic.device_normal((N, K), 71 + i, 0.02, dev))
        ops.append((a, a_s, q, s, fb.gemm_workspace_bytes(M, N, K)))
    a, a_s, q, s, nb = ops[1]
    want = fb.fp8_gemm(a, a_s, q, s, ws=torch.zeros(nb, dtype=torch.uint8, device=dev))
    shared = torch.zeros(max(o[4] for o in ops), dtype=torch.uint8, device=dev)
    for _ in range(2):
        a1, a1_s, q1, s1, nb1 = ops[0]
        fb.fp8_gemm(a1, a1_s, q1, s1, ws=shared[:nb1])
        got = fb.fp8_gemm(a, a_s, q, s, ws=shared[:nb])
        assert torch.equal(got.view(torch.int16), want.view(torch.int16))
    assert torch.count_nonzero(shared[:64 * 1024]) == 0
    assert fb.last_device_error() == 0


def test_linear_workspace_shared_by_layers_of_different_shapes():
    """The linear layer's workspace keeps the GEMM's tile counters at offset 0
    whatever the shape, so one workspace serves layers of different shapes
    (a small stream-K layer, then a larger one): bit-equal to fresh workspaces."""
    dev = torch.device("cuda")
    shapes = [(300, 576, 1024), (1300, 7000, 640)]
    layers = []
    for i, (M, N, K) in enumerate(shapes):
        x = synthetic.device_activations(M, K, 81 + i, dev)
        q, s = fb.weight_quant(synthetic.device_normal((N, K), 91 + i, 0.02, dev))
        nb = fb.linear_workspace_bytes(M, N, K)
        want = fb.linear(x, q, s, ws=torch.zeros(nb, dtype=torch.uint8, device=dev))
        layers.append((x, q, s, nb, want))
    shared = torch.zeros(max(l[3] for l in layers), dtype=torch.uint8, device=dev)
    for _ in range(2):
        for x, q, s, nb, want in layers:
            got = fb.linear(x, q, s, ws=shared[:nb])
            assert torch.equal(got.view(torch.int16), want.view(torch.int16))
    assert torch.count_nonzero(shared[:64 * 1024]) == 0
    assert fb.last_device_error() == 0


@pytest.mark.parametrize("M,N,K", [(64, 576, 7168), (4096, 7168, 18432)])
def test_gemm_split_paths_deterministic(M, N, K):
    """Split-K clusters (few weight tiles) and stream-K cluster pairs reduce
    partials in a fixed order: two calls give identical bits."""
    dev = torch.device("cuda")
    x = synthetic.device_activations(M, K, 77, dev)
    a, a_s = fb.act_quant(x)
    q, s = fb.weight_quant(synthetic.device_normal((N, K), 78, 0.02, dev))
    c1 = fb.fp8_gemm(a, a_s, q, s)
    c2 = fb.fp8_gemm(a, a_s, q, s)
    assert torch.equal(c1.view(torch.int16), c2.view(torch.int16))
    assert fb.last_device_error() == 0


def test_gemm_edge_cases():
    L = fb.lib()
    a = torch.zeros((4, 256), dtype=torch.float8_e4m3fn, device="cuda")
    a_s = torch.ones((4, 2), device="cuda")
    w = torch.zeros((8, 256), dtype=torch.float8_e4m3fn, device="cuda")
    w_s = torch.ones((1, 2), device="cuda")
    c = torch.full((4, 8), 7.0, dtype=torch.bfloat16, device="cuda")
    ws = fb.workspace(fb.gemm_workspace_bytes(4, 8, 256), torch.device("cuda"))
    p = lambda t: t.data_ptr()
    # K % 128 != 0
    assert L.fp8blk_gemm(p(a), p(a_s), p(w), p(w_s), p(c), 4, 8, 200, 0, p(ws), ws.numel(), None) == 2
    # misaligned operand
    assert L.fp8blk_gemm(p(a) + 8, p(a_s), p(w), p(w_s), p(c), 4, 8, 128, 0, p(ws), ws.numel(), None) == 3
    # workspace too small
    assert L.fp8blk_gemm(p(a), p(a_s), p(w), p(w_s), p(c), 4, 8, 256, 0, p(ws), 16, None) == 4
    # null operand
    assert L.fp8blk_gemm(None, p(a_s), p(w), p(w_s), p(c), 4, 8, 256, 0, p(ws), ws.numel(), None) == 1
    # bad scale format
    assert L.fp8blk_gemm(p(a), p(a_s), p(w), p(w_s), p(c), 4, 8, 256, 5, p(ws), ws.numel(), None) == 8
    # M == 0 and N == 0 are no-ops
    assert L.fp8blk_gemm(None, None, None, None, p(c), 0, 8, 256, 0, None, 0, None) == 0
    assert L.fp8blk_gemm(None, None, None, None, p(c), 4, 0, 256, 0, None, 0, None) == 0
    # K == 0: an empty sum, zeros
    assert L.fp8blk_gemm(None, None, None, None, p(c), 4, 8, 0, 0, None, 0, None) == 0
    torch.cuda.synchronize()
    assert torch.count_nonzero(c.float()) == 0


def test_gemm_unaligned_output_scalar_stores():
    """N % 8 != 0 forces the scalar store path (non-swapped and swapped)."""
    for M, N in ((200, 131), (5, 131)):
        x, w, xq, xs, wq, ws = host_problem(M, N, 256, 9)
        a, a_s, q, s = gpu_quantised(x, w, fb.SCALE_FP32)
        c = fb.fp8_gemm(a, a_s, q, s)
        assert_gemm_close(dev_to_bits(c), oracle.gemm(xq, xs, wq, ws))


# ---- full-size workloads, sampled ------------------------------------------------

def sampled_check(M, N, K, seed, frac=0.0, n_random=48, fmt=fb.SCALE_FP32):
    """Device-generated inputs at full size; the oracle recomputes sampled
    outputs from host copies of the same bf16 / fp32 inputs (quantising the
    needed rows and weight blocks itself)."""
    dev = torch.device("cuda")
    ue = (fmt & ~fb.SCALE_PROMOTE) == fb.SCALE_UE8M0
    x = synthetic.device_activations(M, K, seed, dev, outlier_frac=frac)
    w = synthetic.device_normal((N, K), seed + 1, 0.02, dev)
    a, a_s = fb.act_quant(x, fmt)
    q, s = fb.weight_quant(w, fmt)
    c = fb.fp8_gemm(a, a_s, q, s, scale_fmt=fmt)
    g = np.random.Generator(np.random.PCG64(seed))
    ms = np.concatenate([[0, M - 1, min(127, M - 1), min(128, M - 1)], g.integers(0, M, n_random)])
    ns = np.concatenate([[0, N - 1, min(127, N - 1), min(255, N - 1)], g.integers(0, N, n_random)])
    ms, ns = np.meshgrid(np.unique(ms), np.unique(ns), indexing="ij")
    ms, ns = ms.ravel(), ns.ravel()
    rows = np.unique(ms)
    xb = dev_to_bits(x[torch.from_numpy(rows).to(dev)])
    xq, xs = oracle.act_quant(xb, ue)
    assert np.array_equal(dev_to_bits(a[torch.from_numpy(rows).to(dev)]), xq)
    blocks = np.unique(ns // 128)
    wq_parts, ws_parts = [], []
    for b in blocks:
        qo, so = oracle.weight_quant(w[b * 128:(b + 1) * 128].cpu().numpy(), ue)
        assert np.array_equal(dev_to_bits(q[b * 128:(b + 1) * 128]), qo)
        wq_parts.append(np.pad(qo, ((0, 128 - qo.shape[0]), (0, 0))))
        ws_parts.append(so)
    wq = np.concatenate(wq_parts)
    wsc = np.concatenate(ws_parts)
    row_of = {r: i for i, r in enumerate(rows)}
    blk_of = {b: i for i, b in enumerate(blocks)}
    mi = np.array([row_of[m] for m in ms])
    ni = np.array([blk_of[n // 128] * 128 + n % 128 for n in ns])
    ref = oracle.gemm_points(xq, xs, wq, wsc, mi, ni)
    got = dev_to_bits(c)[ms, ns]
    # rms of the whole output, estimated from the oracle's sampled values (it only sets the absolute floor)
    rms = float(np.sqrt(np.mean(ref ** 2)))
    assert_gemm_close(got, ref, rms=rms, what=f"sampled {M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K", [(4096, 18432, 7168), (4096, 7168, 18432), (2048, 1536, 7168),
                                   (2048, 576, 7168), (2048, 24576, 1536), (2048, 32768, 512),
                                   (64, 24576, 1536), (64, 32768, 512), (64, 576, 7168), (100, 10944, 2048)])
def test_gemm_full_size_sampled(M, N, K):
    sampled_check(M, N, K, 4000 + M % 97 + N % 89, frac=0.01)


@pytest.mark.parametrize("mma", [True, False])
@pytest.mark.parametrize("M,N,K", [(1300, 7000, 640), (4096, 18432, 7168), (4096, 7168, 18432)])
def test_gemm_ue8m0_tensor_core_scaling_sampled(M, N, K, mma):
    """Power-of-two scales on 128 x 256 tiles: the tensor core applies the
    UE8M0 scales itself (block-scaled MMA, one accumulator over the whole K
    range). 1300 x 7000 x 640: cluster pairs, a ragged row tile, a partial
    weight block, stream-K parts, 5 K blocks (a scale group of 4 and one of
    1); 7168 and 18432: 14 and 36 scale groups through the 8-slot ring.
    mma False: the same problems through the per-block promotion (the
    FP8BLK_SCALE_PROMOTE flag of the call)."""
    fmt = fb.SCALE_UE8M0 if mma else fb.SCALE_UE8M0 | fb.SCALE_PROMOTE
    sampled_check(M, N, K, 5000 + M % 97 + N % 89, frac=0.01, fmt=fmt)
    assert fb.last_device_error() == 0


def test_gemm_ue8m0_flags_scales_that_are_not_powers_of_two():
    """Under UE8M0 the tensor core takes only the exponent of each scale: fp32
    weight scales that are not powers of two set the device error bit 1 << 7."""
    dev = torch.device("cuda")
    a, a_s = fb.act_quant(synthetic.device_activations(1300, 640, 91, dev), fb.SCALE_UE8M0)
    q, s = fb.weight_quant(synthetic.device_normal((7000, 640), 92, 0.02, dev))
    assert fb.last_device_error() == 0
    fb.fp8_gemm(a, a_s, q, s, scale_fmt=fb.SCALE_UE8M0)
    assert fb.last_device_error() & (1 << 7)
    assert fb.last_device_error() == 0


def test_linear_chain_reads_the_previous_output():
    """Two dense linears back to back on one stream, the second reading the
    first's output (M > 128: the first stores through TMA boxes; the second's
    act_quant may launch early and reads x after its dependency wait), over
    reused buffers, against the same calls with a synchronisation between
    them: the first kernel's stores are in memory when it completes."""
    dev = torch.device("cuda")
    M, D, H = 300, 512, 1024
    q1, s1 = fb.weight_quant(synthetic.device_normal((H, D), 71, 0.02, dev))
    q2, s2 = fb.weight_quant(synthetic.device_normal((D, H), 72, 0.02, dev))
    xs = [synthetic.device_activations(M, D, 73 + r, dev) for r in range(3)]
    mid = torch.empty((M, H), dtype=torch.bfloat16, device=dev)
    outs = [torch.empty((M, D), dtype=torch.bfloat16, device=dev) for _ in xs]
    ws1 = fb.workspace(fb.linear_workspace_bytes(M, H, D), dev, "chain1")
    ws2 = fb.workspace(fb.linear_workspace_bytes(M, D, H), dev, "chain2")
    for x, o in zip(xs, outs):
        fb.linear(x, q1, s1, out=mid, ws=ws1)
        fb.linear(mid, q2, s2, out=o, ws=ws2)
    torch.cuda.synchronize()
    for x, o in zip(xs, outs):
        m = fb.linear(x, q1, s1)
        torch.cuda.synchronize()
        ref = fb.linear(m, q2, s2)
        torch.cuda.synchronize()
        assert torch.equal(o.view(torch.int16), ref.view(torch.int16))
    assert fb.last_device_error() == 0


def test_linear_matches_quant_then_gemm():
    x, w, xq, xs, wq, ws = host_problem(8, 10944, 2048, 21, 0.01)
    xd = bits_to_dev_bf16(x)
    q, s = fb.weight_quant(torch.from_numpy(w).cuda())
    y = fb.linear(xd, q, s)
    a, a_s = fb.act_quant(xd)
    c = fb.fp8_gemm(a, a_s, q, s)
    assert torch.equal(y.view(torch.int16), c.view(torch.int16))
    assert_gemm_close(dev_to_bits(y), oracle.gemm(xq, xs, wq, ws))


def test_linear_kernel_count():
    """fp8blk_linear_kernels names the launches of fp8blk_linear: act_quant
    fused into the GEMM (1) only for M <= 2 where the decode GEMM does not
    take the shape."""
    assert fb.linear_kernels(1, 10944, 2048) == 2    # act_quant + the slice-per-SM decode GEMM
    assert fb.linear_kernels(8, 10944, 2048) == 2
    assert fb.linear_kernels(2, 10944, 7168) == 1    # slices too large: the fused kernel
    assert fb.linear_kernels(64, 10944, 2048) == 2
    assert fb.linear_kernels(3, 0, 2048) == 0
    with pytest.raises(fb.Fp8BlkError):
        fb.linear_kernels(1, 10, 100)


@pytest.mark.parametrize("M", [1, 8, 64])
@pytest.mark.parametrize("pinned", [True, False])
def test_linear_host_buffers(M, pinned):
    """Host x and y: pinned buffers are read and written in place by the
    kernels, pageable ones go through staging copies; both give the device
    layer's bits."""
    x, w, xq, xs, wq, ws = host_problem(M, 10944, 2048, 22, 0.01)
    q, s = fb.weight_quant(torch.from_numpy(w).cuda())
    xh = torch.from_numpy(x.view(np.int16).copy()).view(torch.bfloat16)
    yh = torch.empty((M, 10944), dtype=torch.bfloat16)
    if pinned:
        xh, yh = xh.pin_memory(), yh.pin_memory()
    fb.linear_host(xh, q, s, yh)
    torch.cuda.current_stream().synchronize()
    y = fb.linear(bits_to_dev_bf16(x), q, s)
    assert torch.equal(yh.view(torch.int16), y.cpu().view(torch.int16))


# ---- decode linear with act_quant fused into the GEMM (M <= 32) ----------------

@pytest.mark.parametrize("M,N,K", [(1, 10944, 2048), (2, 320, 256), (1, 1000, 7168), (2, 576, 9984),
                                   (2, 32768, 512), (1, 129, 4096), (8, 10944, 2048), (32, 4096, 1024),
                                   (2, 11000, 384), (1, 7300, 512), (2, 10944, 7168)])
@pytest.mark.parametrize("fmt", [fb.SCALE_FP32, fb.SCALE_UE8M0])
def test_fused_decode_linear(M, N, K, fmt):
    """fp8blk_linear (for M <= 2 act_quant runs inside the GEMM kernel: weight
    slices of 48..80 rows where N allows, else whole 128-row tiles with 8
    weight stages up to K = 5888 and 4 beyond): same bits as act_quant +
    fp8_gemm on the same kind of schedule (each output element summed over K
    in order by one CTA, N <= 128 * SMs), and within the GEMM tolerance of the
    oracle."""
    ue = (fmt & ~fb.SCALE_PROMOTE) == fb.SCALE_UE8M0
    x, w, xq, xs, wq, ws = host_problem(M, N, K, 3000 + M + N, 0.01, ue8m0=ue)
    xd = bits_to_dev_bf16(x)
    q, s = fb.weight_quant(torch.from_numpy(w).cuda(), fmt)
    y = fb.linear(xd, q, s, scale_fmt=fmt)
    a, a_s = fb.act_quant(xd, fmt)
    c = fb.fp8_gemm(a, a_s, q, s, scale_fmt=fmt)
    if -(-N // 128) <= torch.cuda.get_device_properties(0).multi_processor_count:
        assert torch.equal(y.view(torch.int16), c.view(torch.int16))
    assert_gemm_close(dev_to_bits(c), oracle.gemm(xq, xs, wq, ws), what=f"act_quant + fp8_gemm {M}x{N}x{K}")
    assert_gemm_close(dev_to_bits(y), oracle.gemm(xq, xs, wq, ws), what=f"fused linear {M}x{N}x{K}")
    assert fb.last_device_error() == 0
