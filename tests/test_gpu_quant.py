"""GPU parity of act_quant, weight_quant and weight_dequant against the CPU
oracle: bit-exact codes, scales and bf16 outputs, through the C ABI."""
import numpy as np
import pytest
import torch

import fp8_block_scaled_quant_gb300 as fb
import oracle
import synthetic
from helpers import bits_to_dev_bf16, dev_to_bits

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("M,K,frac", [(1, 128, 0.0), (16, 256, 0.0), (8, 2048, 0.01), (64, 2048, 0.01),
                                      (3, 7168, 0.0), (257, 384, 0.05), (4096, 7168, 0.0), (33, 18432, 0.01)])
@pytest.mark.parametrize("fmt", [fb.SCALE_FP32, fb.SCALE_UE8M0])
def test_act_quant_bit_exact(M, K, frac, fmt):
    x = synthetic.activations(M, K, 100 + M + K, outlier_frac=frac)
    q, s = fb.act_quant(bits_to_dev_bf16(x), fmt)
    torch.cuda.synchronize()
    qo, so = oracle.act_quant(x, fmt == fb.SCALE_UE8M0)
    assert np.array_equal(dev_to_bits(q), qo)
    assert np.array_equal(s.cpu().numpy().view(np.uint32), so.view(np.uint32))


def test_act_quant_special_blocks():
    """All-zero blocks, negative zeros, tiny values (clamp), subnormal
    results, one huge element per block, ties of the e4m3 rounding."""
    M, K = 6, 512
    x = synthetic.activations(M, K, 7)
    x[0, :128] = 0
    x[0, 128:256] = 0x8000                                    # -0.0
    x[1, :128] = synthetic.to_bf16_bits(np.full(128, 1e-6, np.float32))   # amax < 1e-4
    x[2, 5] = synthetic.to_bf16_bits(np.array([3e4], np.float32))[0]      # tiny rest -> subnormal codes
    tie = np.float32(448.0) * np.array([1.0, 0.5, 272 / 448, 304 / 448, 0.0, -1.0] * 22, np.float32)[:128]
    x[3, :128] = synthetic.to_bf16_bits(tie)
    x[4] = synthetic.to_bf16_bits(-np.abs(synthetic.bf16_bits_to_f32(x[4])))
    for fmt in (fb.SCALE_FP32, fb.SCALE_UE8M0):
        q, s = fb.act_quant(bits_to_dev_bf16(x), fmt)
        qo, so = oracle.act_quant(x, fmt == fb.SCALE_UE8M0)
        assert np.array_equal(dev_to_bits(q), qo)
        assert np.array_equal(s.cpu().numpy().view(np.uint32), so.view(np.uint32))


def test_act_quant_all_bf16_values():
    """Every finite bf16 bit pattern passes through the kernel once (as
    2^16 / 128 blocks): the encoder and the scale rule agree with the oracle
    over the whole input range."""
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    v = synthetic.bf16_bits_to_f32(bits)
    bits = bits[np.isfinite(v)]
    bits = bits[: (bits.size // 128) * 128].reshape(-1, 128)
    g = np.random.Generator(np.random.PCG64(3))
    for fmt in (fb.SCALE_FP32, fb.SCALE_UE8M0):
        for perm in (False, True):
            x = g.permutation(bits.ravel()).reshape(bits.shape) if perm else bits
            q, s = fb.act_quant(bits_to_dev_bf16(np.ascontiguousarray(x)), fmt)
            qo, so = oracle.act_quant(x, fmt == fb.SCALE_UE8M0)
            assert np.array_equal(dev_to_bits(q), qo)
            assert np.array_equal(s.cpu().numpy().view(np.uint32), so.view(np.uint32))


def test_act_quant_errors():
    x = torch.zeros((4, 100), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(fb.Fp8BlkError):
        fb.act_quant(x)
    L = fb.lib()
    x = torch.zeros((4, 128), dtype=torch.bfloat16, device="cuda")
    q = torch.empty((4, 128), dtype=torch.uint8, device="cuda")
    s = torch.empty((4, 1), dtype=torch.float32, device="cuda")
    assert L.fp8blk_act_quant(x.data_ptr(), 4, 100, q.data_ptr(), s.data_ptr(), 0, None) == 2
    assert L.fp8blk_act_quant(None, 4, 128, q.data_ptr(), s.data_ptr(), 0, None) == 1
    assert L.fp8blk_act_quant(x.data_ptr() + 2, 4, 128, q.data_ptr(), s.data_ptr(), 0, None) == 3
    assert L.fp8blk_act_quant(x.data_ptr(), 4, 128, q.data_ptr(), s.data_ptr(), 7, None) == 8
    assert L.fp8blk_act_quant(x.data_ptr(), 0, 128, None, None, 0, None) == 0


@pytest.mark.parametrize("N,K", [(320, 256), (576, 7168), (130, 200), (1, 1), (128, 128), (1000, 4000)])
@pytest.mark.parametrize("fmt", [fb.SCALE_FP32, fb.SCALE_UE8M0])
def test_weight_quant_bit_exact(N, K, fmt):
    w = synthetic.weights(N, K, 200 + N + K)
    q, s = fb.weight_quant(torch.from_numpy(w).cuda(), fmt)
    qo, so = oracle.weight_quant(w, fmt == fb.SCALE_UE8M0)
    assert np.array_equal(dev_to_bits(q), qo)
    assert np.array_equal(s.cpu().numpy().view(np.uint32), so.view(np.uint32))


@pytest.mark.parametrize("N,K", [(320, 256), (576, 7168), (130, 200), (1, 1), (129, 16), (1000, 4000),
                                 (18432, 7168)])
def test_weight_dequant_bit_exact(N, K):
    if N * K > 10_000_000:
        w = synthetic.device_normal((N, K), 9, 0.02, "cuda")
        q, s = fb.weight_quant(w)
        out = fb.weight_dequant(q, s)
        # the oracle quantises the same fp32 weight itself; check codes, then a
        # band of whole rows (edges included) of the dequantised output
        rows = np.r_[0:256, 9000:9128, N - 200:N]
        wh = w[torch.from_numpy(rows).cuda()].cpu().numpy()
        blocks = np.unique(rows // 128)
        for b in blocks:
            r0 = b * 128
            qo, so = oracle.weight_quant(w[r0:r0 + 128].cpu().numpy())
            assert np.array_equal(dev_to_bits(q[r0:r0 + 128]), qo)
            assert np.array_equal(s[b].cpu().numpy().view(np.uint32), so[0].view(np.uint32))
            got = dev_to_bits(out[r0:r0 + 128])
            assert np.array_equal(got, oracle.weight_dequant(qo, so))
        del wh
        return
    w = synthetic.weights(N, K, 300 + N + K)
    qo, so = oracle.weight_quant(w)
    q = torch.from_numpy(qo).cuda().view(torch.float8_e4m3fn)
    out = fb.weight_dequant(q, torch.from_numpy(so).cuda())
    assert np.array_equal(dev_to_bits(out), oracle.weight_dequant(qo, so))


def test_weight_dequant_scalar_path_unaligned():
    """An output offset by one element takes the scalar kernel; same bits."""
    N, K = 130, 256
    w = synthetic.weights(N, K, 11)
    qo, so = oracle.weight_quant(w)
    q = torch.from_numpy(qo).cuda().view(torch.float8_e4m3fn)
    big = torch.empty(N * K + 8, dtype=torch.bfloat16, device="cuda")
    out = big[1:1 + N * K].view(N, K)
    fb.weight_dequant(q, torch.from_numpy(so).cuda(), out=out)
    assert np.array_equal(dev_to_bits(out), oracle.weight_dequant(qo, so))


def test_weight_dequant_every_code_and_scale():
    """All 256 codes (NaN codes excluded by the oracle's decode compare) times
    a spread of scales, including ones that round in bf16."""
    codes = np.arange(256, dtype=np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0
    q = np.tile(codes, (128 * 4, 1))[:, :256]
    s = np.array([[1.0, 3.0e-3], [0.1234567, 2.0 ** -20], [7.77e3, 1e-30], [1.5, 0.3]], np.float32)
    qd = torch.from_numpy(q).cuda().view(torch.float8_e4m3fn)
    out = fb.weight_dequant(qd, torch.from_numpy(s).cuda())
    assert np.array_equal(dev_to_bits(out), oracle.weight_dequant(q, s))
