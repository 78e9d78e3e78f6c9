"""GPU parity of the MLA absorb projections against the CPU oracle.

Both sides use the dequantised weight bf16(fp32(code) * scale) and bf16
activations. The oracle rounds the exact (fp64) sum to bf16; the kernel rounds
its fp32 sum to bf16. Where the two sums straddle a rounding boundary the
results differ by one bf16 step, which is at most 2^-7 |ref| (the step of a
value in [2^e, 2^(e+1)) is 2^(e-7)). Tolerance per element: 2^-7 |ref| plus
1e-3 of the output's rms for sums that cancel."""
import numpy as np
import pytest
import torch

import fp8_block_scaled_quant_gb300 as fb
import oracle
import synthetic
from helpers import bits_to_dev_bf16, dev_to_bits

pytestmark = pytest.mark.gpu
DN = DV = 128


def close(got_bits, ref_bits, rms=None, what=""):
    got = synthetic.bf16_bits_to_f32(got_bits).astype(np.float64)
    ref = synthetic.bf16_bits_to_f32(ref_bits).astype(np.float64)
    if rms is None:
        rms = float(np.sqrt(np.mean(ref ** 2)))
    bad = np.abs(got - ref) > 2.0 ** -7 * np.abs(ref) + 1e-3 * rms
    assert not bad.any(), f"{what}: {bad.sum()} of {bad.size} outside, e.g. {got[bad][:4]} vs {ref[bad][:4]}"


def weights(H, C, seed):
    return oracle.weight_quant(synthetic.weights(H * (DN + DV), C, seed))


def dev_w(wq, ws):
    return torch.from_numpy(wq).cuda().view(torch.float8_e4m3fn), torch.from_numpy(ws).cuda()


# (20, 320, 128) and (33, 160, 256): 320 tiles, more than one per SM, so
# persistent CTAs cycle both accumulator buffers and the operand ring.
@pytest.mark.parametrize("T,H,C", [(5, 3, 256), (130, 2, 512), (1, 4, 512), (257, 1, 128), (20, 320, 128),
                                   (33, 160, 256)])
@pytest.mark.parametrize("mode", ["qk", "v"])
def test_mla_full_compare(T, H, C, mode):
    wq, ws = weights(H, C, 300 + T + H)
    width = DN if mode == "qk" else C
    a = synthetic.activations(T, H * width, 301 + T)
    out = fb.mla_absorb(bits_to_dev_bf16(a).view(T, H, width), *dev_w(wq, ws), mode)
    ref = oracle.mla_absorb(a, wq, ws, H, DN, DV, mode)
    close(dev_to_bits(out), ref, what=f"mla {mode} T={T} H={H} C={C}")
    assert fb.last_device_error() == 0


@pytest.mark.parametrize("T", [64, 2048])
@pytest.mark.parametrize("mode", ["qk", "v"])
def test_mla_full_size_sampled(T, mode):
    """128 heads, kv_lora 512 (the 671B MLA); the oracle recomputes sampled
    tokens of sampled heads (a sub-problem with only those heads' weights)."""
    H, C = 128, 512
    wq, ws = weights(H, C, 400 + T)
    width = DN if mode == "qk" else C
    a = synthetic.activations(T, H * width, 401 + T)
    out = dev_to_bits(fb.mla_absorb(bits_to_dev_bf16(a).view(T, H, width), *dev_w(wq, ws), mode))
    tokens = np.array(sorted({0, 1, T // 2, T - 1}))
    heads = np.array([0, 63, 127])
    rows = np.concatenate([np.arange(h * (DN + DV), (h + 1) * (DN + DV)) for h in heads])
    srows = np.concatenate([np.arange(2 * h, 2 * h + 2) for h in heads])
    sub = a.reshape(T, H, width)[tokens][:, heads].reshape(len(tokens), -1)
    ref = oracle.mla_absorb(sub, wq[rows], ws[srows], len(heads), DN, DV, mode)
    got = out[tokens][:, heads]
    # rms of the whole output, estimated from the oracle's sampled rows
    rms = float(np.sqrt(np.mean(synthetic.bf16_bits_to_f32(ref).astype(np.float64) ** 2)))
    close(got, ref, rms=rms, what=f"mla {mode} sampled T={T}")
    assert fb.last_device_error() == 0


def test_mla_chain_reads_the_previous_kernels_output():
    """qk then v on its output, back to back on one stream: the v kernel may
    start while qk still runs (it loads wkv_b early) but must read qk's
    output only once qk has completed, and qk may overwrite its output only
    after the v launch before it has read it. Checked against the same calls
    with a synchronisation between them, over several rounds that reuse the
    buffers."""
    T, H, C = 300, 128, 512
    wq, ws = weights(H, C, 500)
    w, s = dev_w(wq, ws)
    qs = [bits_to_dev_bf16(synthetic.activations(T, H * DN, 501 + r)).view(T, H, DN) for r in range(3)]
    mid = torch.empty((T, H, C), dtype=torch.bfloat16, device="cuda")
    outs = [torch.empty((T, H, DV), dtype=torch.bfloat16, device="cuda") for _ in qs]
    for q, o in zip(qs, outs):
        fb.mla_absorb(q, w, s, "qk", out=mid)
        fb.mla_absorb(mid, w, s, "v", out=o)
    torch.cuda.synchronize()
    for q, o in zip(qs, outs):
        m = fb.mla_absorb(q, w, s, "qk")
        torch.cuda.synchronize()
        ref = fb.mla_absorb(m, w, s, "v")
        torch.cuda.synchronize()
        assert torch.equal(o.view(torch.int16), ref.view(torch.int16))
    assert fb.last_device_error() == 0


@pytest.mark.parametrize("mode", ["qk", "v"])
def test_mla_many_tiles_per_cta_match_one_tile_per_cta(mode):
    """The 128-head layer at 300 tokens gives each persistent CTA about ten
    tiles, some of whose 32-row quarters lie wholly past T (the last token
    tile holds 44 rows), so each epilogue warp alternates tiles it stores
    and tiles it skips while reusing its staging slab. The same heads run 8
    at a time (one tile per CTA) must give the same bits."""
    T, H, C = 300, 128, 512
    wq, ws = weights(H, C, 600)
    w, s = dev_w(wq, ws)
    width = DN if mode == "qk" else C
    x = bits_to_dev_bf16(synthetic.activations(T, H * width, 601)).view(T, H, width)
    full = fb.mla_absorb(x, w, s, mode)
    for h0 in range(0, H, 8):
        part = fb.mla_absorb(x[:, h0:h0 + 8].contiguous(), w[h0 * (DN + DV):(h0 + 8) * (DN + DV)],
                             s[2 * h0:2 * (h0 + 8)], mode)
        assert torch.equal(part.view(torch.int16), full[:, h0:h0 + 8].view(torch.int16)), f"heads {h0}..{h0 + 7}"
    assert fb.last_device_error() == 0


def test_mla_argument_errors():
    L = fb.lib()
    x = torch.zeros((4, 2, 128), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros((512, 256), dtype=torch.float8_e4m3fn, device="cuda")
    s = torch.ones((4, 2), dtype=torch.float32, device="cuda")
    y = torch.zeros((4, 2, 256), dtype=torch.bfloat16, device="cuda")
    p = lambda t: t.data_ptr()
    assert L.fp8blk_mla_absorb_qk(p(x), p(w), p(s), p(y), 4, 2, 64, 128, 256, None) == 2     # dn != 128
    assert L.fp8blk_mla_absorb_qk(p(x), p(w), p(s), p(y), 4, 2, 128, 128, 200, None) == 2    # C % 128
    assert L.fp8blk_mla_absorb_qk(None, p(w), p(s), p(y), 4, 2, 128, 128, 256, None) == 1
    assert L.fp8blk_mla_absorb_qk(p(x) + 2, p(w), p(s), p(y), 4, 2, 128, 128, 256, None) == 3
    assert L.fp8blk_mla_absorb_v(None, None, None, None, 0, 2, 128, 128, 256, None) == 0     # T == 0
