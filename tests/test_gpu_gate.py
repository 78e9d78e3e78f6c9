"""GPU parity of the MoE gate against the CPU oracle.

The expert ids are integers decided by floating-point comparisons. The kernel
takes those decisions in fp32 with CUDA's expf (within 2 ulp); the oracle
computes the scores in fp64 and rounds them to fp32 once. The two therefore
agree on every token except at near-ties, where two experts' keys differ by
a few fp32 ulps. Such tokens are checked for validity instead: position by
position, the keys of the kernel's experts must equal the oracle's within
1e-5 (the fp32 rounding of the scores), and with group-limited routing every
chosen expert must come from a kept group (the best topk_groups groups, up to
a tie at the cut within fp32 noise). Such tokens must also be rare. Weights are
compared wherever the ids agree: within 4e-6 relative for sigmoid scores (a
few roundings of fp32 operations), and within 2e-5 for softmax scores, whose
fp32 sum over the E experts carries up to E roundings."""
import numpy as np
import pytest
import torch
from scipy.special import expit, softmax

import fp8_block_scaled_quant_gb300 as fb
import oracle
import synthetic

pytestmark = pytest.mark.gpu

# (T, E, groups, kept groups, k, sigmoid, bias, route_scale, normalize): the
# 671B / V3.1 gate, the 236B gate, the 16B gate (section 3.3 of the guide),
# and edge variants.
CASES = [
    (4096, 256, 8, 4, 8, True, True, 2.5, True),
    (1000, 160, 8, 3, 6, False, False, 16.0, True),
    (777, 64, 1, 1, 6, False, False, 1.0, False),
    (33, 256, 8, 4, 8, True, False, 2.5, True),
    (65, 256, 8, 4, 8, True, True, 1.0, False),
    (9, 32, 32, 5, 5, True, False, 1.0, True),
    (17, 96, 4, 4, 32, False, True, 1.0, True),
]


def keys(l, b, sigmoid):
    l64 = l.astype(np.float64)
    s = (expit(l64) if sigmoid else softmax(l64, axis=1)).astype(np.float32)
    return s + b if b is not None else s


def group_scores(z, G, bias):
    """[T, G]: a group's largest key (no bias) or the sum of its two largest (bias)."""
    T, E = z.shape
    zg = np.sort(z.reshape(T, G, E // G).astype(np.float64), axis=2)
    return zg[:, :, -2:].sum(axis=2) if bias else zg[:, :, -1]


@pytest.mark.parametrize("T,E,G,TG,k,sigmoid,use_bias,scale,norm", CASES)
def test_gate_matches_oracle(T, E, G, TG, k, sigmoid, use_bias, scale, norm):
    l = synthetic.gate_logits(T, E, synthetic.SEED_GATE + E)
    b = synthetic.gate_bias(E, synthetic.SEED_GATE) if use_bias else None
    want_idx, want_w = oracle.moe_gate(l, b, G, TG, k, sigmoid, scale, norm)
    dev = torch.device("cuda")
    idx, w = fb.moe_gate(torch.from_numpy(l).to(dev), None if b is None else torch.from_numpy(b).to(dev), G, TG, k,
                         fb.SCORE_SIGMOID if sigmoid else fb.SCORE_SOFTMAX, scale, norm)
    torch.cuda.synchronize()
    idx, w = idx.cpu().numpy(), w.cpu().numpy()
    same = np.all(idx == want_idx, axis=1)
    z = keys(l, b, sigmoid)
    gs = group_scores(z, G, b is not None) if G > 1 else None
    for t in np.nonzero(~same)[0]:
        got_z = z[t, idx[t].astype(np.int64)]
        ref_z = z[t, want_idx[t].astype(np.int64)]
        assert len(set(idx[t].tolist())) == k
        assert np.allclose(got_z, ref_z, rtol=0, atol=1e-5), f"token {t}: {idx[t]} vs {want_idx[t]}"
        if gs is not None:
            # every chosen expert lies in a kept group: one of the TG best groups
            # (the oracle's own, or one whose score ties the cut within fp32 noise)
            kept = set(np.argsort(-gs[t], kind="stable")[:TG].tolist())
            cut = np.sort(gs[t])[::-1][TG - 1]
            for e in idx[t]:
                g = int(e) // (E // G)
                assert g in kept or gs[t, g] >= cut - 2e-5, f"token {t}: expert {e} from a dropped group"
    assert (~same).sum() <= max(1, T // 500)
    assert np.allclose(w[same], want_w[same], rtol=4e-6 if sigmoid else 2e-5, atol=0)
    assert fb.last_device_error() == 0


@pytest.mark.parametrize("T,E,G,TG,k,sigmoid,use_bias,scale,norm", CASES + [(4097, 256, 8, 4, 8, True, True, 2.5, True),
                                                                      (1, 64, 1, 1, 6, False, False, 1.0, True)])
def test_route_is_gate_then_permute(T, E, G, TG, k, sigmoid, use_bias, scale, norm):
    """fp8blk_moe_route (the gate kernel also ranks the pairs and builds the
    bases) gives exactly fp8blk_moe_gate's ids and weights, and exactly the
    oracle's permutation of those ids (an integer stable sort: bit-exact)."""
    l = synthetic.gate_logits(T, E, synthetic.SEED_GATE + E + 1)
    b = synthetic.gate_bias(E, synthetic.SEED_GATE + 1) if use_bias else None
    dev = torch.device("cuda")
    ld = torch.from_numpy(l).to(dev)
    bd = None if b is None else torch.from_numpy(b).to(dev)
    sf = fb.SCORE_SIGMOID if sigmoid else fb.SCORE_SOFTMAX
    gi, gw = fb.moe_gate(ld, bd, G, TG, k, sf, scale, norm)
    for _ in range(2):   # twice: the workspace's arrival counter is left at zero
        idx, w, counts, offsets, perm = fb.moe_route(ld, bd, G, TG, k, sf, scale, norm)
        torch.cuda.synchronize()
        assert torch.equal(idx, gi) and torch.equal(w.view(torch.int32), gw.view(torch.int32))
        co, oo, po = oracle.moe_permute(idx.cpu().numpy(), E)
        assert np.array_equal(counts.cpu().numpy(), co)
        assert np.array_equal(offsets.cpu().numpy(), oo)
        assert np.array_equal(perm.cpu().numpy(), po)
    assert fb.last_device_error() == 0


def test_route_no_tokens():
    dev = torch.device("cuda")
    l = torch.zeros((0, 256), dtype=torch.float32, device=dev)
    idx, w, counts, offsets, perm = fb.moe_route(l, None, 8, 4, 8)
    torch.cuda.synchronize()
    assert int(counts.abs().sum()) == 0 and int(offsets.abs().sum()) == 0


def test_gate_feeds_the_permutation():
    """Gate output straight into the routing permutation: the per-expert
    counts are the bincount of the gate's ids."""
    T, E = 512, 256
    dev = torch.device("cuda")
    l = torch.from_numpy(synthetic.gate_logits(T, E, 21)).to(dev)
    b = torch.from_numpy(synthetic.gate_bias(E, 21)).to(dev)
    idx, w = fb.moe_gate(l, b, 8, 4, 8, fb.SCORE_SIGMOID, 2.5, True)
    counts, offsets, perm = fb.moe_permute(idx, E)
    torch.cuda.synchronize()
    assert np.array_equal(counts.cpu().numpy(), np.bincount(idx.cpu().numpy().ravel(), minlength=E))
    assert int(offsets[-1]) == T * 8


def test_gate_argument_errors():
    L = fb.lib()
    dev = torch.device("cuda")
    l = torch.zeros((4, 256), dtype=torch.float32, device=dev)
    idx = torch.empty((4, 8), dtype=torch.int32, device=dev)
    w = torch.empty((4, 8), dtype=torch.float32, device=dev)
    p = lambda t: t.data_ptr()
    f = fb._set_types("fp8blk_moe_gate", [fb.ctypes.c_void_p] * 2 + [fb.ctypes.c_int64] * 5 +
                      [fb.ctypes.c_int, fb.ctypes.c_float, fb.ctypes.c_int] + [fb.ctypes.c_void_p] * 3)
    assert f(p(l), None, 4, 256, 8, 4, 8, 2, 1.0, 1, p(idx), p(w), None) == 8        # bad score_func
    assert f(p(l), None, 4, 200, 8, 4, 8, 1, 1.0, 1, p(idx), p(w), None) == 2        # E % 32
    assert f(p(l), None, 4, 256, 3, 2, 8, 1, 1.0, 1, p(idx), p(w), None) == 2        # groups must divide 32
    assert f(p(l), None, 4, 256, 8, 1, 33, 1, 1.0, 1, p(idx), p(w), None) == 2       # topk > one group of 32
    assert f(p(l), None, 4, 256, 8, 4, 8, 1, float("inf"), 1, p(idx), p(w), None) == 8
    assert f(None, None, 4, 256, 8, 4, 8, 1, 1.0, 1, p(idx), p(w), None) == 1
    assert f(None, None, 0, 256, 8, 4, 8, 1, 1.0, 1, None, None, None) == 0          # T == 0: nothing to do
    torch.cuda.synchronize()
    del L
