"""Pins for the oracle's block-scaled GEMM, SwiGLU chain and MoE routing.

GEMM ("Administrator & Developer Guide", 8.5.3 fp8_gemm_kernel): pinned by
(a) the dequantise-then-matmul formulation of the same product (the guide's
6.3 "bf16" path: weight_dequant then a plain linear), computed with numpy's
fp64 matmul on independently dequantised operands; (b) an exact integer closed
form; (c) the zero-padding rule; (d) scale linearity. MoE (6.4 MoE expert
routing): the permutation against numpy's bincount / stable argsort, and the
token output against per-expert slices taken with numpy."""
import numpy as np
import pytest
import torch

import oracle
import synthetic


def dequant_rows(q, s_rows):
    """fp64 dequantised activation: decode(q[m, k]) * s[m, k // 128]."""
    return oracle.e4m3_decode_array(q) * np.repeat(s_rows.astype(np.float64), 128, axis=1)


def dequant_blocks(q, s):
    N, K = q.shape
    sv = np.repeat(np.repeat(s.astype(np.float64), 128, 0), 128, 1)[:N, :K]
    return oracle.e4m3_decode_array(q) * sv


def make_problem(M, N, K, seed, ue8m0=False):
    x = synthetic.activations(M, K, seed)
    w = synthetic.weights(N, K, seed + 100)
    qa, a_s = oracle.act_quant(x, ue8m0)
    qw, w_s = oracle.weight_quant(w, ue8m0)
    return qa, a_s, qw, w_s


@pytest.mark.parametrize("M,N,K", [(1, 1, 128), (3, 5, 256), (8, 8, 128), (7, 130, 384), (16, 320, 256)])
@pytest.mark.parametrize("ue8m0", [False, True])
def test_gemm_matches_dequantised_matmul(M, N, K, ue8m0):
    qa, a_s, qw, w_s = make_problem(M, N, K, 40 + M + N, ue8m0)
    ref = oracle.gemm(qa, a_s, qw, w_s)
    alt = dequant_rows(qa, a_s) @ dequant_blocks(qw, w_s).T
    assert np.allclose(ref, alt, rtol=1e-12, atol=1e-12 * np.abs(alt).max())


def test_gemm_brute_force_triple_loop():
    qa, a_s, qw, w_s = make_problem(2, 3, 256, 50)
    A = dequant_rows(qa, a_s)
    W = dequant_blocks(qw, w_s)
    ref = oracle.gemm(qa, a_s, qw, w_s)
    for m in range(2):
        for n in range(3):
            acc = 0.0
            for k in range(256):
                acc += A[m, k] * W[n, k]
            assert abs(acc - ref[m, n]) <= 1e-12 * max(1.0, abs(acc))


def test_gemm_integer_closed_form():
    """Unit scales and small-integer codes give an exact integer product."""
    g = np.random.Generator(np.random.PCG64(51))
    vals = np.array([-2.0, -1.0, 0.0, 1.0, 2.0], np.float32)
    codes = oracle.e4m3_encode_array(vals)
    ia = g.integers(0, 5, (6, 384))
    iw = g.integers(0, 5, (9, 384))
    qa, qw = codes[ia], codes[iw]
    ref = oracle.gemm(qa, np.ones((6, 3), np.float32), qw, np.ones((1, 3), np.float32))
    exact = vals[ia].astype(np.int64) @ vals[iw].astype(np.int64).T
    assert np.array_equal(ref, exact.astype(np.float64))


def test_gemm_padded_edge_contributes_nothing():
    qa, a_s, qw, w_s = make_problem(4, 320, 256, 52)
    ref = oracle.gemm(qa, a_s, qw, w_s)
    qwp = np.zeros((384, 256), np.uint8)
    qwp[:320] = qw
    refp = oracle.gemm(qa, a_s, qwp, w_s)
    assert np.array_equal(refp[:, :320], ref)
    assert np.all(refp[:, 320:] == 0)


def test_gemm_scale_linearity():
    """Doubling one weight block's scale adds exactly that block's
    contribution again, and leaves columns of other blocks unchanged."""
    qa, a_s, qw, w_s = make_problem(5, 256, 384, 53)
    ref = oracle.gemm(qa, a_s, qw, w_s)
    w2 = w_s.copy()
    w2[1, 2] *= 2
    ref2 = oracle.gemm(qa, a_s, qw, w2)
    only = np.zeros_like(w_s)
    only[1, 2] = w_s[1, 2]
    contrib = oracle.gemm(qa, a_s, qw, only)
    assert np.array_equal(ref2[:, :128], ref[:, :128])
    assert np.allclose(ref2[:, 128:] - ref[:, 128:], contrib[:, 128:], rtol=1e-12, atol=1e-15)
    assert np.all(contrib[:, :128] == 0)


def test_gemm_points_match_full():
    qa, a_s, qw, w_s = make_problem(9, 200, 256, 54)
    ref = oracle.gemm(qa, a_s, qw, w_s)
    ms = np.array([0, 8, 3, 4])
    ns = np.array([199, 0, 128, 127])
    assert np.array_equal(oracle.gemm_points(qa, a_s, qw, w_s, ms, ns), ref[ms, ns])


def test_swiglu_matches_library_ops():
    """bf16(bf16(silu(h1)) * h3), against torch's fp32 silu: the fp64 silu
    of the oracle and torch's fp32 one may differ by one bf16 step in rare
    cases."""
    g = np.random.Generator(np.random.PCG64(55))
    h1 = synthetic.to_bf16_bits(g.standard_normal(50_000).astype(np.float32) * 4)
    h3 = synthetic.to_bf16_bits(g.standard_normal(50_000).astype(np.float32))
    u = oracle.swiglu(h1, h3)
    t1 = torch.from_numpy(synthetic.bf16_bits_to_f32(h1)).to(torch.bfloat16)
    t3 = torch.from_numpy(synthetic.bf16_bits_to_f32(h3)).to(torch.bfloat16)
    ref = (torch.nn.functional.silu(t1) * t3).view(torch.int16).numpy().view(np.uint16)
    same = u == ref
    assert same.mean() > 0.999
    ulps = np.abs(u.astype(np.int32) - ref.astype(np.int32))
    assert ulps.max() <= 1


def test_swiglu_closed_forms():
    one = synthetic.to_bf16_bits(np.array([1.0], np.float32))
    import math
    tiny = float(torch.tensor(-64.0 / (1.0 + math.exp(64.0)), dtype=torch.float64)
                 .to(torch.float32).to(torch.bfloat16).to(torch.float32))
    for v, expect in [(0.0, 0.0), (64.0, 64.0), (-64.0, tiny)]:
        h1 = synthetic.to_bf16_bits(np.array([v], np.float32))
        u = synthetic.bf16_bits_to_f32(oracle.swiglu(h1, one))[0]
        assert u == expect
    # silu(1) = 1/(1+e^-1) = 0.7310585786...; bf16 -> 0.73046875
    h1 = synthetic.to_bf16_bits(np.array([1.0], np.float32))
    assert synthetic.bf16_bits_to_f32(oracle.swiglu(h1, one))[0] == np.float32(0.73046875)


def test_moe_permute_against_library():
    idx, _ = synthetic.moe_routing(300, 16, 4, 56, zipf_s=1.2)
    counts, offsets, perm = oracle.moe_permute(idx, 16)
    assert np.array_equal(counts, np.bincount(idx.ravel(), minlength=16))
    assert offsets[0] == 0 and offsets[-1] == idx.size
    assert np.array_equal(np.diff(offsets), counts)
    assert np.array_equal(perm, np.argsort(idx.ravel(), kind="stable"))
    assert np.array_equal(np.sort(perm), np.arange(idx.size))       # a bijection


def test_moe_permute_rejects_bad_index():
    with pytest.raises(ValueError):
        oracle.moe_permute(np.array([[0, 9]], np.int32), 4)


def _moe_problem(T, E, dim, inter, topk, seed):
    x = synthetic.activations(T, dim, seed)
    xq, xs = oracle.act_quant(x)
    w1 = synthetic.weights(E * inter, dim, seed + 1)
    w3 = synthetic.weights(E * inter, dim, seed + 2)
    w2 = synthetic.weights(E * dim, inter, seed + 3)
    # quantise per expert so that no 128x128 block straddles two experts
    w1q, w1s = oracle.weight_quant(w1)
    w3q, w3s = oracle.weight_quant(w3)
    w2q, w2s = oracle.weight_quant(w2)
    idx, wts = synthetic.moe_routing(T, E, topk, seed + 4)
    return xq, xs, idx, wts, w1q, w1s, w3q, w3s, w2q, w2s


def test_moe_token_matches_per_expert_slices():
    E, dim, inter, topk = 4, 256, 256, 2
    xq, xs, idx, wts, w1q, w1s, w3q, w3s, w2q, w2s = _moe_problem(6, E, dim, inter, topk, 57)
    y = oracle.moe_tokens(xq, xs, idx, wts, w1q, w1s, w3q, w3s, w2q, w2s, range(6))
    bi, bd = inter // 128, dim // 128
    for t in range(6):
        acc = np.zeros(dim)
        for j in range(topk):
            e = idx[t, j]
            o = oracle.ffn_rows(xq[t:t + 1], xs[t:t + 1],
                                w1q[e * inter:(e + 1) * inter], w1s[e * bi:(e + 1) * bi],
                                w3q[e * inter:(e + 1) * inter], w3s[e * bi:(e + 1) * bi],
                                w2q[e * dim:(e + 1) * dim], w2s[e * bd:(e + 1) * bd], [0])[0]
            acc += np.float64(wts[t, j]) * synthetic.bf16_bits_to_f32(oracle.bf16_round(o))
        assert np.array_equal(y[t], oracle.bf16_round(acc))


def test_ffn_chain_against_library_composition():
    """The dense chain against a composition of library ops: numpy fp64 matmul
    of dequantised operands, torch's silu and casts, the oracle act_quant
    (pinned above) for the re-quantisation. Within the GEMM tolerance."""
    dim, inter = 256, 384
    x = synthetic.activations(5, dim, 58)
    xq, xs = oracle.act_quant(x)
    w1q, w1s = oracle.weight_quant(synthetic.weights(inter, dim, 59))
    w3q, w3s = oracle.weight_quant(synthetic.weights(inter, dim, 60))
    w2q, w2s = oracle.weight_quant(synthetic.weights(dim, inter, 61))
    got = oracle.ffn_rows(xq, xs, w1q, w1s, w3q, w3s, w2q, w2s, range(5))
    A = dequant_rows(xq, xs)
    h1 = torch.from_numpy(A @ dequant_blocks(w1q, w1s).T).to(torch.bfloat16)
    h3 = torch.from_numpy(A @ dequant_blocks(w3q, w3s).T).to(torch.bfloat16)
    u = (torch.nn.functional.silu(h1) * h3).view(torch.int16).numpy().view(np.uint16)
    uq, us = oracle.act_quant(u)
    ref = dequant_rows(uq, us) @ dequant_blocks(w2q, w2s).T
    tol = 2.0 ** -7 * np.abs(ref) + 1e-3 * np.sqrt(np.mean(ref ** 2))
    assert np.all(np.abs(got - ref) <= tol)


def test_moe_topk1_unit_weight_is_dense_chain():
    E, dim, inter = 3, 256, 256
    xq, xs, idx, wts, w1q, w1s, w3q, w3s, w2q, w2s = _moe_problem(4, E, dim, inter, 1, 62)
    wts = np.ones_like(wts)
    y = oracle.moe_tokens(xq, xs, idx, wts, w1q, w1s, w3q, w3s, w2q, w2s, range(4))
    bi, bd = inter // 128, dim // 128
    for t in range(4):
        e = idx[t, 0]
        o = oracle.ffn_rows(xq[t:t + 1], xs[t:t + 1],
                            w1q[e * inter:(e + 1) * inter], w1s[e * bi:(e + 1) * bi],
                            w3q[e * inter:(e + 1) * inter], w3s[e * bi:(e + 1) * bi],
                            w2q[e * dim:(e + 1) * dim], w2s[e * bd:(e + 1) * bd], [0])[0]
        assert np.array_equal(y[t], oracle.bf16_round(o))


def test_moe_shared_expert_is_routed_plus_dense():
    """With a shared expert stacked after the E routed ones (Guide 8.4 steps 6
    and 8: z = shared MLP of every token, output y + z), each row equals the
    routed-only row y plus the dense chain z of the shared expert, added as
    two bf16 tensors by torch (fp32 add, one bf16 rounding)."""
    E, dim, inter, topk = 4, 256, 256, 2
    xq, xs, idx, wts, w1q, w1s, w3q, w3s, w2q, w2s = _moe_problem(5, E + 1, dim, inter, topk, 63)
    idx = idx % E                       # routed ids only
    bi, bd = inter // 128, dim // 128
    y = oracle.moe_tokens(xq, xs, idx, wts, w1q, w1s, w3q, w3s, w2q, w2s, range(5), n_shared=1)
    routed = oracle.moe_tokens(xq, xs, idx, wts, w1q[:E * inter], w1s[:E * bi], w3q[:E * inter], w3s[:E * bi],
                               w2q[:E * dim], w2s[:E * bd], range(5))
    z = oracle.bf16_round(oracle.ffn_rows(xq, xs, w1q[E * inter:], w1s[E * bi:], w3q[E * inter:], w3s[E * bi:],
                                          w2q[E * dim:], w2s[E * bd:], range(5)))
    as_bf16 = lambda b: torch.from_numpy(b.astype(np.int16)).view(torch.bfloat16)
    want = (as_bf16(routed) + as_bf16(z)).view(torch.int16).numpy().astype(np.uint16)
    assert np.array_equal(y, want)
