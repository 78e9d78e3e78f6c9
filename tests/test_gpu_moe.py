"""GPU parity of the SwiGLU FFN chain and the routed-expert (MoE) path
against the CPU oracle ("Administrator & Developer Guide", 6.4 and 8.4; 1.2
MLP / Expert).

- The routing permutation is integer work: bit-exact.
- The fused w1/w3 GEMM's e4m3 output: every scale and code lies in the
  interval the oracle's fp64 h1, h3 admit (helpers: rules 1-4), and every
  block's largest code matches its own scale.
- The chains (dense FFN, MoE) are graded on every output element with the
  GEMM tolerance |diff| <= 2^-7 |ref| + 1e-3 rms(ref) plus the exact change
  the admissible intermediates permit."""
import numpy as np
import pytest
import torch

import fp8_block_scaled_quant_gb300 as fb
import oracle
import synthetic
from helpers import (admissible_quant, admissible_u, assert_chain_close, assert_gemm_close, assert_quant_admissible,
                     bits_to_dev_bf16, dequant_weight, dev_to_bits, ffn_chain_allowance)

pytestmark = pytest.mark.gpu


def to_dev_q(q):
    return torch.from_numpy(q).cuda().view(torch.float8_e4m3fn)


def to_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


# ---- A5: permutation ------------------------------------------------------------

@pytest.mark.parametrize("T,E,k,zipf", [(4096, 256, 8, 0.0), (4096, 256, 8, 1.2), (1, 4, 2, 0.0),
                                        (3000, 1024, 6, 1.2), (700, 7, 3, 0.0)])
def test_moe_permute_bit_exact(T, E, k, zipf):
    idx, _ = synthetic.moe_routing(T, E, k, 500 + T + E, zipf_s=zipf)
    counts, offsets, perm = fb.moe_permute(to_dev(idx), E)
    co, oo, po = oracle.moe_permute(idx, E)
    assert np.array_equal(counts.cpu().numpy(), co)
    assert np.array_equal(offsets.cpu().numpy(), oo)
    assert np.array_equal(perm.cpu().numpy(), po)


def test_moe_permute_invalid_ids_reported_and_skipped():
    idx, _ = synthetic.moe_routing(50, 8, 2, 7)
    bad = idx.copy()
    bad[4, 1] = 8
    bad[9, 0] = -3
    counts, offsets, perm = fb.moe_permute(to_dev(bad), 8)
    assert fb.last_device_error() != 0          # reported ...
    keep = np.flatnonzero((bad.ravel() >= 0) & (bad.ravel() < 8))
    want = keep[np.argsort(bad.ravel()[keep], kind="stable")]
    assert offsets[-1].item() == keep.size      # ... and left out
    assert np.array_equal(perm[: keep.size].cpu().numpy(), want)
    assert fb.last_device_error() == 0          # the bit was cleared


# ---- A4: fused w1/w3 GEMM with SwiGLU + act_quant --------------------------------



@pytest.mark.parametrize("M,dim,inter", [(5, 256, 384), (130, 512, 256), (300, 256, 1024)])
@pytest.mark.parametrize("fmt", [fb.SCALE_FP32, fb.SCALE_UE8M0, "ue8m0-promotion"])
def test_swiglu_gemm_matches_oracle_chain(M, dim, inter, fmt):
    """UE8M0 scales are applied by the tensor core (block-scaled MMA);
    ue8m0-promotion: the same scales through the per-block promotion."""
    if fmt == "ue8m0-promotion":
        fmt = fb.SCALE_UE8M0 | fb.SCALE_PROMOTE
    ue = (fmt & ~fb.SCALE_PROMOTE) == fb.SCALE_UE8M0
    x = synthetic.activations(M, dim, 600 + M)
    xq, xs = oracle.act_quant(x, ue)
    w1q, w1s = oracle.weight_quant(synthetic.weights(inter, dim, 601 + M), ue)
    w3q, w3s = oracle.weight_quant(synthetic.weights(inter, dim, 602 + M), ue)
    u, us = fb.swiglu_gemm(to_dev_q(xq), to_dev(xs), to_dev_q(w1q), to_dev(w1s), to_dev_q(w3q), to_dev(w3s), fmt)
    H1 = oracle.gemm(xq, xs, w1q, w1s)
    H3 = oracle.gemm(xq, xs, w3q, w3s)
    adm = admissible_quant(*admissible_u(H1, H3), ue)
    assert_quant_admissible(dev_to_bits(u), us.cpu().numpy(), adm, ue, what=f"swiglu {M}x{dim}x{inter}")


# ---- A4 chain: dense FFN ---------------------------------------------------------

@pytest.mark.parametrize("M,dim,inter", [(5, 256, 384), (300, 256, 384), (129, 512, 1024)])
def test_ffn_full_compare(M, dim, inter):
    x = synthetic.activations(M, dim, 700 + M, outlier_frac=0.02)
    w1 = synthetic.weights(inter, dim, 701)
    w3 = synthetic.weights(inter, dim, 702)
    w2 = synthetic.weights(dim, inter, 703)
    w1q, w1s = oracle.weight_quant(w1)
    w3q, w3s = oracle.weight_quant(w3)
    w2q, w2s = oracle.weight_quant(w2)
    xq, xs = oracle.act_quant(x)
    y = fb.ffn(bits_to_dev_bf16(x), to_dev_q(w1q), to_dev(w1s), to_dev_q(w3q), to_dev(w3s), to_dev_q(w2q),
               to_dev(w2s))
    ref, uq, us = oracle.ffn_rows(xq, xs, w1q, w1s, w3q, w3s, w2q, w2s, range(M), return_u=True)
    allow = ffn_chain_allowance(xq, xs, w1q, w1s, w3q, w3s, dequant_weight(w2q, w2s), uq, us)
    assert_chain_close(dev_to_bits(y), ref, allow, what=f"ffn {M}x{dim}x{inter}")
    # repeated call: workspaces were left clean
    y2 = fb.ffn(bits_to_dev_bf16(x), to_dev_q(w1q), to_dev(w1s), to_dev_q(w3q), to_dev(w3s), to_dev_q(w2q),
                to_dev(w2s))
    assert torch.equal(y.view(torch.int16), y2.view(torch.int16))


def test_ffn_workspace_shared_by_layers_of_different_shapes():
    """The FFN's two GEMMs share one GEMM workspace at offset 0 of the FFN
    workspace, so one workspace serves FFNs of different shapes: bit-equal to
    fresh workspaces, counters back at zero."""
    dev = torch.device("cuda")
    shapes = [(300, 256, 1024), (1300, 512, 1024)]
    layers = []
    for i, (M, dim, inter) in enumerate(shapes):
        x = synthetic.device_activations(M, dim, 111 + i, dev)
        qs = [fb.weight_quant(synthetic.device_normal(sh, 121 + 3 * i + j, 0.02, dev))
              for j, sh in enumerate([(inter, dim), (inter, dim), (dim, inter)])]
        args = (x, qs[0][0], qs[0][1], qs[1][0], qs[1][1], qs[2][0], qs[2][1])
        nb = fb.ffn_workspace_bytes(M, dim, inter)
        want = fb.ffn(*args, ws=torch.zeros(nb, dtype=torch.uint8, device=dev))
        layers.append((args, nb, want))
    shared = torch.zeros(max(l[1] for l in layers), dtype=torch.uint8, device=dev)
    for _ in range(2):
        for args, nb, want in layers:
            got = fb.ffn(*args, ws=shared[:nb])
            assert torch.equal(got.view(torch.int16), want.view(torch.int16))
    assert torch.count_nonzero(shared[:64 * 1024]) == 0
    assert fb.last_device_error() == 0


def test_ffn_full_size_sampled_rows():
    """The prefill FFN (x [4096, 7168], inter 18432) on the device; the oracle
    recomputes two whole output rows (one per end of the row range)."""
    M, dim, inter = 4096, 7168, 18432
    dev = torch.device("cuda")
    x = synthetic.device_activations(M, dim, synthetic.SEED_PREFILL, dev)
    ws = [synthetic.device_normal(shape, synthetic.SEED_PREFILL + 10 + i, 0.02, dev)
          for i, shape in enumerate([(inter, dim), (inter, dim), (dim, inter)])]
    qs = [fb.weight_quant(w) for w in ws]
    y = fb.ffn(x, qs[0][0], qs[0][1], qs[1][0], qs[1][1], qs[2][0], qs[2][1])
    rows = np.array([1, M - 2])
    xq, xs = oracle.act_quant(dev_to_bits(x[torch.from_numpy(rows).to(dev)]))
    host_q = [oracle.weight_quant(w.cpu().numpy()) for w in ws]
    for (q, s), (qo, so) in zip(qs, host_q):
        assert np.array_equal(dev_to_bits(q), qo) and np.array_equal(s.cpu().numpy(), so)
    ref, uq, us = oracle.ffn_rows(xq, xs, *host_q[0], *host_q[1], *host_q[2], range(2), return_u=True)
    allow = ffn_chain_allowance(xq, xs, *host_q[0], *host_q[1], dequant_weight(*host_q[2]), uq, us)
    # the tolerance's rms term from the oracle's own rows (an estimate of the whole output's rms)
    assert_chain_close(dev_to_bits(y)[rows], ref, allow, rms=float(np.sqrt(np.mean(ref ** 2))),
                       what="ffn sampled rows")


# ---- A6/A7: routed experts ----------------------------------------------------------

def moe_problem(T, E, dim, inter, k, seed, zipf=0.0, ue8m0=False):
    x = synthetic.activations(T, dim, seed, outlier_frac=0.01)
    xq, xs = oracle.act_quant(x, ue8m0)
    w1q, w1s = oracle.weight_quant(synthetic.weights(E * inter, dim, seed + 1), ue8m0)
    w3q, w3s = oracle.weight_quant(synthetic.weights(E * inter, dim, seed + 2), ue8m0)
    w2q, w2s = oracle.weight_quant(synthetic.weights(E * dim, inter, seed + 3), ue8m0)
    idx, wts = synthetic.moe_routing(T, E, k, seed + 4, zipf_s=zipf)
    return xq, xs, idx, wts, w1q, w1s, w3q, w3s, w2q, w2s


def moe_reference(p, tokens, E, ue8m0=False, wdeq_cache=None):
    """The oracle's MoE output rows (fp64 of its bf16 result) and the chain
    allowance: for each slot j, |w_j| times (one bf16 step of the expert output
    o_j, which a different fp32 summation may round the other way, plus the
    expert's admissible-intermediate allowance)."""
    xq, xs, idx, wts, w1q, w1s, w3q, w3s, w2q, w2s = p
    dim = xq.shape[1]
    inter = w2q.shape[1]
    bi, bd = inter // 128, dim // 128
    tokens = list(tokens)
    ref = synthetic.bf16_bits_to_f32(oracle.moe_tokens(*p, tokens, ue8m0=ue8m0)).astype(np.float64)
    allow = np.zeros((len(tokens), dim))
    cache = {} if wdeq_cache is None else wdeq_cache
    pos = {t: i for i, t in enumerate(tokens)}
    for e in range(E):
        slots = [(t, j) for t in tokens for j in range(idx.shape[1]) if idx[t, j] == e]
        if not slots:
            continue
        rows = np.array([t for t, _ in slots])
        we = (w1q[e * inter:(e + 1) * inter], w1s[e * bi:(e + 1) * bi], w3q[e * inter:(e + 1) * inter],
              w3s[e * bi:(e + 1) * bi])
        w2e = (w2q[e * dim:(e + 1) * dim], w2s[e * bd:(e + 1) * bd])
        o, uq, us = oracle.ffn_rows(xq[rows], xs[rows], *we, *w2e, range(len(rows)), ue8m0=ue8m0, return_u=True)
        if e not in cache:
            cache[e] = dequant_weight(*w2e)
        al = ffn_chain_allowance(xq[rows], xs[rows], *we, cache[e], uq, us, ue8m0)
        for r, (t, j) in enumerate(slots):
            allow[pos[t]] += abs(float(wts[t, j])) * (2.0 ** -7 * np.abs(o[r]) + al[r])
    return ref, allow


def run_moe(p, E, fmt=fb.SCALE_FP32):
    xq, xs, idx, wts, w1q, w1s, w3q, w3s, w2q, w2s = p
    return fb.moe_grouped_gemm(to_dev_q(xq), to_dev(xs), to_dev(idx), to_dev(wts), to_dev_q(w1q), to_dev(w1s),
                               to_dev_q(w3q), to_dev(w3s), to_dev_q(w2q), to_dev(w2s), E, fmt)


@pytest.mark.parametrize("T,E,dim,inter,k,zipf", [(64, 8, 256, 256, 2, 0.0), (96, 16, 512, 384, 4, 1.2),
                                                  (33, 5, 256, 128, 3, 0.0), (300, 4, 256, 256, 1, 0.0)])
@pytest.mark.parametrize("fmt", [fb.SCALE_FP32, fb.SCALE_UE8M0, "ue8m0-promotion"])
def test_moe_full_compare(T, E, dim, inter, k, zipf, fmt):
    """UE8M0: both grouped GEMMs with the scales applied by the tensor core;
    ue8m0-promotion: the same scales through the per-block promotion."""
    if fmt == "ue8m0-promotion":
        fmt = fb.SCALE_UE8M0 | fb.SCALE_PROMOTE
    ue = (fmt & ~fb.SCALE_PROMOTE) == fb.SCALE_UE8M0
    p = moe_problem(T, E, dim, inter, k, 800 + T + E, zipf, ue)
    y = run_moe(p, E, fmt)
    ref, allow = moe_reference(p, range(T), E, ue8m0=ue)
    assert_chain_close(dev_to_bits(y), ref, allow, what=f"moe T={T} E={E}")
    assert fb.last_device_error() == 0


def test_moe_empty_experts_and_invalid_slots():
    T, E, dim, inter = 40, 6, 256, 256
    xq, xs, idx, wts, w1q, w1s, w3q, w3s, w2q, w2s = moe_problem(T, E, dim, inter, 2, 900)
    idx[:, :] = np.where(idx >= 3, idx % 3, idx)     # experts 3..5 get no token
    idx[:, 1] = np.where(idx[:, 1] == idx[:, 0], (idx[:, 0] + 1) % 3, idx[:, 1])
    bad = idx.copy()
    bad[5, 1] = 17                                   # invalid slot: contributes nothing
    y = run_moe((xq, xs, bad, wts, w1q, w1s, w3q, w3s, w2q, w2s), E)
    assert fb.last_device_error() != 0
    idx_ref, wts_ref = bad.copy(), wts.copy()
    idx_ref[5, 1], wts_ref[5, 1] = 0, 0.0
    ref, allow = moe_reference((xq, xs, idx_ref, wts_ref, w1q, w1s, w3q, w3s, w2q, w2s), range(T), E)
    assert_chain_close(dev_to_bits(y), ref, allow, what="moe with empty experts and an invalid slot")


def test_moe_full_size_sampled_tokens():
    """T=4096 tokens, 256 experts (dim 7168, inter 2048), top-8 Zipf(1.2)
    routing on the device; the oracle recomputes two whole output rows from
    its own quantisation of the experts those tokens use."""
    T, E, dim, inter, k = 4096, 256, 7168, 2048, 8
    dev = torch.device("cuda")
    seed = synthetic.SEED_MOE
    x = synthetic.device_activations(T, dim, seed, dev)
    xq_d, xs_d = fb.act_quant(x)
    idx, wts = synthetic.moe_routing(T, E, k, seed, zipf_s=1.2)

    def expert_w(e, which):
        shape = (inter, dim) if which < 2 else (dim, inter)
        return synthetic.device_normal(shape, seed * 100000 + 3 * e + which, 0.02, dev)

    stacks = []
    for which in range(3):
        qs, ss = zip(*[fb.weight_quant(expert_w(e, which)) for e in range(E)])
        stacks.append((torch.cat(qs), torch.cat(ss)))
    y = fb.moe_grouped_gemm(xq_d, xs_d, to_dev(idx), to_dev(wts), stacks[0][0], stacks[0][1], stacks[1][0],
                            stacks[1][1], stacks[2][0], stacks[2][1], E)
    tokens = [3, T - 1]
    rows = torch.tensor(tokens, device=dev)
    xq, xs = oracle.act_quant(dev_to_bits(x[rows]))
    ref, allow = [], []
    for i, t in enumerate(tokens):
        acc, al = np.zeros(dim), np.zeros(dim)
        for j in range(k):
            e = idx[t, j]
            wq = [oracle.weight_quant(expert_w(e, which).cpu().numpy()) for which in range(3)]
            o, uq, us = oracle.ffn_rows(xq[i:i + 1], xs[i:i + 1], *wq[0], *wq[1], *wq[2], [0], return_u=True)
            acc += np.float64(wts[t, j]) * synthetic.bf16_bits_to_f32(oracle.bf16_round(o[0]))
            al += abs(float(wts[t, j])) * (2.0 ** -7 * np.abs(o[0]) + ffn_chain_allowance(
                xq[i:i + 1], xs[i:i + 1], *wq[0], *wq[1], dequant_weight(*wq[2]), uq, us)[0])
        ref.append(synthetic.bf16_bits_to_f32(oracle.bf16_round(acc)).astype(np.float64))
        allow.append(al)
    ref = np.array(ref)
    # the tolerance's rms term from the oracle's own rows (an estimate of the whole output's rms)
    assert_chain_close(dev_to_bits(y)[tokens], ref, np.array(allow), rms=float(np.sqrt(np.mean(ref ** 2))),
                       what="moe sampled tokens")
    assert fb.last_device_error() == 0


@pytest.mark.parametrize("T,E,dim,inter,k", [(64, 8, 256, 256, 2), (33, 5, 256, 128, 3), (200, 3, 512, 256, 1)])
def test_moe_shared_expert(T, E, dim, inter, k):
    """One shared expert stacked after the E routed ones: every token also goes
    through it (weight 1) in the same grouped launches, and the row is
    bf16(y + z) (Guide 8.4 steps 6 and 8). Tolerance: the routed and shared
    chains' allowances plus one bf16 step of y and of z (each is rounded once
    before the sum)."""
    xq, xs, _, _, w1q, w1s, w3q, w3s, w2q, w2s = moe_problem(T, E + 1, dim, inter, k, 950 + T)
    idx, wts = synthetic.moe_routing(T, E, k, 951 + T)
    p = (xq, xs, idx, wts, w1q, w1s, w3q, w3s, w2q, w2s)
    y = fb.moe_grouped_gemm(to_dev_q(xq), to_dev(xs), to_dev(idx), to_dev(wts), to_dev_q(w1q), to_dev(w1s),
                            to_dev_q(w3q), to_dev(w3s), to_dev_q(w2q), to_dev(w2s), E, n_shared=1)
    ref = synthetic.bf16_bits_to_f32(oracle.moe_tokens(*p, range(T), n_shared=1)).astype(np.float64)
    bi, bd = inter // 128, dim // 128
    routed = (xq, xs, idx, wts, w1q[:E * inter], w1s[:E * bi], w3q[:E * inter], w3s[:E * bi], w2q[:E * dim],
              w2s[:E * bd])
    ref_r, allow_r = moe_reference(routed, range(T), E)
    sh = (w1q[E * inter:], w1s[E * bi:], w3q[E * inter:], w3s[E * bi:])
    z, uq, us = oracle.ffn_rows(xq, xs, *sh, w2q[E * dim:], w2s[E * bd:], range(T), return_u=True)
    allow_z = 2.0 ** -7 * np.abs(z) + ffn_chain_allowance(xq, xs, *sh, dequant_weight(w2q[E * dim:], w2s[E * bd:]),
                                                          uq, us)
    allow = allow_r + allow_z + 2.0 ** -8 * (np.abs(ref_r) + np.abs(z))
    assert_chain_close(dev_to_bits(y), ref, allow, what=f"moe + shared expert T={T} E={E}")
    assert fb.last_device_error() == 0
