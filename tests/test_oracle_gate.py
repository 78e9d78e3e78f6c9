"""Pins of the oracle's MoE gate (no GPU).

The gate follows "Administrator & Developer Guide" 8.4 and 3.3 and the MoE
data flow of the "Repository overview" page: scores (sigmoid or softmax),
optional group-limited masking (group score = max without a bias, sum of the
top two with one; the top topk_groups groups stay), top-k experts, the chosen
experts' original scores, normalisation, route_scale. The pins below check it
against library routines (numpy sorting, scipy's expit and softmax), against
invariants that any correct gate satisfies, and against a small case worked
out by hand from those rules."""
import numpy as np
import pytest
from scipy.special import expit, softmax

import oracle
import synthetic


def f32_scores(logits, sigmoid):
    """fp32 scores from scipy (fp64, rounded once): independent of the oracle."""
    l64 = logits.astype(np.float64)
    return (expit(l64) if sigmoid else softmax(l64, axis=1)).astype(np.float32)


@pytest.mark.parametrize("sigmoid", [True, False])
def test_single_group_is_topk_of_the_logits(sigmoid):
    """G = 1, no bias: both score functions are increasing in the logit, so the
    experts are the k largest logits, in descending order, and (unnormalised,
    scale 1) the weights are their scores."""
    T, E, k = 64, 64, 6
    l = synthetic.gate_logits(T, E, 11)
    idx, w = oracle.moe_gate(l, None, 1, 1, k, sigmoid, 1.0, normalize=False)
    top = -np.sort(-l, axis=1)[:, :k]
    assert np.array_equal(np.take_along_axis(l, idx.astype(np.int64), 1), top)
    s = f32_scores(l, sigmoid)
    want = np.take_along_axis(s, idx.astype(np.int64), 1)
    assert np.allclose(w, want, rtol=2.4e-7, atol=0)


def test_normalisation_and_route_scale():
    T, E, k = 32, 160, 6
    l = synthetic.gate_logits(T, E, 12)
    idx, w = oracle.moe_gate(l, None, 8, 3, k, False, 16.0, normalize=True)
    assert np.allclose(w.sum(axis=1), 16.0, rtol=1e-6)
    s = f32_scores(l, False).astype(np.float64)
    sel = np.take_along_axis(s, idx.astype(np.int64), 1)
    assert np.allclose(w, 16.0 * sel / sel.sum(axis=1, keepdims=True), rtol=1e-6)


@pytest.mark.parametrize("E,G,TG,k,sigmoid,use_bias", [(256, 8, 4, 8, True, True), (256, 8, 4, 8, True, False),
                                                       (160, 8, 3, 6, False, False), (64, 4, 2, 6, True, True)])
def test_group_limited_invariants(E, G, TG, k, sigmoid, use_bias):
    """On random logits: the experts are distinct, come from groups that rank
    among the TG best by group score, beat every other expert of those groups,
    appear in descending key order, and carry their (unbiased) scores as
    weights before normalisation."""
    T = 200
    l = synthetic.gate_logits(T, E, 13)
    b = synthetic.gate_bias(E, 13) if use_bias else None
    idx, w = oracle.moe_gate(l, b, G, TG, k, sigmoid, 1.0, normalize=False)
    s = f32_scores(l, sigmoid)
    z = s + b if use_bias else s
    GS = E // G
    zg = z.reshape(T, G, GS)
    gscore = (np.sort(zg, axis=2)[:, :, -2:].sum(axis=2, dtype=np.float32) if use_bias else zg.max(axis=2))
    for t in range(T):
        e = idx[t].astype(np.int64)
        assert len(set(e.tolist())) == k
        groups = set((e // GS).tolist())
        assert len(groups) <= TG
        cut = np.sort(gscore[t])[::-1][TG - 1]
        assert all(gscore[t, g] >= cut for g in groups)
        zs = z[t, e]
        assert np.all(np.diff(zs) <= 0)
        others = [x for g in groups for x in range(g * GS, (g + 1) * GS) if x not in set(e.tolist())]
        assert all(z[t, x] <= zs[-1] for x in others)
        assert np.allclose(w[t], s[t, e], rtol=2.4e-7, atol=0)


def test_worked_example_by_hand():
    """E = 8 experts in G = 4 groups of two, keep TG = 2 groups, k = 3, sigmoid.
    Scores s (by expert): 0.9 0.1 | 0.6 0.55 | 0.7 0.2 | 0.3 0.65.

    No bias: group scores are the group maxima 0.9, 0.6, 0.7, 0.65, so groups 0
    and 2 stay; among experts {0, 1, 4, 5} the three best are 0, 4, 5 (expert
    7, third overall at 0.65, is masked out).

    Zero bias: group scores are top-two sums 1.0, 1.15, 0.9, 0.95, so groups 1
    and 0 stay; the best of {0, 1, 2, 3} are 0, 2, 3.

    Bias +0.5 on expert 6 (z6 = 0.8): group 3 scores 0.8 + 0.65 = 1.45, so
    groups 3 and 1 stay; by key the best of {2, 3, 6, 7} are 6 (0.8), 7 (0.65),
    2 (0.6). Their weights are the unbiased scores 0.3, 0.65, 0.6, divided by
    their sum 1.55 and times route_scale."""
    s = np.array([0.9, 0.1, 0.6, 0.55, 0.7, 0.2, 0.3, 0.65])
    l = np.log(s / (1.0 - s)).astype(np.float32)[None, :]
    idx, _ = oracle.moe_gate(l, None, 4, 2, 3, True, 1.0, normalize=True)
    assert idx.tolist() == [[0, 4, 5]]
    idx, _ = oracle.moe_gate(l, np.zeros(8, np.float32), 4, 2, 3, True, 1.0, normalize=True)
    assert idx.tolist() == [[0, 2, 3]]
    bias = np.zeros(8, np.float32)
    bias[6] = 0.5
    idx, w = oracle.moe_gate(l, bias, 4, 2, 3, True, 2.5, normalize=True)
    assert idx.tolist() == [[6, 7, 2]]
    assert np.allclose(w[0], 2.5 * np.array([0.3, 0.65, 0.6]) / 1.55, rtol=1e-6)


def test_rejects_shapes_outside_the_rules():
    l = synthetic.gate_logits(2, 64, 14)
    with pytest.raises(ValueError):
        oracle.moe_gate(l, None, 5, 2, 4, True)       # E % G != 0
    with pytest.raises(ValueError):
        oracle.moe_gate(l, None, 8, 1, 9, True)       # k > TG * E / G
    with pytest.raises(ValueError):
        oracle.moe_gate(l, np.zeros(64, np.float32), 64, 4, 2, True)   # top-two sum of one-expert groups
