"""Seeded synthetic inputs for the block-scaled FP8 linear-algebra path.

This module is shared by the CUDA path's tests and benchmark and by the CPU
oracle's tests. It holds none of the method's arithmetic: it only draws random
numbers (numpy PCG64 on the host, torch's Philox generator on a device for
weights too large to draw on the host) and rounds them to the storage dtype of
the model (bf16 activations, fp32 master weights). Quantisation, scales,
dequantisation and products live on each side separately.

Workload shapes follow the DeepSeek-V3 inference pages ("Administrator &
Developer Guide", section 3.3 model configs: dim 7168, inter_dim 18432,
moe_inter_dim 2048, 256 routed experts, 8 activated; MLA ranks q_lora 1536,
kv_lora 512, rope 64).
"""
from __future__ import annotations

import numpy as np

BLOCK = 128

# Seeds, one per workload, in the order the workloads are listed.
SEED_PR1 = 0
SEED_DECODE = 1
SEED_PREFILL = 2
SEED_ATTN = 3
SEED_MOE = 4
SEED_GATE = 5


def rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (torch's round-to-nearest-even cast) and
    return the raw uint16 bit patterns."""
    import torch

    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 (exact: a bf16 is the top half of an fp32)."""
    return (b.astype(np.uint32) << 16).view(np.float32)


def activations(M: int, K: int, seed: int, outlier_frac: float = 0.0,
                outlier_mult: float = 20.0) -> np.ndarray:
    """X ~ N(0, 1) of shape [M, K] as bf16 bits. When outlier_frac > 0, that
    fraction of the K channels (outlier_channels(K, seed, outlier_frac)) is
    multiplied by outlier_mult before rounding."""
    ch = outlier_channels(K, seed, outlier_frac)
    x = rng(seed).standard_normal((M, K), dtype=np.float32)
    if ch.size:
        x[:, ch] *= np.float32(outlier_mult)
    return to_bf16_bits(x)


def outlier_channels(K: int, seed: int, outlier_frac: float) -> np.ndarray:
    """The seeded set of outlier channels (sorted int64 indices), drawn from a
    stream of its own so that it does not depend on M."""
    n_out = int(round(outlier_frac * K))
    if n_out <= 0:
        return np.zeros(0, np.int64)
    g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 0x0C4A])))
    return np.sort(g.choice(K, size=n_out, replace=False)).astype(np.int64)


def weights(N: int, K: int, seed: int, std: float = 0.02) -> np.ndarray:
    """Master weight W ~ N(0, std) of shape [N, K], float32, drawn from a
    stream of its own so that a weight and an activation with the same seed
    are independent."""
    g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 0x57])))
    return (g.standard_normal((N, K), dtype=np.float32) * np.float32(std)).astype(np.float32)


def device_normal(shape, seed: int, std: float, device, dtype=None):
    """N(0, std) drawn on a device with torch's seeded generator, for weights
    too large to draw on the host (e.g. the 256 stacked MoE experts). The
    result is float32 unless dtype is given."""
    import torch

    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    t = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    t.mul_(std)
    return t if dtype is None else t.to(dtype)


def device_activations(M: int, K: int, seed: int, device, outlier_frac: float = 0.0,
                       outlier_mult: float = 20.0):
    """Device twin of activations() for sizes that are slow on the host:
    N(0, 1) bf16 [M, K] with a seeded fraction of outlier channels."""
    import torch

    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    x = torch.randn((M, K), generator=g, device=device, dtype=torch.float32)
    ch = outlier_channels(K, seed, outlier_frac)
    if ch.size:
        x[:, torch.from_numpy(ch).to(device)] *= outlier_mult
    return x.to(torch.bfloat16)


def moe_routing(T: int, E: int, topk: int, seed: int, zipf_s: float = 0.0):
    """Top-k routing of T tokens over E experts.

    Logits are log p_e + Gumbel noise, with p uniform (zipf_s == 0) or
    p_e proportional to rank^-zipf_s over a seeded permutation of the experts.
    The k largest logits give k distinct experts per token (sampling without
    replacement); their gate weights are the softmax of the selected logits.
    Returns (indices int32 [T, topk], weights float32 [T, topk])."""
    g = rng(seed)
    if zipf_s > 0.0:
        ranks = np.arange(1, E + 1, dtype=np.float64)
        p = ranks ** (-zipf_s)
        p = p[np.argsort(g.permutation(E))]
    else:
        p = np.ones(E, dtype=np.float64)
    p /= p.sum()
    gumbel = -np.log(-np.log(g.uniform(1e-12, 1.0, size=(T, E))))
    logits = np.log(p)[None, :] + gumbel
    idx = np.argsort(-logits, axis=1, kind="stable")[:, :topk]
    sel = np.take_along_axis(logits, idx, axis=1)
    sel = sel - sel.max(axis=1, keepdims=True)
    w = np.exp(sel)
    w /= w.sum(axis=1, keepdims=True)
    return idx.astype(np.int32), w.astype(np.float32)


def gate_logits(T: int, E: int, seed: int, std: float = 1.0) -> np.ndarray:
    """Gate logits fp32 [T, E] ~ N(0, std^2), one draw per (token, expert)."""
    return (rng(seed).standard_normal((T, E)) * std).astype(np.float32)


def gate_bias(E: int, seed: int, std: float = 0.1) -> np.ndarray:
    """Per-expert gate bias fp32 [E] ~ N(0, std^2)."""
    return (rng(seed + 1000).standard_normal(E) * std).astype(np.float32)
