"""Seeded synthetic inputs for the W4A16 verify linear and the speculative accept step.

This module is shared by the tests, the benchmark and the CPU baseline. It holds
only random-number generation and input *structure* (shapes, distributions,
planted argmaxes); none of the method's arithmetic (no quantisation, no softmax,
no acceptance rule, no argmax). Everything is host-side numpy (PCG64) so the
same seed gives the same bytes on x86 and Arm.

Workload recipes follow "Speculative Decoding Meets Quantization" (Zhang et
al. 2025: 4-bit weight Llama-3-70B target) and the Korean tutorial page
"Speculative Decoding이란?" (section 3, Steps 1-4: K draft tokens, target and
draft distributions, uniforms).
"""
from __future__ import annotations

import numpy as np

# Llama-3-70B verify-pass linear shapes (K = in-features, N = out-features).
LLAMA3_70B_SHAPES = {
    "qkv": (8192, 10240),
    "o": (8192, 8192),
    "gate_up": (8192, 57344),
    "down": (28672, 8192),
}
LLAMA3_70B_LM_HEAD = (8192, 128256)
LLAMA3_VOCAB = 128256
GROUP = 128


def rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def bf16_bits_from_f32(a: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (round-to-nearest-even) and return the
    16-bit patterns. Used only to *make* bf16 inputs; finite inputs assumed."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    lsb = (u >> 16) & 1
    r = (u + np.uint32(0x7FFF) + lsb) >> 16
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32)


def activations(M: int, K: int, seed: int) -> np.ndarray:
    """x[M,K] ~ N(0,1), returned as bf16 bit patterns (uint16)."""
    x = rng(seed).standard_normal((M, K), dtype=np.float32)
    return bf16_bits_from_f32(x)


def weights(N: int, K: int, seed: int, std: float = 0.02) -> np.ndarray:
    """W[N,K] ~ N(0, std^2) float32 (nn.Linear convention: out = x W^T)."""
    return (rng(seed).standard_normal((N, K), dtype=np.float32) * np.float32(std)).astype(np.float32)


def random_codes(N: int, K: int, seed: int) -> np.ndarray:
    """Uniform int4 codes in [-8, 7] as int8, [N, K]."""
    return rng(seed).integers(-8, 8, size=(N, K), dtype=np.int8)


def random_scales_f16(N: int, K: int, seed: int, lo: float = 1e-3, hi: float = 2e-2) -> np.ndarray:
    """Positive fp16 group scales [N, K/128] as uint16 bit patterns."""
    s = rng(seed).uniform(lo, hi, size=(N, K // GROUP)).astype(np.float16)
    return s.view(np.uint16)


def gumbel_max_sample(logits: np.ndarray, g: np.random.Generator) -> np.ndarray:
    """Draw one index per row from softmax(logits) with the Gumbel-max trick
    (argmax of logits + Gumbel noise); this is the synthetic drafter, not part
    of the verify path."""
    u = g.random(logits.shape, dtype=np.float64)
    u = np.clip(u, 1e-300, 1.0)
    z = logits.astype(np.float64) - np.log(-np.log(u))
    return np.argmax(z, axis=-1).astype(np.int32)


def accept_seq_case(B: int, K: int, V: int, seed: int, p_std: float = 3.0, noise_std: float = 1.0):
    """Sequence-draft accept inputs.

    p_logits [B, K+1, V] ~ N(0, p_std^2); q_logits [B, K, V] = p[:, :K] + N(0, noise_std^2);
    draft_ids [B, K] drawn from softmax(q) (Gumbel-max); uniforms [B, K+1] in [0, 1).
    """
    g = rng(seed)
    p = (g.standard_normal((B, K + 1, V), dtype=np.float32) * np.float32(p_std)).astype(np.float32)
    q = (p[:, :K, :] + g.standard_normal((B, K, V), dtype=np.float32) * np.float32(noise_std)).astype(np.float32)
    d = gumbel_max_sample(q, g)
    u = g.random((B, K + 1), dtype=np.float32)
    return p, np.ascontiguousarray(q), d, u


def random_tree_parents(n: int, max_depth: int, g: np.random.Generator) -> np.ndarray:
    """Parent array of an n-node rooted tree (node 0 = root, parent[0] = -1,
    parent[j] < j), each parent drawn uniformly from earlier nodes whose depth
    is below max_depth."""
    parents = np.full(n, -1, dtype=np.int32)
    depth = np.zeros(n, dtype=np.int32)
    for j in range(1, n):
        cand = np.nonzero(depth[:j] < max_depth)[0]
        par = int(cand[g.integers(0, len(cand))])
        parents[j] = par
        depth[j] = depth[par] + 1
    return parents


def greedy_tree_case(B: int, n: int, V: int, seed: int, max_depth: int = 6, match_prob: float = 0.5,
                     p_std: float = 3.0, plant: float = 40.0, per_batch_parents: bool = True):
    """Greedy tree-verify inputs with *planted* argmaxes.

    Each node j gets a planted token t[b, j]; p_logits[b, j, t[b, j]] is set to
    `plant` (far above the N(0, p_std^2) background), so the row's argmax is t
    by construction. A child node's draft token copies its parent's planted
    token with probability match_prob (at most one such sibling per parent),
    otherwise it is a uniformly random other id. draft_ids[:, 0] (root) is -1.
    """
    g = rng(seed)
    p = (g.standard_normal((B, n, V), dtype=np.float32) * np.float32(p_std)).astype(np.float32)
    planted = g.integers(0, V, size=(B, n), dtype=np.int64).astype(np.int32)
    for b in range(B):
        p[b, np.arange(n), planted[b]] = np.float32(plant)
    if per_batch_parents:
        parents = np.stack([random_tree_parents(n, max_depth, g) for _ in range(B)])
    else:
        parents = np.broadcast_to(random_tree_parents(n, max_depth, g), (B, n)).copy()
    draft = np.full((B, n), -1, dtype=np.int32)
    for b in range(B):
        taken = set()
        for j in range(1, n):
            par = int(parents[b, j])
            if par not in taken and g.random() < match_prob:
                draft[b, j] = planted[b, par]
                taken.add(par)
            else:
                t = int(g.integers(0, V - 1))
                draft[b, j] = t if t < planted[b, par] else t + 1
    return p, draft, parents


def greedy_chain_case(B: int, K: int, V: int, seed: int, match_prob: float = 0.8, p_std: float = 3.0,
                      plant: float = 40.0):
    """Greedy sequence-draft inputs: p_logits [B, K+1, V] with planted argmax
    per row, draft_ids [B, K] where d_i copies row (i-1)'s planted token with
    probability match_prob."""
    g = rng(seed)
    p = (g.standard_normal((B, K + 1, V), dtype=np.float32) * np.float32(p_std)).astype(np.float32)
    planted = g.integers(0, V, size=(B, K + 1), dtype=np.int64).astype(np.int32)
    for b in range(B):
        p[b, np.arange(K + 1), planted[b]] = np.float32(plant)
    draft = np.empty((B, K), dtype=np.int32)
    for b in range(B):
        for i in range(K):
            if g.random() < match_prob:
                draft[b, i] = planted[b, i]
            else:
                t = int(g.integers(0, V - 1))
                draft[b, i] = t if t < planted[b, i] else t + 1
    return p, draft


def attention_case(B: int, n: int, H: int, Hkv: int, D: int, lens, Lcap: int, seed: int, tree: bool = True,
                   max_depth: int = 6):
    """Verify-attention inputs (Llama-3 geometry: H query heads over Hkv
    key/value heads of width D): q [B,n,H,D] and the key / value caches
    [B,Hkv,Lcap,D], all N(0,1) as bf16 bit patterns; the committed prefix of
    row b at cache positions 0..lens[b]-1 and the n tree nodes' own keys and
    values at lens[b]..lens[b]+n-1. parents [B,n]: a random tree per row
    (depth < max_depth), or the chain parent[j] = j - 1 when tree is False."""
    g = rng(seed)
    lens = np.asarray(lens, dtype=np.int32)
    assert lens.shape == (B,) and int(lens.max()) + n <= Lcap
    q = bf16_bits_from_f32(g.standard_normal((B, n, H, D), dtype=np.float32))
    k = bf16_bits_from_f32(g.standard_normal((B, Hkv, Lcap, D), dtype=np.float32))
    v = bf16_bits_from_f32(g.standard_normal((B, Hkv, Lcap, D), dtype=np.float32))
    if tree:
        parents = np.stack([random_tree_parents(n, max_depth, g) for _ in range(B)])
    else:
        parents = np.broadcast_to(np.arange(-1, n - 1, dtype=np.int32), (B, n)).copy()
    return q, k, v, lens, parents


def attention_lens(B: int, lo: int, hi: int, seed: int) -> np.ndarray:
    """Ragged committed lengths, uniform in [lo, hi)."""
    return rng(seed).integers(lo, hi, size=B).astype(np.int32)


def accept_tree_case(B: int, n: int, V: int, seed: int, max_depth: int = 6, p_std: float = 3.0,
                     noise: float = 1.0):
    """Stochastic tree-verify inputs: target logits ~ N(0, p_std^2) at every
    node, draft logits = target + N(0, noise^2); a random tree per row (depth
    < max_depth); every child's token drawn from the draft's distribution at
    its parent (Gumbel-max); uniforms U[0, 1) [B, n] (u[:, 0] draws the next
    token, u[:, j] tests node j)."""
    g = rng(seed)
    p = (g.standard_normal((B, n, V), dtype=np.float32) * np.float32(p_std)).astype(np.float32)
    q = (p + g.standard_normal((B, n, V), dtype=np.float32) * np.float32(noise)).astype(np.float32)
    parents = np.stack([random_tree_parents(n, max_depth, g) for _ in range(B)])
    d = np.full((B, n), -1, dtype=np.int32)
    if n > 1:
        for b in range(B):
            d[b, 1:] = gumbel_max_sample(q[b, parents[b, 1:]], g)
    u = g.random((B, n), dtype=np.float32)
    return p, q, d, parents, u
