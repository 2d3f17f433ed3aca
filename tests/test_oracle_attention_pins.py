"""Pins of the oracle's tree-masked verify attention and KV compaction
(the tutorial page "Speculative Decoding이란?", section 10.1 Medusa tree-based
attention, section 10.4 ReDrafter dynamic tree attention, section 8.7 KV cache
reuse) against things other than the oracle itself: PyTorch's scaled
dot-product attention with masks built independently (networkx ancestors),
closed forms, invariances and brute-force indexing."""
import numpy as np
import pytest
import torch

nx = pytest.importorskip("networkx")  # not installed everywhere these tests are collected

import oracle
import synth


def _f(bits):
    return synth.bf16_bits_to_f32(bits).astype(np.float64)


def _nx_tree(parents):
    g = nx.DiGraph()
    g.add_nodes_from(range(len(parents)))
    g.add_edges_from((int(p), j) for j, p in enumerate(parents) if p >= 0)
    return g


def _sdpa_reference(q, k, v, lens, parents):
    """torch SDPA (fp64, CPU) with the tree mask from networkx ancestors."""
    B, n, H, D = q.shape
    Hkv = k.shape[1]
    out = np.empty((B, n, H, D))
    for b in range(B):
        L = int(lens[b])
        T = L + n
        tr = _nx_tree(parents[b])
        mask = np.zeros((n, T), dtype=bool)
        mask[:, :L] = True
        for j in range(n):
            for i in nx.ancestors(tr, j) | {j}:
                mask[j, L + i] = True
        Q = torch.from_numpy(_f(q[b])).permute(1, 0, 2)                      # [H, n, D]
        K = torch.from_numpy(_f(k[b, :, :T])).repeat_interleave(H // Hkv, 0)  # [H, T, D]
        V = torch.from_numpy(_f(v[b, :, :T])).repeat_interleave(H // Hkv, 0)
        o = torch.nn.functional.scaled_dot_product_attention(Q, K, V, attn_mask=torch.from_numpy(mask))
        out[b] = o.permute(1, 0, 2).numpy()
    return out


@pytest.mark.parametrize("tree", [False, True])
def test_matches_sdpa(tree):
    B, n, H, Hkv, D, Lcap = 3, 9, 8, 2, 32, 48
    lens = np.array([0, 5, 30], dtype=np.int32)
    q, k, v, lens, parents = synth.attention_case(B, n, H, Hkv, D, lens, Lcap, seed=5 + tree, tree=tree)
    got = oracle.tree_attention(q, k, v, lens, parents if tree else None)
    want = _sdpa_reference(q, k, v, lens, parents)
    assert np.abs(got - want).max() < 1e-12


def test_identical_keys_give_the_mean_of_the_allowed_values():
    # every key equal: the softmax is uniform over the L + depth(j) + 1 allowed keys
    B, n, H, Hkv, D, Lcap = 2, 12, 4, 4, 16, 40
    lens = np.array([3, 17], dtype=np.int32)
    q, k, v, lens, parents = synth.attention_case(B, n, H, Hkv, D, lens, Lcap, seed=11)
    k[:] = k[0, 0, 0]
    got = oracle.tree_attention(q, k, v, lens, parents)
    for b in range(B):
        L = int(lens[b])
        tr = _nx_tree(parents[b])
        for j in range(n):
            keys = list(range(L)) + [L + i for i in sorted(nx.ancestors(tr, j) | {j})]
            want = _f(v[b][:, keys]).mean(axis=1)  # [Hkv, D]
            assert np.abs(got[b, j] - want).max() < 1e-12


def test_only_the_root_path_and_prefix_matter():
    B, n, H, Hkv, D, Lcap = 2, 16, 4, 2, 16, 64
    lens = np.array([9, 20], dtype=np.int32)
    q, k, v, lens, parents = synth.attention_case(B, n, H, Hkv, D, lens, Lcap, seed=13)
    base = oracle.tree_attention(q, k, v, lens, parents)
    g = synth.rng(14)
    for b in range(B):
        L = int(lens[b])
        tr = _nx_tree(parents[b])
        j = n - 1
        keep = {L + i for i in nx.ancestors(tr, j) | {j}} | set(range(L))
        other = [x for x in range(Lcap) if x not in keep]
        k2, v2 = k.copy(), v.copy()
        k2[b][:, other] = synth.bf16_bits_from_f32(g.standard_normal((Hkv, len(other), D), dtype=np.float32))
        v2[b][:, other] = synth.bf16_bits_from_f32(g.standard_normal((Hkv, len(other), D), dtype=np.float32))
        got = oracle.tree_attention(q, k2, v2, lens, parents)
        assert np.array_equal(got[b, j], base[b, j])
        # and a node off that path does see the change
        assert not np.array_equal(got[b], base[b])


def test_root_with_empty_prefix_returns_its_own_value():
    B, n, H, Hkv, D, Lcap = 1, 4, 2, 1, 8, 8
    q, k, v, lens, parents = synth.attention_case(B, n, H, Hkv, D, [0], Lcap, seed=17)
    got = oracle.tree_attention(q, k, v, lens, parents)
    assert np.array_equal(got[0, 0], np.broadcast_to(_f(v[0, 0, 0]), (H, D)))


def test_grouped_heads_equal_expanded_heads():
    B, n, H, Hkv, D, Lcap = 2, 6, 8, 2, 16, 24
    q, k, v, lens, parents = synth.attention_case(B, n, H, Hkv, D, [4, 11], Lcap, seed=19)
    grouped = oracle.tree_attention(q, k, v, lens, parents)
    ke, ve = np.repeat(k, H // Hkv, axis=1), np.repeat(v, H // Hkv, axis=1)
    expanded = oracle.tree_attention(q, ke, ve, lens, parents)
    assert np.array_equal(grouped, expanded)


def test_scale_is_applied_to_the_scores():
    # doubling q equals doubling the scale
    B, n, H, Hkv, D, Lcap = 1, 5, 2, 1, 16, 16
    q, k, v, lens, parents = synth.attention_case(B, n, H, Hkv, D, [6], Lcap, seed=23)
    q2 = synth.bf16_bits_from_f32(2.0 * synth.bf16_bits_to_f32(q))  # exact: a power of two
    a = oracle.tree_attention(q2, k, v, lens, parents, scale=0.25)
    b = oracle.tree_attention(q, k, v, lens, parents, scale=0.5)
    assert np.abs(a - b).max() < 1e-12


@pytest.mark.parametrize("tree", [False, True])
def test_kv_compact_moves_the_accepted_path(tree):
    layers, B, n, Hkv, D, Lcap = 2, 4, 10, 2, 8, 32
    g = synth.rng(29)
    lens = np.array([0, 3, 12, 21], dtype=np.int32)
    k = g.integers(0, 1 << 16, size=(layers, B, Hkv, Lcap, D), dtype=np.int64).astype(np.uint16)
    v = g.integers(0, 1 << 16, size=(layers, B, Hkv, Lcap, D), dtype=np.int64).astype(np.uint16)
    parents = np.stack([synth.random_tree_parents(n, 5, g) for _ in range(B)]) if tree else \
        np.broadcast_to(np.arange(-1, n - 1, dtype=np.int32), (B, n)).copy()
    node = np.array([0, n - 1, 4, 7], dtype=np.int32)
    k2, v2, new_lens = oracle.kv_compact(k, v, lens, parents if tree else None, node)
    for b in range(B):
        path = nx.shortest_path(_nx_tree(parents[b]), 0, int(node[b]))  # root first
        L = int(lens[b])
        assert new_lens[b] == L + len(path)
        ek, ev = k[:, b].copy(), v[:, b].copy()
        ek[:, :, L:L + len(path)] = k[:, b][:, :, [L + i for i in path]]
        ev[:, :, L:L + len(path)] = v[:, b][:, :, [L + i for i in path]]
        assert np.array_equal(k2[:, b], ek) and np.array_equal(v2[:, b], ev)
        if not tree:
            assert np.array_equal(k2[:, b], k[:, b])  # a chain is already in place


def test_greedy_tree_reports_the_deepest_accepted_node():
    B, n, V = 32, 24, 50
    p, draft, parents = synth.greedy_tree_case(B, n, V, seed=31, max_depth=5, match_prob=0.7)
    acc, nxt, node = oracle.greedy_tree(p, draft, parents, want_node=True)
    for b in range(B):
        tr = _nx_tree(parents[b])
        path = nx.shortest_path(tr, 0, int(node[b]))
        assert len(path) - 1 == acc[b]
        for a, c in zip(path[:-1], path[1:]):  # every edge on the path matches the parent's argmax
            assert draft[b, c] == int(np.argmax(p[b, a]))
        assert nxt[b] == int(np.argmax(p[b, node[b]]))
        # no accepted node is deeper, and none at the same depth has a smaller index
        for j in range(n):
            pj = nx.shortest_path(tr, 0, j)
            ok = all(draft[b, c] == int(np.argmax(p[b, a])) for a, c in zip(pj[:-1], pj[1:]))
            if ok:
                assert len(pj) - 1 < acc[b] or (len(pj) - 1 == acc[b] and j >= node[b])


def test_weighted_abs_values():
    # with all values >= 0 the weighted |v| is the output itself; with v -> -v it is -out
    B, n, H, Hkv, D, Lcap = 2, 7, 4, 2, 16, 32
    q, k, v, lens, parents = synth.attention_case(B, n, H, Hkv, D, [3, 9], Lcap, seed=37)
    vpos = synth.bf16_bits_from_f32(np.abs(synth.bf16_bits_to_f32(v)))
    out, a = oracle.tree_attention(q, k, vpos, lens, parents, want_abs=True)
    assert np.array_equal(out, a)
    vneg = vpos | np.uint16(0x8000)
    out2, a2 = oracle.tree_attention(q, k, vneg, lens, parents, want_abs=True)
    assert np.array_equal(out2, -a) and np.array_equal(a2, a)
