"""Pins of the oracle's stochastic tree acceptance (multi-step speculative
sampling, as SpecInfer defines it for children drawn independently from the
draft's distribution at their parent; the pages give the rule for a sequence
draft only: the tutorial page "Speculative Decoding이란?", section 3 Steps 3-4).

The pins do not restate the rule: the tokens it emits must follow the target
distribution (chi-square over many seeded trials), the acceptance rate of a
first child is sum_x min(P, Q), identical distributions accept every first
child, a token the target gives no mass is never emitted, and a chain gives
the sequence rule's decisions."""
import numpy as np
import pytest

import oracle
import synth

scipy_stats = pytest.importorskip("scipy.stats")


def _softmax(l):
    e = np.exp(l.astype(np.float64) - l.max())
    return e / e.sum()


# root 0 with children 1, 2, 3; node 1: children 4, 5; node 2: child 6; node 3: children 7, 8
PARENTS = np.array([-1, 0, 0, 0, 1, 1, 2, 3, 3], dtype=np.int32)
DEPTH = np.array([0, 1, 1, 1, 2, 2, 2, 2, 2])


def _trials(T, V, seed, p_root, p_mid, p_leaf, q_root, q_mid):
    """T independent trials on one fixed tree shape: node rows p / q per
    depth; every child's token drawn independently from the draft
    distribution at its parent."""
    g = synth.rng(seed)
    n = len(PARENTS)
    p = np.empty((T, n, V), dtype=np.float32)
    q = np.empty((T, n, V), dtype=np.float32)
    for j in range(n):
        p[:, j] = (p_root, p_mid, p_leaf)[DEPTH[j]]
        q[:, j] = (q_root, q_mid, q_mid)[DEPTH[j]]
    d = np.full((T, n), -1, dtype=np.int32)
    for j in range(1, n):
        Qp = _softmax(q[0, PARENTS[j]])
        d[:, j] = g.choice(V, size=T, p=Qp)
    u = g.random((T, n), dtype=np.float32)
    return p, q, d, u


def _emitted(d, acc, nxt, node):
    """The emitted tokens of each trial: the accepted path's draft tokens,
    then the next token."""
    out = []
    for t in range(len(acc)):
        path, j = [], int(node[t])
        while j > 0:
            path.append(int(d[t, j]))
            j = int(PARENTS[j])
        out.append(path[::-1] + [int(nxt[t])])
    return out


def test_emitted_tokens_follow_the_target_distribution():
    V, T = 6, 120000
    g = synth.rng(1)
    p_root, p_mid, p_leaf = (g.normal(0, 1.2, V).astype(np.float32) for _ in range(3))
    q_root, q_mid = (g.normal(0, 1.2, V).astype(np.float32) for _ in range(2))
    p, q, d, u = _trials(T, V, 2, p_root, p_mid, p_leaf, q_root, q_mid)
    acc, nxt, node, _, _ = oracle.spec_accept_tree(p, q, d, PARENTS, u)
    assert np.array_equal(acc, DEPTH[node])
    seqs = _emitted(d, acc, nxt, node)
    for pos, P in ((0, _softmax(p_root)), (1, _softmax(p_mid)), (2, _softmax(p_leaf))):
        tokens = np.array([s[pos] for s in seqs if len(s) > pos])
        counts = np.bincount(tokens, minlength=V)
        _, pval = scipy_stats.chisquare(counts, P * len(tokens))
        assert pval > 1e-4, (pos, pval, counts, P * len(tokens))
    assert (acc == 2).sum() > 1000 and (acc == 0).sum() > 1000  # every depth is exercised


def test_first_child_acceptance_rate_is_the_overlap():
    V, T = 5, 100000
    g = synth.rng(3)
    p_root, p_mid, p_leaf, q_root, q_mid = (g.normal(0, 1.5, V).astype(np.float32) for _ in range(5))
    p, q, d, u = _trials(T, V, 4, p_root, p_mid, p_leaf, q_root, q_mid)
    # node 1, the root's first child, is on the accepted path iff its own test passed
    acc, nxt, node, _, _ = oracle.spec_accept_tree(p, q, d, PARENTS, u)
    path_first = np.array([_first_on_path(int(j)) for j in node])
    rate = np.mean(path_first == 1)
    want = np.minimum(_softmax(p_root), _softmax(q_root)).sum()
    sd = np.sqrt(want * (1 - want) / T)
    assert abs(rate - want) < 5 * sd, (rate, want)


def _first_on_path(j):
    while j > 0 and PARENTS[j] != 0:
        j = int(PARENTS[j])
    return j


def test_identical_distributions_accept_every_first_child():
    V, T = 7, 64
    g = synth.rng(5)
    rows = [g.normal(0, 2, V).astype(np.float32) for _ in range(3)]
    p, q, d, u = _trials(T, V, 6, rows[0], rows[1], rows[2], rows[0], rows[1])
    acc, _, node, _, _ = oracle.spec_accept_tree(p, q, d, PARENTS, u)
    assert np.all(node == 4) and np.all(acc == 2)  # 0 -> 1 -> 4: the first child at every level


def test_a_token_without_target_mass_is_never_emitted():
    V, T, x = 6, 2000, 2
    g = synth.rng(7)
    p_root = g.normal(0, 1, V).astype(np.float32)
    p_root[x] = -60.0  # P(x) ~ 1e-27
    q_root = np.full(V, -60.0, dtype=np.float32)
    q_root[x] = 10.0  # every child of the root drafts x
    p_mid, p_leaf, q_mid = (g.normal(0, 1, V).astype(np.float32) for _ in range(3))
    p, q, d, u = _trials(T, V, 8, p_root, p_mid, p_leaf, q_root, q_mid)
    acc, nxt, node, _, _ = oracle.spec_accept_tree(p, q, d, PARENTS, u)
    assert np.all(d[:, 1:4] == x)
    assert np.all(acc == 0) and np.all(node == 0) and np.all(nxt != x)


def test_a_chain_gives_the_sequence_rule():
    B, K, V = 64, 5, 50
    p, q, d, u = synth.accept_seq_case(B, K, V, seed=9)
    n = K + 1
    parents = np.arange(-1, n - 1, dtype=np.int32)
    qt = np.concatenate([q, np.zeros((B, 1, V), np.float32)], axis=1)  # the leaf's row is never read
    dt = np.concatenate([np.full((B, 1), -1, np.int32), d], axis=1)
    ut = np.concatenate([u[:, K:K + 1], u[:, :K]], axis=1)  # u_0 draws; u_j tests node j
    acc_s, nxt_s, _, ma_s, mc_s = oracle.spec_accept_seq(p, q, d, u)
    acc_t, nxt_t, node_t, ma_t, mc_t = oracle.spec_accept_tree(p, qt, dt, parents, ut)
    assert np.array_equal(acc_t, acc_s) and np.array_equal(node_t, acc_s)
    safe = mc_s > 1e-12
    assert np.array_equal(nxt_t[safe], nxt_s[safe]) and safe.sum() >= B - 1
    assert np.allclose(ma_t, ma_s, rtol=0, atol=1e-12)
