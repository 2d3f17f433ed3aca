"""GPU parity of the stochastic token-tree acceptance (multi-step speculative
sampling; SpecInfer's rule for children drawn independently from the draft's
distribution at their parent) against the CPU oracle, through the C ABI.

Decisions, emitted tokens and the accepted node must match the oracle bit for
bit except where the oracle's fp64 margins put a decision within the
near-tie windows: |u - alpha| < 1e-6, or the draw's CDF boundary within
1e-6 of the sum. The CDF window is wider than the sequence rule's 1e-8
because a residual after k rejections, max(0, P - c_k Q) with c_k up to k,
is formed from fp32 values whose rounding errors scale with P + c_k Q rather
than with the (possibly small) residual itself."""
import numpy as np
import pytest
import torch

import oracle
import speculative_decode_verify_w4a16_gb300 as sv
import synth
from helpers import dev

pytestmark = pytest.mark.gpu
NEAR_TIE, NEAR_TIE_CDF = 1e-6, 1e-6


@pytest.fixture(scope="module", autouse=True)
def _built():
    from speculative_decode_verify_w4a16_gb300 import build
    build.build()
    oracle.build()


def _case(B, n, V, seed, max_depth=6, p_std=3.0, noise=1.0):
    return synth.accept_tree_case(B, n, V, seed, max_depth=max_depth, p_std=p_std, noise=noise)


def _compare(p, q, d, parents, u, what):
    acc_r, nxt_r, node_r, ma, mc = oracle.spec_accept_tree(p, q, d, parents, u)
    t = [torch.from_numpy(np.ascontiguousarray(a)).to(dev()) for a in (p, q, d, parents, u)]
    acc, nxt, node = sv.spec_accept_node(t[0], t[2], q_logits=t[1], tree_parents=t[3], uniforms=t[4])
    torch.cuda.synchronize()
    assert sv.check_device_status() == 0
    acc, nxt, node = acc.cpu().numpy(), nxt.cpu().numpy(), node.cpu().numpy()
    tie = (ma < NEAR_TIE) | (mc < NEAR_TIE_CDF)
    bad = ((acc != acc_r) | (nxt != nxt_r) | (node != node_r)) & ~tie
    print(f"{what}: {int(tie.sum())} near-ties of {len(acc)}; mean depth {acc_r.mean():.2f}; "
          f"differing within the windows {int(((acc != acc_r) | (nxt != nxt_r)) [tie].sum())}")
    assert not bad.any(), np.nonzero(bad)[0][:10]
    assert np.array_equal(acc_r, np.array([_depth(parents[b], node_r[b]) for b in range(len(acc_r))]))
    return tie


def _depth(par, j):
    k = 0
    while j > 0:
        j = int(par[j])
        k += 1
    return k


def test_config_tree_full_vocab():
    """16 sequences, 64-node trees of depth < 6, Llama-3 vocabulary."""
    p, q, d, parents, u = _case(16, 64, 128256, seed=1001)
    tie = _compare(p, q, d, parents, u, "B=16 n=64 V=128256")
    assert tie.sum() == 0


@pytest.mark.parametrize("B,n,V,noise", [(64, 9, 5, 1.0), (128, 17, 1003, 0.5), (32, 33, 32000, 2.0),
                                         (8, 1, 64, 1.0), (4, 200, 4096, 0.3), (40, 24, 131072, 1.0)])
def test_random_cases(B, n, V, noise):
    p, q, d, parents, u = _case(B, n, V, seed=1010 + n + V, noise=noise)
    tie = _compare(p, q, d, parents, u, f"B={B} n={n} V={V}")
    # a token's CDF interval is about 1/V wide, so at large V a few rows fall
    # in the 1e-6 window; they are excluded from the comparison, not failed
    assert tie.sum() <= max(2, B // 8)


def test_many_trials_small_vocabulary():
    """Many independent small trees (the regime of the oracle's chi-square
    pin): every emitted token and the accepted node as the oracle's."""
    p, q, d, parents, u = _case(3000, 9, 6, seed=1020, p_std=1.2, noise=1.2)
    tie = _compare(p, q, d, parents, u, "B=3000 n=9 V=6")
    assert tie.sum() <= 3


def test_chain_matches_the_sequence_kernel():
    B, K, V = 32, 6, 128256
    p, q, d, u = synth.accept_seq_case(B, K, V, seed=1030)
    n = K + 1
    parents = np.broadcast_to(np.arange(-1, n - 1, dtype=np.int32), (B, n)).copy()
    qt = np.concatenate([q, np.zeros((B, 1, V), np.float32)], axis=1)
    dt = np.concatenate([np.full((B, 1), -1, np.int32), d], axis=1)
    ut = np.ascontiguousarray(np.concatenate([u[:, K:K + 1], u[:, :K]], axis=1))
    t = [torch.from_numpy(np.ascontiguousarray(a)).to(dev()) for a in (p, q, d, u, qt, dt, parents, ut)]
    acc_s, nxt_s = sv.spec_accept(t[0], t[2], q_logits=t[1], uniforms=t[3])
    acc_t, nxt_t, node_t = sv.spec_accept_node(t[0], t[5], q_logits=t[4], tree_parents=t[6], uniforms=t[7])
    torch.cuda.synchronize()
    assert sv.check_device_status() == 0
    _, _, _, ma, mc = oracle.spec_accept_seq(p, q, d, u)
    ok = (ma >= NEAR_TIE) & (mc >= NEAR_TIE_CDF)
    assert ok.sum() >= B - 1
    assert torch.equal(acc_t, node_t)
    assert np.array_equal(acc_t.cpu().numpy()[ok], acc_s.cpu().numpy()[ok])
    assert np.array_equal(nxt_t.cpu().numpy()[ok], nxt_s.cpu().numpy()[ok])


def test_bad_draft_id_is_reported_and_skipped():
    p, q, d, parents, u = _case(4, 8, 100, seed=1040)
    d[1, 3] = 100  # out of range
    t = [torch.from_numpy(np.ascontiguousarray(a)).to(dev()) for a in (p, q, d, parents, u)]
    acc, nxt, node = sv.spec_accept_node(t[0], t[2], q_logits=t[1], tree_parents=t[3], uniforms=t[4])
    torch.cuda.synchronize()
    assert sv.check_device_status() == 5  # W4A16_ERR_DEVICE_INPUT
    assert 0 <= int(nxt[1]) < 100
    assert sv.check_device_status() == 0  # the error word was cleared
