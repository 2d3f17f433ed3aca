"""The bounds-checked debug build on the small odd-shaped parity cases.

The library built with -DW4A16_BOUNDS_CHECK=1 (a separate .so outside the
package; the product never loads it) checks every instrumented global index
of its kernels against the buffer it addresses and records a miss in the
device error word (W4A16_ERR_BOUNDS) instead of performing the access; it
never traps. Every entry point runs here through that build on shapes with
ragged tails, split tiles and all token-tile widths: no index may leave its
buffer (status 0 after each call) and the results must still meet the same
bars as the product build's parity tests.
"""
import numpy as np
import pytest
import torch

import oracle
import speculative_decode_verify_w4a16_gb300 as sv
import synth
from helpers import assert_linear_close, bf16_bits, bf16_to_dev, canon_to_dev, dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def bounds_lib():
    from speculative_decode_verify_w4a16_gb300 import _lib, build

    oracle.build()
    path = build.build_bounds()
    with _lib.use_library(path) as L:
        yield L


def _ok():
    torch.cuda.synchronize()
    assert sv.check_device_status() == 0  # W4A16_ERR_BOUNDS would be 7


@pytest.mark.parametrize("M,N,K", [(1, 384, 1152), (3, 640, 3072), (8, 128, 1024), (9, 1152, 2048),
                                   (17, 256, 5120), (40, 640, 3072), (64, 384, 1024), (80, 1024, 2048)])
def test_linear(bounds_lib, M, N, K):
    x = synth.activations(M, K, seed=1100 + M)
    qw, sc = oracle.quantize(synth.weights(N, K, seed=1101 + N))
    w = sv.prepack(*canon_to_dev(qw, sc))
    out = sv.linear(bf16_to_dev(x), w)
    _ok()
    assert_linear_close(bf16_bits(out), oracle.linear(x, qw, sc), f"bounds build {M}x{N}x{K}")


@pytest.mark.parametrize("M", [5, 33, 80])
def test_linear_logits(bounds_lib, M):
    N, K = 1536, 2048
    x = synth.activations(M, K, seed=1110 + M)
    qw, sc = oracle.quantize(synth.weights(N, K, seed=1111))
    logits, stats = sv.linear_logits(bf16_to_dev(x), sv.prepack(*canon_to_dev(qw, sc)))
    _ok()
    _, y = oracle.linear(x, qw, sc, want_y=True)
    got = logits.cpu().numpy().astype(np.float64)
    assert np.abs(got - y).max() <= 1e-3 * np.abs(y).max()
    l = got.reshape(M, -1, 32)
    assert np.array_equal(stats.cpu().numpy()[:, :, 0], l.max(axis=2).astype(np.float32))


def _accept_match(got, want, margins, what):
    (acc, nxt), (acc_r, nxt_r) = got, want
    ma, mc = margins
    tie = (ma < 1e-6) | (mc < 1e-8)
    bad = ((acc.cpu().numpy() != acc_r) | (nxt.cpu().numpy() != nxt_r)) & ~tie
    assert not bad.any(), (what, np.nonzero(bad)[0][:8])


@pytest.mark.parametrize("B,K,V", [(5, 3, 4099), (16, 4, 128256), (2, 1, 2)])
def test_stochastic_sequence_accept(bounds_lib, B, K, V):
    p, q, d, u = synth.accept_seq_case(B, K, V, seed=1120 + K)
    t = [torch.from_numpy(a).to(dev()) for a in (p, q, d, u)]
    got = sv.spec_accept(t[0], t[2], q_logits=t[1], uniforms=t[3])
    _ok()
    acc_r, nxt_r, _, ma, mc = oracle.spec_accept_seq(p, q, d, u)
    _accept_match(got, (acc_r, nxt_r), (ma, mc), f"sequence B={B} K={K} V={V}")


def test_prestat_accept(bounds_lib):
    B, K, V, hidden = 3, 2, 4096, 1024
    x = synth.activations(B * (K + 1), hidden, seed=1125)
    qw, sc = oracle.quantize(synth.weights(V, hidden, seed=1126, std=0.066))
    logits, stats = sv.linear_logits(bf16_to_dev(x), sv.prepack(*canon_to_dev(qw, sc)))
    torch.cuda.synchronize()
    p = logits.cpu().numpy().reshape(B, K + 1, V)
    g = synth.rng(1127)
    q = (p[:, :K] + g.standard_normal((B, K, V), dtype=np.float32)).astype(np.float32)
    d = synth.gumbel_max_sample(q, g)
    u = g.random((B, K + 1), dtype=np.float32)
    qt, dt, ut = (torch.from_numpy(np.ascontiguousarray(a)).to(dev()) for a in (q, d, u))
    got = sv.spec_accept_prestat(logits.view(B, K + 1, V), stats.view(B, K + 1, V // 32, 2), dt, qt, ut)
    _ok()
    acc_r, nxt_r, _, ma, mc = oracle.spec_accept_seq(p, q, d, u)
    _accept_match(got, (acc_r, nxt_r), (ma, mc), "prestat")


def test_greedy_chain_and_tree_accept(bounds_lib):
    p, draft, parents = synth.greedy_tree_case(6, 23, 5003, seed=1130)
    t = [torch.from_numpy(a).to(dev()) for a in (p, draft, parents)]
    acc, nxt, node = sv.spec_accept_node(t[0], t[1], tree_parents=t[2])
    _ok()
    acc_r, nxt_r, node_r = oracle.greedy_tree(p, draft, parents, want_node=True)
    assert np.array_equal(acc.cpu().numpy(), acc_r) and np.array_equal(nxt.cpu().numpy(), nxt_r)
    assert np.array_equal(node.cpu().numpy(), node_r)
    pc, dc = synth.greedy_chain_case(7, 5, 777, seed=1131)
    acc, nxt = sv.spec_accept(torch.from_numpy(pc).to(dev()), torch.from_numpy(dc).to(dev()))
    _ok()
    acc_r, nxt_r = oracle.greedy_chain(pc, dc)
    assert np.array_equal(acc.cpu().numpy(), acc_r) and np.array_equal(nxt.cpu().numpy(), nxt_r)


def test_stochastic_tree_accept(bounds_lib):
    p, q, d, parents, u = synth.accept_tree_case(9, 19, 3001, seed=1135)
    t = [torch.from_numpy(a).to(dev()) for a in (p, q, d, parents, u)]
    acc, nxt, node = sv.spec_accept_node(t[0], t[2], q_logits=t[1], tree_parents=t[3], uniforms=t[4])
    _ok()
    acc_r, nxt_r, node_r, ma, mc = oracle.spec_accept_tree(p, q, d, parents, u)
    tie = (ma < 1e-6) | (mc < 1e-6)
    bad = ((acc.cpu().numpy() != acc_r) | (nxt.cpu().numpy() != nxt_r) | (node.cpu().numpy() != node_r)) & ~tie
    assert not bad.any()


@pytest.mark.parametrize("B,n,H,Hkv,lens,tree,max_len", [(3, 9, 16, 2, [0, 37, 300], True, None),
                                                         (2, 40, 24, 8, [1, 130], True, None),
                                                         (1, 5, 16, 2, [3000], False, 3000),
                                                         (4, 33, 8, 1, [0, 0, 0, 0], True, 0)])
def test_tree_attention(bounds_lib, B, n, H, Hkv, lens, tree, max_len):
    Lcap = max(lens) + n + 24
    q, k, v, lens, parents = synth.attention_case(B, n, H, Hkv, 128, lens, Lcap, seed=1140 + n, tree=tree)
    bf = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev())
    out = sv.tree_attention(bf(q), bf(k), bf(v), torch.from_numpy(lens).to(dev()),
                            torch.from_numpy(parents).to(dev()) if tree else None, max_len=max_len)
    _ok()
    want, absw = oracle.tree_attention(q, k, v, lens, parents if tree else None, want_abs=True)
    got = out.float().cpu().numpy().astype(np.float64)
    assert np.all(np.abs(got - want) <= 1.05 * 2.0 ** -7 * absw + 2.0 ** -8 * np.abs(want) + 1e-6)


def test_kv_compact(bounds_lib):
    layers, B, n, Hkv, D, Lcap = 2, 3, 17, 4, 128, 90
    g = synth.rng(1150)
    lens = np.array([0, 40, 73], dtype=np.int32)
    k = g.integers(0, 1 << 16, size=(layers, B, Hkv, Lcap, D), dtype=np.int64).astype(np.uint16)
    v = g.integers(0, 1 << 16, size=(layers, B, Hkv, Lcap, D), dtype=np.int64).astype(np.uint16)
    parents = np.stack([synth.random_tree_parents(n, 7, g) for _ in range(B)])
    node = np.array([n - 1, 5, 0], dtype=np.int32)
    bf = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev())
    kt, vt = bf(k), bf(v)
    new_lens = sv.kv_compact(kt, vt, torch.from_numpy(lens).to(dev()), torch.from_numpy(node).to(dev()),
                             torch.from_numpy(parents).to(dev()))
    _ok()
    k_r, v_r, lens_r = oracle.kv_compact(k, v, lens, parents, node)
    assert np.array_equal(new_lens.cpu().numpy(), lens_r)
    assert np.array_equal(kt.view(torch.int16).cpu().numpy().view(np.uint16), k_r)
    assert np.array_equal(vt.view(torch.int16).cpu().numpy().view(np.uint16), v_r)
