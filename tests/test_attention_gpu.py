"""GPU parity of the tree-masked verify attention and the accepted-path KV
compaction against the CPU oracle (the tutorial page "Speculative Decoding이란?",
section 10.1 Medusa tree-based attention, section 10.4 ReDrafter dynamic tree
attention, section 8.7 KV cache reuse), through the C ABI.

Attention tolerance, from the arithmetic: the kernel rounds each softmax weight
p_k to bf16 for the weighted sum of the values (an 8-bit significand: relative
error delta <= 2^-8, plus the fp32 score and exponential errors, about 1e-6)
and normalises by the sum of the fp32 weights, so each normalised weight is
within a factor (1 +- delta) of the exact one and the weighted sum moves by at
most about 2^-8 * A, where A = sum_k w_k |v_k| (the oracle reports it);
storing the result in bf16 adds 2^-8 |out|. The bound used keeps a factor of
two beyond that: 1.05 * 2^-7 * A + 2^-8 * |out| + 1e-6."""
import numpy as np
import pytest
import torch

import oracle
import speculative_decode_verify_w4a16_gb300 as sv
import synth
from helpers import dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from speculative_decode_verify_w4a16_gb300 import build
    build.build()
    oracle.build()


def _bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(dev())


def _run(q, k, v, lens, parents, max_len=None):
    out = sv.tree_attention(_bf16(q), _bf16(k), _bf16(v), torch.from_numpy(lens).to(dev()),
                            None if parents is None else torch.from_numpy(parents).to(dev()), max_len=max_len)
    torch.cuda.synchronize()
    assert sv.check_device_status() == 0
    return out.float().cpu().numpy().astype(np.float64)


def _check(got, want, absw, what):
    bound = 1.05 * 2.0 ** -7 * absw + 2.0 ** -8 * np.abs(want) + 1e-6
    worst = float((np.abs(got - want) / bound).max())
    print(f"{what}: max |err| / bound = {worst:.3f}")
    assert worst <= 1.0, what


CASES = [  # B, n, H, Hkv, lens, tree
    (3, 9, 16, 2, [0, 37, 300], True),
    (2, 64, 64, 8, [100, 1000], True),       # Llama-3-70B heads, a full 64-node tree
    (4, 5, 64, 8, [0, 63, 64, 2000], False),  # sequence draft K = 4; lengths at block edges
    (1, 1, 8, 8, [5], False),                 # one query, one head per KV head
    (2, 17, 12, 4, [129, 7], True),           # three query heads per KV head
    (2, 33, 8, 1, [511, 64], True),           # all heads on one KV head
    (2, 24, 64, 8, [300, 77], True),          # 192 query rows: the second 128-row tile half full
    # 70 sequences: above 64 the units are taken in order, one CTA each
    (70, 3, 16, 2, [(37 * i) % 260 for i in range(70)], True),
]


@pytest.mark.parametrize("B,n,H,Hkv,lens,tree", CASES)
def test_tree_attention_matches_oracle(B, n, H, Hkv, lens, tree):
    Lcap = max(lens) + n + 40
    q, k, v, lens, parents = synth.attention_case(B, n, H, Hkv, 128, lens, Lcap, seed=900 + n + H, tree=tree)
    want, absw = oracle.tree_attention(q, k, v, lens, parents if tree else None, want_abs=True)
    got = _run(q, k, v, lens, parents if tree else None)
    _check(got, want, absw, f"B={B} n={n} H={H}/{Hkv} tree={tree}")


def test_one_split_and_many_splits_agree_with_the_oracle():
    # max_len = 0 leaves one key block (one split: rows normalised in the
    # kernel); a long prefix on a small grid takes many splits and the
    # combine. The first case takes two 128-row tiles per CTA (320 query rows
    # per KV head), the others one (40 and 128 rows); the last one has splits
    # holding no key of its first sequence
    cases = [(16, 40, 64, 8, [0] * 16, 0), (1, 5, 16, 2, [3000], 3000), (1, 16, 64, 8, [3000], 3000),
             (2, 16, 64, 8, [100, 3000], 3000)]
    seen = set()
    for B, n, H, Hkv, lens, max_len in cases:
        Lcap = max_len + n + 8
        seen.add(sv.tree_attention_workspace_bytes(B, n, H, Hkv, 128, Lcap, max_len) > 0)
        q, k, v, lens, parents = synth.attention_case(B, n, H, Hkv, 128, lens, Lcap, seed=950 + B)
        want, absw = oracle.tree_attention(q, k, v, lens, parents, want_abs=True)
        _check(_run(q, k, v, lens, parents, max_len=max_len), want, absw, f"B={B} max_len={max_len}")
    assert seen == {False, True}


def test_only_the_root_path_and_prefix_matter_on_the_gpu():
    B, n, H, Hkv, Lcap = 2, 48, 16, 2, 400
    q, k, v, lens, parents = synth.attention_case(B, n, H, Hkv, 128, [70, 200], Lcap, seed=960)
    base = _run(q, k, v, lens, parents)
    g = synth.rng(961)
    j = n - 1
    k2, v2 = k.copy(), v.copy()
    for b in range(B):
        keep = set(range(int(lens[b])))
        i = j
        while i >= 0:
            keep.add(int(lens[b]) + i)
            i = int(parents[b, i])
        other = [x for x in range(Lcap) if x not in keep]
        k2[b][:, other] = synth.bf16_bits_from_f32(g.standard_normal((Hkv, len(other), 128), dtype=np.float32))
        v2[b][:, other] = synth.bf16_bits_from_f32(g.standard_normal((Hkv, len(other), 128), dtype=np.float32))
    got = _run(q, k2, v2, lens, parents)
    assert np.array_equal(got[:, j], base[:, j])
    assert not np.array_equal(got, base)


def test_llama70b_tree_verify_attention_sampled():
    """Llama-3-70B attention geometry (64 query heads on 8 KV heads of 128) at
    the tree-verify configuration (16 sequences, 64-node trees, committed
    lengths 1024..4096), in the launch configuration the benchmark times;
    checked on two sampled sequences."""
    B, n, H, Hkv = 16, 64, 64, 8
    lens = synth.attention_lens(B, 1024, 4096, seed=970)
    Lcap = 4096 + n
    q, k, v, lens, parents = synth.attention_case(B, n, H, Hkv, 128, lens, Lcap, seed=971)
    got = _run(q, k, v, lens, parents, max_len=4096)
    for b in (0, B - 1):
        want, absw = oracle.tree_attention(q[b:b + 1], k[b:b + 1], v[b:b + 1], lens[b:b + 1], parents[b:b + 1],
                                           want_abs=True)
        _check(got[b:b + 1], want, absw, f"sequence {b}")


@pytest.mark.parametrize("tree", [False, True])
def test_kv_compact_matches_oracle(tree):
    layers, B, n, Hkv, D, Lcap = 3, 5, 24, 8, 128, 200
    g = synth.rng(980 + tree)
    lens = np.array([0, 1, 63, 100, 176], dtype=np.int32)
    k = g.integers(0, 1 << 16, size=(layers, B, Hkv, Lcap, D), dtype=np.int64).astype(np.uint16)
    v = g.integers(0, 1 << 16, size=(layers, B, Hkv, Lcap, D), dtype=np.int64).astype(np.uint16)
    if tree:
        parents = np.stack([synth.random_tree_parents(n, 8, g) for _ in range(B)])
        node = g.integers(0, n, size=B).astype(np.int32)
    else:
        parents = None
        node = np.array([0, n - 1, 3, 10, 23], dtype=np.int32)
    k_r, v_r, lens_r = oracle.kv_compact(k, v, lens, parents, node)
    kt, vt = _bf16(k), _bf16(v)
    new_lens = sv.kv_compact(kt, vt, torch.from_numpy(lens).to(dev()), torch.from_numpy(node).to(dev()),
                             None if parents is None else torch.from_numpy(parents).to(dev()), n=n)
    torch.cuda.synchronize()
    assert sv.check_device_status() == 0
    assert np.array_equal(new_lens.cpu().numpy(), lens_r)
    assert np.array_equal(kt.view(torch.int16).cpu().numpy().view(np.uint16), k_r)
    assert np.array_equal(vt.view(torch.int16).cpu().numpy().view(np.uint16), v_r)


def test_accept_reports_the_accepted_node():
    B, n, V = 16, 64, 128256
    p, draft, parents = synth.greedy_tree_case(B, n, V, seed=990)
    acc_r, nxt_r, node_r = oracle.greedy_tree(p, draft, parents, want_node=True)
    t = [torch.from_numpy(a).to(dev()) for a in (p, draft, parents)]
    acc, nxt, node = sv.spec_accept_node(t[0], t[1], tree_parents=t[2])
    torch.cuda.synchronize()
    assert sv.check_device_status() == 0
    assert np.array_equal(acc.cpu().numpy(), acc_r) and np.array_equal(nxt.cpu().numpy(), nxt_r)
    assert np.array_equal(node.cpu().numpy(), node_r)
    # sequence modes: the node is the accepted length
    ps, qs, ds, us = synth.accept_seq_case(8, 4, 4096, seed=991)
    ts = [torch.from_numpy(a).to(dev()) for a in (ps, qs, ds, us)]
    acc, _, node = sv.spec_accept_node(ts[0], ts[2], q_logits=ts[1], uniforms=ts[3])
    torch.cuda.synchronize()
    assert torch.equal(acc, node)
    acc, _, node = sv.spec_accept_node(ts[0], ts[2])
    torch.cuda.synchronize()
    assert torch.equal(acc, node)


def test_verify_step_end_to_end():
    """One tree-verify step of the KV side: attention over the tree, greedy
    acceptance, compaction of the accepted path; then the next step's single
    query attends to the compacted cache exactly as the oracle's, i.e. as if
    only the accepted tokens had ever been written."""
    B, n, H, Hkv, V = 4, 32, 16, 2, 4096
    lens = np.array([10, 200, 64, 0], dtype=np.int32)
    Lcap = 256 + n
    q, k, v, lens, parents = synth.attention_case(B, n, H, Hkv, 128, lens, Lcap, seed=995)
    p, draft, _ = synth.greedy_tree_case(B, n, V, seed=996, per_batch_parents=True)
    # reuse the attention case's trees for the accept step
    p_t, d_t, par_t = (torch.from_numpy(a).to(dev()) for a in (p, draft, parents))
    _, _, node = sv.spec_accept_node(p_t, d_t, tree_parents=par_t)
    kt, vt = _bf16(k), _bf16(v)
    lens_t = torch.from_numpy(lens).to(dev())
    new_lens = sv.kv_compact(kt, vt, lens_t, node, par_t)
    torch.cuda.synchronize()
    assert sv.check_device_status() == 0
    node_h = node.cpu().numpy()
    k_r, v_r, lens_r = oracle.kv_compact(k[None], v[None], lens, parents, node_h)
    assert np.array_equal(new_lens.cpu().numpy(), lens_r)
    # next step: one query per row at the new end of the cache (a chain of one node whose keys are the bonus token's)
    q1 = synth.attention_case(B, 1, H, Hkv, 128, lens_r, Lcap, seed=997)[0]
    k1 = k_r[0].copy()
    v1 = v_r[0].copy()
    got = _run(q1, k1, v1, lens_r, None)
    want, absw = oracle.tree_attention(q1, k1, v1, lens_r, None, want_abs=True)
    _check(got, want, absw, "next step")
