"""Pins for the CPU oracle: each test ties the oracle to something other than
itself (a library routine, a closed form, brute force, or the pages' worked
example), so that a dropped term, a wrong index or a transposed operand in the
oracle fails here. CPU only."""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# --------------------------------------------------------------- rounding

def test_bf16_round_matches_torch():
    g = synth.rng(1)
    vals = np.concatenate([
        g.standard_normal(20000).astype(np.float32) * np.float32(10.0) ** g.integers(-30, 30, 20000).astype(np.float32),
        # exact ties between two bf16 neighbours (round half to even)
        (np.arange(1, 2000, dtype=np.uint32) << 16 | 0x8000).view(np.float32),
        np.array([0.0, -0.0, 1.0, -1.0, 3.0e38, -3.0e38, 1e-40, -1e-40], dtype=np.float32),
    ])
    ref = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.bf16_round(float(v)) for v in vals], dtype=np.uint16)
    assert np.array_equal(got, ref)


def _bf16_exact(bits: int):
    """The value of a bf16 bit pattern as an exact Fraction (None for inf/nan)."""
    from fractions import Fraction
    sign = -1 if bits & 0x8000 else 1
    e = (bits >> 7) & 0xFF
    m = bits & 0x7F
    if e == 0xFF:
        return None
    if e == 0:
        return sign * Fraction(m, 2 ** 133)
    return sign * Fraction(128 + m) * Fraction(2) ** (e - 134)


def _bf16_rne_brute_force(v: float) -> int:
    """Round-to-nearest-even of a double onto the bf16 grid by its definition:
    among the finite bf16 values around v pick the nearest in exact rational
    arithmetic, on a tie the one with an even last significand bit; past the
    largest finite bf16 by half a step or more, infinity."""
    from fractions import Fraction
    fv = Fraction(v)
    base = int(np.array([v], dtype=np.float32).view(np.uint32)[0] >> 16)
    if v == 0:
        return base  # +0 / -0 keep their sign bit
    cands = []
    for b in range(base - 2, base + 3):
        b &= 0xFFFF
        val = _bf16_exact(b)
        if val is not None and ((val > 0) == (v > 0) or val == 0):
            cands.append((abs(val - fv), b & 1, (b & 0x8000) != (base & 0x8000), b))
    cands.sort()
    best = cands[0][-1]
    big = _bf16_exact(0x7F7F)
    if abs(fv) >= big + (big - _bf16_exact(0x7F7E)) / 2:
        return 0xFF80 if v < 0 else 0x7F80
    return best


def test_bf16_round_from_f64_matches_definition():
    g = synth.rng(5)
    vals = list(g.standard_normal(3000) * 10.0 ** g.integers(-40, 38, 3000))
    # just above / below / on a tie between bf16 neighbours, by less than fp32 can see
    # (an fp32 intermediate would land on the tie and round to even instead)
    for b in list(range(0x3F80, 0x3F90)) + [0x0001, 0x0080, 0x4780, 0x7F00, 0x8123, 0xC2F1]:
        lo, hi = _bf16_exact(b), _bf16_exact(b + 1)
        mid = float((lo + hi) / 2)
        step = float(hi - lo)
        vals += [mid, mid + step * 2.0 ** -20, mid - step * 2.0 ** -20, mid + step * 2.0 ** -40]
    vals += [0.0, -0.0, 1e-45, -1e-45, 2.0 ** -140, 2.0 ** -134, 3.4e38, -3.4e38, 3.39e38]
    for v in vals:
        assert oracle.bf16_round_f64(v) == _bf16_rne_brute_force(v), v
    # the case a float intermediate gets wrong: 1 + 2^-8 + 2^-30 lies above the tie
    assert oracle.bf16_round_f64(1.0 + 2.0 ** -8 + 2.0 ** -30) == 0x3F81
    assert oracle.bf16_round(np.float32(1.0 + 2.0 ** -8 + 2.0 ** -30)) == 0x3F80


def test_f16_round_matches_numpy():
    g = synth.rng(2)
    vals = np.concatenate([g.uniform(-65000, 65000, 5000), g.uniform(-1e-3, 1e-3, 5000),
                           g.uniform(-1e-6, 1e-6, 2000)]).astype(np.float32)
    ref = vals.astype(np.float16).view(np.uint16)
    got = np.array([oracle.f16_round(float(v)) for v in vals], dtype=np.uint16)
    assert np.array_equal(got, ref)


# ------------------------------------------------------------ 4-bit format

def test_pack_known_words():
    # nibble j of word = code of k = 8*w + j, two's complement, little nibble first
    codes = np.array([[1, 2, 3, 4, 5, 6, 7, -8], [-1, 0, 0, 0, 0, 0, 0, 0]], dtype=np.int8)
    qw = oracle.pack_codes(codes)
    assert qw.tolist() == [[0x87654321], [0x0000000F]]


def test_pack_unpack_all_codes_all_positions():
    # every code in every nibble position: row r, word w holds code ((r + j + w) mod 16) - 8 at nibble j
    N, K = 16, 64
    codes = np.empty((N, K), dtype=np.int8)
    for r in range(N):
        for k in range(K):
            codes[r, k] = ((r + k % 8 + k // 8) % 16) - 8
    qw = oracle.pack_codes(codes)
    for r in range(N):
        for w in range(K // 8):
            word = int(qw[r, w])
            for j in range(8):
                nib = (word >> (4 * j)) & 0xF
                assert (nib - 16 if nib >= 8 else nib) == codes[r, 8 * w + j]
    assert np.array_equal(oracle.unpack_codes(qw, K), codes)


def test_dequant_index_mapping_with_power_of_two_scales():
    # one nonzero code per group; every (row, group) has its own power-of-two scale,
    # so the product lands exactly and any index slip shows up
    N, K = 8, 512
    G = K // 128
    g = synth.rng(3)
    codes = np.zeros((N, K), dtype=np.int8)
    pos = g.integers(0, 128, size=(N, G))
    vals = g.integers(1, 8, size=(N, G)) * np.where(g.random((N, G)) < 0.5, -1, 1)
    for n in range(N):
        for gi in range(G):
            codes[n, gi * 128 + pos[n, gi]] = vals[n, gi]
    exps = (np.arange(N * G).reshape(N, G) % 20) - 14
    scales = (2.0 ** exps).astype(np.float16).view(np.uint16)
    w = oracle.dequantize(oracle.pack_codes(codes), scales, K)
    expect = np.zeros((N, K), dtype=np.float64)
    for n in range(N):
        for gi in range(G):
            expect[n, gi * 128 + pos[n, gi]] = vals[n, gi] * 2.0 ** exps[n, gi]
    assert np.array_equal(w.astype(np.float64), expect)


# ---------------------------------------------------------------- quantiser

def test_quantizer_invariants():
    N, K = 64, 1024
    w = synth.weights(N, K, seed=4)
    w[3, 128:256] = 0.0  # an all-zero group
    qw, sc = oracle.quantize(w)
    codes = oracle.unpack_codes(qw, K).astype(np.float64)
    s = sc.view(np.float16).astype(np.float64)
    G = K // 128
    for n in range(N):
        for gi in range(G):
            grp = w[n, gi * 128:(gi + 1) * 128].astype(np.float64)
            q = codes[n, gi * 128:(gi + 1) * 128]
            a = np.abs(grp).max()
            if a == 0:
                assert s[n, gi] == 0 and np.all(q == 0)
                continue
            # scale is the fp16 rounding of the fp32 quotient max|w|/7
            assert sc[n, gi] == np.float16(np.float32(a) / np.float32(7.0)).view(np.uint16)
            assert np.abs(q).max() == 7
            assert q.min() >= -8 and q.max() <= 7
            assert np.all(np.abs(grp - q * s[n, gi]) <= s[n, gi] / 2 * (1 + 1e-6))


def test_quantizer_roundtrip_of_representable_weights():
    # weights that are exactly q*s with max|q| = 7 per group come back unchanged
    N, K = 32, 512
    codes = np.clip(synth.random_codes(N, K, seed=5), -7, 7)
    codes[:, ::128] = 7
    scales = synth.random_scales_f16(N, K, seed=6)
    w = oracle.dequantize(oracle.pack_codes(codes), scales, K)
    qw, sc = oracle.quantize(w)
    assert np.array_equal(sc, scales)
    assert np.array_equal(oracle.unpack_codes(qw, K), codes)


# ------------------------------------------------------------------ linear

def _bf16_to_f32(b):
    return synth.bf16_bits_to_f32(b)


def test_linear_one_hot_selects_columns_of_x():
    # W[n, perm[n]] = 1 (scale 1): out[m, n] = x[m, perm[n]] exactly
    M, N, K = 5, 256, 256
    g = synth.rng(7)
    perm = g.permutation(K)[:N]
    codes = np.zeros((N, K), dtype=np.int8)
    codes[np.arange(N), perm] = 1
    scales = np.full((N, K // 128), np.float16(1.0)).view(np.uint16)
    x = synth.activations(M, K, seed=8)
    out = oracle.linear(x, oracle.pack_codes(codes), scales)
    assert np.array_equal(out, x[:, perm])


def test_linear_identity_input_gives_dequantized_weight_transposed():
    K = 256
    N = 384
    x = synth.bf16_bits_from_f32(np.eye(K, dtype=np.float32))
    codes = synth.random_codes(N, K, seed=9)
    scales = synth.random_scales_f16(N, K, seed=10)
    qw = oracle.pack_codes(codes)
    out = oracle.linear(x, qw, scales)  # [K, N]
    wt = torch.from_numpy(oracle.dequantize(qw, scales, K).T.copy()).to(torch.bfloat16)
    assert np.array_equal(out, wt.view(torch.int16).numpy().view(np.uint16))


@pytest.mark.parametrize("M,N,K", [(1, 128, 128), (4, 256, 512), (7, 384, 1024)])
def test_linear_matches_torch_fp64_matmul(M, N, K):
    x = synth.activations(M, K, seed=11 + M)
    qw, sc = oracle.quantize(synth.weights(N, K, seed=12 + M))
    out, y = oracle.linear(x, qw, sc, want_y=True)
    w = torch.from_numpy(oracle.dequantize(qw, sc, K)).double()
    xt = torch.from_numpy(_bf16_to_f32(x)).double()
    ref = xt @ w.T
    bound = (xt.abs() @ w.abs().T) * 1e-13
    assert torch.all((torch.from_numpy(y) - ref).abs() <= bound)
    # the output is y rounded once, directly, to bf16 (checked by the definition on every element)
    ref_bf16 = np.array([_bf16_rne_brute_force(v) for v in y.ravel()], dtype=np.uint16).reshape(out.shape)
    assert np.array_equal(out, ref_bf16)


def test_linear_cols_equals_full():
    M, N, K = 3, 256, 256
    x = synth.activations(M, K, seed=13)
    qw, sc = oracle.quantize(synth.weights(N, K, seed=14))
    full = oracle.linear(x, qw, sc)
    cols = np.array([0, 5, 127, 128, 255], dtype=np.int64)
    assert np.array_equal(oracle.linear_cols(x, qw, sc, cols), full[:, cols])


# ------------------------------------------------------------- accept step

def _softmax64(l):
    import scipy.special
    return scipy.special.softmax(l.astype(np.float64), axis=-1)


def test_accept_p_equals_q_accepts_everything():
    B, K, V = 64, 6, 50
    p, q, d, u = synth.accept_seq_case(B, K, V, seed=20)
    q = np.ascontiguousarray(p[:, :K])
    acc, nxt, alpha, margin_alpha, margin_cdf = oracle.spec_accept_seq(p, q, d, u)
    assert np.all(acc == K)
    assert np.all(alpha == 1.0)
    assert np.allclose(margin_alpha, 1.0 - u[:, :K].max(axis=1), rtol=0, atol=1e-15)


def test_accept_alpha_matches_library_softmax():
    B, K, V = 8, 4, 300
    p, q, d, u = synth.accept_seq_case(B, K, V, seed=21)
    u[:, :K] = 0.0  # accept all: every alpha is evaluated
    acc, nxt, alpha, margin_alpha, _ = oracle.spec_accept_seq(p, q, d, u)
    P = _softmax64(p[:, :K])
    Q = _softmax64(q)
    b_idx, i_idx = np.meshgrid(np.arange(B), np.arange(K), indexing="ij")
    ref = np.minimum(1.0, P[b_idx, i_idx, d] / Q[b_idx, i_idx, d])
    assert np.allclose(alpha, ref, rtol=1e-12, atol=0)
    assert np.all(acc == K)
    assert np.allclose(margin_alpha, ref.min(axis=1), rtol=1e-12, atol=0)  # |0 - alpha_i| = alpha_i


NEG = -1000.0  # exp(NEG - max) underflows to exactly 0 in fp64: a token with zero probability


def _rows(*ps):
    """Logit rows whose softmax is exactly the given dyadic distributions: each
    p lists how many tokens share the mass equally (the rest get NEG), e.g. 2
    gives (1/2, 1/2, 0, 0) on V = 4."""
    out = np.full((len(ps), 4), NEG, dtype=np.float32)
    for i, k in enumerate(ps):
        out[i, :k] = 0.0
    return out


def test_accept_margins_exact_on_dyadic_rows():
    """alpha_i = 1, 1/2, 1/4 (target mass 1, 1/2, 1/4 on token 0; draft mass 1
    on token 0). u = (7/8, 3/8, 5/16): accepted, accepted, rejected; the
    smallest |u_i - alpha_i| is 1/16. The residual max(0, P - Q) at the
    rejection is (0, 1/4, 1/4, 1/4), S = 3/4; u_4 = 3/8 gives t = u_4 S = 9/32,
    inside token 2's interval [1/4, 1/2): margin_cdf = (9/32 - 1/4) / S = 1/24."""
    p = _rows(1, 2, 4, 4)[None]
    q = _rows(1, 1, 1)[None]
    d = np.zeros((1, 3), dtype=np.int32)
    u = np.array([[0.875, 0.375, 0.3125, 0.375]], dtype=np.float32)
    acc, nxt, alpha, margin_alpha, margin_cdf = oracle.spec_accept_seq(p, q, d, u)
    assert acc[0] == 2 and nxt[0] == 2
    assert alpha[0].tolist() == [1.0, 0.5, 0.25]
    assert margin_alpha[0] == 0.0625
    assert abs(margin_cdf[0] - 1.0 / 24.0) < 1e-16
    # the same rows, u_4 moved to the upper part of token 2's interval: the
    # nearer end is now the upper one, (1/2 - t) / S with t = (5/8)(3/4)
    u2 = u.copy()
    u2[0, 3] = 0.625
    acc2, nxt2, _, _, margin_cdf2 = oracle.spec_accept_seq(p, q, d, u2)
    assert acc2[0] == 2 and nxt2[0] == 2
    assert abs(margin_cdf2[0] - (0.5 - 0.625 * 0.75) / 0.75) < 1e-16
    # the first decision within 2^-12 of alpha: that is the margin
    u3 = u.copy()
    u3[0, 0] = 1.0 - 2.0 ** -12
    assert oracle.spec_accept_seq(p, q, d, u3)[3][0] == 2.0 ** -12


def test_accept_margin_cdf_of_the_extra_token():
    """All drafts accepted (p == q): the extra token comes from the last target
    row, uniform over 4 tokens; u = 0.5625 puts t 1/16 past token 2's start."""
    p = _rows(1, 4)[None]
    q = _rows(1)[None]
    d = np.zeros((1, 1), dtype=np.int32)
    u = np.array([[0.5, 0.5625]], dtype=np.float32)
    acc, nxt, alpha, margin_alpha, margin_cdf = oracle.spec_accept_seq(p, q, d, u)
    assert acc[0] == 1 and nxt[0] == 2
    assert margin_alpha[0] == 0.5
    assert margin_cdf[0] == 0.0625


def _first_token(acc, nxt, d):
    return np.where(acc > 0, d[:, 0], nxt)


def test_emitted_token_distribution_equals_target():
    """Exactness (section 5 of the tutorial page): the first emitted token is
    distributed as the target's p, whatever the draft q. 10^6 seeded trials on
    V = 8, chi-square."""
    import scipy.stats
    B, K, V = 1_000_000, 2, 8
    g = synth.rng(22)
    pl = (g.standard_normal((K + 1, V)) * 1.5).astype(np.float32)
    ql = (pl[:K] + g.standard_normal((K, V)) * 1.5).astype(np.float32)
    p = np.broadcast_to(pl, (B, K + 1, V)).copy()
    q = np.broadcast_to(ql, (B, K, V)).copy()
    Qd = _softmax64(ql)
    d = np.stack([g.choice(V, size=B, p=Qd[i]) for i in range(K)], axis=1).astype(np.int32)
    u = g.random((B, K + 1), dtype=np.float32)
    acc, nxt, alpha, _, _ = oracle.spec_accept_seq(p, q, d, u)
    P1 = _softmax64(pl[0])
    counts = np.bincount(_first_token(acc, nxt, d), minlength=V)
    stat, pval = scipy.stats.chisquare(counts, B * P1)
    assert pval > 1e-4, (counts, B * P1)
    # acceptance at position 1 happens with probability sum_x min(P, Q) (= 1 - TV)
    beta = np.minimum(P1, Qd[0]).sum()
    rate = np.mean(acc >= 1)
    assert abs(rate - beta) < 5 * math.sqrt(beta * (1 - beta) / B)
    # given acceptance at 1, the second token is again distributed as the target row 2
    sel = acc >= 1
    tok2 = np.where(acc[sel] >= 2, d[sel, 1], nxt[sel])
    P2 = _softmax64(pl[1])
    stat2, pval2 = scipy.stats.chisquare(np.bincount(tok2, minlength=V), sel.sum() * P2)
    assert pval2 > 1e-4


def test_extra_token_after_full_acceptance_follows_last_target_row():
    import scipy.stats
    B, K, V = 400_000, 3, 8
    g = synth.rng(23)
    pl = (g.standard_normal((K + 1, V)) * 1.2).astype(np.float32)
    p = np.broadcast_to(pl, (B, K + 1, V)).copy()
    q = np.ascontiguousarray(p[:, :K])
    d = g.integers(0, V, size=(B, K)).astype(np.int32)
    u = g.random((B, K + 1), dtype=np.float32)
    acc, nxt, _, _, _ = oracle.spec_accept_seq(p, q, d, u)
    assert np.all(acc == K)
    stat, pval = scipy.stats.chisquare(np.bincount(nxt, minlength=V), B * _softmax64(pl[K]))
    assert pval > 1e-4


def test_expected_tokens_per_step_closed_form_and_worked_count():
    """i.i.d. acceptance beta per position gives E[tokens per target call] =
    (1 - beta^(K+1)) / (1 - beta); with K = 5, beta = 0.8 that puts 100 tokens
    at 20-30 target calls (worked count, section 4 of the tutorial page)."""
    fx = json.load(open(os.path.join(GOLDEN, "worked_count.json")))
    K, beta = fx["K"], fx["acceptance"]
    V, B = 4, 400_000
    # target p = (beta, 1 - beta, 0, 0); draft q = (1, 0, 0, 0): sum min(P, Q) = beta
    big = np.float32(60.0)
    pl = np.log(np.array([beta, 1 - beta, 1e-30, 1e-30])).astype(np.float32)
    ql = np.array([big, 0, 0, 0], dtype=np.float32)
    p = np.broadcast_to(pl, (B, K + 1, V)).copy()
    q = np.broadcast_to(ql, (B, K, V)).copy()
    d = np.zeros((B, K), dtype=np.int32)
    u = synth.rng(24).random((B, K + 1), dtype=np.float32)
    acc, nxt, _, _, _ = oracle.spec_accept_seq(p, q, d, u)
    mean_tokens = np.mean(acc + 1)
    expect = (1 - beta ** (K + 1)) / (1 - beta)
    sd = np.std(acc + 1) / math.sqrt(B)
    assert abs(mean_tokens - expect) < 5 * sd
    calls = fx["tokens"] / mean_tokens
    assert fx["calls_min"] <= calls <= fx["calls_max"]
    # after a rejection the corrected distribution max(0, p - q) puts all mass on token 1
    assert np.all(nxt[acc < K] == 1)


# ------------------------------------------------------------------- greedy

def test_greedy_page_example():
    fx = json.load(open(os.path.join(GOLDEN, "g4_greedy_paris.json")))
    V = fx["V"]
    rows = fx["target_argmax_rows"]
    p = np.zeros((1, len(rows), V), dtype=np.float32)
    for i, t in enumerate(rows):
        p[0, i, t] = 5.0
    d = np.array([fx["draft"]], dtype=np.int32)
    acc, nxt = oracle.greedy_chain(p, d)
    assert acc[0] == fx["expected_accepted_len"] and nxt[0] == fx["expected_next_token"]
    # the same case as a tree (a chain: parent[j] = j - 1)
    parents = np.arange(-1, len(rows) - 1, dtype=np.int32)
    dt = np.concatenate([[-1], fx["draft"]]).astype(np.int32)[None]
    acc2, nxt2 = oracle.greedy_tree(p, dt, parents)
    assert acc2[0] == acc[0] and nxt2[0] == nxt[0]


def test_greedy_argmax_ties_take_smallest_index():
    V = 37
    p = np.zeros((3, 2, V), dtype=np.float32)
    p[0, 0, [4, 9, 30]] = 2.0
    p[1, 0, [0, 36]] = 1.0
    p[2, 0, :] = -1.0
    p[:, 1, 7] = 1.0
    d = np.array([[4], [36], [0]], dtype=np.int32)
    acc, nxt = oracle.greedy_chain(p, d)
    assert acc.tolist() == [1, 0, 1]
    assert nxt.tolist() == [7, int(np.argmax(p[1, 0])), 7]


def test_greedy_chain_equals_tree_with_linear_parents():
    B, K, V = 32, 7, 100
    p, d = synth.greedy_chain_case(B, K, V, seed=30, match_prob=0.7)
    acc, nxt = oracle.greedy_chain(p, d)
    parents = np.arange(-1, K, dtype=np.int32)
    dt = np.concatenate([np.full((B, 1), -1, np.int32), d], axis=1)
    acc2, nxt2 = oracle.greedy_tree(p, dt, parents)
    assert np.array_equal(acc, acc2) and np.array_equal(nxt, nxt2)
    assert 0 < acc.mean() < K  # the case exercises partial acceptance


def _brute_force_tree(p, draft, parents):
    """Enumerate every node, walk its root path edge by edge, keep the deepest
    fully matching one (smallest index on ties)."""
    n = len(parents)
    best, best_depth = 0, 0
    for j in range(n):
        path = []
        v = j
        while v != 0:
            path.append(v)
            v = int(parents[v])
        ok = all(int(draft[v]) == int(np.argmax(p[int(parents[v])])) for v in path)
        if ok and len(path) > best_depth:
            best, best_depth = j, len(path)
    return best_depth, int(np.argmax(p[best]))


def test_greedy_tree_brute_force_small_trees():
    g = synth.rng(31)
    for trial in range(300):
        n = int(g.integers(1, 9))
        V = 4
        parents = synth.random_tree_parents(n, max_depth=int(g.integers(1, 6)), g=g)
        p = g.integers(-2, 3, size=(1, n, V)).astype(np.float32)  # many ties
        draft = g.integers(0, V, size=(1, n)).astype(np.int32)
        draft[0, 0] = -1
        acc, nxt = oracle.greedy_tree(p, draft, parents)
        assert (acc[0], nxt[0]) == _brute_force_tree(p[0], draft[0], parents)


def test_greedy_tree_planted_generator_paths():
    B, n, V = 16, 64, 1000
    p, draft, parents = synth.greedy_tree_case(B, n, V, seed=32)
    acc, nxt = oracle.greedy_tree(p, draft, parents)
    for b in range(B):
        assert (acc[b], nxt[b]) == _brute_force_tree(p[b], draft[b], parents[b])
    assert acc.max() >= 2
