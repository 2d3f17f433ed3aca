"""The lm_head of the verify pass with fused softmax statistics
(w4a16_linear_logits) and the accept step that takes them
(spec_accept_prestat), against the CPU oracle.

The accept rule is the tutorial page's section 3 Steps 3-4 (alpha =
min(1, p/q), first rejection, corrected distribution); p is the softmax of
the target's lm_head logits ("Speculative Decoding Meets Quantization": the
verify forward of the 4-bit target). Accept decisions and emitted tokens must
be bit-exact against the oracle run on the same logits, outside the near-tie
windows of test_accept_gpu.
"""
import numpy as np
import pytest
import torch

import oracle
import speculative_decode_verify_w4a16_gb300 as sv
import synth
from helpers import bf16_to_dev, canon_to_dev, dev

pytestmark = pytest.mark.gpu
NEAR_TIE, NEAR_TIE_CDF = 1e-6, 1e-8


@pytest.fixture(scope="module", autouse=True)
def _built():
    from speculative_decode_verify_w4a16_gb300 import build
    build.build()
    oracle.build()


def _fp32_bound(x, qw, sc, K):
    """Error bound of an fp32 tensor-core sum of the exact bf16 products x_k w_k:
    at most K/16 MMA accumulations (16 products each) and K/128 split-K
    fix-ups chained, each adding at most 2^-22 (one truncated fp32 rounding,
    doubled) of sum_k |x_k w_k|."""
    w = oracle.dequantize(qw, sc, K).astype(np.float64)
    a = np.abs(synth.bf16_bits_to_f32(x).astype(np.float64)) @ np.abs(w).T
    return (K // 16 + K // 128 + 2) * 2.0 ** -22 * a


def _check_logits(got, y, bound, what):
    err = np.abs(got.astype(np.float64) - y)
    worst = float((err / bound).max())
    print(f"{what}: max |err| / bound = {worst:.3g}")
    assert worst <= 1.0, what


def _stats_reference(logits):
    """(max, sum exp(l - max)) per 32-logit slice, in fp64 from the given fp32 logits."""
    l = logits.astype(np.float64).reshape(logits.shape[0], -1, 32)
    mx = l.max(axis=2)
    return mx, np.exp(l - mx[:, :, None]).sum(axis=2)


@pytest.mark.parametrize("M", [1, 4, 9, 16, 40, 80])
def test_logits_and_slice_statistics(M):
    N, K = 1536, 3072  # 12 row tiles, 24 groups: split tiles and a ragged last item
    x = synth.activations(M, K, seed=800 + M)
    qw, sc = oracle.quantize(synth.weights(N, K, seed=801 + M))
    w = sv.prepack(*canon_to_dev(qw, sc))
    logits, stats = sv.linear_logits(bf16_to_dev(x), w)
    torch.cuda.synchronize()
    assert sv.check_device_status() == 0
    got = logits.cpu().numpy()
    _, y = oracle.linear(x, qw, sc, want_y=True)
    _check_logits(got, y, _fp32_bound(x, qw, sc, K), f"M={M}")
    mx, z = _stats_reference(got)
    st = stats.cpu().numpy()
    assert np.array_equal(st[:, :, 0], mx.astype(np.float32))  # the maximum of the same fp32 values
    assert np.allclose(st[:, :, 1], z, rtol=2e-6, atol=0)      # 32 terms, accurate exp, fp32 sum


def _accept_case(B, K, V, hidden, seed, want_oracle_logits=False):
    """Target logits from the fused lm_head of a W ~ N(0, 0.066^2) int4 weight
    (logits ~ N(0, 3^2), the task's accept distribution) and draft = target +
    N(0, 1), draft ids drawn from softmax(q), uniforms U[0, 1)."""
    g = synth.rng(seed)
    x = synth.activations(B * (K + 1), hidden, seed=seed + 1)
    wt = torch.from_numpy(synth.weights(V, hidden, seed=seed + 2, std=0.066)).to(dev())
    qw, sc = sv.quantize(wt)
    del wt
    w = sv.prepack(qw, sc)
    logits, stats = sv.linear_logits(bf16_to_dev(x), w)
    torch.cuda.synchronize()
    p = logits.cpu().numpy().reshape(B, K + 1, V)
    q = (p[:, :K] + g.standard_normal((B, K, V), dtype=np.float32)).astype(np.float32)
    d = synth.gumbel_max_sample(q, g)
    u = g.random((B, K + 1), dtype=np.float32)
    out = [logits.view(B, K + 1, V), stats.view(B, K + 1, V // 32, 2), p, np.ascontiguousarray(q), d, u]
    if want_oracle_logits:
        _, y = oracle.linear(x, qw.cpu().numpy().view(np.uint32), sc.cpu().numpy().view(np.uint16), want_y=True)
        out.append(y.reshape(B, K + 1, V))
    return out


@pytest.mark.parametrize("B,K,V,hidden", [(16, 4, 128256, 2048), (8, 7, 32768, 1024), (3, 1, 4096, 1024)])
def test_fused_accept_matches_oracle(B, K, V, hidden):
    logits, stats, p, q, d, u = _accept_case(B, K, V, hidden, seed=810 + K)
    qt, dt, ut = (torch.from_numpy(a).to(dev()) for a in (q, d, u))
    acc, nxt = sv.spec_accept_prestat(logits, stats, dt, qt, ut)
    torch.cuda.synchronize()
    assert sv.check_device_status() == 0
    acc, nxt = acc.cpu().numpy(), nxt.cpu().numpy()
    acc_r, nxt_r, _, margin_alpha, margin_cdf = oracle.spec_accept_seq(p, q, d, u)
    tie = (margin_alpha < NEAR_TIE) | (margin_cdf < NEAR_TIE_CDF)
    bad = ((acc != acc_r) | (nxt != nxt_r)) & ~tie
    print(f"B={B} K={K} V={V}: {int(tie.sum())} near-ties; mean accepted {acc_r.mean():.2f}")
    assert not bad.any(), np.nonzero(bad)[0][:10]
    # the unfused accept on the same logits makes the same decisions
    acc2, nxt2 = sv.spec_accept(logits.contiguous(), dt, q_logits=qt, uniforms=ut)
    torch.cuda.synchronize()
    same = (acc2.cpu().numpy() == acc) & (nxt2.cpu().numpy() == nxt)
    assert np.all(same | tie)


@pytest.mark.parametrize("B,K,V,hidden", [(16, 4, 4096, 1024), (3, 1, 4096, 1024)])
def test_fused_accept_matches_oracle_on_oracle_logits(B, K, V, hidden):
    """The fused path's decisions against the oracle's accept on the oracle's
    own lm_head (fp64 sums rounded to fp32). The two logit sets differ by the
    GPU's fp32 accumulation, at most delta; alpha = P(d) / Q(d) then moves by
    a factor within exp(+-2 delta) and a CDF boundary, relative to the sum,
    by about 4 delta, so rows within those distances of a decision (plus the
    usual near-tie windows) are excluded. A draw's CDF interval is about 1/V
    wide, so the vocabulary is kept small enough (4096) that few rows fall
    inside the 8 delta window."""
    logits, stats, p, q, d, u, y = _accept_case(B, K, V, hidden, seed=840 + K, want_oracle_logits=True)
    delta = float(np.abs(p.astype(np.float64) - y).max())
    assert delta < 1e-4, delta
    qt, dt, ut = (torch.from_numpy(a).to(dev()) for a in (q, d, u))
    acc, nxt = sv.spec_accept_prestat(logits, stats, dt, qt, ut)
    torch.cuda.synchronize()
    assert sv.check_device_status() == 0
    acc_r, nxt_r, _, margin_alpha, margin_cdf = oracle.spec_accept_seq(y.astype(np.float32), q, d, u)
    tie = (margin_alpha < NEAR_TIE + 4 * delta) | (margin_cdf < NEAR_TIE_CDF + 8 * delta)
    bad = ((acc.cpu().numpy() != acc_r) | (nxt.cpu().numpy() != nxt_r)) & ~tie
    print(f"B={B} K={K} V={V}: logits differ by <= {delta:.2e}; {int(tie.sum())} rows within the windows")
    assert not bad.any(), np.nonzero(bad)[0][:10]
    assert tie.sum() <= max(1, B // 4)


def test_llama70b_lm_head_fused_sampled():
    """The Llama-3-70B lm_head (8192 -> 128256) at the accept configuration's
    80 verify positions (B = 16, K = 4), checked on sampled vocabulary columns."""
    M, K, N = 80, 8192, 128256
    wt = torch.from_numpy(synth.weights(N, K, seed=820)).to(dev())
    qw, sc = sv.quantize(wt)
    del wt
    w = sv.prepack(qw, sc)
    x = synth.activations(M, K, seed=821)
    logits, stats = sv.linear_logits(bf16_to_dev(x), w)
    torch.cuda.synchronize()
    assert sv.check_device_status() == 0
    g = synth.rng(822)
    cols = np.unique(np.concatenate([np.arange(0, 128), np.arange(N - 128, N), g.integers(0, N, 256)]))
    qw_h = qw.cpu().numpy().view(np.uint32)
    sc_h = sc.cpu().numpy().view(np.uint16)
    _, y = oracle.linear_cols(x, qw_h, sc_h, cols, want_y=True)
    _check_logits(logits.cpu().numpy()[:, cols], y, _fp32_bound(x, qw_h[cols], sc_h[cols], K), "lm_head M=80")
    lg = logits.cpu().numpy()
    mx, z = _stats_reference(lg)
    st = stats.cpu().numpy()
    assert np.array_equal(st[:, :, 0], mx.astype(np.float32))
    assert np.allclose(st[:, :, 1], z, rtol=2e-6, atol=0)


@pytest.mark.parametrize("M", [5, 80])
def test_logits_not_16_byte_aligned(M):
    """Logits that start 4 bytes past a 16-byte boundary take the per-element
    store path (tiles are otherwise written by TMA stores): the same values,
    and the floats around the output untouched."""
    N, K = 640, 2048
    x = synth.activations(M, K, seed=830 + M)
    qw, sc = oracle.quantize(synth.weights(N, K, seed=831 + M))
    w = sv.prepack(*canon_to_dev(qw, sc))
    xd = bf16_to_dev(x)
    ref, ref_stats = sv.linear_logits(xd, w)
    buf = torch.full((M * N + 8,), 7.0, dtype=torch.float32, device=dev())
    logits = buf[1:1 + M * N].view(M, N)
    assert logits.data_ptr() % 16 == 4
    _, stats = sv.linear_logits(xd, w, logits=logits)
    torch.cuda.synchronize()
    assert sv.check_device_status() == 0
    assert torch.equal(logits, ref) and torch.equal(stats, ref_stats)
    assert buf[0].item() == 7.0 and torch.all(buf[1 + M * N:] == 7.0)
