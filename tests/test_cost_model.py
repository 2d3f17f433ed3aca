"""Pins of the verify-cost model (host arithmetic, no GPU)."""
import json
import math
import os

import numpy as np
import pytest

import oracle
import synth
from speculative_decode_verify_w4a16_gb300 import cost_model as cm

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
TIMES = {1: 8000.0, 4: 8500.0, 64: 13000.0}  # a made-up verify stack, microseconds


def test_expected_tokens_equals_the_accepted_run_distribution():
    # accepted run j < K has probability alpha^j (1 - alpha), j = K has alpha^K;
    # the target adds one token either way
    for alpha in (0.0, 0.3, 0.7, 0.9, 1.0):
        for K in (0, 1, 4, 8):
            probs = [alpha ** j * (1 - alpha) for j in range(K)] + [alpha ** K]
            assert math.isclose(sum(probs), 1.0)
            mean = sum(p * (j + 1) for j, p in enumerate(probs))
            assert math.isclose(cm.expected_tokens(alpha, K), mean, rel_tol=1e-12, abs_tol=1e-12)
    assert cm.expected_tokens(0.0, 5) == 1.0 and cm.expected_tokens(1.0, 5) == 6.0
    with pytest.raises(ValueError):
        cm.expected_tokens(1.2, 4)


def test_expected_tokens_matches_the_accept_rule_on_the_worked_count():
    """Section 4 of the tutorial page: K = 5 at 80 % acceptance needs 20-30
    target calls for 100 tokens. The oracle's accept rule on a target/draft
    pair with sum min(P, Q) = 0.8 gives the model's tokens per call."""
    fx = json.load(open(os.path.join(GOLDEN, "worked_count.json")))
    K, beta = fx["K"], fx["acceptance"]
    B, V = 200_000, 4
    pl = np.log(np.array([beta, 1 - beta, 1e-30, 1e-30])).astype(np.float32)
    ql = np.array([60.0, 0, 0, 0], dtype=np.float32)  # the draft always proposes token 0
    p = np.broadcast_to(pl, (B, K + 1, V)).copy()
    q = np.broadcast_to(ql, (B, K, V)).copy()
    d = np.zeros((B, K), dtype=np.int32)
    u = synth.rng(31).random((B, K + 1), dtype=np.float32)
    acc, _, _, _, _ = oracle.spec_accept_seq(p, q, d, u)
    tokens = acc + 1
    model = cm.expected_tokens(beta, K)
    assert abs(tokens.mean() - model) < 5 * tokens.std() / math.sqrt(B)
    assert fx["calls_min"] <= fx["tokens"] / model <= fx["calls_max"]


def test_verify_time_interpolates_between_measured_counts_only():
    assert cm.verify_time(TIMES, 1) == 8000.0 and cm.verify_time(TIMES, 64) == 13000.0
    assert cm.verify_time(TIMES, 34) == pytest.approx(8500.0 + 4500.0 * 30 / 60)
    assert cm.verify_time(TIMES, 2) == pytest.approx(8000.0 + 500.0 / 3)
    for m in (0, 65):
        with pytest.raises(ValueError):
            cm.verify_time(TIMES, m)


def test_speedup_relation():
    # plain decoding: one token per decode step and nothing drafted
    assert cm.speedup(1.0, 8000.0, 0.0, 8000.0) == 1.0
    # only ratios matter
    a = cm.speedup(3.2, 9000.0, 400.0, 8000.0)
    assert cm.speedup(3.2, 9.0, 0.4, 8.0) == pytest.approx(a)
    assert a == pytest.approx(3.2 * 8000.0 / 9400.0)
    with pytest.raises(ValueError):
        cm.speedup(1.0, 0.0, 0.0, 1.0)


def test_sequence_tree_and_hierarchical_steps():
    s = cm.sequence_step(TIMES, 0.8, 4, 0.05)
    assert s["verify"] == pytest.approx(cm.verify_time(TIMES, 5))
    assert s["draft"] == pytest.approx(4 * 0.05 * 8000.0)
    assert s["speedup"] == pytest.approx(cm.expected_tokens(0.8, 4) * 8000.0 / (s["verify"] + s["draft"]))
    t = cm.tree_step(TIMES, 4.5, 64, 0.3)
    assert t["speedup"] == pytest.approx(4.5 * 8000.0 / (13000.0 + 2400.0))
    h = cm.hierarchical_step(TIMES, 0.8, 4, 0.3, 0.1)
    # the same target verify as the sequence draft, drafted by tree + intermediate model
    assert h["verify"] == s["verify"] and h["draft"] == pytest.approx(0.4 * 8000.0)


def test_break_even_tau_equalises_the_two_speedups():
    for alpha in (0.7, 0.8, 0.9):
        for K in (4, 8):
            tau = cm.break_even_tau(TIMES, alpha, K, 0.05, 64, 0.3)
            assert cm.tree_step(TIMES, tau, 64, 0.3)["speedup"] == pytest.approx(
                cm.sequence_step(TIMES, alpha, K, 0.05)["speedup"])
    # a verify cost that does not grow with M: the tree breaks even with the
    # sequence's own tokens when both drafts cost the same
    flat = {1: 100.0, 64: 100.0}
    assert cm.break_even_tau(flat, 0.8, 4, 0.0, 64, 0.0) == pytest.approx(cm.expected_tokens(0.8, 4))


def test_table_and_cli(tmp_path):
    rows = cm.table(TIMES)
    assert len(rows) == 6 and {r["K"] for r in rows} == {4, 8}
    line = {"stack_verify_forward": {str(m): {"us": t} for m, t in TIMES.items()} | {"ratio_m64_m1": 1.625}}
    path = tmp_path / "bench.json"
    path.write_text(json.dumps(line) + "\n")
    assert cm.times_from_bench(line) == TIMES
    # the current line's summary and the --detail file
    assert cm.times_from_bench({"summary": {"stack_us": {str(m): t for m, t in TIMES.items()}}}) == TIMES
    assert cm.times_from_bench({"line": {}, "stack": {str(m): {"us": t} for m, t in TIMES.items()}
                                | {"ratio_m64_m1": 1.625}}) == TIMES
    assert cm.main([str(path)]) == 0
