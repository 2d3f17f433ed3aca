"""Verify-cost model of one speculative step on a 4-bit-weight target.

Host arithmetic only. It combines the measured time of the target's verify
forward at M tokens (this library's W4A16 linears over the 80-layer stack, as
bench.py reports it) with two facts from the pages:

* the speedup relation of the tutorial page "Speculative Decoding이란?"
  (closing summary): speedup ~ accepted tokens per verification divided by
  (verification cost + draft cost), the costs in units of one plain decode step;
* the tokens one verification yields under the acceptance rule (same page,
  section 3 Steps 3-4; section 4's worked count: K = 5 at 80 % acceptance
  needs 20-30 target calls for 100 tokens).

With these it compares the verify shapes that "Speculative Decoding Meets
Quantization" weighs on a 4-bit target (abstract; "The Compatibility
Problem"; "The Hierarchical Framework"): a sequence draft of K tokens
(verify at M = K + 1), a tree draft of `nodes` tokens (verify at M = nodes),
and the hierarchical scheme, in which an intermediate model turns the tree
draft into a sequence draft so that the target verifies M = K + 1 tokens.

Readings (the pages give no cost model):
* Draft tokens are accepted independently with probability alpha, so the
  accepted run of a K-token sequence draft is geometric truncated at K, and
  the target always adds one token (the corrected draw or the extra token).
* The verify time is read at measured token counts (bench.py measures the
  stack at M = 1, 4, 5, 9, 16, 32, 48, 64, i.e. at K + 1 for K = 4 and 8 and at
  the tree sizes); between two measured counts it is interpolated linearly
  (used only for counts the bench did not measure), never extrapolated.
* A tree draft's tokens per verification (tau) depends on the drafter and the
  tree, which no synthetic input fixes, so the model reports the break-even
  tau: what the tree must yield to match a sequence draft.

Usage: python -m speculative_decode_verify_w4a16_gb300.cost_model BENCH.json
(one JSON line of bench.py with its stack figures, or the file bench.py
--detail writes).
"""
from __future__ import annotations

import argparse
import json
import math
from typing import Mapping


def expected_tokens(alpha: float, K: int) -> float:
    """Mean tokens per verification of a K-token sequence draft whose tokens
    are each accepted with probability alpha: sum_{j=0..K} alpha^j, i.e.
    (1 - alpha^(K+1)) / (1 - alpha), and K + 1 at alpha = 1."""
    if not 0.0 <= alpha <= 1.0 or K < 0:
        raise ValueError("alpha must lie in [0, 1] and K must be >= 0")
    if alpha == 1.0:
        return float(K + 1)
    return (1.0 - alpha ** (K + 1)) / (1.0 - alpha)


def verify_time(times: Mapping[int, float], M: int) -> float:
    """Verify-forward time at M tokens from measured {M: time}, linear between
    the two nearest measured token counts. Raises ValueError outside them."""
    ms = sorted(int(m) for m in times)
    if not ms or M < ms[0] or M > ms[-1]:
        raise ValueError(f"M = {M} outside the measured token counts {ms}")
    t = {int(m): float(v) for m, v in times.items()}
    if M in t:
        return t[M]
    hi = next(m for m in ms if m > M)
    lo = max(m for m in ms if m < M)
    return t[lo] + (t[hi] - t[lo]) * (M - lo) / (hi - lo)


def speedup(tokens: float, verify: float, draft: float, decode: float) -> float:
    """Tokens per verification times the plain decode time, over the time of
    one speculative step (verification + drafting)."""
    if verify <= 0 or draft < 0 or decode <= 0:
        raise ValueError("times must be positive (draft may be 0)")
    return tokens * decode / (verify + draft)


def sequence_step(times: Mapping[int, float], alpha: float, K: int, draft_per_token: float) -> dict:
    """A K-token sequence draft: the drafter runs K steps of `draft_per_token`
    (in units of one plain decode step), the target verifies M = K + 1."""
    decode = verify_time(times, 1)
    verify = verify_time(times, K + 1)
    draft = K * draft_per_token * decode
    tokens = expected_tokens(alpha, K)
    return {"tokens": tokens, "verify": verify, "draft": draft, "speedup": speedup(tokens, verify, draft, decode)}


def tree_step(times: Mapping[int, float], tau: float, nodes: int, draft_cost: float) -> dict:
    """A tree draft of `nodes` tokens yielding tau tokens per verification;
    drafting costs `draft_cost` plain decode steps; the target verifies M = nodes."""
    decode = verify_time(times, 1)
    verify = verify_time(times, nodes)
    draft = draft_cost * decode
    return {"tokens": tau, "verify": verify, "draft": draft, "speedup": speedup(tau, verify, draft, decode)}


def hierarchical_step(times: Mapping[int, float], alpha: float, K: int, tree_draft_cost: float,
                      intermediate_cost: float) -> dict:
    """The hierarchical scheme: a tree drafter (`tree_draft_cost` decode steps)
    and an intermediate model that checks the tree (`intermediate_cost`)
    hand the target a K-token sequence accepted token by token with
    probability alpha; the target verifies M = K + 1."""
    decode = verify_time(times, 1)
    verify = verify_time(times, K + 1)
    draft = (tree_draft_cost + intermediate_cost) * decode
    tokens = expected_tokens(alpha, K)
    return {"tokens": tokens, "verify": verify, "draft": draft, "speedup": speedup(tokens, verify, draft, decode)}


def break_even_tau(times: Mapping[int, float], alpha: float, K: int, draft_per_token: float, nodes: int,
                   tree_draft_cost: float) -> float:
    """Tokens per verification a `nodes`-token tree draft must yield to match
    the speedup of a K-token sequence draft at acceptance alpha."""
    seq = sequence_step(times, alpha, K, draft_per_token)
    decode = verify_time(times, 1)
    return seq["speedup"] * (verify_time(times, nodes) + tree_draft_cost * decode) / decode


def table(times: Mapping[int, float], alphas=(0.7, 0.8, 0.9), Ks=(4, 8), draft_per_token: float = 0.05,
          nodes: int = 64, tree_draft_cost: float = 0.3) -> list[dict]:
    """Sequence-draft speedup and the tree's break-even tau for each (alpha, K)
    that the measured token counts cover (acceptance 70-90 % and draft length
    4-8 are the tutorial's typical values, section 7)."""
    rows = []
    ms = sorted(int(m) for m in times)
    for K in Ks:
        if K + 1 > ms[-1] or nodes > ms[-1]:
            continue
        for a in alphas:
            s = sequence_step(times, a, K, draft_per_token)
            rows.append({"alpha": a, "K": K, "tokens": round(s["tokens"], 3),
                         "verify_over_decode": round(s["verify"] / verify_time(times, 1), 3),
                         "speedup_sequence": round(s["speedup"], 3),
                         "tree_verify_over_decode": round(verify_time(times, nodes) / verify_time(times, 1), 3),
                         "break_even_tau": round(break_even_tau(times, a, K, draft_per_token, nodes, tree_draft_cost), 3)})
    return rows


def times_from_bench(line: Mapping) -> dict[int, float]:
    """{M: microseconds} of the verify stack from a bench.py JSON line
    (summary.stack_us), the --detail file (stack) or an older line
    (stack_verify_forward)."""
    if "line" in line and isinstance(line.get("stack"), Mapping):
        st = {k: v["us"] for k, v in line["stack"].items() if isinstance(v, Mapping)}
    elif "summary" in line and "stack_us" in line["summary"]:
        st = line["summary"]["stack_us"]
    else:
        st = {k: v["us"] for k, v in line["stack_verify_forward"].items() if isinstance(v, Mapping)}
    out = {int(k): float(v) for k, v in st.items() if str(k).isdigit()}
    if 1 not in out:
        raise ValueError("the bench line has no M = 1 stack time")
    if any(not math.isfinite(v) or v <= 0 for v in out.values()):
        raise ValueError("stack times must be positive")
    return out


def main(argv=None) -> int:
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("bench_json", help="file holding one bench.py JSON line")
    ap.add_argument("--draft-per-token", type=float, default=0.05,
                    help="sequence drafter cost per drafted token, in plain decode steps")
    ap.add_argument("--tree-draft-cost", type=float, default=0.3,
                    help="cost of drafting one tree, in plain decode steps")
    ap.add_argument("--nodes", type=int, default=64)
    args = ap.parse_args(argv)
    with open(args.bench_json) as f:
        text = f.read()
    try:
        line = json.loads(text)
    except json.JSONDecodeError:
        line = json.loads(text.splitlines()[0])
    times = times_from_bench(line)
    print(json.dumps({"verify_us": times, "rows": table(times, draft_per_token=args.draft_per_token,
                                                       nodes=args.nodes, tree_draft_cost=args.tree_draft_cost)}))
    return 0


if __name__ == "__main__":
    raise SystemExit(main())
