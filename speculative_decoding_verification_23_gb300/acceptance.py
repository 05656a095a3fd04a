"""Acceptance statistics of verification runs (host side, on kernel outputs).

With x_i drawn from the draft distribution q_i, position i of a mentored
verification is accepted with probability

    a_i = sum_v min(q_i(v), pi_i(v)) = 1 - TV(pi_i, q_i) = 1 - max(0, d_i - D),

since pi - q = (1 - theta)(p - q) gives TV(pi, q) = (1 - theta) d and
theta = min(1, D / d) ("What I Gave Up to Make Speculative Decoding Faster",
section "A knob for accepting more draft tokens").  Positions are decided
with independent uniforms, so a round with K drafts accepts j of them with
probability a_0 ... a_{j-1} (1 - a_j), the first rejection ending the round.

`acceptance_report` compares observed accepted counts with these
expectations: per position the rate among the rounds that reached it, and
for every K' <= K the accepted and emitted tokens per round of a round cut
to its first K' drafts (the same uniforms decide the same first K'
positions, so the accepted count of the shorter round is min(accepted, K')).
"""
from __future__ import annotations

import math
from typing import Dict, Iterable, List, Sequence

import numpy as np


def expected_acceptance(d: Sequence[float], D: float) -> np.ndarray:
    """a_i = 1 - max(0, d_i - D) per position."""
    d = np.asarray(d, dtype=np.float64)
    return 1.0 - np.maximum(0.0, d - float(D))


def expected_accepted(a: Sequence[float], K: int) -> float:
    """Expected accepted drafts of a round with the first K positions:
    sum over j = 1..K of a_0 ... a_{j-1}."""
    a = np.asarray(a, dtype=np.float64)[:K]
    return float(np.sum(np.cumprod(a)))


def expected_emitted(a: Sequence[float], K: int, bonus: bool = True) -> float:
    """Expected tokens emitted per round: the accepted drafts plus one token
    (the correction after a rejection, or the bonus after full acceptance;
    without the bonus a fully accepted round adds none)."""
    a = np.asarray(a, dtype=np.float64)[:K]
    full = float(np.prod(a)) if K > 0 else 1.0
    return expected_accepted(a, K) + (1.0 if bonus else 1.0 - full)


def acceptance_report(accepted: Sequence[int], d: Sequence[float], D: float,
                      ks: Iterable[int] = (1, 2, 4, 8)) -> Dict:
    """Observed against expected acceptance over rounds of K = len(d) drafts.

    accepted: accepted drafts of each round (0..K); d: TV of each position
    (rounds that share their rows share d).  Returns per position the rounds
    that reached it, the observed and expected rates and a z-score (binomial
    standard error), and per K' the accepted and emitted tokens per round,
    observed and expected (with and without the bonus)."""
    acc = np.asarray(accepted, dtype=np.int64)
    K = len(d)
    a = expected_acceptance(d, D)
    positions: List[Dict] = []
    for i in range(K):
        reach = int(np.sum(acc >= i))
        passed = int(np.sum(acc >= i + 1))
        rate = passed / reach if reach else float("nan")
        sd = math.sqrt(a[i] * (1.0 - a[i]) / reach) if reach else float("nan")
        z = (rate - a[i]) / sd if reach and sd > 0 else (0.0 if reach and rate == a[i] else float("nan"))
        positions.append(dict(i=i, reached=reach, accepted=passed, rate=rate, expected=float(a[i]), z=z))
    sweep = []
    for k in ks:
        if k > K:
            continue
        cut = np.minimum(acc, k)
        sweep.append(dict(K=int(k),
                          accepted=float(np.mean(cut)),
                          expected_accepted=expected_accepted(a, k),
                          emitted=float(np.mean(cut + 1)),
                          expected_emitted=expected_emitted(a, k, bonus=True),
                          emitted_no_bonus=float(np.mean(cut + (cut < k))),
                          expected_emitted_no_bonus=expected_emitted(a, k, bonus=False)))
    return dict(D=float(D), rounds=int(acc.size), d=[float(x) for x in d], positions=positions, k_sweep=sweep)
