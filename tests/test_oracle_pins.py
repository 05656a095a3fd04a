"""Pins for the CPU oracle: values the pages print, closed forms, invariants,
library routines and brute force on tiny inputs.  No GPU."""
import json
import math
import os

import numpy as np
import pytest
import scipy.special
import scipy.stats

import oracle
from oracle import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _logits(p):
    return np.log(np.asarray(p, dtype=np.float64)).astype(np.float32)


def _grid(n):
    return ((np.arange(n) + 0.5) / n).astype(np.float32)


def _one(zt, zd, x, u, D, T=1.0, alpha=1.0, top_p=1.0, hist=()):
    return O.verify_request(np.asarray(zt), np.asarray(zd), np.asarray(x), np.asarray(hist, dtype=np.int64),
                            T, alpha, top_p, D, np.asarray(u, dtype=np.float32))


# --------------------------------------------------------------------------
# The worked example (Speculative Decoding note, "Warum eine Korrektur ...")
# --------------------------------------------------------------------------

def _output_distribution(p, q, D, n_accept=3000, n_fin=3000):
    """Exact stratified integration of the oracle's first emitted token with
    x ~ q (weights q(x)) and midpoint grids over u_0 and u_fin."""
    zt = np.stack([_logits(p), _logits(p)])
    zd = _logits(q)[None, :]
    V = len(p)
    acc_mass = np.zeros(V)
    for x in range(V):
        n_acc = sum(_one(zt, zd, [x], [u, 0.5], D)["accepted"] == 1 for u in _grid(n_accept))
        acc_mass[x] = q[x] * n_acc / n_accept
    # the correction distribution: force a rejection at a token with pi/q < 1
    res = _one(zt, zd, [0], [0.0, 0.5], D)
    ratio = [(1 - res["theta"][0]) * p[v] / q[v] + res["theta"][0] for v in range(V)]
    xr = int(np.argmin(ratio))
    assert ratio[xr] < 0.99
    corr = np.zeros(V)
    for u in _grid(n_fin):
        r = _one(zt, zd, [xr], [0.999, u], D)
        assert r["accepted"] == 0
        corr[r["tokens"][0]] += 1
    corr /= n_fin
    return acc_mass, corr, acc_mass + (1 - acc_mass.sum()) * corr


def test_worked_example_lossless():
    g = _load("worked_example.json")
    p, q = np.array(g["p"]), np.array(g["q"])
    acc, corr, out = _output_distribution(p, q, D=0.0)
    np.testing.assert_allclose(acc, g["accepted_mass"], atol=1e-4)
    assert abs((1 - acc.sum()) - g["remaining_mass"]) < 1e-4
    np.testing.assert_allclose(corr, g["remaining_split"], atol=1e-4)
    np.testing.assert_allclose(out, p, atol=2e-4)
    # the naive correction drawn from p itself would give a different output
    naive = acc + (1 - acc.sum()) * p
    np.testing.assert_allclose(naive, g["naive_correction_from_p"], atol=2e-4)
    assert np.max(np.abs(out - np.array(g["naive_correction_from_p"]))) > 0.05


def test_worked_example_mentored_budget():
    """Derived closed forms for the same rows: TV = 0.4; D = 0.2 gives
    theta = 0.5 and pi = [0.4, 0.4, 0.2]; the output follows pi."""
    g = _load("worked_example.json")
    p, q = np.array(g["p"]), np.array(g["q"])
    zt = np.stack([_logits(p), _logits(p)])
    zd = _logits(q)[None, :]
    r = _one(zt, zd, [0], [0.5, 0.5], D=0.2)
    assert abs(r["tv"][0] - 0.4) < 1e-6
    assert abs(r["theta"][0] - 0.5) < 1e-5
    _, _, out = _output_distribution(p, q, D=0.2)
    np.testing.assert_allclose(out, [0.4, 0.4, 0.2], atol=2e-4)


# --------------------------------------------------------------------------
# Endpoints of the TV budget (mentored decoding section)
# --------------------------------------------------------------------------

def _random_rows(rng, V, K, scale=2.0):
    zt = (scale * rng.standard_normal((K + 1, V))).astype(np.float32)
    zd = (scale * rng.standard_normal((K, V))).astype(np.float32)
    return zt, zd


def test_budget_zero_uses_p_exactly():
    rng = np.random.default_rng(1)
    for _ in range(50):
        V, K = 7, 3
        zt, zd = _random_rows(rng, V, K)
        x = rng.integers(0, V, K)
        u = rng.random(K + 1).astype(np.float32)
        r = _one(zt, zd, x, u, D=0.0, T=0.9)
        for i in range(K):
            assert r["theta"][i] == 0.0 or r["tv"][i] == 0.0
            want = float(u[i]) * r["q_x"][i] < r["p_x"][i]
            assert r["accept"][i] == want


def test_budget_one_accepts_everything():
    rng = np.random.default_rng(2)
    for _ in range(50):
        V, K = 9, 4
        zt, zd = _random_rows(rng, V, K, 4.0)
        x = rng.integers(0, V, K)
        u = rng.random(K + 1).astype(np.float32)
        r = _one(zt, zd, x, u, D=1.0, T=0.8, alpha=1.3, hist=[1, 2, 2])
        assert r["theta"] == [1.0] * K
        assert r["accepted"] == K
        assert r["tokens"][:K] == [int(t) for t in x]
        assert 0 <= r["tokens"][K] < V


def test_equal_distributions_never_reject():
    rng = np.random.default_rng(3)
    for D in (0.0, 0.3, 1.0):
        for _ in range(20):
            V, K = 6, 3
            zt, _ = _random_rows(rng, V, K)
            zd = zt[:K].copy()
            x = rng.integers(0, V, K)
            u = rng.random(K + 1).astype(np.float32)
            r = _one(zt, zd, x, u, D=D, T=0.7)
            assert r["tv"] == [0.0] * K and r["theta"] == [1.0] * K
            assert r["accepted"] == K


# --------------------------------------------------------------------------
# Closed form of the acceptance probability: sum_v min(q, pi) = 1 - max(0, d - D)
# --------------------------------------------------------------------------

@pytest.mark.parametrize("D", [0.0, 0.1, 0.25, 0.6])
def test_acceptance_probability_closed_form(D):
    rng = np.random.default_rng(int(D * 100) + 7)
    V = 6
    p = scipy.special.softmax(rng.standard_normal(V) * 1.5)
    q = scipy.special.softmax(rng.standard_normal(V) * 1.5)
    zt = np.stack([_logits(p), _logits(p)])
    zd = _logits(q)[None, :]
    n = 4000
    prob = 0.0
    for x in range(V):
        n_acc = sum(_one(zt, zd, [x], [u, 0.5], D)["accepted"] == 1 for u in _grid(n))
        prob += q[x] * n_acc / n
    d = 0.5 * np.abs(p - q).sum()
    assert abs(prob - (1 - max(0.0, d - D))) < 2.5e-4 * V


# --------------------------------------------------------------------------
# Chi-square: first emitted token ~ pi_0, with x drawn by an independent sampler
# --------------------------------------------------------------------------

def _first_token_counts(rng, p_rows_logits, q_rows_logits, D, n, T=1.0):
    V = p_rows_logits.shape[1]
    K = q_rows_logits.shape[0]
    q0 = scipy.special.softmax(q_rows_logits.astype(np.float64) / T, axis=1)
    counts = np.zeros(V, dtype=np.int64)
    for _ in range(n):
        x = np.array([rng.choice(V, p=q0[i]) for i in range(K)])
        u = rng.random(K + 1).astype(np.float32)
        r = _one(p_rows_logits, q_rows_logits, x, u, D, T=T)
        counts[r["tokens"][0]] += 1
    return counts


def _pi0(zt, zd, D, T=1.0):
    p = scipy.special.softmax(zt[0].astype(np.float64) / T)
    q = scipy.special.softmax(zd[0].astype(np.float64) / T)
    d = 1.0 - np.minimum(p, q).sum()          # TV by an independent identity
    th = 1.0 if d <= D else D / d
    return (1 - th) * p + th * q


@pytest.mark.parametrize("V,K,D", [(3, 1, 0.0), (5, 2, 0.25), (8, 1, 0.5), (5, 1, 0.1)])
def test_chi_square_first_token(V, K, D):
    rng = np.random.default_rng(100 + V * 10 + K)
    zt = (1.5 * rng.standard_normal((K + 1, V))).astype(np.float32)
    zd = (1.5 * rng.standard_normal((K, V))).astype(np.float32)
    n = 12000
    counts = _first_token_counts(rng, zt, zd, D, n, T=0.9)
    pi = _pi0(zt, zd, D, T=0.9)
    _, pval = scipy.stats.chisquare(counts, pi * n)
    assert pval > 1e-3, (counts, pi * n)


def test_chi_square_detects_naive_correction(monkeypatch):
    """Negative control: plant the naive correction (draw from p, not from the
    residual) in the oracle; the same chi-square must reject it."""
    monkeypatch.setattr(O, "residual", lambda p, q: p.copy())
    rng = np.random.default_rng(5)
    V, K, D = 3, 1, 0.0
    p = np.array([0.2, 0.5, 0.3])
    q = np.array([0.6, 0.3, 0.1])
    zt = np.stack([_logits(p), _logits(p)])
    zd = _logits(q)[None, :]
    n = 12000
    counts = _first_token_counts(rng, zt, zd, D, n)
    _, pval = scipy.stats.chisquare(counts, p * n)
    assert pval < 1e-6


# --------------------------------------------------------------------------
# Brute force on a tiny case: the joint law of the emitted sequence, K = 2
# --------------------------------------------------------------------------

def test_joint_sequence_law_brute_force():
    rng = np.random.default_rng(11)
    V, K, D, T, N = 3, 2, 0.3, 1.0, 12
    zt = (1.5 * rng.standard_normal((K + 1, V))).astype(np.float32)
    zd = (1.5 * rng.standard_normal((K, V))).astype(np.float32)
    x = [int(np.argmax(zd[0])), int(np.argmax(zd[1]))]
    g = _grid(N)
    seen = {}
    for u0 in g:
        for u1 in g:
            for uf in g:
                r = _one(zt, zd, x, [u0, u1, uf], D, T=T)
                seq = tuple(t for t in r["tokens"] if t >= 0)
                seen[seq] = seen.get(seq, 0) + 1
    # the expected grid counts, computed independently with scipy
    P = scipy.special.softmax(zt.astype(np.float64) / T, axis=1)
    Q = scipy.special.softmax(zd.astype(np.float64) / T, axis=1)

    def frac_below(a):   # grid points u with u < a
        return int(np.sum(g.astype(np.float64) < a))

    def frac_in(w, v):   # grid points landing on token v under inverse CDF
        c = np.cumsum(w) / w.sum()
        lo = c[v - 1] if v else 0.0
        return int(np.sum((g >= lo) & (g < c[v])))

    want = {}
    a, res = [], []
    for i in range(K):
        d = 1 - np.minimum(P[i], Q[i]).sum()
        th = 1.0 if d <= D else D / d
        pi = (1 - th) * P[i] + th * Q[i]
        a.append(frac_below(pi[x[i]] / Q[i][x[i]]))
        res.append(np.maximum(P[i] - Q[i], 0))
    for v in range(V):
        want[(v,)] = (N - a[0]) * N * frac_in(res[0], v)
        want[(x[0], v)] = want.get((x[0], v), 0) + a[0] * (N - a[1]) * frac_in(res[1], v)
        want[(x[0], x[1], v)] = a[0] * a[1] * frac_in(P[2], v)
    want = {k: c for k, c in want.items() if c}
    assert seen == want


# --------------------------------------------------------------------------
# Building blocks against library routines and independent identities
# --------------------------------------------------------------------------

def test_softmax_matches_scipy():
    rng = np.random.default_rng(21)
    for V in (1, 2, 17, 1000):
        z = rng.standard_normal(V) * 5
        np.testing.assert_allclose(O.softmax(z), scipy.special.softmax(z), rtol=1e-12, atol=1e-15)


def test_tv_identities():
    rng = np.random.default_rng(22)
    for _ in range(20):
        p = scipy.special.softmax(rng.standard_normal(50) * 3)
        q = scipy.special.softmax(rng.standard_normal(50) * 3)
        d = O.tv_distance(p, q)
        assert abs(d - (1.0 - np.minimum(p, q).sum())) < 1e-12
        assert abs(d - np.maximum(p - q, 0).sum()) < 1e-12
    assert O.tv_distance(p, p) == 0.0


def test_theta_rule():
    assert O.mentored_theta(0.0, 0.0) == 1.0       # d = 0 -> theta = 1
    assert O.mentored_theta(0.4, 0.2) == pytest.approx(0.5, rel=1e-7)
    assert O.mentored_theta(0.3, 0.5) == 1.0
    assert O.mentored_theta(0.7, 1.0) == 1.0
    assert O.mentored_theta(0.5, 0.0) == 0.0


def _top_p_brute(p, top_p):
    """The largest threshold among the distinct values whose kept mass
    reaches top_p; keep everything at or above it."""
    best = None
    for tau in sorted(set(p.tolist()), reverse=True):
        if p[p >= tau].sum() >= top_p:
            best = tau
            break
    keep = p >= best
    out = np.where(keep, p, 0.0)
    return out / out.sum()


def test_top_p_hand_cases():
    p = np.array([0.5, 0.3, 0.2])
    out, _ = O.top_p_filter(p, np.float32(0.75))
    np.testing.assert_allclose(out, [0.625, 0.375, 0.0])
    out, _ = O.top_p_filter(p, np.float32(0.85))
    np.testing.assert_allclose(out, p)
    out, _ = O.top_p_filter(np.array([0.4, 0.3, 0.3]), np.float32(0.5))
    np.testing.assert_allclose(out, [0.4, 0.3, 0.3])   # ties at tau are kept
    out, _ = O.top_p_filter(p, np.float32(1.0))
    np.testing.assert_allclose(out, p)


def test_top_p_matches_brute_force():
    rng = np.random.default_rng(23)
    for _ in range(200):
        V = int(rng.integers(1, 12))
        z = np.round(rng.standard_normal(V) * 2, 1)     # repeated values -> ties
        p = scipy.special.softmax(z)
        tp = float(np.float32(rng.uniform(0.05, 1.0)))
        out, _ = O.top_p_filter(p, tp)
        np.testing.assert_allclose(out, _top_p_brute(p, tp), rtol=1e-12, atol=1e-15)


def test_repetition_penalty_hand_case():
    z = np.array([2.0, -2.0, 1.0, 0.5, 0.0], dtype=np.float32)
    out = O.apply_repetition_penalty(z, O.penalty_set([0, 1, 1], [4]), 2.0)
    np.testing.assert_array_equal(out, np.array([1.0, -4.0, 1.0, 0.5, 0.0], dtype=np.float32))
    out = O.apply_repetition_penalty(z, [0, 1, 2], 1.0)
    np.testing.assert_array_equal(out, z)
    # fp32 rounding of the division, as the kernels do it
    out = O.apply_repetition_penalty(np.array([1.0], np.float32), [0], 1.1)
    assert out[0] == np.float32(np.float32(1.0) / np.float32(1.1))


def test_inverse_cdf_grid_frequencies():
    w = np.array([0.0, 0.25, 0.0, 0.5, 0.25])
    n = 4000
    counts = np.zeros(5)
    for u in _grid(n):
        v, _ = O.inverse_cdf(w, u)
        counts[v] += 1
    np.testing.assert_allclose(counts / n, w / w.sum(), atol=1 / n)
    assert counts[0] == 0 and counts[2] == 0


def test_inverse_cdf_unnormalised_and_edges():
    w = np.array([0.0, 3.0, 1.0])
    assert O.inverse_cdf(w, 0.0)[0] == 1
    assert O.inverse_cdf(w, np.float32(0.74))[0] == 1
    assert O.inverse_cdf(w, np.float32(0.76))[0] == 2
    assert O.inverse_cdf(w, np.float32(1 - 2 ** -24))[0] == 2


# --------------------------------------------------------------------------
# Greedy longest-prefix verification (Adaptive-SpecDecode-Lab, implementation)
# --------------------------------------------------------------------------

def test_greedy_argmax_matches_numpy_with_ties():
    rng = np.random.default_rng(31)
    for _ in range(100):
        V, K = 20, 3
        zt = rng.integers(-3, 4, size=(K + 1, V)).astype(np.float32)   # many exact ties
        x = rng.integers(0, V, K)
        r = O.greedy_request(zt, x, np.zeros(0, np.int64), 1.0)
        assert r["argmax"][0] == int(np.argmax(zt[0]))
        j = r["accepted"]
        assert all(r["argmax"][i] == x[i] for i in range(j))
        assert j == K or r["argmax"][j] != x[j]


def test_greedy_full_match_emits_bonus_and_mismatch_emits_correction():
    V, K = 10, 3
    zt = np.zeros((K + 1, V), np.float32)
    for i, t in enumerate([4, 7, 1, 9]):
        zt[i, t] = 5.0
    r = O.greedy_request(zt, np.array([4, 7, 1]), np.zeros(0, np.int64), 1.0)
    assert r["accepted"] == 3 and r["tokens"] == [4, 7, 1, 9]
    r = O.greedy_request(zt, np.array([3, 7, 1]), np.zeros(0, np.int64), 1.0)
    assert r["accepted"] == 0 and r["tokens"] == [4, -1, -1, -1]
    r = O.greedy_request(zt, np.array([4, 7, 2]), np.zeros(0, np.int64), 1.0)
    assert r["accepted"] == 2 and r["tokens"] == [4, 7, 1, -1]


def test_greedy_penalty_changes_argmax():
    V = 6
    zt = np.array([[3.0, 2.9, 0, 0, 0, 0], [0, 0, 0, 4.0, 3.9, 0]], np.float32)
    # history holds token 0: 3.0/1.1 < 2.9, so token 1 wins row 0
    r = O.greedy_request(zt, np.array([1]), np.array([0]), 1.1)
    assert r["argmax"][0] == 1 and r["accepted"] == 1
    # the accepted draft (token 1) is penalised in row 1 only if it matters: token 3 stays
    assert r["tokens"] == [1, 3]


# --------------------------------------------------------------------------
# Status handling
# --------------------------------------------------------------------------

def test_invalid_requests_get_status_and_minus_one():
    V, K = 8, 2
    zt = np.zeros((K + 1, V), np.float32)
    zd = np.zeros((K, V), np.float32)
    u = np.full(K + 1, 0.5, np.float32)
    r = _one(zt, zd, [0, 9], u, D=0.5)
    assert r["status"] & O.STATUS_BAD_TOKEN and r["tokens"] == [-1] * 3 and r["accepted"] == -1
    r = _one(zt, zd, [0, 1], u, D=0.5, T=0.0)
    assert r["status"] & O.STATUS_BAD_PARAM
    r = _one(zt, zd, [0, 1], u, D=1.5)
    assert r["status"] & O.STATUS_BAD_PARAM
    r = _one(zt, zd, [0, 1], u, D=0.5, top_p=0.0)
    assert r["status"] & O.STATUS_BAD_PARAM
    bad = zt.copy()
    bad[1, 3] = np.nan
    r = _one(bad, zd, [0, 1], u, D=0.5)
    assert r["status"] & O.STATUS_BAD_LOGITS
    bad = zd.copy()
    bad[0, 2] = np.inf
    r = _one(zt, bad, [0, 1], u, D=0.5)
    assert r["status"] & O.STATUS_BAD_LOGITS
    r = _one(zt, zd, [0, 1], u, D=0.5, hist=[8])
    assert r["status"] & O.STATUS_BAD_TOKEN


def test_empty_draft_emits_bonus_only():
    V = 5
    zt = np.log(np.array([[0.1, 0.2, 0.3, 0.25, 0.15]])).astype(np.float32)
    r = _one(zt, np.zeros((0, V), np.float32), [], [np.float32(0.35)], D=0.5)
    assert r["accepted"] == 0 and r["tokens"] == [2]


def test_no_bonus_variant():
    rng = np.random.default_rng(41)
    zt, zd = _random_rows(rng, 6, 2)
    r = O.verify_request(zt, zd, np.array([1, 2]), np.zeros(0, np.int64), 1.0, 1.0, 1.0, 1.0,
                         np.array([0.1, 0.2, 0.3], np.float32), bonus=False)
    assert r["accepted"] == 2 and r["tokens"] == [1, 2, -1]


# ------------------------------------------------ draft confidence early stop
# ("Adaptive-SpecDecode-Lab" README, section "Confidence-guided early stop")

def _conf(z, x, hist=(), T=1.0, alpha=1.0, thr=0.5):
    return O.draft_confidence_request(np.asarray(z, np.float32), np.asarray(x, np.int64),
                                      np.asarray(hist, np.int64), T, alpha, thr)


def test_confidence_worked_distribution():
    """p = [0.2, 0.5, 0.3] as logits ln p: the top-1 probability is 0.5."""
    z = np.log([[0.2, 0.5, 0.3]])
    r = _conf(z, [1], thr=0.4)
    assert r["conf"][0] == pytest.approx(0.5, abs=1e-7)
    assert r["k_eff"] == 1


def test_confidence_uniform_is_one_over_v():
    V = 1000
    r = _conf(np.zeros((3, V)), [1, 2, 3], thr=0.5)
    np.testing.assert_allclose(r["conf"], 1.0 / V, rtol=1e-12)
    assert r["k_eff"] == 1          # the first draft is already below 0.5: stop after it


def test_confidence_temperature_by_hand():
    """T = 0.5 squares the probabilities: [0.04, 0.25, 0.09] / 0.38."""
    z = np.log([[0.2, 0.5, 0.3]]).astype(np.float32)
    r = _conf(z, [0], T=0.5)
    p = np.array([0.2, 0.5, 0.3], np.float64)
    zf = z.astype(np.float64)[0]   # the fp32 logits the oracle sees
    e = np.exp(zf / 0.5)
    assert r["conf"][0] == pytest.approx(e.max() / e.sum(), rel=1e-12)
    assert r["conf"][0] == pytest.approx(0.25 / 0.38, abs=1e-6)
    del p


def test_confidence_penalty_on_history_and_preceding_drafts():
    """alpha = 4 on a negative logit multiplies it: ln 0.8 -> 4 ln 0.8."""
    z = np.log([[0.8, 0.2], [0.8, 0.2]]).astype(np.float32)
    r = _conf(z, [0, 1], alpha=4.0, thr=0.5)
    assert r["conf"][0] == pytest.approx(0.8, abs=1e-6)            # nothing penalised yet
    pen = 0.8 ** 4
    assert r["conf"][1] == pytest.approx(pen / (pen + 0.2), abs=1e-6)  # draft 0 penalised in row 1
    r2 = _conf(z, [0, 1], hist=[0], alpha=4.0, thr=0.5)
    assert r2["conf"][0] == pytest.approx(pen / (pen + 0.2), abs=1e-6)


def test_confidence_stops_after_the_first_low_token():
    """Two-token rows with top-1 probability 0.9, 0.7, 0.55, 0.95 and a 0.6
    threshold: the drafter proposes three tokens (the third is the first
    below the threshold and is still verified)."""
    c = [0.9, 0.7, 0.55, 0.95]
    z = np.log([[v, 1 - v] for v in c])
    r = _conf(z, [0, 0, 1, 0], thr=0.6)
    np.testing.assert_allclose(r["conf"], [max(v, 1 - v) for v in c], atol=1e-6)
    assert r["k_eff"] == 3
    assert _conf(z[[0, 1, 3]], [0, 0, 0], thr=0.6)["k_eff"] == 3   # never below: all K kept
    assert _conf(z[:0], [], thr=0.6)["k_eff"] == 0


def test_confidence_status():
    z = np.zeros((2, 4), np.float32)
    assert _conf(z, [0, 7])["status"] & O.STATUS_BAD_TOKEN
    assert _conf(z, [0, 1], T=0.0)["status"] & O.STATUS_BAD_PARAM
    zb = z.copy(); zb[1, 2] = np.nan
    assert _conf(zb, [0, 1])["status"] & O.STATUS_BAD_LOGITS


def test_confidence_no_drafts_checks_history_against_v():
    """A request without drafts still has a vocabulary: valid history tokens
    are valid, out-of-range ones are flagged."""
    z = np.zeros((0, 10), np.float32)
    assert _conf(z, [], hist=[3, 9])["status"] == 0
    assert _conf(z, [], hist=[10])["status"] & O.STATUS_BAD_TOKEN
