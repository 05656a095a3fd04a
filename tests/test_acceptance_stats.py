"""The acceptance-statistics report (host side): its expectations against
closed forms and the oracle's distributions, and its observed statistics
on rounds simulated from a known acceptance law."""
import numpy as np

from speculative_decoding_verification_23_gb300 import acceptance as A
from speculative_decoding_verification_23_gb300 import workload as W

import oracle


def test_expected_counts_closed_forms():
    assert A.expected_accepted([1.0] * 8, 8) == 8.0
    assert A.expected_accepted([0.5] * 4, 4) == 0.5 + 0.25 + 0.125 + 0.0625
    assert A.expected_accepted([0.3, 0.9], 1) == 0.3
    # the bonus adds one token to every round; without it a fully accepted
    # round adds none
    a = [0.5, 0.5]
    assert A.expected_emitted(a, 2, bonus=True) == 0.75 + 1.0
    assert A.expected_emitted(a, 2, bonus=False) == 0.75 + 0.75
    np.testing.assert_allclose(A.expected_acceptance([0.1, 0.4, 0.7], 0.4), [1.0, 1.0, 0.7])


def test_expected_acceptance_matches_the_oracles_distributions():
    """sum_v min(q, pi) computed from the oracle's processed rows equals
    1 - max(0, d - D) for every budget."""
    b = W.acceptance_trials(0.0, 1, V=512, K=3, dtype="f32")
    r = b.request(0)
    for D in (0.0, 0.2, 0.5, 1.0):
        for i in range(3):
            p = oracle.process_row(r["z_target"][i], [], 1.0, float(r["T"]), 1.0)[0]
            q = oracle.process_row(r["z_draft"][i], [], 1.0, float(r["T"]), 1.0)[0]
            d = oracle.tv_distance(p, q)
            pi = (1.0 - oracle.mentored_theta(d, D)) * p + oracle.mentored_theta(d, D) * q
            np.testing.assert_allclose(np.minimum(q, pi).sum(), A.expected_acceptance([d], D)[0], atol=1e-12)


def test_report_on_simulated_rounds():
    rng = np.random.default_rng(3)
    a = np.array([0.9, 0.7, 0.8, 0.6])
    n = 20000
    u = rng.random((n, 4))
    ok = u < a
    acc = np.where(ok.all(axis=1), 4, np.argmin(ok, axis=1))
    d = 1.0 - a          # with D = 0 the law is a_i = 1 - d_i
    rep = A.acceptance_report(acc, d, 0.0, ks=(1, 2, 4))
    for pos in rep["positions"]:
        assert abs(pos["z"]) < 5, pos
    for s in rep["k_sweep"]:
        assert abs(s["accepted"] - s["expected_accepted"]) < 0.05, s
        assert abs(s["emitted_no_bonus"] - s["expected_emitted_no_bonus"]) < 0.05, s
    assert rep["positions"][0]["reached"] == n


def test_trials_share_rows_and_draw_fresh_drafts():
    b = W.acceptance_trials(0.5, 8, V=256, K=3, dtype="f32")
    r0, r5 = b.request(0), b.request(5)
    np.testing.assert_array_equal(r0["z_target"], r5["z_target"])
    np.testing.assert_array_equal(r0["z_draft"], r5["z_draft"])
    assert b.draft_tokens.shape == (24,) and b.uniforms.shape == (32,)
    assert len({tuple(b.request(t)["x"]) for t in range(8)}) > 1
