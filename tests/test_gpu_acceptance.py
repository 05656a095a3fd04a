"""Acceptance law of the GPU path: with drafts drawn from q, position i is
accepted with probability 1 - max(0, d_i - D) ("What I Gave Up to Make
Speculative Decoding Faster", section "A knob for accepting more draft
tokens").  Thousands of rounds over the same rows (one request each, fresh
drafts and uniforms) against that law, with d_i from spec_tv_budget checked
against the oracle."""
import numpy as np
import pytest

import speculative_decoding_verification_23_gb300 as sv
from speculative_decoding_verification_23_gb300 import acceptance as A
from speculative_decoding_verification_23_gb300 import workload as W

import oracle
import parity as PR

pytestmark = pytest.mark.gpu

RESIDENT, STREAMING = 2, 4


def _tv(batch, round_=0):
    """d_i of the shared rows (those of `round_`) from the GPU, checked against the oracle."""
    one = W.acceptance_trials(float(batch.tv_budget[0]), 1, round_=round_, V=batch.V, K=batch.k(0), dtype=batch.dtype)
    tv, _, _, _ = PR.run_tv(one)
    r = one.request(0)
    ref = oracle.tv_budget_request(r["z_target"], r["z_draft"], r["x"], r["hist"], r["T"], r["alpha"], r["top_p"],
                                   r["D"])
    np.testing.assert_allclose(tv, ref["tv"], atol=1e-5)
    return tv


@pytest.mark.parametrize("variant", [RESIDENT, STREAMING], ids=["resident", "streaming"])
@pytest.mark.parametrize("D", [0.0, 0.15, 0.4, 1.0])
def test_per_position_acceptance_follows_the_budget(D, variant):
    n, K = 3000, 4
    batch = W.acceptance_trials(D, n, V=2048, K=K, dtype="f32")
    d = _tv(batch)
    tok, acc, st = PR.run_sample(batch, flags=variant)
    assert (st == 0).all()
    rep = A.acceptance_report(acc, d, D, ks=(1, 2, 4))
    for pos in rep["positions"]:
        assert pos["reached"] > 50, pos
        assert abs(pos["z"]) < 5, pos
    if D >= 1.0:
        assert (acc == K).all()
    # the same rounds without the bonus: the same decisions, one token less
    # when every draft was accepted
    tok_nb, acc_nb, _ = PR.run_sample(batch, flags=variant | sv.SPEC_NO_BONUS)
    np.testing.assert_array_equal(acc_nb, acc)
    last = tok_nb.reshape(n, K + 1)[:, K]
    assert (last[acc == K] == -1).all()


def test_k_sweep_matches_the_expected_tokens_per_round():
    n, K, D = 3000, 4, 0.1
    batch = W.acceptance_trials(D, n, V=2048, K=K, dtype="f32", round_=1)
    d = _tv(batch, round_=1)
    np.testing.assert_array_equal(batch.request(0)["z_target"],
                                  W.acceptance_trials(D, 1, round_=1, V=2048, K=K, dtype="f32").request(0)["z_target"])
    _, acc, _ = PR.run_sample(batch)
    rep = A.acceptance_report(acc, d, D, ks=(1, 2, 4))
    for s in rep["k_sweep"]:
        # binomial-scale tolerance on a mean of n rounds
        assert abs(s["accepted"] - s["expected_accepted"]) < 5 * np.sqrt(s["K"] / n) + 1e-3, s
        assert abs(s["emitted_no_bonus"] - s["expected_emitted_no_bonus"]) < 5 * np.sqrt(s["K"] / n) + 1e-3, s
