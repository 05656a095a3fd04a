"""GPU parity of spec_verify_greedy against the oracle: bit-exact, no
tolerance (the argmax compares fp32 penalised logits, lowest id on ties)."""
import numpy as np
import pytest

from speculative_decoding_verification_23_gb300 import workload as W

import parity as PR

pytestmark = pytest.mark.gpu


def _check(batch):
    got = PR.run_greedy(batch)
    ref = PR.oracle_greedy(batch)
    np.testing.assert_array_equal(got[0], ref["tokens"])
    np.testing.assert_array_equal(got[1], ref["accepted"])
    np.testing.assert_array_equal(got[2], ref["status"])
    return got, ref


@pytest.mark.parametrize("K", [1, 2, 4, 8])
def test_greedy_qwen3_single(K):
    """B=1, V=151936 bf16, rho=0.95, drafts = draft-row argmax."""
    _check(W.greedy_single(K))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("V", [7, 8192, 8193, 20000])
def test_greedy_ties_and_penalty(dtype, V):
    rng = np.random.default_rng(V)
    batch = W.make_batch(B=5, V=V, K=[0, 1, 3, 8, 2], dtype=dtype, seed=V, rep_penalty=[1.0, 1.5, 1.1, 0.7, 2.0],
                         hist_len=6, greedy_drafts=True, rho=0.99)
    # integer logits: many exact ties, so the lowest-id rule decides
    batch.target[:, :V] = rng.integers(-4, 5, size=(batch.target.shape[0], V)).astype(np.float32)
    # make some drafts match the target argmax so prefixes are long
    for b in range(batch.B):
        d0 = int(batch.cu_draft[b])
        for i in range(batch.k(b)):
            if rng.random() < 0.7:
                batch.draft_tokens[d0 + i] = int(np.argmax(batch.target[d0 + b + i, :V]))
    _check(batch)


def test_greedy_batched_full_size():
    _check(W.batched(0))


def test_greedy_invalid_inputs():
    batch = W.make_batch(B=4, V=300, K=[2, 2, 2, 2], dtype="f32", seed=9, greedy_drafts=True, hist_len=3,
                         rep_penalty=1.2)
    batch.draft_tokens[0] = -1
    batch.target[3 + 1, 5] = np.inf
    batch.rep_penalty[2] = 0.0
    got, ref = _check(batch)
    assert list(got[2] != 0) == [True, True, True, False]
