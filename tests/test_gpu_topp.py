"""GPU parity of the top-p path (row-cut and finish kernels) against the
oracle, on the cases that leave its common route:

- cuts deeper than the candidate window below the row maximum (the select
  reads the row again from global memory);
- rows so flat that the candidates overflow shared memory, and kept sets
  too large to list (the finish kernel scans those rows in full, as it does
  for requests with top_p = 1);
- repetition penalties, exact ties at the cut, a zero residual, top_p = 1
  next to filtering requests, invalid requests, and the TV quantities.

Tokens, accepted counts and status bit-exact except at the oracle's near
ties; probabilities, TV and theta within 1e-5."""
import numpy as np
import pytest

from speculative_decoding_verification_23_gb300 import workload as W

import parity as PR

pytestmark = pytest.mark.gpu

CUT = 0            # no hint: top-p batches take the row-cut path


def _check(batch, max_near=None, flags=CUT, tv=True):
    got = PR.run_sample(batch, flags=flags)
    ref = PR.oracle_sample(batch, bonus=not (flags & 1))
    bad, near = PR.compare_sample(batch, got, ref)
    PR.record_near((batch.name or "top-p B=%d V=%d %s" % (batch.B, batch.V, batch.dtype)) + " [row-cut]", near,
                   batch.B)
    assert not bad, bad[:3]
    assert near <= (max_near if max_near is not None else max(1, batch.B // 4)), near
    if tv:
        # a near tie at a cut may move one token in or out of a kept set,
        # which moves the TV by about that token's mass: those requests are
        # excused here too
        clear = [b for b in range(batch.B) if not ref["near_tie"][b]]
        assert PR.compare_tv(batch, PR.run_tv(batch, flags=flags), ref, clear) < PR.TOL_PROB
    return got, ref


VIA_ROW = 1 << 16   # row record flag: the cut was selected over the row in global memory


def _paths(batch):
    """The row records the row-cut kernel leaves in the workspace: how many
    rows took the global select, and how many kept sets went unlisted."""
    import torch

    import speculative_decoding_verification_23_gb300 as sv
    from speculative_decoding_verification_23_gb300.device_batch import to_device

    db = to_device(batch)
    total = int(batch.cu_draft[-1])
    ws = sv.make_workspace(batch.B, total, batch.V)
    sv.spec_verify_sample(db.args(flags=CUT), workspace=ws)
    torch.cuda.synchronize()
    nr = 2 * total + batch.B
    rec = ws[:nr * 32].cpu().numpy().view(np.int32).reshape(nr, 8)
    return int(np.sum((rec[:, 5] & VIA_ROW) != 0)), int(np.sum(rec[:, 3] < 0))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_deep_cuts_beyond_the_window(dtype):
    """Rows of one dominant token over a flat tail of 63 (logits 0.25 N(0,1)
    on a 1/64 grid, so some tie): the dominant logit sits 9.75 above the
    tail's largest, 14 log2 units at T = 1, beyond the 13-unit candidate
    window, and a top_p above its mass cuts 14.5 to 15 units down, in the
    tail.  The tail's tokens keep probabilities near 5e-5, far above the
    1e-6 near-tie margin."""
    batch = W.make_batch(B=8, V=64, K=[2, 3, 1, 4, 2, 1, 3, 2], dtype=dtype, seed=801, rho=0.8, temperature=1.0,
                         top_p=[0.9985, 0.9990, 0.9993, 0.9996] * 2, tv_budget=[0.0, 0.5, 0.3, 0.8] * 2)
    V = batch.V
    rng = np.random.default_rng(801)
    for rows in (batch.target, batch.draft):
        for r in range(rows.shape[0]):
            z = (np.round(0.25 * rng.standard_normal(V) * 64) / 64).astype(np.float32)
            top = int(rng.integers(0, V))
            z[top] = np.float32(np.round((np.max(z) + 9.75) * 16) / 16)     # exact in bf16
            rows[r, :V] = z
    _check(batch, max_near=2)
    via_row, _ = _paths(batch)
    assert via_row > 0


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_flat_rows_overflow_the_candidates(dtype):
    """Nearly flat rows of 12000 tokens: every token is a candidate, more
    than shared memory holds, and the select reads the row from global
    memory.  Each token carries about 1e-4 of the mass, so one row in a few
    dozen lands within 1e-6 of top_p (a near tie)."""
    batch = W.make_batch(B=8, V=12000, K=[1, 2, 3, 2, 1, 2, 1, 3], dtype=dtype, seed=802, rho=0.9, temperature=1.0,
                         logit_scale=0.3, top_p=[0.3, 0.6, 0.9, 0.97] * 2, tv_budget=[0.2, 0.5, 0.0, 1.0] * 2)
    _check(batch, max_near=3)
    via_row, _ = _paths(batch)
    assert via_row >= batch.B        # most rows (the flattest hold more than 10240 candidates)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_kept_sets_too_large_to_list(dtype):
    """Kept sets of more than 32768 tokens are not listed: the finish kernel
    scans those rows in full with the cut as a mask.  (At 3e-5 of the mass
    a token, near ties are common: two of the three requests here.)"""
    batch = W.make_batch(B=3, V=40000, K=[1, 2, 1], dtype=dtype, seed=803, rho=0.95, temperature=1.0,
                         logit_scale=0.2, top_p=[0.95, 0.98, 0.9], tv_budget=[0.3, 0.6, 1.0])
    _check(batch, max_near=2)
    _, unlisted = _paths(batch)
    assert unlisted > 0


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_penalties_with_top_p(dtype):
    batch = W.make_batch(B=5, V=40000, K=[3, 0, 5, 8, 2], dtype=dtype, seed=803, rho=0.85,
                         temperature=[0.7, 1.0, 0.9, 1.2, 0.8], rep_penalty=[1.3, 1.0, 0.8, 1.1, 1.5], hist_len=60,
                         top_p=[0.9, 0.8, 0.95, 0.5, 0.7], tv_budget=[0.1, 0.5, 0.25, 0.75, 0.0])
    _check(batch)


def test_ties_at_the_cut():
    """bf16 logits on a coarse scale: many tokens share a logit, and the cut
    keeps every token tied with the last one it needs."""
    batch = W.make_batch(B=4, V=5000, K=[2, 2, 3, 1], dtype="bf16", seed=804, rho=0.9, temperature=1.0,
                         logit_scale=0.6, top_p=[0.2, 0.5, 0.7, 0.9], tv_budget=0.4)
    z = batch.target[:, :batch.V]
    batch.target[:, :batch.V] = np.round(z * 4.0) / 4.0       # exact in bf16, heavy ties
    zd = batch.draft[:, :batch.V]
    batch.draft[:, :batch.V] = np.round(zd * 4.0) / 4.0
    _check(batch)


def test_top_p_one_next_to_filtering_requests():
    batch = W.make_batch(B=4, V=30000, K=[2, 4, 3, 1], dtype="f32", seed=805, rho=0.9, temperature=0.8,
                         top_p=[1.0, 0.9, 1.0, 0.6], tv_budget=0.5)
    _check(batch)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_zero_residual_correction_from_p(dtype):
    """Draft rows equal to the target rows and a drafted token with -inf
    logits in both: the draft is rejected with zero residual mass and the
    correction comes from p~."""
    batch = W.make_batch(B=3, V=3000, K=[2, 3, 1], dtype=dtype, seed=806, rho=0.8, temperature=0.9,
                         top_p=[0.9, 0.6, 0.95], tv_budget=[0.0, 0.4, 1.0])
    for b in range(batch.B):
        d0, d1 = int(batch.cu_draft[b]), int(batch.cu_draft[b + 1])
        off = d0 + b
        batch.draft[d0:d1] = batch.target[off:off + (d1 - d0)]
        x = int(batch.draft_tokens[d0])
        batch.target[off, x] = -np.inf
        batch.draft[d0, x] = -np.inf
    got, _ = _check(batch)
    assert np.all(got[2] == 0) and list(got[1]) == [0, 0, 0]


def test_invalid_inputs_set_status():
    batch = W.make_batch(B=7, V=500, K=[2] * 7, dtype="f32", seed=807, hist_len=4, rep_penalty=1.1,
                         top_p=0.9)
    batch.draft_tokens[1] = 500                 # request 0: token out of range
    batch.temperature[1] = 0.0                  # request 1: T = 0
    batch.target[2 * 3 + 1, 7] = np.nan         # request 2: NaN logit
    batch.tv_budget[3] = 1.5                    # request 3: D > 1
    batch.hist[4 * 4] = -3                      # request 4: bad history token
    batch.top_p[5] = 0.0                        # request 5: top_p = 0
    tok, acc, st = PR.run_sample(batch, flags=CUT)
    ref = PR.oracle_sample(batch)
    assert list(st[:6] != 0) == [True] * 6 and st[6] == 0
    np.testing.assert_array_equal(st, ref["status"])
    for b in range(6):
        assert acc[b] == -1 and np.all(tok[3 * b:3 * b + 3] == -1)
    bad, _ = PR.compare_sample(batch, (tok, acc, st), ref, [6])
    assert not bad
    tv = PR.run_tv(batch, flags=CUT)
    assert np.all(np.isnan(tv[0][:12])) and np.all(np.isfinite(tv[0][12:]))


def test_no_bonus_flag():
    """D = 1 accepts every draft that q~ keeps (a draft outside q's nucleus
    has q~(x) = 0 and is rejected); a request that accepts all of its drafts
    then emits no bonus token."""
    batch = W.make_batch(B=4, V=2000, K=[2, 3, 0, 4], dtype="bf16", seed=808, top_p=0.8, tv_budget=1.0)
    got, _ = _check(batch, flags=1, tv=False)
    tok, acc, _ = got
    assert acc[2] == 0 and tok[3 + 4] == -1
    full = [b for b in range(batch.B) if acc[b] == batch.k(b)]
    assert len(full) >= 2
    for b in full:
        off = int(batch.cu_draft[b]) + b
        assert tok[off + batch.k(b)] == -1


def test_many_requests_small_vocabulary():
    """B = 600 requests, K in 0..4, V = 700 (the rows are shorter than one
    copy): a sample against the oracle, properties on all."""
    rng = np.random.default_rng(809)
    K = rng.integers(0, 5, size=600)
    batch = W.make_batch(B=600, V=700, K=K, dtype="bf16", seed=809, rho=0.8, temperature=0.9, rep_penalty=1.1,
                         hist_len=6, top_p=0.85, tv_budget=0.5)
    got = PR.run_sample(batch, flags=CUT)
    sample = list(range(0, 600, 23))
    ref = PR.oracle_sample(batch, sample)
    bad, near = PR.compare_sample(batch, got, ref, sample)
    assert not bad and near <= 1, (bad[:2], near)
    tok, acc, st = got
    assert np.all(st == 0) and np.all((acc >= 0) & (acc <= K))
