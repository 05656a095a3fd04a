"""GPU parity of spec_draft_confidence against the oracle: the top-1 draft
probability per row within 1e-5, the confidence-stopped draft count exactly
(except rows whose confidence is within 1e-6 of the threshold)."""
import numpy as np
import pytest

from speculative_decoding_verification_23_gb300 import workload as W

import oracle

pytestmark = pytest.mark.gpu


def _run(batch, threshold):
    import torch

    import speculative_decoding_verification_23_gb300 as sv
    from speculative_decoding_verification_23_gb300.device_batch import to_device

    db = to_device(batch)
    conf, k_eff, st = sv.spec_draft_confidence(db.args(), threshold)
    torch.cuda.synchronize()
    return conf.cpu().numpy().astype(np.float64), k_eff.cpu().numpy(), st.cpu().numpy()


def _check(batch, threshold, requests=None):
    conf, k_eff, st = _run(batch, threshold)
    ref = oracle.draft_confidence_batch(batch, threshold, requests)
    reqs = range(batch.B) if requests is None else requests
    for b in reqs:
        d0, d1 = int(batch.cu_draft[b]), int(batch.cu_draft[b + 1])
        assert st[b] == ref["status"][b], b
        if st[b]:
            assert k_eff[b] == -1 and np.all(np.isnan(conf[d0:d1]))
            continue
        np.testing.assert_allclose(conf[d0:d1], ref["conf"][d0:d1], atol=1e-5, rtol=0)
        if not ref["near_tie"][b]:
            assert k_eff[b] == ref["k_eff"][b], (b, k_eff[b], ref["k_eff"][b], conf[d0:d1])
    return conf, k_eff, st, ref


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("V", [3, 257, 8192, 8193, 50000, 152064])
def test_confidence_shapes(dtype, V):
    """Ragged K including 0, penalties with history, temperatures; V spans
    one chunk, exactly one, a ragged second chunk and many."""
    batch = W.make_batch(B=6, V=V, K=[0, 1, 3, 8, 5, 2], dtype=dtype, seed=5000 + V,
                         rho=[0.3, 0.6, 0.8, 0.9, 0.95, 0.99], temperature=[0.5, 0.7, 1.0, 1.3, 0.9, 0.6],
                         rep_penalty=[1.0, 1.3, 1.1, 0.8, 1.2, 1.0], hist_len=min(24, 3 * V))
    for thr in (0.05, 0.3, 0.6):
        _check(batch, thr)


def test_confidence_greedy_drafts_and_k_sweep():
    """Drafts taken as the draft argmax (the lab's greedy drafter), K 1..8."""
    for K in (1, 2, 4, 8):
        batch = W.greedy_single(K)
        conf, k_eff, st, ref = _check(batch, 0.4)
        assert 1 <= k_eff[0] <= K


def test_confidence_invalid_requests():
    batch = W.make_batch(B=4, V=600, K=[2, 2, 0, 2], dtype="f32", seed=9, hist_len=3, rep_penalty=1.1)
    batch.draft_tokens[1] = 600           # request 0: token out of range
    batch.temperature[1] = -1.0           # request 1: T < 0
    batch.hist[2 * 3] = 9999              # request 2 (no drafts): bad history token
    batch.draft[5, 5] = np.nan            # request 3 (rows 4, 5), row 1: NaN
    conf, k_eff, st, ref = _check(batch, 0.5)
    assert list(st != 0) == [True, True, True, True]


def _sms():
    import torch

    return torch.cuda.get_device_properties(0).multi_processor_count


_KS = [0, 8, 3, 6, 1, 8, 5, 7]


def _wide(V, dtype, seed, **kw):
    """A batch with more draft rows than SMs: the pipelined kernel, one CTA
    per SM streaming whole rows."""
    B = len(_KS) * (_sms() // sum(_KS) + 1)
    reps = B // len(_KS)
    args = dict(rho=[0.3, 0.6, 0.8, 0.9, 0.95, 0.99, 0.5, 0.7] * reps,
                temperature=[0.5, 0.7, 1.0, 1.3, 0.9, 0.6, 2.0, 0.8] * reps,
                rep_penalty=[1.0, 1.3, 1.1, 0.8, 1.2, 1.0, 1.5, 0.9] * reps, hist_len=min(24, 3 * V))
    args.update(kw)
    batch = W.make_batch(B=B, V=V, K=_KS * reps, dtype=dtype, seed=seed, **args)
    assert batch.total_drafts >= _sms()
    return batch


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("V", [3, 1000, 8193, 50000])
def test_confidence_pipelined_shapes(dtype, V):
    """Ragged K including 0, penalties with history, temperatures; V spans
    one partial segment, one stage, a ragged last stage and many stages."""
    batch = _wide(V, dtype, 7000 + V)
    for thr in (0.05, 0.3, 0.6):
        _check(batch, thr)


def test_confidence_pipelined_batched_workload():
    """The batched workload (B=64, K=8, V=152064, bf16, 512-token histories
    with a 1.1 penalty): 512 rows over the SMs, several rows per CTA."""
    _check(W.batched(), 0.45)


def test_confidence_pipelined_invalid_requests():
    batch = _wide(600, "f32", 11, hist_len=3, rep_penalty=1.1)
    cu = batch.cu_draft
    batch.draft_tokens[int(cu[1]) + 1] = 600          # request 1: token out of range
    batch.temperature[2] = -1.0                        # request 2: T < 0
    batch.hist[8 * 3] = 9999                           # request 8 (no drafts): bad history token
    batch.draft[int(cu[3]) + 2, 5] = np.nan            # request 3, row 2: NaN
    batch.draft[int(cu[5]) + 4, 7] = np.inf            # request 5, row 4: +inf
    conf, k_eff, st, ref = _check(batch, 0.5)
    assert st[1] and st[2] and st[3] and st[5] and st[8]
    assert not st[4] and not st[6]


def _run_args(db, args, threshold):
    import torch

    import speculative_decoding_verification_23_gb300 as sv

    conf, k_eff, st = sv.spec_draft_confidence(args, threshold)
    torch.cuda.synchronize()
    return conf.cpu().numpy().astype(np.float64), k_eff.cpu().numpy(), st.cpu().numpy()


@pytest.mark.parametrize("wide", [False, True], ids=["chunked", "pipelined"])
def test_confidence_draft_count_above_max_k(wide):
    """A request with more drafts than the call's max_k is reported (status
    bit 8, k_eff = -1, NaN confidences); the other requests are unaffected."""
    from speculative_decoding_verification_23_gb300.device_batch import to_device

    if wide:
        batch = _wide(3000, "bf16", 21, rep_penalty=1.2)
        max_k = 5
    else:
        batch = W.make_batch(B=6, V=3000, K=[0, 1, 3, 8, 5, 2], dtype="bf16", seed=22, hist_len=9,
                             rep_penalty=1.2)
        max_k = 4
    assert batch.total_drafts <= batch.B * max_k
    db = to_device(batch)
    args = db.args()
    args.max_k = max_k
    conf, k_eff, st = _run_args(db, args, 0.4)
    ref = oracle.draft_confidence_batch(batch, 0.4, None)
    for b in range(batch.B):
        d0, d1 = int(batch.cu_draft[b]), int(batch.cu_draft[b + 1])
        if d1 - d0 > max_k:
            assert st[b] & 8 and k_eff[b] == -1 and np.all(np.isnan(conf[d0:d1])), b
            continue
        assert st[b] == ref["status"][b], b
        np.testing.assert_allclose(conf[d0:d1], ref["conf"][d0:d1], atol=1e-5, rtol=0)
        if not ref["near_tie"][b]:
            assert k_eff[b] == ref["k_eff"][b], b
