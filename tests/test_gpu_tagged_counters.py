"""Arrival counters without a clearing launch.

The greedy, cluster, pipelined and confidence kernels count each request's
arrivals (the top-p path, its pool's fill) on a 64-bit word tagged with the
call: a word that carries another call's tag, or any bytes the memory
happened to hold, counts as no arrival.
So a workspace full of random bytes, and one that earlier calls left behind,
give the oracle's results, and a call enqueues its kernel alone.  Under
stream capture a call captures a clear of its counters (tag 0), so a graph
replays correctly however often it runs."""
import numpy as np
import pytest

import speculative_decoding_verification_23_gb300 as sv
from speculative_decoding_verification_23_gb300 import workload as W

import oracle
import parity as PR

pytestmark = pytest.mark.gpu

RESIDENT, STREAMING = 2, 4


def _small(dtype="bf16", top_p=1.0, seed=301):
    return W.make_batch(B=6, V=50000, K=[0, 1, 3, 5, 8, 2], dtype=dtype, seed=seed,
                        rho=[0.3, 0.6, 0.8, 0.9, 0.95, 0.99], temperature=[0.5, 0.7, 1.0, 1.3, 0.9, 0.6],
                        rep_penalty=[1.0, 1.3, 1.1, 0.8, 1.2, 1.0], hist_len=20, top_p=top_p,
                        tv_budget=[0.0, 0.2, 0.5, 0.75, 1.0, 0.1])


def _noise_workspace(batch, seed):
    import torch

    ws = sv.make_workspace(batch.B, int(batch.cu_draft[-1]), batch.V)
    g = torch.Generator(device="cpu").manual_seed(seed)
    ws.copy_(torch.randint(0, 256, (ws.numel(),), dtype=torch.uint8, generator=g))
    return ws


def _host(ts):
    return [t.cpu().numpy().astype(np.int64) for t in ts]


def _check_sample(batch, got, ref):
    bad, near = PR.compare_sample(batch, got, ref)
    assert not bad, bad[:2]
    assert near <= 1


@pytest.mark.parametrize("flags,top_p", [(RESIDENT, 1.0), (STREAMING, 1.0), (STREAMING, [0.9, 0.5, 0.95, 0.3, 1.0, 0.7]),
                                         (0, [0.9, 0.5, 0.95, 0.3, 1.0, 0.7])],
                         ids=["resident", "pipelined", "cluster-top-p", "row-cut-top-p"])
def test_sample_on_a_random_workspace_and_repeated(flags, top_p):
    import torch

    from speculative_decoding_verification_23_gb300.device_batch import to_device

    batch = _small(top_p=top_p)
    ref = PR.oracle_sample(batch)
    db = to_device(batch)
    ws = _noise_workspace(batch, 11)
    for _ in range(3):          # the later calls find the earlier calls' counters
        got = _host(sv.spec_verify_sample(db.args(flags=flags), workspace=ws))
        _check_sample(batch, got, ref)
    torch.cuda.synchronize()


def test_greedy_on_a_random_workspace_and_repeated():
    from speculative_decoding_verification_23_gb300.device_batch import to_device

    batch = _small(seed=302)
    ref = PR.oracle_greedy(batch)
    db = to_device(batch)
    ws = _noise_workspace(batch, 12)
    for _ in range(3):
        tok, acc, st = _host(sv.spec_verify_greedy(db.args(), workspace=ws))
        np.testing.assert_array_equal(tok, ref["tokens"])
        np.testing.assert_array_equal(acc, ref["accepted"])
        np.testing.assert_array_equal(st, ref["status"])


def test_confidence_on_a_random_workspace_and_repeated():
    from speculative_decoding_verification_23_gb300.device_batch import to_device

    batch = _small(dtype="f32", seed=303)
    ref = oracle.draft_confidence_batch(batch, 0.3, None)
    db = to_device(batch)
    ws = _noise_workspace(batch, 13)
    for _ in range(3):
        conf, k_eff, st = sv.spec_draft_confidence(db.args(), 0.3, workspace=ws)
        conf, k_eff, st = conf.cpu().numpy().astype(np.float64), k_eff.cpu().numpy(), st.cpu().numpy()
        for b in range(batch.B):
            assert st[b] == ref["status"][b]
            d0, d1 = int(batch.cu_draft[b]), int(batch.cu_draft[b + 1])
            np.testing.assert_allclose(conf[d0:d1], ref["conf"][d0:d1], atol=1e-5, rtol=0)
            if not ref["near_tie"][b]:
                assert k_eff[b] == ref["k_eff"][b]


@pytest.mark.parametrize("entry", ["greedy", "sample-resident"])
def test_graph_replays(entry):
    """A call captured into a CUDA graph (the clear of its counters captured
    with it) gives the oracle's results on every replay."""
    import torch

    from speculative_decoding_verification_23_gb300.device_batch import to_device

    batch = _small(seed=304)
    db = to_device(batch)
    ws = _noise_workspace(batch, 14)
    n = int(batch.cu_draft[-1]) + batch.B
    outs = [torch.full((n,), -7, dtype=torch.int32, device="cuda"),
            torch.full((batch.B,), -7, dtype=torch.int32, device="cuda"),
            torch.full((batch.B,), -7, dtype=torch.int32, device="cuda")]
    if entry == "greedy":
        call = lambda: sv.spec_verify_greedy(db.args(), workspace=ws, out_tokens=outs[0], out_accepted=outs[1],
                                             out_status=outs[2])
        ref = PR.oracle_greedy(batch)
    else:
        call = lambda: sv.spec_verify_sample(db.args(flags=RESIDENT), workspace=ws, out_tokens=outs[0],
                                             out_accepted=outs[1], out_status=outs[2])
        ref = PR.oracle_sample(batch)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        call()                  # outside capture: a tagged call
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    for _ in range(3):
        for o in outs:
            o.fill_(-7)
        g.replay()
        torch.cuda.synchronize()
        got = _host(outs)
        if entry == "greedy":
            for x, k in zip(got, ("tokens", "accepted", "status")):
                np.testing.assert_array_equal(x, ref[k])
        else:
            _check_sample(batch, got, ref)
