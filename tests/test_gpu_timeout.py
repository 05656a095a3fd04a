"""Device-side timeouts of the split-vocabulary sampling kernel.

With the wait bound set far below what a call needs (spec_set_wait_cycles),
waits run out: the kernel raises its abort flag, every CTA stops, and the
requests left unfinished report SPEC_STATUS_TIMEOUT, while the call itself
returns and the CUDA context stays usable.  No fault, trap or endless wait
is involved: every wait in the kernel is bounded, and the wait for copies in
flight before a CTA exits keeps its own fixed bound.  The default bound,
restored afterwards, gives the usual results again."""
import numpy as np
import pytest

import speculative_decoding_verification_23_gb300 as sv
from speculative_decoding_verification_23_gb300 import workload as W

import parity as PR

pytestmark = pytest.mark.gpu

SPLIT = 8


@pytest.fixture()
def short_waits():
    sv.load_library()
    prev = sv.set_wait_cycles(20000)          # about 10 us at 2 GHz
    yield
    sv.set_wait_cycles(prev)


def _batch():
    return W.make_batch(B=16, V=152064, K=8, dtype="bf16", seed=91, rho=0.9, temperature=0.8, rep_penalty=1.1,
                        hist_len=64, tv_budget=[0.0, 0.25, 0.5, 0.75] * 4)


def test_setter_returns_the_previous_bound():
    sv.load_library()
    first = sv.set_wait_cycles(12345)
    assert sv.set_wait_cycles(0) == 12345
    assert sv.set_wait_cycles(first) == 4000000000


def test_waits_that_run_out_set_timeout_and_the_call_returns(short_waits):
    import torch

    batch = _batch()
    tok, acc, st = PR.run_sample(batch, flags=SPLIT)
    assert set(np.unique(st)) <= {0, sv.SPEC_STATUS_TIMEOUT}, np.unique(st)
    assert (st == sv.SPEC_STATUS_TIMEOUT).any()
    for b in np.nonzero(st == sv.SPEC_STATUS_TIMEOUT)[0]:
        off = int(batch.cu_draft[b]) + b
        assert acc[b] == -1 and np.all(tok[off:off + batch.k(b) + 1] == -1)
    # the context is intact: a plain device operation still works
    x = torch.arange(1024, device="cuda", dtype=torch.float32)
    assert float(x.sum()) == 1024 * 1023 / 2


def test_default_bound_gives_the_oracle_results_again(short_waits):
    batch = _batch()
    PR.run_sample(batch, flags=SPLIT)        # runs out
    sv.set_wait_cycles(0)
    got = PR.run_sample(batch, flags=SPLIT)
    ref = PR.oracle_sample(batch, [0, 5, 10, 15])
    bad, near = PR.compare_sample(batch, got, ref, [0, 5, 10, 15])
    assert not bad and near <= 1, (bad[:2], near)
    assert np.all(got[2] == 0)
