"""Helpers shared by the GPU parity tests: run the CUDA path through the C
ABI and compare it with the oracle request by request."""
import numpy as np

import oracle

TOL_PROB = 1e-5     # probabilities, TV and theta: absolute, fp32 kernels vs fp64 oracle

# Near ties seen by the GPU parity tests: (case, near ties, requests
# compared).  The test session prints them at its end (conftest.py).
NEAR_TIES = []


def record_near(case, near, n):
    NEAR_TIES.append((str(case), int(near), int(n)))


def run_sample(batch, *, flags=0, device="cuda", db=None):
    import torch

    import speculative_decoding_verification_23_gb300 as sv
    from speculative_decoding_verification_23_gb300.device_batch import to_device

    db = db or to_device(batch, device)
    tok, acc, st = sv.spec_verify_sample(db.args(flags=flags), device=torch.device(device))
    torch.cuda.synchronize()
    return tok.cpu().numpy().astype(np.int64), acc.cpu().numpy().astype(np.int64), st.cpu().numpy().astype(np.int64)


def run_tv(batch, *, flags=0, device="cuda", db=None):
    import torch

    import speculative_decoding_verification_23_gb300 as sv
    from speculative_decoding_verification_23_gb300.device_batch import to_device

    db = db or to_device(batch, device)
    tv, th, px, qx = sv.spec_tv_budget(db.args(flags=flags), device=torch.device(device))
    torch.cuda.synchronize()
    return [t.cpu().numpy().astype(np.float64) for t in (tv, th, px, qx)]


def run_greedy(batch, *, device="cuda", db=None):
    import torch

    import speculative_decoding_verification_23_gb300 as sv
    from speculative_decoding_verification_23_gb300.device_batch import to_device

    db = db or to_device(batch, device)
    tok, acc, st = sv.spec_verify_greedy(db.args(), device=torch.device(device))
    torch.cuda.synchronize()
    return tok.cpu().numpy().astype(np.int64), acc.cpu().numpy().astype(np.int64), st.cpu().numpy().astype(np.int64)


def compare_sample(batch, got, ref, requests=None):
    """Bit-exact tokens/accepted/status for every request the oracle does not
    flag as a near tie.  Returns (list of mismatching requests, #near ties)."""
    tok, acc, st = got
    bad, near = [], 0
    for b in (range(batch.B) if requests is None else requests):
        off = int(batch.cu_draft[b]) + b
        K = batch.k(b)
        if ref["near_tie"][b]:
            near += 1
            continue
        same = (np.array_equal(tok[off:off + K + 1], ref["tokens"][off:off + K + 1])
                and acc[b] == ref["accepted"][b] and st[b] == ref["status"][b])
        if not same:
            bad.append((b, tok[off:off + K + 1].tolist(), ref["tokens"][off:off + K + 1].tolist(),
                        int(acc[b]), int(ref["accepted"][b]), int(st[b]), int(ref["status"][b]),
                        float(ref["margin"][b])))
    return bad, near


def compare_tv(batch, got, ref, requests=None):
    """Max absolute error of tv, theta, p(x), q(x) over the positions of the
    given requests (valid ones only)."""
    tv, th, px, qx = got
    err = 0.0
    for b in (range(batch.B) if requests is None else requests):
        if ref["status"][b]:
            continue
        d0, d1 = int(batch.cu_draft[b]), int(batch.cu_draft[b + 1])
        for name, g in (("tv", tv), ("theta", th), ("p_x", px), ("q_x", qx)):
            e = np.max(np.abs(g[d0:d1] - ref[name][d0:d1])) if d1 > d0 else 0.0
            err = max(err, float(e))
    return err


def oracle_sample(batch, requests=None, **kw):
    return oracle.verify_batch(batch, requests, **kw)


def oracle_greedy(batch, requests=None):
    return oracle.greedy_batch(batch, requests)
