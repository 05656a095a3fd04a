"""spec_verify_sample_static: sampling with the library's fixed per-device
scratch instead of a caller's workspace.  Its results must equal those of
spec_verify_sample on the same inputs; two calls back to back on one stream
check that each call starts from cleared counters."""
import ctypes

import numpy as np
import pytest

import speculative_decoding_verification_23_gb300 as sv
from speculative_decoding_verification_23_gb300 import workload as W


def _fake_args(B, total, V, max_k=8):
    """Host-only arguments whose pointers are never dereferenced: the call
    must reject the batch before it touches a device."""
    a = sv.SpecArgs()
    a.B, a.V, a.total_drafts, a.max_k, a.dtype = B, V, total, max_k, sv.SPEC_F32
    fake = 1 << 20                          # 16-byte aligned, never read
    for f in ("cu_draft", "target_logits", "draft_logits", "draft_tokens", "temperature", "tv_budget",
              "uniforms"):
        setattr(a, f, fake)
    a.ld_target = a.ld_draft = 16
    return a


def test_oversize_batch_is_rejected_on_the_host():
    import __graft_entry__

    __graft_entry__.build()
    lib = sv.load_library()
    a = _fake_args(B=200000, total=0, V=10)
    rc = lib.spec_verify_sample_static(ctypes.byref(a), 1 << 20, 1 << 20, 1 << 20, None)
    assert rc == sv.SPEC_ERR_STATIC_SCRATCH
    assert "SPEC_STATIC_SCRATCH_BYTES" in sv.status_string(rc)


def _run(fn, db, **kw):
    import torch

    out = [torch.full((db.n_tokens,), -7, dtype=torch.int32, device="cuda"),
           torch.full((db.B,), -7, dtype=torch.int32, device="cuda"),
           torch.full((db.B,), -7, dtype=torch.int32, device="cuda")]
    fn(db.args(), out_tokens=out[0], out_accepted=out[1], out_status=out[2], **kw)
    return out


@pytest.mark.gpu
def test_two_calls_in_a_row_match_the_workspace_path():
    import torch

    from speculative_decoding_verification_23_gb300.device_batch import to_device

    small = W.make_batch(B=6, V=50000, K=[0, 1, 3, 5, 8, 2], dtype="bf16", seed=77,
                         rho=[0.3, 0.6, 0.8, 0.9, 0.95, 0.99], temperature=[0.5, 0.7, 1.0, 1.3, 0.9, 0.6],
                         rep_penalty=[1.0, 1.3, 1.1, 0.8, 1.2, 1.0], hist_len=20,
                         tv_budget=[0.0, 0.2, 0.5, 0.75, 1.0, 0.1])
    dbs = [to_device(small), to_device(W.batched(0))]
    for db in dbs:
        db.n_tokens = int(db.draft_tokens.numel()) + db.B
    ref = [_run(sv.spec_verify_sample, db) for db in dbs]
    torch.cuda.synchronize()
    # back to back on one stream: the second call's counters were left
    # non-zero by the first and must be cleared by the call itself
    got = [_run(sv.spec_verify_sample_static, db) for db in dbs]
    torch.cuda.synchronize()
    for r, g in zip(ref, got):
        for x, y in zip(r, g):
            np.testing.assert_array_equal(x.cpu().numpy(), y.cpu().numpy())
    assert int(got[1][2].abs().max()) == 0 and int(got[1][1].min()) >= 0


@pytest.mark.gpu
def test_oversize_batch_with_device_tensors_leaves_outputs_untouched():
    import torch

    B, V = 200000, 8
    target = torch.zeros((B, V), dtype=torch.float32, device="cuda")
    cu = torch.zeros(B + 1, dtype=torch.int32, device="cuda")
    ones = torch.ones(B, dtype=torch.float32, device="cuda")
    args = sv.make_args(target=target, cu_draft=cu, draft_tokens=None, V=V, draft=None, temperature=ones,
                        tv_budget=ones, uniforms=torch.zeros(B, dtype=torch.float32, device="cuda"), max_k=0)
    tok = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    acc = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    with pytest.raises(sv.SpecError) as e:
        sv.spec_verify_sample_static(args, out_tokens=tok, out_accepted=acc)
    assert e.value.code == sv.SPEC_ERR_STATIC_SCRATCH
    torch.cuda.synchronize()
    assert int(tok.max()) == -7 and int(acc.max()) == -7
