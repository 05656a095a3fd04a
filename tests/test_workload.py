"""The seeded input generator: determinism, packed layout, value recipe."""
import numpy as np

from speculative_decoding_verification_23_gb300 import workload as W


def test_deterministic_and_seed_dependent():
    a = W.make_batch(B=3, V=100, K=[2, 0, 3], dtype="f32", seed=7, hist_len=5)
    b = W.make_batch(B=3, V=100, K=[2, 0, 3], dtype="f32", seed=7, hist_len=5)
    c = W.make_batch(B=3, V=100, K=[2, 0, 3], dtype="f32", seed=8, hist_len=5)
    for f in ("target", "draft", "draft_tokens", "hist", "uniforms"):
        np.testing.assert_array_equal(getattr(a, f), getattr(b, f))
    assert not np.array_equal(a.target, c.target)


def test_packed_layout_and_padding():
    bt = W.make_batch(B=3, V=13, K=[2, 0, 3], dtype="bf16", seed=1, hist_len=4)
    assert bt.ld == 16 and bt.ld % 8 == 0
    assert list(bt.cu_draft) == [0, 2, 2, 5]
    assert bt.target.shape == (5 + 3, 16) and bt.draft.shape == (5, 16)
    assert np.all(bt.target[:, 13:] == 0) and np.all(bt.draft[:, 13:] == 0)
    assert bt.uniforms.shape == (8,)
    assert np.all((bt.uniforms >= 0) & (bt.uniforms < 1))
    # uniforms are multiples of 2^-24
    assert np.all(np.floor(bt.uniforms.astype(np.float64) * 2 ** 24) == bt.uniforms.astype(np.float64) * 2 ** 24)
    r = bt.request(2)
    assert r["z_target"].shape == (4, 13) and r["z_draft"].shape == (3, 13) and r["u"].shape == (4,)
    assert np.all((bt.draft_tokens >= 0) & (bt.draft_tokens < 13))
    assert np.all((bt.hist >= 0) & (bt.hist < 13))


def test_bf16_values_are_bf16_exact():
    bt = W.make_batch(B=1, V=64, K=2, dtype="bf16", seed=3)
    bits = bt.target.view(np.uint32)
    assert np.all(bits & 0xFFFF == 0)


def test_draft_correlation_follows_rho():
    bt = W.make_batch(B=1, V=20000, K=1, dtype="f32", seed=4, rho=0.8)
    zt, zd = bt.target[0, :20000], bt.draft[0, :20000]
    c = np.corrcoef(zt, zd)[0, 1]
    assert 0.75 < c < 0.85


def test_greedy_drafts_are_draft_argmax():
    bt = W.make_batch(B=2, V=300, K=3, dtype="f32", seed=5, greedy_drafts=True)
    for g in range(bt.total_drafts):
        assert bt.draft_tokens[g] == int(np.argmax(bt.draft[g, :300]))


def test_named_workloads_small_shapes():
    t = W.tiny()
    assert (t.B, t.V, t.max_k, t.dtype) == (1, 1024, 4, "f32")
    assert float(t.tv_budget[0]) == 0.75 and float(t.temperature[0]) == np.float32(0.7)
