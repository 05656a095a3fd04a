"""Seeded synthetic inputs for the verification step (shared by the tests, the
oracle comparisons and ``bench.py``).

This module holds no arithmetic of the verification method itself: no
penalty, temperature, softmax, top-p, total variation, acceptance test or
inverse-CDF sampling.  It only draws the *inputs* the method consumes:

* target logits ``z_p = 3*N(0,1) + b(rank)`` with a Zipf(1.1) rank bias
  ``b(rank) = -1.1 * ln(rank)`` over a per-row random assignment of ranks to
  token ids;
* draft logits ``z_q = rho*z_p + sqrt(1-rho^2) * 3*N(0,1)`` (rho = 0.8 gives
  ``0.8 z_p + 0.6 N(0, 3^2)``);
* draft tokens, drawn by the *draft model's own sampler*: Gumbel-max over the
  temperature-scaled draft logits (optionally restricted to the draft row's
  ``draft_topk`` largest logits), or the draft row's argmax for greedy
  workloads.  Gumbel-max is a different algorithm from anything the verifier
  runs, so a mistake here cannot hide one in the verifier;
* history tokens, uniform over ``[0, V)``;
* per-request scalars (temperature, repetition penalty, top-p, TV budget D);
* uniforms ``u = (uint32 >> 8) * 2^-24`` in ``[0, 1)``, exactly representable
  in fp32: ``u[off_b + i]`` for the K_b acceptance tests of request b and
  ``u[off_b + K_b]`` for its final (correction or bonus) draw.

Rows are packed ragged: request b owns draft rows ``cu_draft[b] ..
cu_draft[b+1]-1`` and target rows ``off_b .. off_b + K_b`` with
``off_b = cu_draft[b] + b``.  Every logit buffer has a row stride ``ld`` that
is a multiple of 8 elements (16-byte rows in bf16, 32-byte rows in fp32), the
padding filled with zeros.

The logits are produced in fp32; for bf16 workloads they are rounded to bf16
(round-to-nearest-even, via torch's CPU cast) and the *rounded* values are
what both the oracle and the GPU consume.

The five named workloads are the pages' settings restated as synthetic inputs
(the pages' prompts and models are not available): a tiny fp32 case, a
Qwen2.5-shaped single request with a TV-budget sweep, greedy longest-prefix
verification with Qwen3's vocabulary, the batched 64-request case and a
ragged 256-request case with top-p.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence

import numpy as np

QWEN25_VOCAB = 152064
QWEN3_VOCAB = 151936

DTYPE_F32 = "f32"
DTYPE_BF16 = "bf16"


@dataclasses.dataclass
class Batch:
    """One packed batch of verification inputs (host numpy arrays)."""

    B: int
    V: int
    ld: int
    dtype: str                      # "f32" or "bf16": the dtype the GPU reads
    cu_draft: np.ndarray            # int32 [B+1]
    target: np.ndarray              # float32 [sum K + B, ld]; bf16-exact values for bf16
    draft: np.ndarray               # float32 [sum K, ld]
    draft_tokens: np.ndarray        # int32 [sum K]
    cu_hist: np.ndarray             # int32 [B+1]
    hist: np.ndarray                # int32 [cu_hist[B]]
    temperature: np.ndarray         # float32 [B]
    rep_penalty: np.ndarray         # float32 [B]
    top_p: np.ndarray               # float32 [B]
    tv_budget: np.ndarray           # float32 [B]
    uniforms: np.ndarray            # float32 [sum K + B]
    name: str = ""

    @property
    def total_drafts(self) -> int:
        return int(self.cu_draft[-1])

    @property
    def max_k(self) -> int:
        k = np.diff(self.cu_draft)
        return int(k.max()) if k.size else 0

    def k(self, b: int) -> int:
        return int(self.cu_draft[b + 1] - self.cu_draft[b])

    def request(self, b: int) -> dict:
        """Unpacked inputs of request b (views; logits cut to the V live columns)."""
        d0, d1 = int(self.cu_draft[b]), int(self.cu_draft[b + 1])
        off = d0 + b
        K = d1 - d0
        h0, h1 = int(self.cu_hist[b]), int(self.cu_hist[b + 1])
        return dict(
            z_target=self.target[off:off + K + 1, :self.V],
            z_draft=self.draft[d0:d1, :self.V],
            x=self.draft_tokens[d0:d1],
            hist=self.hist[h0:h1],
            T=self.temperature[b],
            alpha=self.rep_penalty[b],
            top_p=self.top_p[b],
            D=self.tv_budget[b],
            u=self.uniforms[off:off + K + 1],
        )

    def logit_bytes(self) -> int:
        """Bytes of logits one call reads: (2*sum K + B) rows of V entries."""
        s = 2 if self.dtype == DTYPE_BF16 else 4
        return (2 * self.total_drafts + self.B) * self.V * s


def round_up(x: int, m: int) -> int:
    return (x + m - 1) // m * m


def bf16_round(a: np.ndarray) -> np.ndarray:
    """Round fp32 -> bf16 (nearest-even) and return the rounded values as fp32."""
    import torch

    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return t.to(torch.bfloat16).to(torch.float32).numpy()


def uniforms_from_bits(bits: np.ndarray) -> np.ndarray:
    """uint32 -> fp32 uniforms in [0,1): (bits >> 8) * 2^-24, exact in fp32."""
    return ((bits.astype(np.uint32) >> np.uint32(8)).astype(np.float64) * 2.0 ** -24).astype(np.float32)


def _rank_bias(rng: np.random.Generator, rows: int, V: int, exponent: float = 1.1) -> np.ndarray:
    """Zipf rank bias -exponent*ln(rank): a seeded permutation of the ranks,
    rotated by a random per-row shift, so each row assigns ranks to token ids
    differently."""
    table = (-exponent * np.log(np.arange(1, V + 1, dtype=np.float64))).astype(np.float32)
    perm = rng.permutation(V).astype(np.int64)
    shift = rng.integers(0, V, size=rows, dtype=np.int64)
    out = np.empty((rows, V), dtype=np.float32)
    base = np.arange(V, dtype=np.int64)
    for r in range(rows):
        out[r] = table[perm[(base + shift[r]) % V]]
    return out


def _gumbel_sample(rng: np.random.Generator, z: np.ndarray, T: float, topk: Optional[int]) -> int:
    """The draft model's sampler: Gumbel-max over z/T (optionally top-k)."""
    z = z.astype(np.float64)
    if topk is not None and topk < z.size:
        cand = np.argpartition(-z, topk - 1)[:topk]
    else:
        cand = np.arange(z.size)
    g = -np.log(-np.log(rng.random(cand.size)))
    return int(cand[np.argmax(z[cand] / T + g)])


def make_batch(
    *,
    B: int,
    V: int,
    K: Sequence[int] | int,
    dtype: str = DTYPE_BF16,
    seed: int = 0,
    rho: Sequence[float] | float = 0.8,
    temperature: Sequence[float] | float = 0.7,
    rep_penalty: Sequence[float] | float = 1.0,
    hist_len: int = 0,
    top_p: Sequence[float] | float = 1.0,
    tv_budget: Sequence[float] | float = 0.5,
    greedy_drafts: bool = False,
    draft_topk: Optional[int] = None,
    logit_scale: float = 3.0,
    zipf: float = 1.1,
    name: str = "",
) -> Batch:
    """Draw one packed batch.  Every random quantity comes from one PCG64
    stream seeded with ``seed``; nothing depends on the machine."""
    rng = np.random.Generator(np.random.PCG64(seed))

    def per_req(v, kind=np.float32):
        a = np.asarray(v, dtype=np.float64)
        if a.ndim == 0:
            a = np.full(B, float(a))
        assert a.shape == (B,)
        return a.astype(kind)

    Ks = np.asarray(K, dtype=np.int64)
    if Ks.ndim == 0:
        Ks = np.full(B, int(Ks))
    assert Ks.shape == (B,) and (Ks >= 0).all()
    cu_draft = np.zeros(B + 1, dtype=np.int32)
    cu_draft[1:] = np.cumsum(Ks)
    total = int(cu_draft[-1])
    ld = round_up(max(V, 1), 8)

    rhos = per_req(rho, np.float64)
    temps = per_req(temperature)
    pens = per_req(rep_penalty)
    tps = per_req(top_p)
    Ds = per_req(tv_budget)

    n_target = total + B
    target = np.zeros((n_target, ld), dtype=np.float32)
    draft = np.zeros((total, ld), dtype=np.float32)
    bias = _rank_bias(rng, n_target, V, zipf)
    target[:, :V] = logit_scale * rng.standard_normal((n_target, V), dtype=np.float32) + bias
    del bias
    for b in range(B):
        d0, d1 = int(cu_draft[b]), int(cu_draft[b + 1])
        off = d0 + b
        k = d1 - d0
        if k == 0:
            continue
        r = rhos[b]
        noise = rng.standard_normal((k, V), dtype=np.float32)
        draft[d0:d1, :V] = (r * target[off:off + k, :V]
                            + math.sqrt(max(0.0, 1.0 - r * r)) * logit_scale * noise)
    if dtype == DTYPE_BF16:
        target = bf16_round(target)
        draft = bf16_round(draft)
    elif dtype != DTYPE_F32:
        raise ValueError(dtype)

    tokens = np.zeros(total, dtype=np.int32)
    for b in range(B):
        d0, d1 = int(cu_draft[b]), int(cu_draft[b + 1])
        for g in range(d0, d1):
            row = draft[g, :V]
            if greedy_drafts:
                tokens[g] = int(np.argmax(row))
            else:
                tokens[g] = _gumbel_sample(rng, row, float(temps[b]), draft_topk)

    cu_hist = np.zeros(B + 1, dtype=np.int32)
    cu_hist[1:] = np.cumsum(np.full(B, hist_len, dtype=np.int64))
    hist = rng.integers(0, V, size=int(cu_hist[-1]), dtype=np.int64).astype(np.int32)
    uniforms = uniforms_from_bits(rng.integers(0, 2 ** 32, size=total + B, dtype=np.uint64))

    return Batch(B=B, V=V, ld=ld, dtype=dtype, cu_draft=cu_draft, target=target, draft=draft,
                 draft_tokens=tokens, cu_hist=cu_hist, hist=hist, temperature=temps,
                 rep_penalty=pens, top_p=tps, tv_budget=Ds, uniforms=uniforms, name=name)


# --------------------------------------------------------------------------
# The named workloads.  Seeds: workload index * 10**6 + round.
# --------------------------------------------------------------------------

def tiny(round_: int = 0) -> Batch:
    """B=1, K=4, V=1024, fp32; T=0.7, no penalty, D=0.75, drafts from q."""
    return make_batch(B=1, V=1024, K=4, dtype=DTYPE_F32, seed=0 * 10 ** 6 + round_, rho=0.8,
                      temperature=0.7, rep_penalty=1.0, tv_budget=0.75, name="tiny")


def qwen25_single(D: float = 0.5, round_: int = 0) -> Batch:
    """B=1, K=8, V=152064, bf16, rho=0.9; T=0.7, penalty 1.1 over 256 history tokens."""
    return make_batch(B=1, V=QWEN25_VOCAB, K=8, dtype=DTYPE_BF16, seed=1 * 10 ** 6 + round_,
                      rho=0.9, temperature=0.7, rep_penalty=1.1, hist_len=256, tv_budget=D,
                      name=f"qwen25_single_D{D}")


def greedy_single(K: int = 8, round_: int = 0) -> Batch:
    """B=1, V=151936, bf16, rho=0.95, drafts = argmax of the draft rows."""
    return make_batch(B=1, V=QWEN3_VOCAB, K=K, dtype=DTYPE_BF16, seed=2 * 10 ** 6 + 10 * K + round_,
                      rho=0.95, temperature=1.0, rep_penalty=1.0, greedy_drafts=True,
                      name=f"greedy_K{K}")


def batched(round_: int = 0, B: int = 64) -> Batch:
    """B=64, K=8, V=152064, bf16; rho~U[0.6,0.98], T~U[0.5,1.0], penalty 1.1
    over 512 history tokens, D_b = {0,.25,.5,.75,1}[b mod 5]."""
    rng = np.random.Generator(np.random.PCG64(3 * 10 ** 6 + 500_000 + round_))
    rho = rng.uniform(0.6, 0.98, size=B)
    temp = rng.uniform(0.5, 1.0, size=B)
    D = np.array([(0.0, 0.25, 0.5, 0.75, 1.0)[b % 5] for b in range(B)])
    return make_batch(B=B, V=QWEN25_VOCAB, K=8, dtype=DTYPE_BF16, seed=3 * 10 ** 6 + round_,
                      rho=rho, temperature=temp, rep_penalty=1.1, hist_len=512, tv_budget=D,
                      name="batched")


def ragged_top_p(round_: int = 0, B: int = 256) -> Batch:
    """B=256, K_b~U{1..8}, V=152064, fp32; rho~U[0.5,0.99], T=0.8, top-p 0.9, D=0.5."""
    rng = np.random.Generator(np.random.PCG64(4 * 10 ** 6 + 500_000 + round_))
    K = rng.integers(1, 9, size=B)
    rho = rng.uniform(0.5, 0.99, size=B)
    return make_batch(B=B, V=QWEN25_VOCAB, K=K, dtype=DTYPE_F32, seed=4 * 10 ** 6 + round_,
                      rho=rho, temperature=0.8, rep_penalty=1.0, top_p=0.9, tv_budget=0.5,
                      draft_topk=16, name="ragged_top_p")


def acceptance_trials(D: float, n: int, round_: int = 0, V: int = QWEN25_VOCAB, K: int = 8,
                      dtype: str = DTYPE_BF16, rho: float = 0.9, temperature: float = 0.7, draws: int = 0) -> Batch:
    """``n`` verification rounds over the same rows (the Qwen2.5-shaped
    request: rho = 0.9, T = 0.7; no repetition penalty, so the draft
    distribution does not depend on earlier drafts): request t is one round,
    its drafts drawn afresh by the draft sampler (Gumbel-max over the draft
    rows / T), its uniforms fresh.  The rounds' accepted counts then sample
    the acceptance law of these rows."""
    base = make_batch(B=1, V=V, K=K, dtype=dtype, seed=5 * 10 ** 6 + round_, rho=rho, temperature=temperature,
                      rep_penalty=1.0, hist_len=0, tv_budget=D, name="acceptance_base")
    rng = np.random.Generator(np.random.PCG64(6 * 10 ** 6 + 1000 * round_ + draws))
    tokens = np.empty((n, K), dtype=np.int32)
    for i in range(K):
        z = base.draft[i, :V].astype(np.float64) / float(temperature)
        for t0 in range(0, n, 64):
            m = min(64, n - t0)
            g = -np.log(-np.log(rng.random((m, V))))
            tokens[t0:t0 + m, i] = np.argmax(z[None, :] + g, axis=1)
    cu_draft = (np.arange(n + 1, dtype=np.int64) * K).astype(np.int32)
    target = np.tile(base.target, (n, 1))
    draft = np.tile(base.draft, (n, 1))
    uniforms = uniforms_from_bits(rng.integers(0, 2 ** 32, size=n * (K + 1), dtype=np.uint64))

    def full(v):
        return np.full(n, v, dtype=np.float32)

    return Batch(B=n, V=V, ld=base.ld, dtype=dtype, cu_draft=cu_draft, target=target, draft=draft,
                 draft_tokens=tokens.reshape(-1), cu_hist=np.zeros(n + 1, dtype=np.int32),
                 hist=np.zeros(0, dtype=np.int32), temperature=full(temperature), rep_penalty=full(1.0),
                 top_p=full(1.0), tv_budget=full(D), uniforms=uniforms, name=f"acceptance_D{D}")


WORKLOADS = {
    "tiny": tiny,
    "qwen25_single": qwen25_single,
    "greedy_single": greedy_single,
    "batched": batched,
    "ragged_top_p": ragged_top_p,
}
