"""Plain, slow CPU oracle for the speculative-decoding verification step.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import
it.  It shares no code with the CUDA path and imports nothing from it.

Everything is numpy, one request at a time, in fp64, written as the steps of
the method in the order the pages give them:

* "What I Gave Up to Make Speculative Decoding Faster", section "A knob for
  accepting more draft tokens": p and q are taken after temperature and
  repetition penalty; d = TV(p,q) = 1/2 sum|p-q|; theta = min(1, D/d) with
  theta = 1 when d = 0; pi = (1-theta) p + theta q; a drafted x ~ q is
  accepted with probability min(1, pi(x)/q(x)); after a rejection the
  replacement is drawn from the normalised positive residual max(p-q, 0).
* "Speculative Decoding" (note), section "Warum eine Korrektur noetig ist":
  the lossless rule min(1, p/q), the residual max(0, p-q), q(x) > 0 for a
  drafted token, no rejection when p = q; temperature and top-p are part of
  both distributions; the accepted prefix is kept up to the first rejection.
* "Adaptive-SpecDecode-Lab" README, section "实现" (implementation): greedy
  longest-prefix acceptance, the target's correction on a mismatch and a
  bonus token when every draft matches.
* The same README, section "Confidence-guided early stop": after each draft
  token the drafter reads its top-1 probability from the logits it has and
  stops proposing below a threshold; the low-confidence token is still
  verified.

Readings where the pages are silent (the same readings the kernels implement):

* Repetition penalty (named only): for every distinct token of the request's
  history plus the drafts that precede the row, z' = z/alpha if z > 0 else
  z*alpha.  The penalised logit is an fp32 value (the precision logits are
  carried in; the same rounding the kernels do), so greedy argmax decisions
  are taken in fp32 on both sides.  Then temperature: z'' = z'/T in fp64.
* Top-p: sort descending, tau = the probability at the first k whose
  cumulative sum reaches top_p, keep every token with p >= tau (ties at tau
  kept), renormalise; applied to p and q separately, before TV.
* TV is clamped to [0,1]; theta = 1 if d <= D else D/d (the same as
  min(1, D/d), and theta = 1 at d = 0).
* Acceptance is the strict comparison u*q(x) < pi(x) with u in [0,1).
* The residual and the bonus are drawn by inverse CDF in token-id order with
  one final uniform: the smallest v whose inclusive prefix sum exceeds u*R.
  If rounding leaves no such v, the last v with positive mass; if R = 0, the
  same draw from p.
* A bonus token from the last target row follows a fully accepted draft
  (``bonus=False`` emits none, as the mentored-decoding engine does).
* Draft confidence is the largest probability of the draft distribution
  after repetition penalty and temperature (top-p does not enter: the
  drafter reads it from its logits); the drafter keeps the first token whose
  confidence is below the threshold and stops after it.

Near ties: every decision whose margin (in units of the uniform it consumes)
is below ``NEAR_TIE`` is reported; the fp32 kernels may decide those either
way.
"""
from __future__ import annotations

import math
from typing import Dict, Iterable, List, Optional, Tuple

import numpy as np

NEAR_TIE = 1e-6

# Per-request status bits (same meaning as the library's; defined here
# independently).
STATUS_OK = 0
STATUS_BAD_TOKEN = 1
STATUS_BAD_PARAM = 2
STATUS_BAD_LOGITS = 4
STATUS_BAD_K = 8

MAX_K = 32


# ---------------------------------------------------------------------------
# Logit processing
# ---------------------------------------------------------------------------

def penalty_set(hist: Iterable[int], drafts_before: Iterable[int]) -> List[int]:
    """Tokens penalised for a row: the history plus the preceding drafts of
    the round, each once (the autoregressive target at that position has
    seen exactly these tokens)."""
    return sorted(set(int(t) for t in hist) | set(int(t) for t in drafts_before))


def apply_repetition_penalty(z: np.ndarray, tokens: Iterable[int], alpha: float) -> np.ndarray:
    """z' = z/alpha for positive, z*alpha for non-positive logits of the
    penalised tokens; fp32 arithmetic (correctly rounded)."""
    out = np.array(z, dtype=np.float32, copy=True)
    a = np.float32(alpha)
    for t in tokens:
        zt = out[t]
        out[t] = np.float32(zt / a) if zt > 0 else np.float32(zt * a)
    return out


def apply_temperature(z: np.ndarray, T: float) -> np.ndarray:
    """z'' = z'/T, in fp64."""
    return np.asarray(z, dtype=np.float64) / float(np.float32(T))


def softmax(x: np.ndarray) -> np.ndarray:
    """Max-subtracted softmax in fp64."""
    x = np.asarray(x, dtype=np.float64)
    m = np.max(x)
    e = np.exp(x - m)
    return e / np.sum(e)


def top_p_filter(p: np.ndarray, top_p: float) -> Tuple[np.ndarray, float]:
    """Nucleus filter.  Returns (filtered renormalised p, margin).

    The margin is the distance of the decision from a tie: how close the
    cumulative mass at the cut (or just before it) is to top_p, and how close
    the cut probability is, relatively, to its neighbours in the sorted
    order (two nearly equal probabilities may tie in fp32)."""
    tp = float(np.float32(top_p))
    if tp >= 1.0:
        return p.copy(), math.inf
    order = np.argsort(-p, kind="stable")
    s = p[order]
    c = np.cumsum(s)
    hit = np.nonzero(c >= tp)[0]
    k = int(hit[0]) if hit.size else p.size - 1
    tau = s[k]
    keep = p >= tau
    out = np.where(keep, p, 0.0)
    out = out / np.sum(out)
    margin = abs(c[k] - tp)
    if k > 0:
        margin = min(margin, abs(c[k - 1] - tp))
    # relative gaps to the neighbouring distinct probabilities
    above = s[:k][s[:k] > tau]
    below = s[k + 1:][s[k + 1:] < tau]
    if above.size:
        margin = min(margin, (above[-1] - tau) / above[-1])
    if below.size and tau > 0:
        margin = min(margin, (tau - below[0]) / tau)
    return out, margin


def process_row(z: np.ndarray, pen_tokens: Iterable[int], alpha: float, T: float,
                top_p: float) -> Tuple[np.ndarray, float]:
    """Penalty -> temperature -> softmax -> top-p.  Returns (dist, top-p margin)."""
    zp = apply_repetition_penalty(z, pen_tokens, alpha)
    return top_p_filter(softmax(apply_temperature(zp, T)), top_p)


# ---------------------------------------------------------------------------
# Mentored decoding quantities
# ---------------------------------------------------------------------------

def tv_distance(p: np.ndarray, q: np.ndarray) -> float:
    """d = 1/2 sum_x |p(x) - q(x)|, clamped to [0, 1]."""
    d = 0.5 * float(np.sum(np.abs(p - q)))
    return min(max(d, 0.0), 1.0)


def mentored_theta(d: float, D: float) -> float:
    """theta = min(1, D/d), theta = 1 when d = 0 (written as d <= D ? 1 : D/d)."""
    D = float(np.float32(D))
    return 1.0 if d <= D else D / d


def mixture_at(p_x: float, q_x: float, theta: float) -> float:
    """pi(x) = (1 - theta) p(x) + theta q(x)."""
    return (1.0 - theta) * p_x + theta * q_x


def accept_draft(u: float, pi_x: float, q_x: float) -> Tuple[bool, float]:
    """Accept x with probability min(1, pi(x)/q(x)) using uniform u:
    accept iff u*q(x) < pi(x).  Returns (accepted, margin |u - pi/q|)."""
    u = float(np.float32(u))
    acc = u * q_x < pi_x
    margin = abs(u - pi_x / q_x) if q_x > 0 else math.inf
    return bool(acc), margin


def residual(p: np.ndarray, q: np.ndarray) -> np.ndarray:
    """max(p - q, 0) (unnormalised)."""
    return np.maximum(p - q, 0.0)


def inverse_cdf(w: np.ndarray, u: float) -> Tuple[int, float]:
    """Draw from weights w (>= 0, unnormalised) with uniform u: the smallest v
    whose inclusive prefix sum exceeds u*sum(w); the last v with w > 0 if
    rounding leaves none.  Returns (token, margin in units of u)."""
    u = float(np.float32(u))
    c = np.cumsum(np.asarray(w, dtype=np.float64))
    R = c[-1]
    t = u * R
    hit = np.nonzero(c > t)[0]
    if hit.size:
        v = int(hit[0])
    else:
        v = int(np.nonzero(w > 0)[0][-1])
    lo = c[v - 1] if v > 0 else 0.0
    margin = min(abs(t - lo), abs(c[v] - t)) / R if R > 0 else math.inf
    return v, margin


# ---------------------------------------------------------------------------
# One request
# ---------------------------------------------------------------------------

def _finite_row(z: np.ndarray) -> bool:
    z = np.asarray(z, dtype=np.float32)
    return not (np.isnan(z).any() or np.isposinf(z).any() or np.isneginf(z).all())


def validate_request(V: int, z_target, z_draft, x, hist, T, alpha, top_p, D,
                     *, sampling: bool) -> int:
    """Status bits for one request (0 = valid)."""
    st = STATUS_OK
    K = len(x)
    if K > MAX_K:
        st |= STATUS_BAD_K
    toks = list(int(t) for t in x) + list(int(t) for t in hist)
    if any(t < 0 or t >= V for t in toks):
        st |= STATUS_BAD_TOKEN
    a = float(np.float32(alpha))
    if not (math.isfinite(a) and a > 0):
        st |= STATUS_BAD_PARAM
    if sampling:
        Tv, tp, Dv = (float(np.float32(v)) for v in (T, top_p, D))
        if not (math.isfinite(Tv) and Tv > 0):
            st |= STATUS_BAD_PARAM
        if not (tp > 0 and tp <= 1):
            st |= STATUS_BAD_PARAM
        if not (Dv >= 0 and Dv <= 1):
            st |= STATUS_BAD_PARAM
        rows = list(z_target) + list(z_draft)
        if any(not _finite_row(r) for r in rows):
            st |= STATUS_BAD_LOGITS
    else:
        zt = np.asarray(z_target, dtype=np.float32)
        if np.isnan(zt).any() or np.isposinf(zt).any():
            st |= STATUS_BAD_LOGITS
    return st


def verify_request(z_target: np.ndarray, z_draft: np.ndarray, x: np.ndarray, hist: np.ndarray,
                   T: float, alpha: float, top_p: float, D: float, u: np.ndarray,
                   *, bonus: bool = True) -> Dict:
    """Mentored speculative sampling for one request.

    z_target: [K+1, V] logits for [last committed, d1..dK]; z_draft: [K, V];
    x: the K drafted tokens; u: K acceptance uniforms then the final one.

    Returns a dict with ``tokens`` (K+1 slots: accepted prefix, then the
    correction or bonus, then -1), ``accepted``, ``status`` and the
    per-position quantities ``tv``, ``theta``, ``p_x``, ``q_x``, ``accept``
    (evaluated at every position), ``near_tie`` and ``margin``.
    """
    z_target = np.asarray(z_target)
    z_draft = np.asarray(z_draft)
    K = len(x)
    V = z_target.shape[1]
    out_tokens = [-1] * (K + 1)
    res = dict(tokens=out_tokens, accepted=-1, status=0, tv=[math.nan] * K,
               theta=[math.nan] * K, p_x=[math.nan] * K, q_x=[math.nan] * K,
               accept=[False] * K, near_tie=False, margin=math.inf)
    st = validate_request(V, z_target, z_draft, x, hist, T, alpha, top_p, D, sampling=True)
    res["status"] = st
    if st:
        return res

    p_rows, q_rows, tp_margin_p, tp_margin_q = [], [], [], []
    for i in range(K + 1):
        pen = penalty_set(hist, x[:i])
        p, mp = process_row(z_target[i], pen, alpha, T, top_p)
        p_rows.append(p)
        tp_margin_p.append(mp)
        if i < K:
            q, mq = process_row(z_draft[i], pen, alpha, T, top_p)
            q_rows.append(q)
            tp_margin_q.append(mq)

    acc_margin = []
    for i in range(K):
        p, q = p_rows[i], q_rows[i]
        d = tv_distance(p, q)
        th = mentored_theta(d, D)
        xi = int(x[i])
        pi_x = mixture_at(p[xi], q[xi], th)
        a, m = accept_draft(u[i], pi_x, q[xi])
        res["tv"][i], res["theta"][i] = d, th
        res["p_x"][i], res["q_x"][i] = float(p[xi]), float(q[xi])
        res["accept"][i] = a
        acc_margin.append(m)

    j = next((i for i in range(K) if not res["accept"][i]), K)
    if j < K:
        r = residual(p_rows[j], q_rows[j])
        w = r if np.sum(r) > 0 else p_rows[j]
        tok, fin_margin = inverse_cdf(w, u[K])
        n_emit = j + 1
    elif bonus:
        tok, fin_margin = inverse_cdf(p_rows[K], u[K])
        n_emit = K + 1
    else:
        tok, fin_margin = None, math.inf
        n_emit = K
    for i in range(j):
        out_tokens[i] = int(x[i])
    if tok is not None:
        out_tokens[j] = int(tok)
    res["accepted"] = j

    margins = acc_margin[:min(j + 1, K)] + [fin_margin]
    margins += tp_margin_p[:j + 1] + tp_margin_q[:min(j + 1, K)]
    res["margin"] = min(margins) if margins else math.inf
    res["near_tie"] = res["margin"] < NEAR_TIE
    res["n_emit"] = n_emit
    return res


def greedy_request(z_target: np.ndarray, x: np.ndarray, hist: np.ndarray, alpha: float) -> Dict:
    """Greedy longest-prefix verification for one request.

    g_i = argmax of the penalised target row i (lowest id on exact ties; the
    comparison is made on the fp32 penalised logits); j = first i < K with
    g_i != x_i (K if none); emit x_0..x_{j-1} then g_j (the correction, or the
    bonus g_K when every draft matches)."""
    z_target = np.asarray(z_target)
    K = len(x)
    V = z_target.shape[1]
    out_tokens = [-1] * (K + 1)
    res = dict(tokens=out_tokens, accepted=-1, status=0, argmax=[-1] * (K + 1))
    st = validate_request(V, z_target, [], x, hist, 1.0, alpha, 1.0, 0.0, sampling=False)
    res["status"] = st
    if st:
        return res
    g = []
    for i in range(K + 1):
        zp = apply_repetition_penalty(z_target[i], penalty_set(hist, x[:i]), alpha)
        g.append(int(np.argmax(zp)))
    res["argmax"] = g
    j = next((i for i in range(K) if g[i] != int(x[i])), K)
    for i in range(j):
        out_tokens[i] = int(x[i])
    out_tokens[j] = g[j]
    res["accepted"] = j
    return res


def tv_budget_request(z_target, z_draft, x, hist, T, alpha, top_p, D) -> Dict:
    """Per-position d, theta, p(x), q(x) (no sampling)."""
    K = len(x)
    u = np.zeros(K + 1, dtype=np.float32)
    r = verify_request(z_target, z_draft, x, hist, T, alpha, top_p, D, u)
    return dict(tv=r["tv"], theta=r["theta"], p_x=r["p_x"], q_x=r["q_x"], status=r["status"])


# ---------------------------------------------------------------------------
# Packed batches (the layout the library uses)
# ---------------------------------------------------------------------------

def _unpack(batch, b):
    return batch.request(b)


def verify_batch(batch, requests: Optional[Iterable[int]] = None, *, bonus: bool = True) -> Dict:
    """Run ``verify_request`` over (a subset of) a packed batch.  Returns
    packed ``tokens`` [sum K + B] (-1 where not computed), ``accepted`` [B],
    ``status`` [B], per-position ``tv``, ``theta``, ``p_x``, ``q_x``
    [sum K] and ``near_tie`` [B]."""
    B = batch.B
    total = batch.total_drafts
    reqs = range(B) if requests is None else list(requests)
    out = dict(tokens=np.full(total + B, -1, np.int64), accepted=np.full(B, -1, np.int64),
               status=np.zeros(B, np.int64), tv=np.full(total, np.nan), theta=np.full(total, np.nan),
               p_x=np.full(total, np.nan), q_x=np.full(total, np.nan),
               near_tie=np.zeros(B, bool), margin=np.full(B, np.inf), computed=np.zeros(B, bool))
    for b in reqs:
        a = _unpack(batch, b)
        r = verify_request(a["z_target"], a["z_draft"], a["x"], a["hist"], a["T"], a["alpha"],
                           a["top_p"], a["D"], a["u"], bonus=bonus)
        d0 = int(batch.cu_draft[b])
        off = d0 + b
        K = batch.k(b)
        out["tokens"][off:off + K + 1] = r["tokens"]
        out["accepted"][b] = r["accepted"]
        out["status"][b] = r["status"]
        out["tv"][d0:d0 + K] = r["tv"]
        out["theta"][d0:d0 + K] = r["theta"]
        out["p_x"][d0:d0 + K] = r["p_x"]
        out["q_x"][d0:d0 + K] = r["q_x"]
        out["near_tie"][b] = r["near_tie"]
        out["margin"][b] = r["margin"]
        out["computed"][b] = True
    return out


# ---------------------------------------------------------------------------
# Draft confidence early stop ("Adaptive-SpecDecode-Lab" README, section
# "Confidence-guided early stop": after each draft token the draft's own
# top-1 probability is read from the logits it already has; below the
# threshold, drafting stops, and that low-confidence token is still verified)
# ---------------------------------------------------------------------------

def draft_confidence_request(z_draft: np.ndarray, x: np.ndarray, hist: np.ndarray, T: float, alpha: float,
                             threshold: float) -> Dict:
    """Per draft row i: conf_i = max_v q_i(v), q_i the draft distribution
    after repetition penalty (history plus the drafts before row i) and
    temperature.  k_eff = i + 1 for the first i with conf_i < threshold, else
    K: the number of drafts a confidence-stopped drafter would have proposed.
    Returns conf [K], k_eff, status, and per row the margin |conf - threshold|
    (a decision closer than NEAR_TIE is a near tie)."""
    K = len(x)
    V = np.asarray(z_draft).shape[1]   # [K, V] even when K = 0
    st = STATUS_OK
    if K > MAX_K:
        st |= STATUS_BAD_K
    if any(int(t) < 0 or int(t) >= V for t in list(x) + list(hist)):
        st |= STATUS_BAD_TOKEN
    a = float(np.float32(alpha))
    Tv = float(np.float32(T))
    if not (math.isfinite(a) and a > 0) or not (math.isfinite(Tv) and Tv > 0):
        st |= STATUS_BAD_PARAM
    if any(not _finite_row(r) for r in z_draft):
        st |= STATUS_BAD_LOGITS
    conf = np.full(K, np.nan)
    margin = np.full(K, np.inf)
    if st:
        return dict(conf=conf, k_eff=-1, status=st, margin=margin)
    k_eff = K
    for i in range(K):
        zp = apply_repetition_penalty(z_draft[i], penalty_set(hist, x[:i]), alpha)
        conf[i] = float(np.max(softmax(apply_temperature(zp, T))))
        margin[i] = abs(conf[i] - float(np.float32(threshold)))
        if k_eff == K and conf[i] < float(np.float32(threshold)):
            k_eff = i + 1
    return dict(conf=conf, k_eff=k_eff, status=st, margin=margin)


def draft_confidence_batch(batch, threshold: float, requests: Optional[Iterable[int]] = None) -> Dict:
    """``draft_confidence_request`` over (a subset of) a packed batch:
    conf [sum K], k_eff [B], status [B], near_tie [B] (a row whose early-stop
    decision lies within NEAR_TIE of the threshold, up to k_eff)."""
    B = batch.B
    total = batch.total_drafts
    reqs = range(B) if requests is None else list(requests)
    out = dict(conf=np.full(total, np.nan), k_eff=np.full(B, -1, np.int64), status=np.zeros(B, np.int64),
               near_tie=np.zeros(B, bool))
    for b in reqs:
        a = _unpack(batch, b)
        r = draft_confidence_request(a["z_draft"], a["x"], a["hist"], a["T"], a["alpha"], threshold)
        d0 = int(batch.cu_draft[b])
        out["conf"][d0:d0 + len(a["x"])] = r["conf"]
        out["k_eff"][b] = r["k_eff"]
        out["status"][b] = r["status"]
        upto = r["k_eff"] if r["k_eff"] > 0 else 0
        out["near_tie"][b] = bool(np.any(r["margin"][:upto] < NEAR_TIE))
    return out


def greedy_batch(batch, requests: Optional[Iterable[int]] = None) -> Dict:
    B = batch.B
    total = batch.total_drafts
    reqs = range(B) if requests is None else list(requests)
    out = dict(tokens=np.full(total + B, -1, np.int64), accepted=np.full(B, -1, np.int64),
               status=np.zeros(B, np.int64), computed=np.zeros(B, bool))
    for b in reqs:
        a = _unpack(batch, b)
        r = greedy_request(a["z_target"], a["x"], a["hist"], a["alpha"])
        off = int(batch.cu_draft[b]) + b
        K = batch.k(b)
        out["tokens"][off:off + K + 1] = r["tokens"]
        out["accepted"][b] = r["accepted"]
        out["status"][b] = r["status"]
        out["computed"][b] = True
    return out
