"""Pins for the oracle's near-tie margins.

A margin is the distance, in units of the uniform a decision consumes, from
that decision to a tie; requests with a margin below ``NEAR_TIE`` (1e-6) are
counted instead of compared bit for bit.  A margin in the wrong units, or a
decision left out of a request's minimum, would silently excuse real
mismatches, so each margin is pinned here to a hand-computed value on inputs
that are exact in binary, and the composition of a request's margin is pinned
to which decisions the method actually consumes:

* the acceptance test u*q(x) < pi(x) ("What I Gave Up to Make Speculative
  Decoding Faster", section "A knob for accepting more draft tokens") has
  the threshold pi(x)/q(x) on u;
* an inverse-CDF draw (the residual or bonus token) has the thresholds
  C(v)/R on u, C the inclusive prefix mass;
* top-p ("Speculative Decoding" note, section "Warum eine Korrektur noetig
  ist") is decided by the cumulative mass against top_p and by the order of
  nearly equal probabilities.

Only the decisions that reach the output count: the acceptance tests of
positions 0..j (j the first rejection), the final draw, and the top-p cuts
of the rows those read (p rows 0..j, q rows 0..min(j, K-1)).  Each
``_pin_*`` helper below is also run against a planted mistake (a margin
scaled by 10, or a margin dropped) and must fail there.
"""
import math

import numpy as np
import pytest

from oracle import oracle as O

F32 = np.float32


def _one(zt, zd, x, u, D, T=1.0, top_p=1.0):
    return O.verify_request(np.asarray(zt, F32), np.asarray(zd, F32), np.asarray(x), np.zeros(0, np.int64),
                            T, 1.0, top_p, D, np.asarray(u, F32))


# ---------------------------------------------------------------- accept_draft

def _pin_accept_margin():
    # pi/q = 0.3/0.6 = 0.5; u sits 8 float32 ulps (2^-24 each) above it
    u = F32(0.5 + 8 * 2.0 ** -24)
    acc, m = O.accept_draft(u, 0.3, 0.6)
    assert not acc
    assert abs(m - 8 * 2.0 ** -24) < 1e-15            # units of u, not of q or pi
    assert m < O.NEAR_TIE
    # the same threshold with a 60x smaller q: the margin does not scale with q
    acc, m = O.accept_draft(u, 0.005, 0.01)
    assert not acc and abs(m - 8 * 2.0 ** -24) < 1e-15
    # 64 ulps below (2^-25 each, 1.9e-6) is not a tie; the draft is accepted
    acc, m = O.accept_draft(F32(0.5 - 64 * 2.0 ** -25), 0.3, 0.6)
    assert acc and abs(m - 64 * 2.0 ** -25) < 1e-15 and m >= O.NEAR_TIE


def test_accept_margin():
    _pin_accept_margin()


# ----------------------------------------------------------------- inverse_cdf

def _pin_inverse_cdf_margin():
    w = np.array([1.0, 2.0, 1.0])                     # R = 4: boundaries at u = 1/4 and 3/4
    u = F32(0.25 + 2.0 ** -23)
    v, m = O.inverse_cdf(w, u)
    assert v == 1 and abs(m - 2.0 ** -23) < 1e-15      # distance to the boundary 1/4, in u units
    v, m = O.inverse_cdf(w, F32(0.625))
    assert v == 1 and abs(m - 0.125) < 1e-15           # nearest boundary is 3/4
    # zero weights: the boundary between tokens 1 and 3 is u = 1/2
    w = np.array([0.0, 0.5, 0.0, 0.5])
    v, m = O.inverse_cdf(w, F32(0.5))
    assert v == 3 and m == 0.0
    v, m = O.inverse_cdf(w, F32(0.5 - 2.0 ** -25))
    assert v == 1 and abs(m - 2.0 ** -25) < 1e-15


def test_inverse_cdf_margin():
    _pin_inverse_cdf_margin()


# ---------------------------------------------------------------- top_p_filter

def _pin_top_p_margins():
    p = np.array([0.5, 0.25, 0.25])                    # cumulative 0.5, 0.75, 1 (exact)
    # top_p 2^-23 above the cumulative mass 0.75: the cut moves to the third token
    out, m = O.top_p_filter(p, F32(0.75 + 2.0 ** -23))
    np.testing.assert_array_equal(out, p)
    assert abs(m - 2.0 ** -23) < 1e-15
    # exactly at the cumulative mass: a tie
    _, m = O.top_p_filter(p, F32(0.75))
    assert m == 0.0
    # far from the cumulative masses (0.5 and 0.75 against 0.6)
    _, m = O.top_p_filter(p, F32(0.6))
    assert abs(m - (float(F32(0.6)) - 0.5)) < 1e-15
    # two probabilities 2^-24 apart relatively: the one just below the cut
    # is excluded, and the relative gap is the margin
    p = np.array([0.5, 0.25, 0.25 - 2.0 ** -26, 2.0 ** -26])
    out, m = O.top_p_filter(p, F32(0.6))
    np.testing.assert_allclose(out, [2 / 3, 1 / 3, 0.0, 0.0], rtol=1e-15)
    assert abs(m - 2.0 ** -24) < 1e-18
    # the same gap above the cut: [0.25 + 2^-26] is just above tau = 0.25
    p = np.array([0.25 + 2.0 ** -26, 0.25, 0.5 - 2.0 ** -26])
    _, m = O.top_p_filter(p, F32(0.8))
    assert abs(m - 2.0 ** -26 / (0.25 + 2.0 ** -26)) < 1e-18


def test_top_p_margins():
    _pin_top_p_margins()


# ----------------------------------------------- which decisions a request counts

# Rows with exact small-integer logits at T = 1, D = 0 (pi = p): thresholds
# p(x)/q(x) are computed here from the oracle's reported p(x), q(x), and the
# uniforms are placed at chosen distances from them.
_ZT = np.array([[2.0, 0.0, 1.0, -1.0],
                [0.0, 1.5, -0.5, 0.5],
                [1.0, -1.0, 0.0, 2.0],
                [0.3, 0.2, 0.1, 0.0]], F32)
_ZD = np.array([[1.0, 0.5, 2.0, 0.0],
                [1.5, 0.0, 0.0, 1.0],
                [0.0, 0.0, 2.5, 0.0]], F32)
_X = [2, 0, 2]       # q > p at each position, so each can be rejected


def _thresholds():
    r = _one(_ZT, _ZD, _X, [0.0, 0.0, 0.0, 0.5], D=0.0)
    return [r["p_x"][i] / r["q_x"][i] for i in range(3)]


def _residual_boundaries(j):
    """Boundaries C(v)/R of the residual draw at position j, from an
    independent softmax of the same rows."""
    def sm(z):
        e = np.exp(z.astype(np.float64) - z.max())
        return e / e.sum()
    r = np.maximum(sm(_ZT[j]) - sm(_ZD[j]), 0.0)
    return np.cumsum(r)[:-1] / r.sum()


def _pin_request_margin_composition():
    t = _thresholds()
    assert all(0.05 < x < 0.95 for x in t)
    bnd = _residual_boundaries(1)
    mid = float(F32(0.5 * (bnd[0] + bnd[1]))) if len(bnd) > 1 else 0.5
    # accept 0 (u0 0.05 below), reject 1 (u1 0.05 above), position 2 sits on
    # its threshold: it comes after the first rejection and must not count
    u = [F32(t[0] - 0.05), F32(t[1] + 0.05), F32(t[2]), F32(mid)]
    r = _one(_ZT, _ZD, _X, u, D=0.0)
    assert r["accepted"] == 1
    fin = min(abs(mid - b) for b in bnd)
    want = min(abs(float(u[0]) - t[0]), abs(float(u[1]) - t[1]), fin)
    assert abs(r["margin"] - want) < 1e-9 and not r["near_tie"]
    # the rejected position's own test counts ...
    u1 = list(u)
    u1[1] = F32(t[1] * (1 + 2e-7))
    r = _one(_ZT, _ZD, _X, u1, D=0.0)
    assert r["accepted"] == 1 and r["near_tie"] and r["margin"] < 1e-6
    # ... and so does an accepted one before it
    u0 = list(u)
    u0[0] = F32(t[0] * (1 - 2e-7))
    r = _one(_ZT, _ZD, _X, u0, D=0.0)
    assert r["accepted"] == 1 and r["near_tie"]
    # the final draw counts: u_fin on a residual boundary
    uf = list(u)
    uf[3] = F32(bnd[0])
    r = _one(_ZT, _ZD, _X, uf, D=0.0)
    assert r["accepted"] == 1 and r["near_tie"] and r["margin"] < 1e-7
    # full acceptance: every test and the bonus draw count
    ua = [F32(t[0] - 0.05), F32(t[1] - 0.05), F32(t[2] * (1 - 2e-7)), F32(0.5)]
    r = _one(_ZT, _ZD, _X, ua, D=0.0)
    assert r["accepted"] == 3 and r["near_tie"]


def test_request_margin_composition():
    _pin_request_margin_composition()


# Top-p rows (top_p = 3/4): logits ln 2, 0, 0 give probabilities 1/2, 1/4,
# 1/4 up to the float32 rounding of ln 2, which puts that row's cut on a tie;
# the other rows are at least 0.04 from any tie.  Drafts x = [0, 2] have
# q(x) > p(x), so either position can be rejected; a tie row keeps that
# (its 1/2 sits on the draft token in a q row, elsewhere in a p row).
_LN2 = float(F32(math.log(2.0)))


def _tie_row(kind, row):
    z = np.array([0.0, 0.0, 0.0, -30.0], F32)
    x = [0, 2, 1][row]
    z[x if kind == "q" else (x + 1) % 3] = _LN2
    return z


_P_ROWS = np.array([[0.7, -0.2, 1.8, -30.0],     # p0 = [0.25, 0, 0.75] after the cut
                    [0.0, 1.3, 0.4, -30.0],      # p1 = [0, 0.71, 0.29]
                    [1.9, 0.0, -1.1, -30.0]], F32)
_Q_ROWS = np.array([[1.0, 0.0, 0.2, -30.0],      # q0 = [0.69, 0, 0.31]
                    [0.0, 0.3, 1.5, -30.0]], F32)  # q1 = [0, 0.23, 0.77]


def _topp_request(tie, reject_at):
    """`tie` = ("p"|"q", row) replaced by the tie row; reject_at = 0, 1 or
    None (accept both drafts)."""
    zt, zd = _P_ROWS.copy(), _Q_ROWS.copy()
    (zt if tie[0] == "p" else zd)[tie[1]] = _tie_row(*tie)
    x = [0, 2]
    base = _one(zt, zd, x, [0.0, 0.0, 0.5], D=0.0, top_p=0.75)
    t = [base["p_x"][i] / base["q_x"][i] for i in range(2)]
    assert all(v > 0.2 for v in t), t
    u = [0.0, 0.0, 0.37]
    if reject_at is not None:
        assert t[reject_at] < 0.9, t
        u[reject_at] = F32(t[reject_at] + 0.05)
    r = _one(zt, zd, x, u, D=0.0, top_p=0.75)
    assert r["accepted"] == (2 if reject_at is None else reject_at)
    return r


def _pin_top_p_composition():
    # the rows read up to a rejection at 0 are p row 0 and q row 0
    assert _topp_request(("q", 0), 0)["near_tie"]
    assert _topp_request(("p", 0), 0)["near_tie"]
    assert not _topp_request(("q", 1), 0)["near_tie"]
    assert not _topp_request(("p", 1), 0)["near_tie"]
    assert not _topp_request(("p", 2), 0)["near_tie"]
    # a rejection at 1 reads the rows of position 1 too, not the bonus row
    assert _topp_request(("p", 1), 1)["near_tie"]
    assert _topp_request(("q", 1), 1)["near_tie"]
    assert not _topp_request(("p", 2), 1)["near_tie"]
    # full acceptance reads every row, the bonus row included
    assert _topp_request(("p", 2), None)["near_tie"]
    assert _topp_request(("q", 1), None)["near_tie"]


def test_top_p_margin_composition():
    _pin_top_p_composition()


# ------------------------------------------------------ planted mistakes (CPU)

def _scaled(fn, k):
    def wrapped(*a, **kw):
        out = fn(*a, **kw)
        return out[0], out[1] * k
    return wrapped


def _dropped(fn):
    def wrapped(*a, **kw):
        return fn(*a, **kw)[0], math.inf
    return wrapped


@pytest.mark.parametrize("name,pin", [
    ("accept_draft", _pin_accept_margin),
    ("inverse_cdf", _pin_inverse_cdf_margin),
    ("top_p_filter", _pin_top_p_margins),
])
def test_scaled_margin_fails_its_pin(monkeypatch, name, pin):
    monkeypatch.setattr(O, name, _scaled(getattr(O, name), 10.0))
    with pytest.raises(AssertionError):
        pin()


@pytest.mark.parametrize("name,pin", [
    ("accept_draft", _pin_request_margin_composition),
    ("inverse_cdf", _pin_request_margin_composition),
    ("top_p_filter", _pin_top_p_composition),
])
def test_dropped_margin_fails_composition(monkeypatch, name, pin):
    monkeypatch.setattr(O, name, _dropped(getattr(O, name)))
    with pytest.raises(AssertionError):
        pin()
