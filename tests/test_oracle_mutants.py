"""Planted mistakes: each copy of the oracle below carries one plausible
error, and at least one of the pins used on the real oracle must reject it.
This shows the pins are strong enough to catch a dropped term, a wrong sign,
a transposed operand, a wrong view, a wrong normalisation, a misplaced
trace ridge or a wrong tie-break -- on the CPU, never on a GPU.
"""

import math

import numpy as np
import pytest

from oracle import ns as ons
from oracle import planning as op
from test_oracle_ns import A, B, C, EPS, svd_closed_form, ridge_closed_form, scalar_map, rel
from test_oracle_planning import load


def ns_variant(t, k, a, b, c, eps, *, view="first", gram="xxt", norm="fro_plus",
               back=True, steps_off=0, order="poly_x"):
    t = np.asarray(t, dtype=np.float64)
    shape = t.shape
    if view == "first":
        g = t.reshape(shape[0], -1)
    else:                                   # mistake: last dim as cols
        g = t.reshape(-1, shape[-1])
    tr = g.shape[0] > g.shape[1]
    x = g.T if tr else g
    nrm = math.sqrt(float(np.sum(x * x)))
    if norm == "fro_plus":
        x = x / (nrm + eps)
    elif norm == "fro_max":
        x = x / max(nrm, eps)
    elif norm == "spectral":
        x = x / (np.linalg.norm(x, 2) + eps)
    for _ in range(k + steps_off):
        gm = x @ x.T if gram == "xxt" else x.T @ x
        p = b * gm + c * (gm @ gm)
        if order == "poly_x":
            x = a * x + p @ x
        else:                                # mistake: a folded into the wrong place
            x = (a * gm + p) @ x
    if tr and back:
        x = x.T
    return x.reshape(shape) if x.size == t.size and (not tr or back) else x


def pins_pass(fn) -> bool:
    """Run the NS pins against `fn`; True iff every pin passes."""
    rng = np.random.default_rng(123)
    try:
        for shape in [(40, 70), (70, 40), (32, 32), (8, 3, 2, 2)]:
            t = rng.standard_normal(shape)
            got = np.asarray(fn(t, 5, A, B, C, EPS))
            if got.shape != t.shape or rel(got, svd_closed_form(t, 5)) > 1e-10:
                return False
        t = rng.standard_normal((12, 20))
        t *= 1e-7 / np.linalg.norm(t)
        if rel(fn(t, 5, A, B, C, EPS), svd_closed_form(t, 5)) > 1e-10:
            return False
        d = [1.0, 0.5, 0.1]
        t = np.zeros((3, 5))
        for i, v in enumerate(d):
            t[i, i] = v
        nu = math.sqrt(sum(v * v for v in d)) + EPS
        got = fn(t, 5, A, B, C, EPS)
        for i, v in enumerate(d):
            if abs(got[i, i] - scalar_map(v / nu, 5)) > 1e-13:
                return False
    except Exception:
        return False
    return True


def test_real_oracle_passes_pins():
    assert pins_pass(ons.newton_schulz)


MUTANTS = {
    "dropped c*A@A term": lambda t, k, a, b, c, e: ons.newton_schulz(t, k, a, b, 0.0, e),
    "wrong sign of b": lambda t, k, a, b, c, e: ons.newton_schulz(t, k, a, -b, c, e),
    "a and b swapped": lambda t, k, a, b, c, e: ons.newton_schulz(t, k, b, a, c, e),
    "one step short": lambda t, k, a, b, c, e: ns_variant(t, k, a, b, c, e, steps_off=-1),
    "Gram as X^T X": lambda t, k, a, b, c, e: ns_variant(t, k, a, b, c, e, gram="xtx"),
    "no transpose back": lambda t, k, a, b, c, e: ns_variant(t, k, a, b, c, e, back=False),
    "view as (prod(shape[:-1]), shape[-1])": lambda t, k, a, b, c, e: ns_variant(t, k, a, b, c, e, view="last"),
    "max(norm, eps) normalisation": lambda t, k, a, b, c, e: ns_variant(t, k, a, b, c, e, norm="fro_max"),
    "spectral-norm normalisation": lambda t, k, a, b, c, e: ns_variant(t, k, a, b, c, e, norm="spectral"),
    "a multiplies A instead of X": lambda t, k, a, b, c, e: ns_variant(t, k, a, b, c, e, order="a_gram"),
}


@pytest.mark.parametrize("name", list(MUTANTS))
def test_ns_mutant_is_caught(name):
    assert not pins_pass(MUTANTS[name])


def lpt_variant(works, *, ascending=False, singles_first=True, last_on_tie=False, reverse_ties=False):
    load_ = {}
    for w in works:
        for r in w.candidates:
            load_.setdefault(r, 0)
    single = [w for w in works if len(w.candidates) == 1] if singles_first else []
    multi = [w for w in works if not singles_first or len(w.candidates) > 1]
    if reverse_ties:
        multi = list(reversed(multi))
    multi.sort(key=lambda w: w.cost if ascending else -w.cost)
    out = {}
    for w in single + multi:
        best = w.candidates[0]
        for r in w.candidates[1:]:
            if load_[r] < load_[best] or (last_on_tie and load_[r] == load_[best]):
                best = r
        out[w.tensor_index] = best
        load_[best] += w.cost
    return out


def lpt_pins_pass(fn) -> bool:
    for case in load("planning_hand_cases.json")["lpt"]:
        works = [op.OwnerWork(i, c, cand) for i, (c, cand) in enumerate(zip(case["costs"], case["candidates"]))]
        got = fn(works)
        if [got[i] for i in range(len(case["costs"]))] != case["owners"]:
            return False
    return True


def test_real_lpt_passes_pins():
    assert lpt_pins_pass(op.assign_owner_work)
    assert lpt_pins_pass(lpt_variant)


@pytest.mark.parametrize("kw", [dict(ascending=True), dict(singles_first=False),
                                dict(last_on_tie=True), dict(reverse_ties=True)],
                         ids=["ascending cost", "no single-candidate pass", "last rank on load tie",
                              "reverse index on cost tie"])
def test_lpt_mutant_is_caught(kw):
    assert not lpt_pins_pass(lambda w: lpt_variant(w, **kw))


def ridge_variant(t, k, a, b, c, eps, lam, *, trace_over="m", where="gram"):
    """The oracle's iteration with one planted mistake in the trace ridge."""
    t = np.asarray(t, dtype=np.float64)
    shape = t.shape
    g = t.reshape(shape[0], -1)
    tr = g.shape[0] > g.shape[1]
    x = g.T if tr else g
    x = x / (math.sqrt(float(np.sum(x * x))) + eps)
    m, n = x.shape
    for _ in range(k):
        gm = x @ x.T
        d = {"m": m, "n": n, "one": 1}[trace_over]
        r = lam * np.trace(gm) / d
        if where == "gram":
            gr = gm + r * np.eye(m)
            p = b * gr + c * (gr @ gr)
        elif where == "linear_only":          # mistake: A^2 taken without the ridge
            p = b * (gm + r * np.eye(m)) + c * (gm @ gm)
        else:                                 # mistake: ridge added to B, not to A
            p = b * gm + c * (gm @ gm) + r * np.eye(m)
        x = a * x + p @ x
    if tr:
        x = x.T
    return x.reshape(shape)


def ridge_pins_pass(fn) -> bool:
    rng = np.random.default_rng(321)
    for shape in [(24, 60), (60, 24), (6, 2, 5)]:
        for lam in (1e-5, 0.05):
            t = rng.standard_normal(shape)
            if rel(fn(t, 5, A, B, C, EPS, lam), ridge_closed_form(t, 5, lam)) > 1e-10:
                return False
    return True


def test_real_ridge_passes_pins():
    assert ridge_pins_pass(lambda t, k, a, b, c, e, lam: ons.newton_schulz(t, k, a, b, c, e, ridge=lam))
    assert ridge_pins_pass(lambda t, k, a, b, c, e, lam: ridge_variant(t, k, a, b, c, e, lam))


RIDGE_MUTANTS = {
    "trace divided by n": dict(trace_over="n"),
    "trace not divided": dict(trace_over="one"),
    "A^2 without the ridge": dict(where="linear_only"),
    "ridge added to B": dict(where="poly"),
}


@pytest.mark.parametrize("name", list(RIDGE_MUTANTS))
def test_ridge_mutant_is_caught(name):
    kw = RIDGE_MUTANTS[name]
    assert not ridge_pins_pass(lambda t, k, a, b, c, e, lam: ridge_variant(t, k, a, b, c, e, lam, **kw))


# ------------------------------------------------- the error measure
def err_variant(y, y_ref, *, squared=False, den="ref", norm="fro"):
    y = np.asarray(y, dtype=np.float64)
    y_ref = np.asarray(y_ref, dtype=np.float64)
    d = y - y_ref

    def nrm(v):
        if norm == "maxabs":
            return float(np.max(np.abs(v))) if v.size else 0.0
        if norm == "first_slice":                     # mistake: one row / slice only
            return math.sqrt(float(np.sum(v.reshape(v.shape[0], -1)[0] ** 2)))
        return math.sqrt(float(np.sum(v * v)))

    base = {"ref": nrm(y_ref), "y": nrm(y), "sum": nrm(y) + nrm(y_ref)}[den]
    if base == 0.0:
        return nrm(d)
    r = nrm(d) / base
    return r * r if squared else r


def err_pins_pass(fn) -> bool:
    from test_oracle_ns import ERROR_HAND_CASES
    for y, y_ref, want in ERROR_HAND_CASES:
        if abs(fn(np.array(y), np.array(y_ref)) - want) > 1e-15 * max(1.0, want):
            return False
    return True


def test_real_error_measure_passes_pins():
    assert err_pins_pass(ons.rel_fro_error)


ERR_MUTANTS = {
    "squared ratio": dict(squared=True),
    "||y|| as the denominator": dict(den="y"),
    "||y|| + ||y_ref|| as the denominator": dict(den="sum"),
    "max-abs instead of Frobenius": dict(norm="maxabs"),
    "norm over the first row only": dict(norm="first_slice"),
}


@pytest.mark.parametrize("name", list(ERR_MUTANTS))
def test_error_measure_mutant_is_caught(name):
    kw = ERR_MUTANTS[name]
    assert not err_pins_pass(lambda y, r: err_variant(y, r, **kw)), name
