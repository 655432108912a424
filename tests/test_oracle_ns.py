"""Pins for the float64 Newton-Schulz oracle (CPU only).

Each check compares the oracle with something other than itself: the
singular-value closed form (numpy's SVD as an independent library routine),
the scalar map on diagonal inputs, orthogonal equivariance, transpose
symmetry, a pure-Python brute force on tiny inputs, the zero matrix, and the
singular-value form of the trace ridge.
``test_oracle_mutants.py`` plants plausible mistakes in copies of the oracle
and shows that these pins catch each one.

Definition pinned: Megatron-Core API page owner_planning, ns_cost_fn (view
as (shape[0], prod(shape[1:])), normalise, transpose so rows <= cols,
A = X X^T, X = a X + (b A + c A A) X).
"""

import math

import numpy as np
import pytest

from oracle import ns as ons

A, B, C, EPS = 3.4445, -4.7750, 2.0315, 1e-7


def scalar_map(s, k, a=A, b=B, c=C):
    for _ in range(k):
        s = a * s + b * s ** 3 + c * s ** 5
    return s


def svd_closed_form(t, k, eps=EPS, a=A, b=B, c=C):
    """NS_k(G) = U p^k(sigma / (||G||_F + eps)) V^T, G the 2-D view."""
    t = np.asarray(t, dtype=np.float64)
    g = t.reshape(t.shape[0], -1)
    u, s, vt = np.linalg.svd(g, full_matrices=False)
    nu = math.sqrt(float(np.sum(s * s))) + eps   # ||G||_F from the singular values
    ps = np.array([scalar_map(float(x) / nu, k, a, b, c) for x in s])
    return ((u * ps) @ vt).reshape(t.shape)


def rel(x, y):
    return float(np.linalg.norm(np.asarray(x) - np.asarray(y)) / max(np.linalg.norm(y), 1e-300))


@pytest.mark.parametrize("shape", [(40, 70), (70, 40), (32, 32), (8, 3, 2, 2), (5, 1), (1, 9), (24, 6, 5)])
@pytest.mark.parametrize("k", [1, 5])
def test_svd_closed_form(shape, k):
    rng = np.random.default_rng(abs(hash((shape, k))) % 2**32)
    t = rng.standard_normal(shape)
    got = ons.newton_schulz(t, k, A, B, C, EPS)
    assert got.shape == t.shape
    assert rel(got, svd_closed_form(t, k)) < 1e-10


def test_eps_is_added_to_the_norm():
    # At ||G|| ~ eps the result depends on how eps enters; the closed form uses
    # ||G||_F + eps (the reading stated for the oracle).
    rng = np.random.default_rng(7)
    t = rng.standard_normal((12, 20))
    t *= 1e-7 / np.linalg.norm(t)
    got = ons.newton_schulz(t, 5, A, B, C, EPS)
    assert rel(got, svd_closed_form(t, 5)) < 1e-10
    # and a max(norm, eps) reading would give a visibly different answer
    alt = svd_closed_form(t, 5, eps=0.0)
    assert rel(alt, got) > 1e-2


@pytest.mark.parametrize("m,n", [(6, 10), (10, 6), (7, 7)])
def test_diagonal_scalar_map(m, n):
    d = np.array([1.0, 0.5, 0.1, 0.01, 2.0, 0.3, 0.05][:min(m, n)])
    t = np.zeros((m, n))
    for i, v in enumerate(d):
        t[i, i] = v
    nu = math.sqrt(sum(v * v for v in d)) + EPS
    want = np.zeros((m, n))
    for i, v in enumerate(d):
        want[i, i] = scalar_map(v / nu, 5)
    got = ons.newton_schulz(t, 5, A, B, C, EPS)
    assert np.max(np.abs(got - want)) < 1e-13


def test_scalar_map_values():
    # p^5 on a few starting values (worked by hand from the scalar map)
    assert abs(scalar_map(1.0, 1) - (A + B + C)) < 1e-15
    assert abs(scalar_map(1.0, 1) - 0.701) < 1e-12


@pytest.mark.parametrize("shape", [(16, 24), (24, 16), (20, 20)])
def test_orthogonal_equivariance(shape):
    rng = np.random.default_rng(11)
    x = rng.standard_normal(shape)
    u, _ = np.linalg.qr(rng.standard_normal((shape[0], shape[0])))
    v, _ = np.linalg.qr(rng.standard_normal((shape[1], shape[1])))
    lhs = ons.newton_schulz(u @ x @ v.T, 5, A, B, C, EPS)
    rhs = u @ ons.newton_schulz(x, 5, A, B, C, EPS) @ v.T
    assert rel(lhs, rhs) < 1e-10


@pytest.mark.parametrize("shape", [(9, 14), (14, 9), (11, 11)])
def test_transpose_symmetry(shape):
    rng = np.random.default_rng(3)
    x = rng.standard_normal(shape)
    assert rel(ons.newton_schulz(x.T, 5, A, B, C, EPS), ons.newton_schulz(x, 5, A, B, C, EPS).T) < 1e-12


@pytest.mark.parametrize("shape", [(3, 5), (5, 3), (4, 4), (1, 6), (6, 1), (2, 2)])
def test_brute_force_loops(shape):
    rng = np.random.default_rng(5)
    x = rng.standard_normal(shape)
    want = np.array(ons.newton_schulz_loops(x.tolist(), 5, A, B, C, EPS))
    got = ons.newton_schulz(x, 5, A, B, C, EPS)
    assert np.max(np.abs(got - want)) < 1e-12


def test_zero_matrix():
    z = np.zeros((6, 9))
    assert np.all(ons.newton_schulz(z, 5, A, B, C, EPS) == 0.0)


def test_scale_invariance():
    rng = np.random.default_rng(9)
    x = rng.standard_normal((10, 30))
    assert rel(ons.newton_schulz(37.0 * x, 5, A, B, C, EPS), ons.newton_schulz(x, 5, A, B, C, EPS)) < 1e-6


def test_output_singular_values_in_band():
    # For Gaussian inputs the normalised singular values lie in (0, 1]; after 5
    # steps they land in p^5's image of that interval, not at 1 (5 steps do not
    # orthogonalise exactly).
    rng = np.random.default_rng(1)
    x = rng.standard_normal((64, 256))
    s = np.linalg.svd(ons.newton_schulz(x, 5, A, B, C, EPS), compute_uv=False)
    assert s.min() > 0.6 and s.max() < 1.2


def test_ridge_zero_is_plain():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((10, 30))
    assert np.array_equal(ons.newton_schulz(x, 5, A, B, C, EPS, ridge=0.0),
                          ons.newton_schulz(x, 5, A, B, C, EPS))


def ridge_closed_form(t, k, lam, eps=EPS, a=A, b=B, c=C):
    """NS_k with the trace ridge (A <- A + lam tr(A)/m I before B) through the
    SVD G = U diag(sigma) V^T: A's eigenvalues are sigma_i^2 and tr(A) is their
    sum over the m = min(rows, cols) singular values, so every step is the
    coupled scalar map sigma_i <- a sigma_i + (b q_i + c q_i^2) sigma_i with
    q_i = sigma_i^2 + lam * mean(sigma^2)."""
    t = np.asarray(t, dtype=np.float64)
    g = t.reshape(t.shape[0], -1)
    u, s, vt = np.linalg.svd(g, full_matrices=False)
    nu = math.sqrt(float(np.sum(s * s))) + eps
    sig = [float(x) / nu for x in s]
    m = len(sig)
    for _ in range(k):
        r = lam * sum(x * x for x in sig) / m
        sig = [a * x + (b * (x * x + r) + c * (x * x + r) ** 2) * x for x in sig]
    return ((u * np.array(sig)) @ vt).reshape(t.shape)


@pytest.mark.parametrize("shape", [(24, 60), (60, 24), (16, 16), (6, 2, 5)])
@pytest.mark.parametrize("lam", [1e-5, 0.05])
def test_ridge_closed_form(shape, lam):
    # the trace ridge of the fp32-Gram mode, pinned to its singular-value
    # closed form (a large lam as well, so a wrong trace scale shows)
    rng = np.random.default_rng(abs(hash((shape, lam))) % 2**32)
    t = rng.standard_normal(shape)
    got = ons.newton_schulz(t, 5, A, B, C, EPS, ridge=lam)
    assert rel(got, ridge_closed_form(t, 5, lam)) < 1e-10
    if lam >= 0.05:
        assert rel(got, svd_closed_form(t, 5)) > 1e-3   # the ridge changes the result


def test_useful_flops():
    # k (4 m^2 n + 2 m^3), m = min, n = max; 128x256, 5 steps by hand:
    # 4*128*128*256 = 16777216, 2*128^3 = 4194304, sum 20971520, x5 = 104857600
    assert ons.useful_flops((128, 256), 5) == 104857600
    assert ons.useful_flops((256, 128), 5) == 104857600


# --- the per-matrix error measure every parity check goes through ----------
# Hand-worked values of ||y - y_ref||_F / ||y_ref||_F (and ||y||_F when
# y_ref = 0). Each case is chosen so that a plausible slip gives a different
# number: the squared ratio, the wrong denominator (||y|| instead of
# ||y_ref||), a max-abs or per-row norm, or a norm over one slice only.
ERROR_HAND_CASES = [
    # diff = [[3, 0], [0, -1]]: sqrt(9 + 1) = sqrt(10); ||y_ref|| = 5
    ([[3.0, 0.0], [0.0, 4.0]], [[0.0, 0.0], [0.0, 5.0]], math.sqrt(10.0) / 5.0),
    # diff = [[-1, 1]]: sqrt(2); ||y_ref|| = 2 (||y|| = sqrt(2) would give 1)
    ([[1.0, 1.0]], [[2.0, 0.0]], math.sqrt(2.0) / 2.0),
    # diff = [1, 1, 1, -1]: Frobenius 2 (max-abs 1); ||y_ref|| = 2
    ([[1.0, 1.0, 1.0, 1.0]], [[0.0, 0.0, 0.0, 2.0]], 1.0),
    # rows: row 0 exact, row 1 off by 3 against ||y_ref|| = sqrt(16 + 9) = 5
    # (the mean of per-row errors would be (0 + 3/3) / 2 = 0.5)
    ([[4.0, 0.0], [0.0, 6.0]], [[4.0, 0.0], [0.0, 3.0]], 3.0 / 5.0),
    # a 3-D tensor: the norm runs over every element, not one slice
    ([[[1.0, 0.0]], [[0.0, 2.0]]], [[[1.0, 0.0]], [[0.0, 0.0]]], 2.0),
    # y_ref = 0: the absolute Frobenius norm of y, sqrt(1 + 4 + 4 + 16) = 5
    ([[1.0, 2.0], [2.0, 4.0]], [[0.0, 0.0], [0.0, 0.0]], 5.0),
    # equal inputs: exactly 0
    ([[0.5, -0.25], [2.0, 8.0]], [[0.5, -0.25], [2.0, 8.0]], 0.0),
]


@pytest.mark.parametrize("y,y_ref,want", ERROR_HAND_CASES)
def test_rel_fro_error_hand_cases(y, y_ref, want):
    got = ons.rel_fro_error(np.array(y), np.array(y_ref))
    assert abs(got - want) <= 1e-15 * max(1.0, want), (got, want)


def test_rel_fro_error_properties():
    rng = np.random.default_rng(7)
    y_ref = rng.standard_normal((13, 21))
    d = rng.standard_normal((13, 21))
    d *= 1e-3 * np.linalg.norm(y_ref) / np.linalg.norm(d)
    # a perturbation of relative size 1e-3 measures 1e-3, in either sign
    assert abs(ons.rel_fro_error(y_ref + d, y_ref) - 1e-3) < 1e-15
    assert abs(ons.rel_fro_error(y_ref - d, y_ref) - 1e-3) < 1e-15
    # invariant to a common scale of both arguments
    assert abs(ons.rel_fro_error(4.0 * (y_ref + d), 4.0 * y_ref) - 1e-3) < 1e-15
    # float32 and bfloat16-sized inputs are measured in float64
    y32 = (y_ref + d).astype(np.float32)
    assert abs(ons.rel_fro_error(y32, y_ref) - np.linalg.norm(y32.astype(np.float64) - y_ref)
               / np.linalg.norm(y_ref)) < 1e-15
