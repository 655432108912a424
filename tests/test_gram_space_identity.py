"""The Gram-space form of the iteration (Megatron-LM issue #6720, gram_once),
checked in float64 against the oracle's standard iteration.

With A_j = X_j X_j^T and Q_j = a I + b A'_j + c A'_j^2, where
A'_j = A_j + r_j I and r_j = ridge * tr(A_j) / m (r_j = 0 without the ridge),
one step is X_{j+1} = Q_j X_j. Q_j is symmetric, so
A_{j+1} = Q_j A_j Q_j, and X_k = P_k X_0 with P_0 = I, P_{j+1} = Q_j P_j:
only A_0 and the final product touch the long dimension n. The fp32
Gram-space path computes exactly this; these tests show the identity holds,
so that path is compared with the oracle of the standard iteration.
"""

import math

import numpy as np
import pytest

from oracle import ns as ons

A, B, C, EPS = 3.4445, -4.7750, 2.0315, 1e-7


def gram_space(t, steps, ridge=0.0):
    t = np.asarray(t, dtype=np.float64)
    g = t.reshape(t.shape[0], -1)
    tr = g.shape[0] > g.shape[1]
    x0 = g.T if tr else g
    x0 = x0 / (math.sqrt(float(np.sum(x0 * x0))) + EPS)
    m = x0.shape[0]
    eye = np.eye(m)
    a_j = x0 @ x0.T
    p = eye.copy()
    for _ in range(steps):
        ar = a_j + ridge * (np.trace(a_j) / m) * eye
        q = A * eye + B * ar + C * (ar @ ar)
        a_j = q @ a_j @ q
        p = q @ p
    x = p @ x0
    return (x.T if tr else x).reshape(t.shape)


@pytest.mark.parametrize("shape", [(16, 64), (64, 16), (24, 24), (8, 4, 5)])
@pytest.mark.parametrize("steps", [0, 1, 5])
@pytest.mark.parametrize("ridge", [0.0, 1e-5, 0.05])
def test_gram_space_equals_standard_iteration(shape, steps, ridge):
    rng = np.random.default_rng(abs(hash((shape, steps, ridge))) % 2**32)
    t = rng.standard_normal(shape)
    want = ons.newton_schulz(t, steps, A, B, C, EPS, ridge=ridge)
    assert ons.rel_fro_error(gram_space(t, steps, ridge), want) < 1e-11


def test_ridge_uses_the_unridged_gram_in_the_update():
    # the ridged A'_j only forms Q_j; propagating A'_j instead would change
    # the result whenever the ridge is non-zero
    rng = np.random.default_rng(9)
    t = rng.standard_normal((12, 40))
    ridge = 0.05
    x0 = t / (np.linalg.norm(t) + EPS)
    m = x0.shape[0]
    a_j, p = x0 @ x0.T, np.eye(m)
    for _ in range(5):
        ar = a_j + ridge * (np.trace(a_j) / m) * np.eye(m)
        q = A * np.eye(m) + B * ar + C * (ar @ ar)
        a_j = q @ ar @ q          # the wrong propagation
        p = q @ p
    wrong = p @ x0
    want = ons.newton_schulz(t, 5, A, B, C, EPS, ridge=ridge)
    assert ons.rel_fro_error(wrong, want) > 1e-3
