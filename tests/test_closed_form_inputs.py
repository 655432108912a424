"""The structured full-size input and its closed form, pinned on the CPU.

The GPU parity test at the largest sweep size (8192 x 65536) compares with
the closed form in closed_forms.py, because the float64 oracle cannot run
there in seconds. These tests tie that closed form and the generator to the
oracle on small sizes, and check the generator's exactness claims.
"""

import numpy as np
import pytest
import torch

import workloads
from closed_forms import hadamard_row_norms, row_gains
from oracle import ns as ons

W = workloads


@pytest.mark.parametrize("m,blocks", [(16, 1), (16, 4), (64, 2), (128, 8)])
def test_closed_form_matches_oracle(m, blocks):
    x, r, d = W.gen_hadamard_rows(m, blocks, seed=11 + m + blocks)
    xf = x.double().numpy()
    g = np.array(row_gains(hadamard_row_norms(m, r, d), W.STEPS, W.A_COEF, W.B_COEF, W.C_COEF, W.EPS))
    want = g[:, None] * xf
    got = ons.newton_schulz(xf, W.STEPS, W.A_COEF, W.B_COEF, W.C_COEF, W.EPS)
    assert ons.rel_fro_error(got, want) < 1e-10
    # the tall form: NS(X^T) = NS(X)^T
    got_t = ons.newton_schulz(xf.T.copy(), W.STEPS, W.A_COEF, W.B_COEF, W.C_COEF, W.EPS)
    assert ons.rel_fro_error(got_t, want.T) < 1e-10


def test_generator_rows_are_orthogonal_and_bf16_exact():
    m, blocks = 64, 3
    x, r, d = W.gen_hadamard_rows(m, blocks, seed=5)
    xf = x.double()
    gram = (xf @ xf.T).numpy()
    sq = np.array([ri * ri * m * sum(dj * dj for dj in d) for ri in r])
    assert np.array_equal(gram, np.diag(sq))                    # dyadic: exact in float64
    assert np.allclose(np.array(hadamard_row_norms(m, r, d)) ** 2, sq, rtol=1e-14, atol=0)
    # values as built in float64 survive the bf16 rounding unchanged
    vals = np.unique(np.abs(xf.numpy()))
    exact = {ri * dj for ri in r for dj in d}
    assert set(vals.tolist()) <= exact
    assert torch.equal(x.float().to(torch.bfloat16), x)


def test_generator_is_seeded():
    a = W.gen_hadamard_rows(32, 2, seed=3)
    b = W.gen_hadamard_rows(32, 2, seed=3)
    c = W.gen_hadamard_rows(32, 2, seed=4)
    assert torch.equal(a[0], b[0]) and a[1:] == b[1:]
    assert not torch.equal(a[0], c[0])
