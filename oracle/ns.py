"""Oracle: quintic Newton-Schulz orthogonalisation on the CPU, in float64.

TEST INFRASTRUCTURE ONLY (see the package docstring): never imported by the
product path.

Definition followed: Megatron-Core API page
``core.distributed.fsdp.src.megatron_fsdp.experimental.owner_planning``,
entry ``ns_cost_fn``. A tensor is viewed as (rows, cols) = (shape[0],
prod(shape[1:])); after normalisation and a transpose that makes
rows <= cols, each step with scalar coefficients (a, b, c) is

    A = X @ X.T
    X = a * X + (b * A + c * (A @ A)) @ X

Readings where the page is silent (each is listed in the design notes):

* normalisation is X / (||X||_F + eps), eps added to the norm (not a max);
* the same (a, b, c) is used in every step;
* the result is transposed back and reshaped to the input's shape, because
  ``route_from_ns_home`` (page ``core.optimizer.layer_sharded_a2a``) hands
  out (P/S, Q) shards of a (P, Q) result;
* optional trace ridge (issue #6720 pairs an fp32/TF32 Gram with a trace ridge):
  A <- A + ridge * (trace(A) / m) * I before B is formed. The issue names
  the ridge but not its form; the oracle's ridge is pinned to the
  singular-value closed form of this reading.

The matrix products use numpy's float64 matmul (a library primitive); the
operation order is exactly the page's, with no fusion or reordering.
"""

from __future__ import annotations

import math

import numpy as np


def view_2d_shape(shape) -> tuple[int, int]:
    """(rows, cols) = (shape[0], prod(shape[1:])) -- ns_cost_fn, owner_planning page."""
    if len(shape) < 2:
        raise ValueError("Newton-Schulz needs a tensor with at least 2 dims")
    rows = int(shape[0])
    cols = 1
    for s in shape[1:]:
        cols *= int(s)
    return rows, cols


def newton_schulz(t, steps: int, a: float, b: float, c: float, eps: float,
                  ridge: float = 0.0) -> np.ndarray:
    """Return NS_k(t) in float64 with t's shape (owner_planning page, ns_cost_fn).

    ``t`` is any array with ndim >= 2; it is converted to float64 first (exact
    for bf16 and fp32 inputs).
    """
    t = np.asarray(t, dtype=np.float64)
    shape = t.shape
    rows, cols = view_2d_shape(shape)
    g = t.reshape(rows, cols)
    transposed = rows > cols
    x = g.T if transposed else g
    # normalise by the Frobenius norm plus eps
    x = x / (math.sqrt(float(np.sum(x * x))) + eps)
    m = x.shape[0]
    for _ in range(steps):
        gram = x @ x.T
        if ridge > 0.0:
            gram = gram + ridge * (np.trace(gram) / m) * np.eye(m)
        poly = b * gram + c * (gram @ gram)
        x = a * x + poly @ x
    if transposed:
        x = x.T
    return np.ascontiguousarray(x).reshape(shape)


def newton_schulz_loops(t, steps: int, a: float, b: float, c: float,
                        eps: float) -> list[list[float]]:
    """Same iteration in pure-Python loops, for tiny 2-D inputs only.

    Written independently of numpy (nested lists, explicit sums) so that it
    can cross-check ``newton_schulz`` by brute force. Returns the result as a
    list of rows in the input's (rows, cols) orientation.
    """
    rows = len(t)
    cols = len(t[0])
    if rows > cols:
        x = [[float(t[i][j]) for i in range(rows)] for j in range(cols)]
    else:
        x = [[float(v) for v in row] for row in t]
    m, n = len(x), len(x[0])
    sq = 0.0
    for i in range(m):
        for j in range(n):
            sq += x[i][j] * x[i][j]
    scale = 1.0 / (math.sqrt(sq) + eps)
    x = [[x[i][j] * scale for j in range(n)] for i in range(m)]
    for _ in range(steps):
        gram = [[sum(x[i][k] * x[j][k] for k in range(n)) for j in range(m)]
                for i in range(m)]
        gram2 = [[sum(gram[i][k] * gram[k][j] for k in range(m)) for j in range(m)]
                 for i in range(m)]
        poly = [[b * gram[i][j] + c * gram2[i][j] for j in range(m)] for i in range(m)]
        x = [[a * x[i][j] + sum(poly[i][k] * x[k][j] for k in range(m))
              for j in range(n)] for i in range(m)]
    if rows > cols:
        x = [[x[j][i] for j in range(m)] for i in range(n)]
    return x


def rel_fro_error(y, y_ref) -> float:
    """||y - y_ref||_F / ||y_ref||_F in float64 (per-matrix error measure)."""
    y = np.asarray(y, dtype=np.float64)
    y_ref = np.asarray(y_ref, dtype=np.float64)
    den = math.sqrt(float(np.sum(y_ref * y_ref)))
    num = math.sqrt(float(np.sum((y - y_ref) ** 2)))
    if den == 0.0:
        return num
    return num / den


def useful_flops(shape, steps: int) -> int:
    """Useful flops of one NS call: steps * (4 m^2 n + 2 m^3), m = min, n = max.

    Per step the Gram is 2 m^2 n, A @ A is 2 m^3 and B @ X is 2 m^2 n.
    """
    rows, cols = view_2d_shape(shape)
    m, n = min(rows, cols), max(rows, cols)
    return steps * (4 * m * m * n + 2 * m * m * m)
