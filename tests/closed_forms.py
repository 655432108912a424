"""Closed forms of Newton-Schulz on structured inputs (test arithmetic only).

For X with orthogonal rows, X X^T = diag(sigma^2) and the SVD is
X = I diag(sigma) V^T with V^T's rows the normalised rows of X. The k-step
quintic iteration (owner_planning page, ns_cost_fn) maps every normalised
singular value s = sigma_i / (||X||_F + eps) through p(s) = a s + b s^3 + c s^5
k times and keeps the singular vectors, so row i of NS_k(X) is
g_i * X_i with g_i = p^k(s_i) / sigma_i.
"""

import math


def row_gains(row_norms, steps, a, b, c, eps):
    """g_i = p^k(sigma_i / (||X||_F + eps)) / sigma_i for rows of norms sigma_i."""
    nu = math.sqrt(sum(s * s for s in row_norms)) + eps
    gains = []
    for s in row_norms:
        x = s / nu
        for _ in range(steps):
            x = a * x + b * x ** 3 + c * x ** 5
        gains.append(x / s)
    return gains


def hadamard_row_norms(m, r, d):
    """Row norms of the workloads' Hadamard-structured input: row i has m
    entries of magnitude r_i d_j in every column block j."""
    return [ri * math.sqrt(m * sum(dj * dj for dj in d)) for ri in r]
