"""Kronecker factors of a layer Hessian from samples, in fp64.

TEST INFRASTRUCTURE ONLY (see the package docstring).

The summary page "FastKron: Efficient Quantization with Kronecker-Factored
Hessians" (its section on the Hessians) factorises the expected Hessian of a
linear layer, E[a a^T (x) g g^T] with a the input activation and g the loss
gradient at the layer output (the per-sample gradient of W is g a^T, and
vec(g a^T) = a (x) g in the column-major vec order), in two ways:

* K-FAC-style independence assumption: ``A = E[a a^T]``, ``B = E[g g^T]``;
* one step of a Shampoo-style power iteration for the best Kronecker
  approximation, started from the identity: ``A = E[tr(g^T g) a a^T]``,
  ``B = E[tr(a^T a) g g^T]``.

Expectations are sample means over the N rows of X (a_t) and G (g_t); the
pages print the formulas without normalisation, and a common scale does not
change the GPTQ result (the solver is invariant to A -> cA, B -> cB).
"""

import numpy as np


def kfac_factors(X, G):
    """K-FAC factors ``(A, B) = (X^T X / N, G^T G / N)`` (fp64); either input
    may be None (then its factor is None)."""
    A = B = None
    if X is not None:
        X = np.asarray(X, dtype=np.float64)
        A = X.T @ X / X.shape[0]
    if G is not None:
        G = np.asarray(G, dtype=np.float64)
        B = G.T @ G / G.shape[0]
    return A, B


def shampoo_factors(X, G):
    """One power-iteration step from the identity:
    ``A = (1/N) sum_t |g_t|^2 a_t a_t^T``, ``B = (1/N) sum_t |a_t|^2 g_t g_t^T``."""
    X = np.asarray(X, dtype=np.float64)
    G = np.asarray(G, dtype=np.float64)
    N = X.shape[0]
    wa = np.sum(X * X, axis=1)
    wg = np.sum(G * G, axis=1)
    A = (X * wg[:, None]).T @ X / N
    B = (G * wa[:, None]).T @ G / N
    return A, B
