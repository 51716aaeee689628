"""Factor preparation in fp64: damping, RevCholesky, update factor.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Reading of the pages (the summary page "FastKron: Efficient Quantization with
Kronecker-Factored Hessians", Corollary 3.4, names ``L(A) = RevCholesky(A)``
but never defines it):

* RevCholesky(A) is the lower-triangular L with ``A = L^T L``.  It is the
  Cholesky factorisation run from the last index to the first; with J the
  index-reversal permutation, ``L = J chol(J A J)^T J``.  This is the only
  reading under which the Corollary 3.4 proxy ``||L(B) dW L(A)^T||_F^2`` equals
  the quadratic loss ``vec(dW)^T (A (x) B) vec(dW)``.
* The factor that drives the GPTQ updates is ``U = L^{-T}``: upper triangular,
  with ``U^T U = A^{-1}``.  It is therefore also the upper Cholesky factor of
  ``A^{-1}`` (the "Hinv" factor of one-sided GPTQ).  Its diagonal is
  ``1 / diag(L)``.
* Damping (not on the pages; the plain GPTQ convention) adds
  ``damp * mean(diag(A)) * I`` once, before factorising.
"""

import numpy as np
import scipy.linalg as sla


def damp(A, damp_frac):
    """Return ``A + damp_frac * mean(diag(A)) * I`` in fp64 (a new array)."""
    A = np.array(A, dtype=np.float64, copy=True)
    if damp_frac:
        lam = float(damp_frac) * float(np.mean(np.diag(A)))
        A[np.diag_indices_from(A)] += lam
    return A


def rev_cholesky(A):
    """Lower-triangular L with ``A = L^T L`` (RevCholesky, Corollary 3.4).

    Computed as ``J chol(J A J)^T J``: ``np.linalg.cholesky`` gives the lower G
    with ``JAJ = G G^T``; then ``A = (J G J)(J G J)^T`` and ``L = (J G J)^T``.
    Raises ``np.linalg.LinAlgError`` when A is not positive definite.
    """
    A = np.asarray(A, dtype=np.float64)
    G = np.linalg.cholesky(A[::-1, ::-1])
    return np.ascontiguousarray(G.T[::-1, ::-1])


def update_factor(L):
    """``U = L^{-T}`` (upper triangular), from the lower RevCholesky factor."""
    n = L.shape[0]
    Linv = sla.solve_triangular(L, np.eye(n), lower=True)
    U = np.ascontiguousarray(Linv.T)
    return np.triu(U)


def lower_from_update(U):
    """Inverse map of :func:`update_factor`: ``L = U^{-T}`` (lower)."""
    n = U.shape[0]
    Uinv = sla.solve_triangular(np.asarray(U, np.float64), np.eye(n), lower=False)
    return np.tril(np.ascontiguousarray(Uinv.T))


def prepare(A, damp_frac):
    """Damping, RevCholesky and update factor of one Kronecker factor.

    Returns ``(L, U)`` in fp64 for the damped matrix.
    """
    Ad = damp(A, damp_frac)
    L = rev_cholesky(Ad)
    return L, update_factor(L)
