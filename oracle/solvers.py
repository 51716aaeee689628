"""GPTQ on vec(W) with a Kronecker Hessian A (x) B, written out several ways.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Conventions (summary page "FastKron: Efficient Quantization with
Kronecker-Factored Hessians", problem set-up and section 3):

* W is m x n; rows i index outputs (B side, m x m), columns j index inputs
  (A side, n x n).  vec is column-major, entry (i, j) -> k = i + m j, so the
  Hessian is ``np.kron(A, B)`` and ``(A (x) B) vec(X) = vec(B X A^T)``
  (Proposition 3.1, the identity that lets each vec step be written on the
  m x n matrix).
* GPTQ on a vector x with Hessian H and ``U = chol_upper(H^{-1})``: for k in
  order, ``q_k = Q(x_k)``, ``e_k = (x_k - q_k) / U_kk``,
  ``x_{k'} -= e_k U_{k,k'}`` for every later k'.
* With ``U_A``, ``U_B`` the update factors of A and B (``U^T U = A^{-1}``,
  upper), ``chol_upper(H^{-1}) = U_A (x) U_B``.  Unvectorised, entry (i, j)
  has scaled error ``E_ij = (w_ij - q_ij) l^B_i l^A_j`` with
  ``l = 1/diag(U)``, and it updates ``w_{i'j'} -= U_B[i,i'] E_ij U_A[j,j']``,
  which is non-zero only for ``i' >= i, j' >= j`` (section 3: an entry only
  updates the entries to its bottom-right).

Every solver returns a :class:`SolveResult`; ``preround`` holds the value each
entry had when it was rounded.  ``s`` is either a per-row scale vector (with
``qmin``/``qmax``; the workloads' symmetric per-row grid) or a
:class:`quantizer.Grid` (per-entry scale and zero point, e.g. column groups or
an asymmetric grid; then ``qmin``/``qmax`` are ignored).  ``guide``/``guide_tol`` (optional, every
solver): where the solver's own pre-rounding value is a near tie (see
``quantizer.near_tie``), take the guide's code instead of its own decision.
"""

import numpy as np

from .quantizer import Grid, quantize_codes, near_tie


class SolveResult:
    """codes, pre-rounding values, V = s c and scaled errors E (all m x n fp64)."""

    def __init__(self, codes, preround, V, E, overrides=0):
        self.codes = codes
        self.preround = preround
        self.V = V
        self.E = E
        self.overrides = overrides


def _as64(*arrs):
    return [np.array(a, dtype=np.float64, copy=True) for a in arrs]


def gptq_rows(W, UA, s, qmin=None, qmax=None, guide=None, guide_tol=1e-4):
    """Textbook one-sided GPTQ (Hessian A (x) I_m): every row independently.

    ``UA`` is the upper Cholesky factor of ``A^{-1}``.  Columns are processed
    left to right; the error of column j, divided by ``UA[j, j]``, is pushed
    into the columns to its right along row j of ``UA``.  This is the special
    case B = I of the two-sided problem (ainews article on BaKron: one-sided
    GPTQ uses a Hessian of the form A (x) I).
    """
    X, UA = _as64(W, UA)
    m, n = X.shape
    grid = Grid.of(s, qmin, qmax, m, n)
    rows = np.arange(m)
    C = np.zeros((m, n))
    P = np.zeros((m, n))
    E = np.zeros((m, n))
    n_over = 0
    for j in range(n):
        x = X[:, j].copy()
        P[:, j] = x
        c, o = grid.decide(x, rows, j, None if guide is None else guide[:, j], guide_tol)
        n_over += o
        C[:, j] = c
        err = (x - grid.value(c, rows, j)) / UA[j, j]
        E[:, j] = err
        X[:, j + 1:] -= np.outer(err, UA[j, j + 1:])
    return SolveResult(C, P, grid.values(C), E, n_over)


def naive_vec_gptq(W, s, qmin=None, qmax=None, A=None, B=None, UA=None, UB=None,
                   guide=None, guide_tol=1e-4):
    """BaKron-naive: GPTQ on vec(W) with the explicit mn x mn Hessian.

    Either the Hessian factors ``A`` (n x n), ``B`` (m x m) are given, and the
    explicit ``H = A (x) B`` is inverted, or the update factors ``UA``, ``UB``
    are given, and ``H^{-1} = (UA^T UA) (x) (UB^T UB)`` is formed explicitly.
    In both cases the mn x mn upper Cholesky factor of ``H^{-1}`` is computed
    directly from the explicit matrix (no Kronecker structure is used), and
    GPTQ runs over k = i + m j in increasing order.  ``mn`` sequential steps,
    ``O(m^2 n^2)`` work per step set (section 3, BaKron-naive).
    """
    W = np.asarray(W, dtype=np.float64)
    m, n = W.shape
    grid = Grid.of(s, qmin, qmax, m, n)
    if A is not None:
        H = np.kron(np.asarray(A, np.float64), np.asarray(B, np.float64))
        Hinv = np.linalg.inv(H)
        Hinv = 0.5 * (Hinv + Hinv.T)
    else:
        UA = np.asarray(UA, np.float64)
        UB = np.asarray(UB, np.float64)
        Hinv = np.kron(UA.T @ UA, UB.T @ UB)
    U = np.linalg.cholesky(Hinv).T
    x = W.reshape(-1, order="F").copy()
    rows = np.arange(m * n) % m
    cols = np.arange(m * n) // m
    g = None if guide is None else np.asarray(guide, np.float64).reshape(-1, order="F")
    c = np.zeros(m * n)
    pre = np.zeros(m * n)
    e = np.zeros(m * n)
    n_over = 0
    for k in range(m * n):
        pre[k] = x[k]
        ri, cj = rows[k:k + 1], cols[k:k + 1]
        ck, o = grid.decide(x[k:k + 1], ri, cj, None if g is None else g[k:k + 1], guide_tol)
        n_over += o
        c[k] = ck[0]
        e[k] = (x[k] - grid.value(ck, ri, cj)[0]) / U[k, k]
        x[k + 1:] -= e[k] * U[k, k + 1:]
    C = c.reshape((m, n), order="F")
    return SolveResult(C, pre.reshape((m, n), order="F"), grid.values(C),
                       e.reshape((m, n), order="F"), n_over)


def _diag_entries(d, m, n):
    i = np.arange(max(0, d - n + 1), min(d, m - 1) + 1)
    return i, d - i


def antidiag(W, UA, UB, s, qmin=None, qmax=None, guide=None, guide_tol=1e-4):
    """BaKron-antidiagonal (the YAQA-equivalent variant, section 3).

    For each anti-diagonal d = i + j in increasing order: quantise every entry
    on it at once (they are mutually independent), form the scaled errors
    ``E_d``, then subtract ``U_B^T E_d U_A`` from every entry on a later
    anti-diagonal.  ``m + n - 1`` sequential steps, ``O(m^2 n^2)`` work.  The
    product is taken only over the rows/columns the update can reach (rows
    >= the smallest active row, columns >= the smallest active column).
    """
    X, UA, UB = _as64(W, UA, UB)
    m, n = X.shape
    grid = Grid.of(s, qmin, qmax, m, n)
    lA = 1.0 / np.diag(UA)
    lB = 1.0 / np.diag(UB)
    S = np.add.outer(np.arange(m), np.arange(n))
    C = np.zeros((m, n))
    P = np.zeros((m, n))
    E = np.zeros((m, n))
    n_over = 0
    for d in range(m + n - 1):
        i, j = _diag_entries(d, m, n)
        x = X[i, j].copy()
        P[i, j] = x
        gd = None if guide is None else np.asarray(guide)[i, j]
        c, o = grid.decide(x, i, j, gd, guide_tol)
        n_over += o
        C[i, j] = c
        e = (x - grid.value(c, i, j)) * lB[i] * lA[j]
        E[i, j] = e
        i0, j0 = int(i[0]), int(j[-1])
        Z = e[:, None] * UA[j, j0:]           # row r: E_{i_r j_r} U_A[j_r, j0:]
        delta = UB[i, i0:].T @ Z              # sum_r U_B[i_r, i'] Z[r, j']
        later = S[i0:, j0:] > d
        X[i0:, j0:] -= np.where(later, delta, 0.0)
    return SolveResult(C, P, grid.values(C), E, n_over)


def recursive_vec(W, UA, UB, s, qmin=None, qmax=None, guide=None, guide_tol=1e-4):
    """BaKron-recursive (Theorem 3.2 names it; the pages do not describe it).

    Reading: divide and conquer over the linear vec order k = i + m j.
    ``rec(k0, k1)``: process ``[k0, km)``, push the errors of ``[k0, km)``
    into ``[km, k1)`` with one Kronecker product ``U_B^T E U_A`` restricted to
    the target range, then process ``[km, k1)``.  mn single-entry leaves;
    intended for tiny shapes only.
    """
    X, UA, UB = _as64(W, UA, UB)
    m, n = X.shape
    grid = Grid.of(s, qmin, qmax, m, n)
    lA = 1.0 / np.diag(UA)
    lB = 1.0 / np.diag(UB)
    K = np.arange(m)[:, None] + m * np.arange(n)[None, :]
    C = np.zeros((m, n))
    P = np.zeros((m, n))
    E = np.zeros((m, n))
    gd = None if guide is None else np.asarray(guide, np.float64)
    n_over = [0]

    def leaf(k):
        i, j = k % m, k // m
        x = X[i:i + 1, j]
        P[i, j] = x[0]
        c, o = grid.decide(x, np.array([i]), np.array([j]),
                           None if gd is None else gd[i:i + 1, j], guide_tol)
        n_over[0] += o
        C[i, j] = c[0]
        E[i, j] = (x[0] - grid.value(c[0], i, j)) * lB[i] * lA[j]

    def rec(k0, k1):
        if k1 - k0 == 1:
            leaf(k0)
            return
        km = (k0 + k1) // 2
        rec(k0, km)
        src = (K >= k0) & (K < km)
        dst = (K >= km) & (K < k1)
        delta = UB.T @ np.where(src, E, 0.0) @ UA
        X[dst] -= delta[dst]
        rec(km, k1)

    if m * n:
        rec(0, m * n)
    return SolveResult(C, P, grid.values(C), E, n_over[0])


def bakron(W, UA, UB, s, qmin=None, qmax=None, leaf_width=1, guide=None,
           guide_tol=1e-4):
    """BaKron: anti-diagonal parallelism + divide and conquer over anti-diagonals.

    Section 3 of the summary page: process the first half of the
    anti-diagonals recursively, propagate their error into the second half,
    then process the second half recursively.  ``rec(d0, d1)`` keeps the
    invariant that every entry on anti-diagonals ``[d0, d1)`` already holds
    the updates of all anti-diagonals ``< d0``.  Leaves of ``leaf_width``
    anti-diagonals run the anti-diagonal steps restricted to the leaf band.
    The propagation is ``U_B^T E_P U_A`` with ``E_P`` the errors of band
    ``[d0, dm)``, applied to band ``[dm, d1)``; it is taken over the bounding
    boxes of the two bands.
    """
    X, UA, UB = _as64(W, UA, UB)
    m, n = X.shape
    grid = Grid.of(s, qmin, qmax, m, n)
    lA = 1.0 / np.diag(UA)
    lB = 1.0 / np.diag(UB)
    S = np.add.outer(np.arange(m), np.arange(n))
    C = np.zeros((m, n))
    P = np.zeros((m, n))
    E = np.zeros((m, n))
    gd = None if guide is None else np.asarray(guide, np.float64)
    n_over = [0]

    def box(d0, d1):
        return (max(0, d0 - n + 1), min(m - 1, d1 - 1) + 1,
                max(0, d0 - m + 1), min(n - 1, d1 - 1) + 1)

    def leaf(d0, d1):
        for d in range(d0, d1):
            i, j = _diag_entries(d, m, n)
            x = X[i, j].copy()
            P[i, j] = x
            c, o = grid.decide(x, i, j, None if gd is None else gd[i, j], guide_tol)
            n_over[0] += o
            C[i, j] = c
            e = (x - grid.value(c, i, j)) * lB[i] * lA[j]
            E[i, j] = e
            if d + 1 < d1:
                r0, r1, c0, c1 = box(d + 1, d1)
                Z = e[:, None] * UA[j][:, c0:c1]
                delta = UB[i][:, r0:r1].T @ Z
                Sb = S[r0:r1, c0:c1]
                inside = (Sb > d) & (Sb < d1)
                X[r0:r1, c0:c1] -= np.where(inside, delta, 0.0)

    def propagate(d0, dm, d1):
        pr0, pr1, pc0, pc1 = box(d0, dm)
        qr0, qr1, qc0, qc1 = box(dm, d1)
        Sp = S[pr0:pr1, pc0:pc1]
        Ep = np.where((Sp >= d0) & (Sp < dm), E[pr0:pr1, pc0:pc1], 0.0)
        delta = UB[pr0:pr1, qr0:qr1].T @ Ep @ UA[pc0:pc1, qc0:qc1]
        Sq = S[qr0:qr1, qc0:qc1]
        X[qr0:qr1, qc0:qc1] -= np.where((Sq >= dm) & (Sq < d1), delta, 0.0)

    def rec(d0, d1):
        if d1 - d0 <= leaf_width:
            leaf(d0, d1)
            return
        dm = (d0 + d1) // 2
        rec(d0, dm)
        propagate(d0, dm, d1)
        rec(dm, d1)

    if m and n:
        rec(0, m + n - 1)
    return SolveResult(C, P, grid.values(C), E, n_over[0])


def bakron_tiled_order_check(W, UA, UB, s, qmin=None, qmax=None, tile=4):
    """GPTQ one entry at a time in the tile-anti-diagonal order.

    Tiles of ``tile x tile`` are taken by tile anti-diagonal I + J; inside a
    tile, entries go by their own anti-diagonal, then by row.  Each entry, once
    rounded, immediately updates every not-yet-rounded entry to its
    bottom-right.  This is the processing order a tiled GPU sweep uses; by
    Theorem 3.2 (any order that rounds an entry after all entries to its
    top-left gives the same output) it must reproduce the other variants.
    Raises ``ValueError`` if the order is not such an order.
    """
    X, UA, UB = _as64(W, UA, UB)
    m, n = X.shape
    grid = Grid.of(s, qmin, qmax, m, n)
    lA = 1.0 / np.diag(UA)
    lB = 1.0 / np.diag(UB)
    order = []
    M = -(-m // tile)
    N = -(-n // tile)
    for D in range(M + N - 1):
        for I in range(max(0, D - N + 1), min(D, M - 1) + 1):
            J = D - I
            ents = [(i, j) for i in range(I * tile, min(m, (I + 1) * tile))
                    for j in range(J * tile, min(n, (J + 1) * tile))]
            ents.sort(key=lambda t: (t[0] + t[1], t[0]))
            order.extend(ents)
    done = np.zeros((m, n), dtype=bool)
    C = np.zeros((m, n))
    P = np.zeros((m, n))
    E = np.zeros((m, n))
    for (i, j) in order:
        if not done[:i + 1, :j + 1].sum() == (i + 1) * (j + 1) - 1:
            raise ValueError("order rounds (%d,%d) before an entry to its top-left" % (i, j))
        x = X[i, j]
        P[i, j] = x
        c = grid.decide(np.array([x]), np.array([i]), np.array([j]))[0][0]
        C[i, j] = c
        e = (x - grid.value(c, i, j)) * lB[i] * lA[j]
        E[i, j] = e
        done[i, j] = True
        upd = np.outer(UB[i, i:], UA[j, j:]) * e
        upd[0, 0] = 0.0
        X[i:, j:] -= np.where(done[i:, j:], 0.0, upd)
    return SolveResult(C, P, grid.values(C), E)
