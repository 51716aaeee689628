"""GPTQ on vec(W) with Hessian A (x) B in the row-accumulator form, in C.

TEST INFRASTRUCTURE ONLY (see the package docstring).

The same output as the other solvers in ``solvers.py`` (Theorem 3.2 of the
summary page "FastKron: Efficient Quantization with Kronecker-Factored
Hessians": any order that rounds an entry after all entries to its top-left),
computed in m n (m + n) fp64 flops instead of the bounding-box products of
``solvers.bakron``, so the whole-solve comparison reaches the full workload
sizes.  The arithmetic is in ``rowacc.c`` (plain C, the entries of one
anti-diagonal in parallel with OpenMP); ``build_c.py`` compiles it into
``librowacc.so`` next to this file.
"""

import ctypes
import os

import numpy as np

from .solvers import SolveResult

HERE = os.path.dirname(os.path.abspath(__file__))
LIB = os.path.join(HERE, "librowacc.so")
_lib = None


def _load():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB):
            from . import build_c
            build_c.build()
        lib = ctypes.CDLL(LIB)
        P = ctypes.c_void_p
        lib.rowacc_solve.restype = ctypes.c_longlong
        lib.rowacc_solve.argtypes = [P, P, P, P, ctypes.c_int64, ctypes.c_int64, ctypes.c_int,
                                     ctypes.c_double, ctypes.c_double, P, ctypes.c_double, P, P, P]
        lib.rowacc_solve_blocked.restype = ctypes.c_longlong
        lib.rowacc_solve_blocked.argtypes = lib.rowacc_solve.argtypes + [ctypes.c_int]
        lib.rowacc_threads.restype = ctypes.c_int
        lib.rowacc_threads.argtypes = [ctypes.c_int]
        _lib = lib
    return _lib


def threads(want=0):
    """Set (want > 0) and return the number of threads the solve uses."""
    return int(_load().rowacc_threads(int(want)))


def _ptr(a):
    return ctypes.c_void_p(a.ctypes.data)


def rowacc(W, UA, UB, s, qmin=None, qmax=None, guide=None, guide_tol=1e-4, rows_per_block=0):
    """GPTQ output for W (m x n) with update factors UA (n x n), UB (m x m) and
    the per-row grid ``s`` (fp32 scales, codes clamped to [qmin, qmax]; both
    None: no clamp).  ``guide``: codes taken at the solver's own near ties.
    ``rows_per_block`` 0: anti-diagonal traversal (``rowacc_solve``); k > 0:
    blocks of k rows (``rowacc_solve_blocked``, the same arithmetic per entry,
    column sums grouped by block; for the full workload sizes).
    Returns a :class:`SolveResult` (codes, preround, V = s c, E)."""
    lib = _load()
    W = np.ascontiguousarray(W, dtype=np.float64)
    UA = np.ascontiguousarray(UA, dtype=np.float64)
    UB = np.ascontiguousarray(UB, dtype=np.float64)
    s32 = np.ascontiguousarray(s, dtype=np.float32)
    m, n = W.shape
    assert UA.shape == (n, n) and UB.shape == (m, m) and s32.shape == (m,)
    clamp = qmin is not None and qmax is not None
    assert clamp or (qmin is None and qmax is None), "clamp both ends or neither"
    g = None if guide is None else np.ascontiguousarray(guide, dtype=np.float64)
    codes = np.empty((m, n))
    pre = np.empty((m, n))
    E = np.empty((m, n))
    args = [_ptr(W), _ptr(UA), _ptr(UB), _ptr(s32), m, n, int(clamp),
            float(qmin) if clamp else 0.0, float(qmax) if clamp else 0.0,
            None if g is None else _ptr(g), float(guide_tol), _ptr(codes), _ptr(pre), _ptr(E)]
    if rows_per_block > 0:
        over = lib.rowacc_solve_blocked(*args, int(rows_per_block))
    else:
        over = lib.rowacc_solve(*args)
    if over < 0:
        raise MemoryError("rowacc: scratch allocation failed")
    V = s32.astype(np.float64)[:, None] * codes
    return SolveResult(codes, pre, V, E, int(over))
