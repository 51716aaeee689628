"""Base quantizer Q: per-row symmetric uniform grid, and the near-tie rule.

TEST INFRASTRUCTURE ONLY (see the package docstring).

The pages call BaKron modular in the base quantizer (abstract of "BaKron:
Efficient Quantization with Kronecker-Factored Hessians") and fix no grid; the
workloads use a per-row symmetric b-bit grid:

* scale ``s_i = max_j |W_ij| / qmax`` with ``qmax = 2^(b-1) - 1``, taken on the
  ORIGINAL weights; an all-zero row gets ``s_i = 1``;
* code ``c = clamp(round_half_even(x / s_i), qmin, qmax)``, value ``q = s_i c``.

The rounding decision is taken in fp32 on both sides (the pages' kernel is a
float32 kernel): ``x`` is rounded to fp32, divided by the fp32 scale with one
IEEE fp32 division, then rounded half-to-even.  ``qmin``/``qmax`` of ``None``
mean no clamp (the unit-step round-to-nearest used for the Corollary 3.4
check).
"""

import numpy as np


def row_scale(W, qmax):
    """Per-row scale in fp32: ``fl32(max_j |W_ij|) / fl32(qmax)``; zero rows -> 1."""
    W32 = np.asarray(W, dtype=np.float32)
    amax = np.max(np.abs(W32), axis=1) if W32.shape[1] else np.zeros(W32.shape[0], np.float32)
    s = (amax / np.float32(qmax)).astype(np.float32)
    s[amax == 0] = np.float32(1.0)
    return s


def quantize_codes(x, s, qmin=None, qmax=None):
    """Codes ``clamp(rint(fl32(x) / fl32(s)), qmin, qmax)`` returned as float64."""
    t = np.asarray(x, dtype=np.float64).astype(np.float32) / np.asarray(s, dtype=np.float32)
    c = np.rint(t).astype(np.float64)
    if qmin is not None:
        c = np.maximum(c, float(qmin))
    if qmax is not None:
        c = np.minimum(c, float(qmax))
    return c


def near_tie(x, s, qmin=None, qmax=None, tol=1e-4):
    """True where ``x / s`` lies within ``tol`` (grid units) of a rounding boundary.

    A boundary ``k + 1/2`` counts only when it separates two codes that the
    clamp can both produce (``qmin <= k`` and ``k + 1 <= qmax``); outside the
    clamp range the decision does not depend on which side of it x falls.
    """
    t = np.asarray(x, dtype=np.float64) / np.asarray(s, dtype=np.float64)
    k = np.floor(t)
    near = np.abs(t - (k + 0.5)) < tol
    if qmin is not None:
        near &= k >= qmin
    if qmax is not None:
        near &= (k + 1) <= qmax
    return near
