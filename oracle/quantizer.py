"""Base quantizers Q (uniform grids) and the near-tie rule.

TEST INFRASTRUCTURE ONLY (see the package docstring).

The pages call BaKron modular in the base quantizer (abstract of "BaKron:
Efficient Quantization with Kronecker-Factored Hessians") and fix no grid.  A
grid gives every entry (i, j) a scale s_ij, an integer zero point z_ij and a
code range [qmin, qmax]:

* code ``c = clamp(round_half_even(x / s_ij) + z_ij, qmin, qmax)``, value
  ``q = s_ij (c - z_ij)``;
* the workloads use the per-row symmetric b-bit grid: ``s_i = max_j |W_ij| /
  qmax`` with ``qmax = 2^(b-1) - 1``, ``qmin = -2^(b-1)``, ``z = 0``, taken on
  the ORIGINAL weights; an all-zero row gets ``s_i = 1``;
* :func:`symmetric_grid` and :func:`asymmetric_grid` generalise it to groups
  of ``group`` consecutive columns per row (the scale of a group is taken on
  the group's original weights, like the per-row scale).  The asymmetric
  grid is the min-max grid with the range widened to contain zero (the usual
  GPTQ convention; the pages name none): ``lo = min(min W_G, 0)``,
  ``hi = max(max W_G, 0)``, ``s = (hi - lo) / (2^b - 1)``, ``z = rint(-lo / s)``,
  codes ``[0, 2^b - 1]``; an all-zero group gets ``s = 1``, ``z = 0``.

The rounding decision is taken in fp32 on both sides (the pages' kernel is a
float32 kernel): ``x`` is rounded to fp32, divided by the fp32 scale with one
IEEE fp32 division, then rounded half-to-even; the grid parameters are formed
in fp32.  ``qmin``/``qmax`` of ``None`` mean no clamp (the unit-step
round-to-nearest used for the Corollary 3.4 check).
"""

import numpy as np


def row_scale(W, qmax):
    """Per-row scale in fp32: ``fl32(max_j |W_ij|) / fl32(qmax)``; zero rows -> 1."""
    W32 = np.asarray(W, dtype=np.float32)
    amax = np.max(np.abs(W32), axis=1) if W32.shape[1] else np.zeros(W32.shape[0], np.float32)
    s = (amax / np.float32(qmax)).astype(np.float32)
    s[amax == 0] = np.float32(1.0)
    return s


def quantize_codes(x, s, qmin=None, qmax=None, z=0.0):
    """Codes ``clamp(rint(fl32(x) / fl32(s)) + z, qmin, qmax)`` returned as float64."""
    t = np.asarray(x, dtype=np.float64).astype(np.float32) / np.asarray(s, dtype=np.float32)
    c = np.rint(t).astype(np.float64) + np.asarray(z, dtype=np.float64)
    if qmin is not None:
        c = np.maximum(c, float(qmin))
    if qmax is not None:
        c = np.minimum(c, float(qmax))
    return c


def near_tie(x, s, qmin=None, qmax=None, tol=1e-4, z=0.0):
    """True where ``x / s`` lies within ``tol`` (grid units) of a rounding boundary.

    A boundary ``k + 1/2`` counts only when it separates two codes that the
    clamp can both produce (``qmin <= k + z`` and ``k + 1 + z <= qmax``);
    outside the clamp range the decision does not depend on which side of it x
    falls.
    """
    t = np.asarray(x, dtype=np.float64) / np.asarray(s, dtype=np.float64)
    k = np.floor(t) + np.asarray(z, dtype=np.float64)
    near = np.abs(t - (np.floor(t) + 0.5)) < tol
    if qmin is not None:
        near &= k >= qmin
    if qmax is not None:
        near &= (k + 1) <= qmax
    return near


class Grid:
    """Per-entry grid of an m x n matrix: scale ``S`` and zero point ``Z``
    (m x n, fp64 holding fp32 / integer values) and the code range."""

    def __init__(self, S, Z=None, qmin=None, qmax=None):
        self.S = np.asarray(S, dtype=np.float64)
        self.Z = np.zeros_like(self.S) if Z is None else np.asarray(Z, dtype=np.float64)
        self.qmin, self.qmax = qmin, qmax

    @staticmethod
    def of(s, qmin, qmax, m, n):
        """``s`` itself if it is a Grid, else the per-row grid of scales ``s``."""
        if isinstance(s, Grid):
            return s
        s = np.asarray(s, dtype=np.float64)
        return Grid(np.repeat(s[:, None], n, axis=1), None, qmin, qmax)

    def decide(self, x, i, j, guide=None, guide_tol=1e-4):
        """Codes of the entries (i, j) with pre-rounding values x; where a
        guide is given, its code is taken at the entries' own near ties.
        Returns (codes, number of guided decisions that changed a code)."""
        S, Z = self.S[i, j], self.Z[i, j]
        c = quantize_codes(x, S, self.qmin, self.qmax, Z)
        n_over = 0
        if guide is not None:
            nt = near_tie(x, S, self.qmin, self.qmax, guide_tol, Z)
            g = np.asarray(guide, dtype=np.float64)
            n_over = int(np.count_nonzero(nt & (g != c)))
            c = np.where(nt, g, c)
        return c, n_over

    def value(self, c, i, j):
        return self.S[i, j] * (c - self.Z[i, j])

    def values(self, C):
        return self.S * (np.asarray(C, dtype=np.float64) - self.Z)


def _group_reduce(W32, group, fn, init):
    m, n = W32.shape
    g = n if (not group or group >= n) else int(group)
    ng = -(-n // g)
    out = np.full((m, ng), init, dtype=np.float32)
    for k in range(ng):
        out[:, k] = fn(W32[:, k * g:(k + 1) * g], axis=1)
    return out, g


def _expand(P, g, n):
    return np.repeat(np.asarray(P, dtype=np.float64), g, axis=1)[:, :n]


def symmetric_grid(W, bits, group=None):
    """Symmetric b-bit grid per row (group None or >= n) or per group of
    ``group`` columns: ``s = fl32(max |W_G|) / fl32(2^(b-1) - 1)`` (zero groups
    -> 1), ``z = 0``, codes ``[-2^(b-1), 2^(b-1) - 1]``.  Returns
    ``(Grid, s (m x groups, fp32), z (m x groups, fp32))``."""
    W32 = np.asarray(W, dtype=np.float32)
    qmax = (1 << (bits - 1)) - 1
    amax, g = _group_reduce(np.abs(W32), group, np.max, 0.0)
    s = (amax / np.float32(qmax)).astype(np.float32)
    s[amax == 0] = np.float32(1.0)
    z = np.zeros_like(s)
    n = W32.shape[1]
    return Grid(_expand(s, g, n), _expand(z, g, n), -(qmax + 1), qmax), s, z


def asymmetric_grid(W, bits, group=None):
    """Min-max b-bit grid with zero in range (see the module docstring), per
    row or per group of ``group`` columns, all in fp32.  Returns
    ``(Grid, s, z)`` like :func:`symmetric_grid`."""
    W32 = np.asarray(W, dtype=np.float32)
    levels = np.float32((1 << bits) - 1)
    lo, g = _group_reduce(W32, group, np.min, 0.0)
    hi, _ = _group_reduce(W32, group, np.max, 0.0)
    lo = np.minimum(lo, np.float32(0.0))
    hi = np.maximum(hi, np.float32(0.0))
    span = (hi - lo).astype(np.float32)
    s = (span / levels).astype(np.float32)
    zero = span == 0
    s[zero] = np.float32(1.0)
    z = np.rint((-lo / s).astype(np.float32)).astype(np.float32)
    z[zero] = np.float32(0.0)
    z = np.clip(z, np.float32(0.0), levels).astype(np.float32)
    n = W32.shape[1]
    return Grid(_expand(s, g, n), _expand(z, g, n), 0, int(levels)), s, z
