"""Output certificate, proxy loss, Corollary 3.4 bound, code comparison.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Certificate (derived from the GPTQ recursion, independent of how V was made):
GPTQ leaves ``x - q = U^T e`` on vec(W), so ``e = L vec(W - V)`` with
``L = U^{-T} = L_A (x) L_B``; unvectorised ``E = L_B (W - V) L_A^T``.  Every
entry's pre-rounding value is then ``w~_ij = V_ij + E_ij / (l^B_i l^A_j)``
with ``l = diag(L)``, and a candidate V is the GPTQ output exactly when every
code equals ``Q_i(w~_ij)``.  By induction over any processing order this
replays all decisions with the candidate's own history ("teacher forcing"),
so one flipped near-tie does not cascade into the count.

Proxy loss and bound (summary page "FastKron: Efficient Quantization with
Kronecker-Factored Hessians", Corollary 3.4 and the remark after it):
``||L(B)(V - W)L(A)^T||_F^2 = vec(V - W)^T (A (x) B) vec(V - W)``, and for an
unclamped unit-step round-to-nearest quantizer it is at most
``1/4 tr(A) tr(B)``; the proof route gives the tighter
``1/4 sum_j l^A_j^2 sum_i l^B_i^2`` (each ``|e_k| <= l_k / 2`` and
``l_k^2 <= H_kk``).
"""

import numpy as np

from .factors import lower_from_update
from .quantizer import Grid, quantize_codes, near_tie


def proxy_loss(W, V, LA, LB):
    """``||L_B (V - W) L_A^T||_F^2`` in fp64."""
    D = np.asarray(V, np.float64) - np.asarray(W, np.float64)
    M = np.asarray(LB, np.float64) @ D @ np.asarray(LA, np.float64).T
    return float(np.sum(M * M))


def cor34_bound(A, B):
    """Corollary 3.4: ``1/4 tr(A) tr(B)``."""
    return 0.25 * float(np.trace(np.asarray(A, np.float64))) * float(np.trace(np.asarray(B, np.float64)))


def cor34_tight_bound(LA, LB):
    """``1/4 sum_j L_A[j,j]^2 sum_i L_B[i,i]^2`` (<= cor34_bound)."""
    return 0.25 * float(np.sum(np.diag(LA) ** 2)) * float(np.sum(np.diag(LB) ** 2))


def certificate(W, V, codes, UA, UB, s, qmin=None, qmax=None, tol=1e-4,
                max_frac=1e-3):
    """Replay every rounding decision of a candidate output (teacher forcing).

    Returns a dict: ``wt`` (replayed pre-rounding values), ``mismatch`` (codes
    that differ from the replay), ``near_mismatch`` (of those, the ones whose
    replayed value is within ``tol`` grid units of a rounding boundary),
    ``bad`` (mismatches that are not near ties) and ``ok``: no bad mismatch and
    at most ``max_frac`` of the entries mismatched.
    """
    W = np.asarray(W, np.float64)
    V = np.asarray(V, np.float64)
    codes = np.asarray(codes, np.float64)
    m, n = W.shape
    g = Grid.of(s, qmin, qmax, m, n)
    LA = lower_from_update(UA)
    LB = lower_from_update(UB)
    E = LB @ (W - V) @ LA.T
    wt = V + E / np.outer(np.diag(LB), np.diag(LA))
    replay = quantize_codes(wt, g.S, g.qmin, g.qmax, g.Z)
    mism = replay != codes
    nt = near_tie(wt, g.S, g.qmin, g.qmax, tol, g.Z)
    n_m = int(np.count_nonzero(mism))
    bad = int(np.count_nonzero(mism & ~nt))
    return {
        "wt": wt, "mismatch": n_m, "near_mismatch": n_m - bad, "bad": bad,
        "ok": bad == 0 and n_m <= max_frac * max(1, m * n),
        "loss": float(np.sum(E * E)),
    }


def compare_codes(codes_test, codes_ref, preround_ref, s, qmin=None, qmax=None,
                  tol=1e-4, max_frac=1e-3):
    """Direct code comparison under the near-tie rule.

    Codes must be equal except where the reference's pre-rounding value lies
    within ``tol`` grid units of a rounding boundary, and at most
    ``max_frac`` of the entries may differ.  Returns a dict with the counts
    and ``ok``.
    """
    a = np.asarray(codes_test, np.float64)
    b = np.asarray(codes_ref, np.float64)
    diff = a != b
    g = Grid.of(s, qmin, qmax, a.shape[0], a.shape[1])
    nt = near_tie(preround_ref, g.S, g.qmin, g.qmax, tol, g.Z)
    n_d = int(np.count_nonzero(diff))
    bad = int(np.count_nonzero(diff & ~nt))
    return {"diff": n_d, "bad": bad,
            "ok": bad == 0 and n_d <= max_frac * max(1, a.size)}
