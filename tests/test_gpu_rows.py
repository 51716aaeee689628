"""GPU parity of the one-sided path (B = I: bakron_quantize with UB = NULL)
against the fp64 oracle's textbook per-row GPTQ.

With B = I every row is its own GPTQ problem with Hessian A, so the oracle
(``oracle.gptq_rows``) can check any subset of rows of a full-size solve
exactly.  Comparison rule as in the two-sided tests: the oracle is re-run
guided by the GPU codes (it takes the GPU decision only at its own near
ties, |x/s - (k + 1/2)| < 1e-4 grid units) and must then reproduce the GPU
codes exactly, with at most 0.1% guided decisions; pre-rounding values agree
to 1e-4 grid units; V = s * code bit for bit.
"""

import numpy as np
import pytest

import oracle as O
from kronecker_factored_gptq_gb300 import workloads as WL

from _gpu_helpers import TOL, MAX_FRAC, LOSS_RTOL, oracle_grid, shared_factors, to_dev

pytestmark = pytest.mark.gpu


def variants():
    from kronecker_factored_gptq_gb300 import bakron as kb
    v = [0]
    if kb.default_opts().use_3xtf32 == 1:
        v.append(1)
    return v


def rows_quantize(W, UA32, s32, qmin, qmax, use_tc=1, preround=True):
    from kronecker_factored_gptq_gb300 import bakron as kb
    dW, dUA, ds = to_dev(W, UA32, s32)
    V, c, p = kb.bakron_quantize(dW, dUA, None, ds, qmin, qmax, want_preround=preround,
                                 opts=kb.default_opts(use_3xtf32=use_tc))
    return (V.cpu().numpy(), c.cpu().numpy().astype(np.float64),
            None if p is None else p.cpu().numpy())


def check_rows(W, UA32, s32, qmin, qmax, V, codes, pre=None, rows=None):
    """Guided oracle on the given rows (all by default)."""
    oq = oracle_grid(qmin, qmax)
    rows = np.arange(W.shape[0]) if rows is None else rows
    Wr, cr, sr = W[rows], codes[rows], s32[rows]
    UA = UA32.astype(np.float64)
    g = O.gptq_rows(Wr, UA, sr, *oq, guide=cr, guide_tol=TOL)
    diff = int(np.count_nonzero(g.codes != cr))
    assert diff == 0, "GPU codes differ from the guided oracle at %d entries (not near ties)" % diff
    assert g.overrides <= max(1, MAX_FRAC * cr.size), g.overrides
    np.testing.assert_array_equal(V[rows], (sr[:, None] * cr.astype(np.float32)).astype(np.float32))
    if pre is not None:
        err = np.max(np.abs(pre[rows] - g.preround) / sr[:, None])
        assert err < TOL, "pre-rounding values off by %.3g grid units" % err
    # proxy loss of the rows against the unguided oracle: ||(V - W) L_A^T||^2
    ref = O.gptq_rows(Wr, UA, sr, *oq)
    LA = O.lower_from_update(UA)
    I = np.eye(len(rows))
    l_gpu = O.proxy_loss(Wr, V[rows], LA, I)
    V_ref = (sr[:, None] * ref.codes.astype(np.float32)).astype(np.float32)
    l_ref = O.proxy_loss(Wr, V_ref, LA, I)
    assert abs(l_gpu - l_ref) <= LOSS_RTOL * abs(l_ref) + 1e-30, (l_gpu, l_ref)
    return g


@pytest.mark.parametrize("use_tc", variants())
@pytest.mark.parametrize("m,n,bits", [(64, 64, 4), (128, 128, 3), (200, 328, 4), (300, 260, 2),
                                      (1, 300, 4), (257, 1, 4), (129, 384, 4), (77, 600, 3)])
def test_rows_parity(use_tc, m, n, bits):
    w = WL.random_problem(m, n, seed=m * 3 + n, bits=bits)
    UA32, _ = shared_factors(w.A, w.damp_A, w.B, w.damp_B)
    s = O.row_scale(w.W, w.qmax)
    V, c, pre = rows_quantize(w.W, UA32, s, w.qmin, w.qmax, use_tc)
    check_rows(w.W, UA32, s, w.qmin, w.qmax, V, c, pre)


def test_rows_matches_two_sided_with_identity():
    """The row path and the two-sided solver given U_B = I solve the same
    problem: both reproduce the guided oracle, and they agree with each other
    except where a near tie was decided differently (then only later entries
    of that row move)."""
    from kronecker_factored_gptq_gb300 import bakron as kb
    w = WL.random_problem(260, 400, seed=21)
    UA32, _ = shared_factors(w.A, w.damp_A, w.B, w.damp_B)
    s = O.row_scale(w.W, w.qmax)
    V1, c1, p1 = rows_quantize(w.W, UA32, s, w.qmin, w.qmax)
    dW, dUA, dI, ds = to_dev(w.W, UA32, np.eye(260, dtype=np.float32), s)
    V2, c2, _ = kb.bakron_quantize(dW, dUA, dI, ds, w.qmin, w.qmax)
    c2 = c2.cpu().numpy().astype(np.float64)
    diff = c1 != c2
    nt = O.near_tie(p1, s[:, None], w.qmin, w.qmax, TOL)
    for i in np.unique(np.nonzero(diff)[0]):
        first = np.nonzero(diff[i])[0][0]
        assert nt[i, first], "row %d first differs at %d, not a near tie" % (i, first)
    assert np.count_nonzero(diff.any(axis=1)) <= max(1, MAX_FRAC * 260)


def test_rows_unclamped_cor34_bound():
    """Corollary 3.4 per row with B = I on an unclamped unit grid:
    ||(V - W) L_A^T||^2 <= 1/4 sum_j l_j^2 <= 1/4 tr(A_damped)."""
    from kronecker_factored_gptq_gb300 import bakron as kb
    w = WL.random_problem(150, 270, seed=22)
    UA32, _ = shared_factors(w.A, w.damp_A, w.B, w.damp_B)
    W10 = (10.0 * w.W).astype(np.float32)
    ones = np.ones(150, np.float32)
    V, c, pre = rows_quantize(W10, UA32, ones, kb.INT32_MIN, kb.INT32_MAX)
    check_rows(W10, UA32, ones, kb.INT32_MIN, kb.INT32_MAX, V, c, pre)
    LA = O.lower_from_update(UA32.astype(np.float64))
    D = (V.astype(np.float64) - W10) @ LA.T
    per_row = np.sum(D * D, axis=1)
    bound = 0.25 * np.sum(np.diag(LA) ** 2)
    Ad = np.linalg.inv(UA32.astype(np.float64).T @ UA32.astype(np.float64))
    assert np.all(per_row <= bound * (1 + 1e-6)) and bound <= 0.25 * np.trace(Ad) * (1 + 1e-9)


def test_rows_nonfinite_input():
    from kronecker_factored_gptq_gb300 import bakron as kb
    w = WL.random_problem(130, 140, seed=23)
    UA32, _ = shared_factors(w.A, w.damp_A, w.B, w.damp_B)
    s = O.row_scale(w.W, w.qmax)
    W = w.W.copy()
    W[70, 90] = np.nan
    dW, dUA, ds = to_dev(W, UA32, s)
    with pytest.raises(kb.BakronError) as ei:
        kb.bakron_quantize(dW, dUA, None, ds, w.qmin, w.qmax)
    assert ei.value.status == 3


def test_rows_full_size_sampled_rows():
    """8192 x 8192 (the headline workload's W and A, B = I) through the same
    sequence a user runs: row grid, preparation of A alone on the GPU, then
    the row path.  Rows are independent, so sampled rows are exact problems
    for the oracle (with the GPU's own fp32 factor)."""
    import torch
    from kronecker_factored_gptq_gb300 import bakron as kb
    w = WL.load("c8192", seed=0, device="cuda")
    dW, dA = to_dev(w.W, w.A)
    s = kb.bakron_rowscale(dW, w.qmax)
    UA, _, _, _, info = kb.bakron_prepare(dA, w.damp_A)
    assert info[0] == -1
    V, c, pre = kb.bakron_quantize(dW, UA, None, s, w.qmin, w.qmax, want_preround=True)
    torch.cuda.synchronize()
    rng = np.random.default_rng(5)
    rows = np.unique(np.concatenate([[0, 1, w.m - 1], rng.choice(w.m, 13, replace=False)]))
    s32 = s.cpu().numpy()
    np.testing.assert_array_equal(s32, O.row_scale(w.W, w.qmax))
    check_rows(w.W, UA.cpu().numpy(), s32, w.qmin, w.qmax, V.cpu().numpy(),
               c.cpu().numpy().astype(np.float64), pre.cpu().numpy(), rows=rows)
