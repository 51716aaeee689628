"""GPU parity at the full workload sizes, in the launch configuration the
benchmark times: per-row grid, factor preparation and the solve all on the
GPU with the default options (tcgen05 3xTF32 propagation), exactly the
``Solver.solve`` sequence of the benchmark step.

Workloads: 1024 x 1024, 4096 x 4096, 4096 x 14336, 14336 x 4096 and
8192 x 8192 (kronecker_factored_gptq_gb300.workloads).  The 64 x 64 case and
ragged small shapes are in test_gpu_parity.py.

The oracle cannot redo a whole solve above 1024 x 1024, so the checks are
  * outputs the oracle computes exactly: entry (i, j) depends only on
    W[:i+1, :j+1] and the leading blocks of the factors (updates only move
    to the bottom-right), so the top 128 rows and the leftmost 128 columns
    are complete GPTQ problems of their own.  The oracle re-runs them guided
    by the GPU codes (only at its own near ties) and must reproduce them;
  * properties that hold at any size: row scales bit-exact, factor residuals
    on sampled columns, every rounding decision replayed in fp64 (the
    certificate), and Corollary 3.4's bound on an unclamped unit-step grid
    (input W * 10, same factors);
  * at 1024 x 1024 the whole solve against the oracle, the B = I reduction
    to per-row GPTQ, and the full variant against the anti-diagonal kernel.
Solve checks use the GPU's own fp32 factors, upcast, on the oracle side.
"""

import numpy as np
import pytest

import oracle as O
from kronecker_factored_gptq_gb300 import workloads as WL

from _gpu_helpers import TOL, MAX_FRAC, check_parity, corner_check, oracle_grid, to_dev

pytestmark = pytest.mark.gpu

FULL = ["c1024", "c4096", "mlp4096x14336", "mlp14336x4096", "c8192"]
STRIP = 128
EPS32 = float(np.finfo(np.float32).eps)


@pytest.fixture(scope="module", params=FULL)
def run(request):
    import torch
    from kronecker_factored_gptq_gb300 import bakron as kb
    w = WL.load(request.param, seed=0, device="cuda")
    dW, dA, dB = to_dev(w.W, w.A, w.B)
    solver = kb.Solver(w.m, w.n, qmin=w.qmin, qmax=w.qmax)
    V, codes = solver.solve(dW, dA, w.damp_A, dB, w.damp_B)
    r = {"w": w, "s": solver.scale.cpu().numpy(), "V": V.cpu().numpy(),
         "codes": codes.cpu().numpy().astype(np.float64),
         "UA": solver.UA.cpu().numpy(), "UB": solver.UB.cpu().numpy()}
    # the same preparation again, now also returning L, for the residuals
    UA2, UB2, LA, LB, info = kb.bakron_prepare(dA, w.damp_A, dB, w.damp_B, want_L=True)
    r["info"] = info
    r["UA2"], r["UB2"] = UA2.cpu().numpy(), UB2.cpu().numpy()
    r["LA"], r["LB"] = LA.cpu().numpy(), LB.cpu().numpy()
    # unclamped unit-step grid on W * 10 with the same factors (Corollary 3.4)
    W10 = (10.0 * w.W).astype(np.float32)
    (dW10,) = to_dev(W10)
    ones = torch.ones(w.m, dtype=torch.float32, device="cuda")
    Vu, cu, _ = kb.bakron_quantize(dW10, solver.UA, solver.UB, ones, kb.INT32_MIN, kb.INT32_MAX,
                                   workspace=solver.ws_q)
    r["W10"], r["Vu"], r["cu"] = W10, Vu.cpu().numpy(), cu.cpu().numpy().astype(np.float64)
    del solver, dW, dA, dB, dW10
    torch.cuda.empty_cache()
    return r


def test_rowscale_bit_exact(run):
    w = run["w"]
    np.testing.assert_array_equal(run["s"], O.row_scale(w.W, w.qmax))


def test_prepare_residuals(run):
    """Backward residual ||(L^T L - A~)[:, S]|| and inverse residual
    ||(L U^T - I)[:, S]|| on sampled columns S, A~ the damped factor, both in
    fp64; bounds n * eps32 relative (normwise Cholesky and triangular-inverse
    bounds).  The preparation is deterministic: two runs agree bit for bit."""
    w = run["w"]
    assert run["info"] == (-1, -1)
    np.testing.assert_array_equal(run["UA"], run["UA2"])
    np.testing.assert_array_equal(run["UB"], run["UB2"])
    rng = np.random.default_rng(1)
    for X, damp, U, L in ((w.A, w.damp_A, run["UA"], run["LA"]),
                          (w.B, w.damp_B, run["UB"], run["LB"])):
        k = X.shape[0]
        S = np.unique(np.concatenate([[0, k - 1], rng.choice(k, size=min(k, 96), replace=False)]))
        Xd = O.damp(X.astype(np.float64), damp)
        L64 = L.astype(np.float64)
        U64 = U.astype(np.float64)
        assert not np.any(np.triu(L64, 1)) and not np.any(np.tril(U64, -1))
        np.testing.assert_allclose(np.diag(U64), 1.0 / np.diag(L64), rtol=1e-5)
        R1 = L64.T @ L64[:, S] - Xd[:, S]
        res = np.linalg.norm(R1) / np.linalg.norm(Xd[:, S])
        assert res < k * EPS32, ("cholesky residual", res)
        R2 = L64 @ U64[S, :].T
        R2[S, np.arange(len(S))] -= 1.0
        inv = np.linalg.norm(R2) / (np.linalg.norm(L64) * np.linalg.norm(U64[S, :]))
        assert inv < k * EPS32, ("inverse residual", inv)


def test_certificate(run):
    """Every rounding decision of the GPU output, replayed in fp64 from its
    own history, agrees except at near ties (at most 0.1%)."""
    w = run["w"]
    s, codes = run["s"], run["codes"]
    np.testing.assert_array_equal(run["V"], (s[:, None] * codes.astype(np.float32)).astype(np.float32))
    cert = O.certificate(w.W, run["V"], codes, run["UA"].astype(np.float64),
                         run["UB"].astype(np.float64), s, *oracle_grid(w.qmin, w.qmax),
                         tol=TOL, max_frac=MAX_FRAC)
    assert cert["ok"], "certificate: %d mismatches, %d not near ties" % (cert["mismatch"], cert["bad"])


def test_top_rows_exact(run):
    w = run["w"]
    if w.m <= 1024 and w.n <= 1024:
        pytest.skip("whole solve checked against the oracle below")
    corner_check(w.W, run["UA"], run["UB"], run["s"], w.qmin, w.qmax, run["codes"], STRIP, w.n,
                 variant="bakron")


def test_left_columns_exact(run):
    w = run["w"]
    if w.m <= 1024 and w.n <= 1024:
        pytest.skip("whole solve checked against the oracle below")
    corner_check(w.W, run["UA"], run["UB"], run["s"], w.qmin, w.qmax, run["codes"], w.m, STRIP,
                 variant="bakron")


def test_cor34_unclamped(run):
    """Corollary 3.4: with an unclamped unit-step grid the proxy loss is at
    most (1/4) sum(l_A^2) sum(l_B^2) <= (1/4) tr(A~) tr(B~); the run also
    passes its certificate."""
    from kronecker_factored_gptq_gb300 import bakron as kb
    w = run["w"]
    ones = np.ones(w.m, np.float32)
    np.testing.assert_array_equal(run["Vu"], run["cu"].astype(np.float32))
    UA, UB = run["UA"].astype(np.float64), run["UB"].astype(np.float64)
    cert = O.certificate(run["W10"], run["Vu"], run["cu"], UA, UB, ones,
                         *oracle_grid(kb.INT32_MIN, kb.INT32_MAX), tol=TOL, max_frac=MAX_FRAC)
    assert cert["ok"], (cert["mismatch"], cert["bad"])
    LA_diag = 1.0 / np.diag(UA)
    LB_diag = 1.0 / np.diag(UB)
    tight = 0.25 * float(np.sum(LA_diag ** 2)) * float(np.sum(LB_diag ** 2))
    trace = O.cor34_bound(O.damp(w.A.astype(np.float64), w.damp_A),
                          O.damp(w.B.astype(np.float64), w.damp_B))
    assert cert["loss"] <= tight, (cert["loss"], tight)
    assert tight <= trace * (1 + 1e-5), (tight, trace)


def test_c1024_whole_solve(run):
    w = run["w"]
    if w.name != "c1024":
        pytest.skip("oracle runs the whole solve at 1024 x 1024 only")
    check_parity(w.W, run["UA"], run["UB"], run["s"], w.qmin, w.qmax, run["V"], run["codes"],
                 variant="bakron")


def test_c1024_b_identity(run):
    """B = I: the solve is per-row GPTQ with Hessian A (oracle ``gptq_rows``).
    Rows are independent, so a near-tie flip cascades only along its row."""
    from kronecker_factored_gptq_gb300 import bakron as kb
    w = run["w"]
    if w.name != "c1024":
        pytest.skip("B = I run at 1024 x 1024")
    I = np.eye(w.m, dtype=np.float32)
    dW, dUA, dI, ds = to_dev(w.W, run["UA"], I, run["s"])
    _, c, _ = kb.bakron_quantize(dW, dUA, dI, ds, w.qmin, w.qmax)
    c = c.cpu().numpy().astype(np.float64)
    one = O.gptq_rows(w.W, run["UA"].astype(np.float64), run["s"], w.qmin, w.qmax)
    diff = c != one.codes
    nt = O.near_tie(one.preround, run["s"][:, None], w.qmin, w.qmax, TOL)
    bad_rows = np.unique(np.nonzero(diff)[0])
    for i in bad_rows:
        assert nt[i, np.nonzero(diff[i])[0][0]]
    assert len(bad_rows) <= max(1, MAX_FRAC * w.m)


def test_c1024_full_vs_antidiag(run):
    """The anti-diagonal kernel, guided by the full variant's codes, returns
    them exactly with at most 0.1% guided decisions."""
    from kronecker_factored_gptq_gb300 import bakron as kb
    w = run["w"]
    if w.name != "c1024":
        pytest.skip("the anti-diagonal kernel does O(m^2 n^2) work; run at 1024 x 1024")
    dW, dUA, dUB, ds, dc = to_dev(w.W, run["UA"], run["UB"], run["s"], run["codes"].astype(np.int8))
    V2, c2, _, over = kb.bakron_quantize_antidiag(dW, dUA, dUB, ds, w.qmin, w.qmax, guide_codes=dc,
                                                  guide_tol=TOL)
    assert np.array_equal(c2.cpu().numpy().astype(np.float64), run["codes"])
    assert over <= MAX_FRAC * w.m * w.n
    np.testing.assert_array_equal(V2.cpu().numpy(), run["V"])
