"""GPU parity: the CUDA path through the C ABI against the fp64 oracle.

Sizes here are small enough for the oracle to finish in seconds but span
several 128-tiles and ragged tails; the full-size workloads are covered in
test_gpu_workloads.py.  Every solve test runs both propagation paths (fp32
FMA and, where built, tcgen05 3xTF32).
"""

import numpy as np
import pytest

import oracle as O
from kronecker_factored_gptq_gb300 import workloads as WL

from _gpu_helpers import (TOL, MAX_FRAC, check_parity, gpu_quantize, shared_factors, to_dev)

pytestmark = pytest.mark.gpu


def variants():
    from kronecker_factored_gptq_gb300 import bakron as kb
    v = [0]
    if kb.default_opts().use_3xtf32 == 1:
        v.append(1)
    return v


@pytest.fixture(scope="module")
def kb():
    from kronecker_factored_gptq_gb300 import bakron as kb
    kb.lib()
    return kb


def test_rowscale_bit_exact(kb):
    rng = np.random.default_rng(0)
    W = (0.02 * rng.standard_normal((37, 301))).astype(np.float32)
    W[5] = 0.0
    W[7, 3] = -0.9
    for qmax in (1, 3, 7):
        (dW,) = to_dev(W)
        s = kb.bakron_rowscale(dW, qmax).cpu().numpy()
        np.testing.assert_array_equal(s, O.row_scale(W, qmax))


@pytest.mark.parametrize("n", [64, 200, 384, 677, 1300])
def test_prepare_matches_oracle(kb, n):
    w = WL.random_problem(n, n, seed=n, oversample=3)
    dA, dB = to_dev(w.A, w.B)
    UA, UB, LA, LB, info = kb.bakron_prepare(dA, 0.01, dB, 0.02, want_L=True)
    assert info == (-1, -1)
    for X, damp, U, L in ((w.A, 0.01, UA, LA), (w.B, 0.02, UB, LB)):
        Xd = O.damp(X.astype(np.float64), damp)
        Lo, Uo = O.prepare(X.astype(np.float64), damp)
        U = U.cpu().numpy().astype(np.float64)
        L = L.cpu().numpy().astype(np.float64)
        assert np.allclose(np.tril(U, -1), 0) and np.allclose(np.triu(L, 1), 0)
        cond = np.linalg.cond(Xd)
        eps = np.finfo(np.float32).eps
        res = np.linalg.norm(L.T @ L - Xd) / np.linalg.norm(Xd)
        assert res < 50 * n * eps, res
        inv = np.linalg.norm(U @ L.T - np.eye(n))
        assert inv < 50 * n * eps * np.sqrt(cond), inv
        rel = np.linalg.norm(U - Uo) / np.linalg.norm(Uo)
        assert rel < 10 * n * eps * cond, (rel, cond)
        np.testing.assert_allclose(np.diag(U), 1.0 / np.diag(L), rtol=1e-5)


def test_prepare_reports_not_pd(kb):
    rng = np.random.default_rng(3)
    X = rng.standard_normal((150, 150))
    A = (X @ X.T / 150 + np.eye(150)).astype(np.float32)
    A[100, 100] = -5.0   # breaks definiteness at original index 100 or later
    (dA,) = to_dev(A)
    with pytest.raises(kb.BakronError) as ei:
        kb.bakron_prepare(dA, 0.0)
    assert ei.value.status == 2
    assert 0 <= ei.value.info[0] <= 100


@pytest.mark.parametrize("use_tc", variants())
@pytest.mark.parametrize("m,n,bits", [(64, 64, 4), (128, 128, 3), (200, 328, 4), (300, 260, 2),
                                      (1, 300, 4), (257, 1, 4), (129, 384, 4)])
def test_quantize_parity(kb, use_tc, m, n, bits):
    w = WL.random_problem(m, n, seed=m * 7 + n, bits=bits)
    UA32, UB32 = shared_factors(w.A, w.damp_A, w.B, w.damp_B)
    s = O.row_scale(w.W, w.qmax)
    V, c, pre = gpu_quantize(w.W, UA32, UB32, s, w.qmin, w.qmax, use_tc)
    r = check_parity(w.W, UA32, UB32, s, w.qmin, w.qmax, V, c, pre)
    assert r["preround_err_grid_units"] < TOL


@pytest.mark.parametrize("use_tc", variants())
def test_tiny64_workload_against_naive(kb, use_tc):
    w = WL.tiny64(seed=0)
    UA32, UB32 = shared_factors(w.A, w.damp_A, w.B, w.damp_B)
    s = O.row_scale(w.W, w.qmax)
    V, c, pre = gpu_quantize(w.W, UA32, UB32, s, w.qmin, w.qmax, use_tc)
    ref = O.naive_vec_gptq(w.W, s, w.qmin, w.qmax, UA=UA32.astype(np.float64),
                           UB=UB32.astype(np.float64), guide=c)
    assert np.array_equal(ref.codes, c) and ref.overrides <= MAX_FRAC * 64 * 64
    check_parity(w.W, UA32, UB32, s, w.qmin, w.qmax, V, c, pre)


@pytest.mark.parametrize("use_tc", variants())
def test_unclamped_unit_grid_cor34(kb, use_tc):
    w = WL.tiny64(seed=1)
    UA32, UB32 = shared_factors(w.A, w.damp_A, w.B, w.damp_B)
    W10 = (10.0 * w.W).astype(np.float32)
    ones = np.ones(64, np.float32)
    V, c, pre = gpu_quantize(W10, UA32, UB32, ones, kb.INT32_MIN, kb.INT32_MAX, use_tc)
    check_parity(W10, UA32, UB32, ones, kb.INT32_MIN, kb.INT32_MAX, V, c, pre)
    LA = O.lower_from_update(UA32.astype(np.float64))
    LB = O.lower_from_update(UB32.astype(np.float64))
    loss = O.proxy_loss(W10, V, LA, LB)
    Ad = np.linalg.inv(UA32.astype(np.float64).T @ UA32.astype(np.float64))
    Bd = np.linalg.inv(UB32.astype(np.float64).T @ UB32.astype(np.float64))
    assert loss <= O.cor34_tight_bound(LA, LB) <= O.cor34_bound(Ad, Bd) * (1 + 1e-9)


@pytest.mark.parametrize("use_tc", variants())
def test_b_identity_is_rowwise_gptq(kb, use_tc):
    w = WL.random_problem(150, 270, seed=9)
    UA32, _ = shared_factors(w.A, w.damp_A, w.B, w.damp_B)
    I = np.eye(150, dtype=np.float32)
    s = O.row_scale(w.W, w.qmax)
    V, c, pre = gpu_quantize(w.W, UA32, I, s, w.qmin, w.qmax, use_tc)
    one = O.gptq_rows(w.W, UA32.astype(np.float64), s, w.qmin, w.qmax)
    diff = c != one.codes
    nt = O.near_tie(one.preround, s[:, None], w.qmin, w.qmax, TOL)
    # rows are independent here, so a near-tie flip cascades only along its row
    bad_rows = np.unique(np.nonzero(diff)[0])
    for i in bad_rows:
        first = np.nonzero(diff[i])[0][0]
        assert nt[i, first]
    assert len(bad_rows) <= max(1, MAX_FRAC * 150)


def test_antidiag_kernel_parity(kb):
    w = WL.random_problem(96, 160, seed=4)
    UA32, UB32 = shared_factors(w.A, w.damp_A, w.B, w.damp_B)
    s = O.row_scale(w.W, w.qmax)
    dW, dUA, dUB, ds = to_dev(w.W, UA32, UB32, s)
    V, c, pre, over = kb.bakron_quantize_antidiag(dW, dUA, dUB, ds, w.qmin, w.qmax, want_preround=True)
    assert over == 0
    check_parity(w.W, UA32, UB32, s, w.qmin, w.qmax, V.cpu().numpy(),
                 c.cpu().numpy().astype(np.float64), pre.cpu().numpy())


@pytest.mark.parametrize("use_tc", variants())
@pytest.mark.parametrize("m,n", [(256, 384), (520, 300)])
def test_full_vs_antidiag_guided(kb, use_tc, m, n):
    """The full and anti-diagonal GPU variants agree under the near-tie rule:
    the anti-diagonal kernel, guided by the full variant's codes, reproduces
    them exactly with at most 0.1% guided decisions."""
    w = WL.random_problem(m, n, seed=m + n)
    UA32, UB32 = shared_factors(w.A, w.damp_A, w.B, w.damp_B)
    s = O.row_scale(w.W, w.qmax)
    V, c, _ = gpu_quantize(w.W, UA32, UB32, s, w.qmin, w.qmax, use_tc, preround=False)
    dW, dUA, dUB, ds, dc = to_dev(w.W, UA32, UB32, s, c.astype(np.int8))
    V2, c2, _, over = kb.bakron_quantize_antidiag(dW, dUA, dUB, ds, w.qmin, w.qmax, guide_codes=dc,
                                                  guide_tol=TOL)
    assert np.array_equal(c2.cpu().numpy().astype(np.float64), c)
    assert over <= MAX_FRAC * m * n
    np.testing.assert_array_equal(V2.cpu().numpy(), V)


# ------------------------------------------------------------ error paths

def test_nonfinite_input(kb):
    w = WL.random_problem(130, 140, seed=2)
    UA32, UB32 = shared_factors(w.A, w.damp_A, w.B, w.damp_B)
    s = O.row_scale(w.W, w.qmax)
    W = w.W.copy()
    W[70, 90] = np.nan
    dW, dUA, dUB, ds = to_dev(W, UA32, UB32, s)
    for use_tc in variants():
        with pytest.raises(kb.BakronError) as ei:
            kb.bakron_quantize(dW, dUA, dUB, ds, w.qmin, w.qmax, opts=kb.default_opts(use_3xtf32=use_tc))
        assert ei.value.status == 3
    bad_s = s.copy()
    bad_s[3] = 0.0
    (dbs,) = to_dev(bad_s)
    with pytest.raises(kb.BakronError) as ei:
        kb.bakron_quantize(to_dev(w.W)[0], dUA, dUB, dbs, w.qmin, w.qmax)
    assert ei.value.status == 3


def test_code_range(kb):
    w = WL.random_problem(64, 64, seed=5)
    UA32, UB32 = shared_factors(w.A, w.damp_A, w.B, w.damp_B)
    W = (w.W * 1e4).astype(np.float32)
    dW, dUA, dUB, ds = to_dev(W, UA32, UB32, np.ones(64, np.float32))
    with pytest.raises(kb.BakronError) as ei:
        kb.bakron_quantize(dW, dUA, dUB, ds, kb.INT32_MIN, kb.INT32_MAX)
    assert ei.value.status == 4


def test_bounded_wait_times_out_without_hanging(kb):
    """A CTA that never arrives at the grid barrier (host-set test flag): the
    others give up after the spin budget and the call returns TIMEOUT."""
    import time
    w = WL.random_problem(64, 96, seed=6)
    UA32, UB32 = shared_factors(w.A, w.damp_A, w.B, w.damp_B)
    s = O.row_scale(w.W, w.qmax)
    dW, dUA, dUB, ds = to_dev(w.W, UA32, UB32, s)
    opts = kb.default_opts(fault_inject=1, spin_budget_cycles=20_000_000)
    t0 = time.time()
    with pytest.raises(kb.BakronError) as ei:
        kb.bakron_quantize_antidiag(dW, dUA, dUB, ds, w.qmin, w.qmax, opts=opts)
    assert ei.value.status == 5
    assert time.time() - t0 < 30
    # the context is still usable afterwards
    V, c, _, _ = kb.bakron_quantize_antidiag(dW, dUA, dUB, ds, w.qmin, w.qmax)
    check_parity(w.W, UA32, UB32, s, w.qmin, w.qmax, V.cpu().numpy(), c.cpu().numpy().astype(np.float64))


def test_invalid_workspace(kb):
    import torch
    w = WL.random_problem(64, 64, seed=7)
    dW = to_dev(w.W)[0]
    ws = torch.empty(1024, dtype=torch.uint8, device="cuda")
    with pytest.raises(ValueError):
        kb.bakron_quantize(dW, dW, dW, dW[0], -8, 7, workspace=ws)


@pytest.mark.parametrize("one_sided", [False, True])
def test_solve_is_bit_reproducible(kb, one_sided):
    """Every W~ tile receives its propagation updates in a fixed order (the
    deferred chunks that overlap a later propagation are waited for first), so
    two solves of the same input agree bit for bit."""
    import torch
    w = WL.random_problem(1100, 1300, seed=31)
    UA32, UB32 = shared_factors(w.A, w.damp_A, w.B, w.damp_B)
    s = O.row_scale(w.W, w.qmax)
    dW, dUA, dUB, ds = to_dev(w.W, UA32, UB32, s)
    outs = []
    for _ in range(2):
        V, c, pre = kb.bakron_quantize(dW, dUA, None if one_sided else dUB, ds, w.qmin, w.qmax,
                                       want_preround=True)
        torch.cuda.synchronize()
        outs.append((V.cpu().numpy(), c.cpu().numpy(), pre.cpu().numpy()))
    for a, b in zip(outs[0], outs[1]):
        np.testing.assert_array_equal(a, b)
