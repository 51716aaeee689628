"""Seeded input generators: shapes, determinism, definiteness, and the oracle
on the 64 x 64 workload (naive explicit-Hessian GPTQ against the anti-diagonal
and BaKron variants, the certificate and the Corollary 3.4 bound)."""

import numpy as np

import oracle as O
from kronecker_factored_gptq_gb300 import workloads as WL


def test_tiny64_shapes_and_determinism():
    a = WL.tiny64(seed=0)
    b = WL.tiny64(seed=0)
    c = WL.tiny64(seed=1)
    assert a.W.shape == (64, 64) and a.A.shape == (64, 64) and a.B.shape == (64, 64)
    assert a.W.dtype == np.float32 and a.A.dtype == np.float32
    np.testing.assert_array_equal(a.W, b.W)
    np.testing.assert_array_equal(a.A, b.A)
    assert not np.array_equal(a.W, c.W)
    assert (a.bits, a.qmin, a.qmax) == (4, -8, 7)
    np.testing.assert_allclose(np.std(a.W), 0.02, rtol=0.1)


def test_random_problem_ragged():
    w = WL.random_problem(37, 53, seed=3, bits=3)
    assert w.W.shape == (37, 53) and w.A.shape == (53, 53) and w.B.shape == (37, 37)
    assert (w.qmin, w.qmax) == (-4, 3)
    assert np.all(np.linalg.eigvalsh(w.A.astype(np.float64)) > 0)


def test_ar1_rows_covariance():
    X = WL._ar1_rows(np.random.default_rng(0), 6, 200000, 0.9)
    C = X @ X.T / X.shape[1]
    idx = np.arange(6)
    np.testing.assert_allclose(C, 0.9 ** np.abs(idx[:, None] - idx[None, :]), atol=0.02)


def test_haar_is_orthogonal():
    Q = WL._haar_orthogonal(np.random.default_rng(0), 33)
    np.testing.assert_allclose(Q @ Q.T, np.eye(33), atol=1e-12)


def test_oracle_on_tiny64_workload():
    w = WL.tiny64(seed=0)
    LA, UA = O.prepare(w.A, w.damp_A)
    LB, UB = O.prepare(w.B, w.damp_B)
    s = O.row_scale(w.W, w.qmax)
    ref = O.naive_vec_gptq(w.W, s, w.qmin, w.qmax, A=O.damp(w.A, w.damp_A), B=O.damp(w.B, w.damp_B))
    for r in (O.antidiag(w.W, UA, UB, s, w.qmin, w.qmax), O.bakron(w.W, UA, UB, s, w.qmin, w.qmax)):
        np.testing.assert_array_equal(r.codes, ref.codes)
    cert = O.certificate(w.W, ref.V, ref.codes, UA, UB, s, w.qmin, w.qmax)
    assert cert["ok"] and cert["mismatch"] == 0
    # unclamped unit-step run on 10 W: Corollary 3.4
    W10 = 10.0 * w.W.astype(np.float64)
    r = O.bakron(W10, UA, UB, np.ones(64))
    loss = O.proxy_loss(W10, r.V, LA, LB)
    assert loss <= O.cor34_tight_bound(LA, LB) <= O.cor34_bound(O.damp(w.A, w.damp_A), O.damp(w.B, w.damp_B))
