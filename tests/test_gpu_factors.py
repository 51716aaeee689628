"""GPU parity of the Kronecker-factor accumulation (bakron_factors) against
the fp64 oracle (``oracle.kfac_factors``, ``oracle.shampoo_factors``).

The GPU sums in fp32 from a 3xTF32 split (each product keeps hi*hi + hi*lo +
lo*hi; the dropped lo*lo is 2^-22 relative), accumulating every 128 samples
in a fresh tensor-core buffer and the chunks in fp32 registers.  Bound: every
entry within 2e-5 * sqrt(A_ii A_jj) of the fp64 value (A is positive
semidefinite, so this is the Cauchy-Schwarz scale of the summed terms), and a
relative Frobenius error of at most 1e-5.
"""

import numpy as np
import pytest

import oracle as O

from _gpu_helpers import to_dev

pytestmark = pytest.mark.gpu

TOLF = 2e-5


def _check(got, ref):
    got = got.astype(np.float64)
    d = np.sqrt(np.abs(np.diag(ref)))
    scale = np.outer(d, d) + 1e-30
    assert np.max(np.abs(got - ref) / scale) <= TOLF
    assert np.linalg.norm(got - ref) <= 1e-5 * np.linalg.norm(ref) + 1e-30
    np.testing.assert_array_equal(got, got.T)


def _samples(N, n, m, seed):
    rng = np.random.default_rng(seed)
    X = rng.standard_normal((N, n)) * np.exp(rng.standard_normal(n))[None, :]   # heavy channels
    G = rng.standard_normal((N, m))
    return X.astype(np.float32), G.astype(np.float32)


@pytest.mark.parametrize("mode", ["kfac", "shampoo"])
@pytest.mark.parametrize("N,n,m", [(1, 64, 3), (100, 200, 128), (300, 130, 257), (257, 1, 5),
                                   (1000, 384, 96)])
def test_factors_parity(mode, N, n, m):
    from kronecker_factored_gptq_gb300 import bakron as kb
    X, G = _samples(N, n, m, seed=N + n + m)
    dX, dG = to_dev(X, G)
    md = kb.FACTORS_KFAC if mode == "kfac" else kb.FACTORS_SHAMPOO
    A, B = kb.bakron_factors(dX, dG, mode=md)
    ref = O.kfac_factors(X, G) if mode == "kfac" else O.shampoo_factors(X, G)
    _check(A.cpu().numpy(), ref[0])
    _check(B.cpu().numpy(), ref[1])


def test_factors_one_side_only():
    from kronecker_factored_gptq_gb300 import bakron as kb
    X, G = _samples(500, 150, 70, seed=3)
    dX, dG = to_dev(X, G)
    A, B = kb.bakron_factors(dX, None)
    assert B is None
    _check(A.cpu().numpy(), O.kfac_factors(X, None)[0])
    A, B = kb.bakron_factors(None, dG)
    assert A is None
    _check(B.cpu().numpy(), O.kfac_factors(None, G)[1])
    with pytest.raises(kb.BakronError):
        kb.bakron_factors(dX, None, mode=kb.FACTORS_SHAMPOO)


def test_factors_feed_the_solver():
    """K-FAC factors from samples, prepared and solved on the GPU: the solve
    passes the full parity check against the oracle on the same (GPU-made)
    fp32 factors."""
    import torch
    from kronecker_factored_gptq_gb300 import bakron as kb
    from _gpu_helpers import check_parity
    X, G = _samples(2048, 192, 160, seed=4)
    rng = np.random.default_rng(5)
    W = (0.02 * rng.standard_normal((160, 192))).astype(np.float32)
    dX, dG, dW = to_dev(X, G, W)
    A, B = kb.bakron_factors(dX, dG)
    UA, UB, _, _, info = kb.bakron_prepare(A, 0.01, B, 0.01)
    assert info == (-1, -1)
    s = O.row_scale(W, 7)
    UA32, UB32 = UA.cpu().numpy(), UB.cpu().numpy()
    dUA, dUB, ds = to_dev(UA32, UB32, s)
    V, c, pre = kb.bakron_quantize(dW, dUA, dUB, ds, -8, 7, want_preround=True)
    torch.cuda.synchronize()
    check_parity(W, UA32, UB32, s, -8, 7, V.cpu().numpy(), c.cpu().numpy().astype(np.float64),
                 pre.cpu().numpy())


def test_factors_full_size_sampled_rows():
    """N = 16384 samples of 8192 features (the shape of the 8192 x 8192
    workload's activation stream): rows of A checked against fp64 sums."""
    from kronecker_factored_gptq_gb300 import bakron as kb
    N, n = 16384, 8192
    rng = np.random.default_rng(6)
    X = rng.standard_normal((N, n), dtype=np.float32)
    (dX,) = to_dev(X)
    A, _ = kb.bakron_factors(dX, None)
    A = A.cpu().numpy()
    rows = [0, 1, 4095, 8191] + list(rng.choice(n, 4, replace=False))
    X64 = X.astype(np.float64)
    diag = np.einsum("ti,ti->i", X64, X64) / N
    for i in rows:
        ref = X64[:, i] @ X64 / N
        scale = np.sqrt(diag[i] * diag)
        assert np.max(np.abs(A[i] - ref) / scale) <= TOLF, i
    np.testing.assert_array_equal(A[rows][:, rows], A[rows][:, rows].T)
