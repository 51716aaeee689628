"""Whole-solve parity against the fp64 oracle at the full workload sizes.

The oracle's row-accumulator solver (``oracle.rowacc``, plain C, m n (m + n)
fp64 flops on the host cores, traversed by blocks of rows) reaches the full
sizes in seconds to a minute, so here every code of
the GPU solve is compared with the oracle, not only the strips and the
certificate of ``test_gpu_workloads.py``:

* inputs: the workload generator's W, A, B; factors prepared by the ORACLE in
  fp64 and rounded once to fp32, fed to both sides (nothing the oracle reads
  comes from the CUDA path); per-row grid from the oracle's ``row_scale``;
* the GPU solve is ``bakron_quantize`` with the default options, the launch
  configuration the benchmark times;
* rule (summary page "FastKron: Efficient Quantization with Kronecker-Factored
  Hessians", Theorem 3.2 and Corollary 3.4): the oracle, guided by the GPU
  codes only at its own near ties (within 1e-4 grid units of a rounding
  boundary), must reproduce every code, with at most 0.1% guided decisions;
  V = s c exactly; the proxy loss ||L(B)(V-W)L(A)^T||_F^2 of the GPU output
  within FULL_LOSS_RTOL relative of the unguided oracle's (see below);
* the GPU's own factor preparation against the oracle's fp64 factors, within
  10 n eps cond (the forward error bound of the Cholesky and triangular
  inverse), cond from Lanczos estimates of the extreme eigenvalues.

The 1024 x 1024 workload is compared with the numpy oracle in
``test_gpu_workloads.py``.
"""

import numpy as np
import pytest

import oracle as O
from kronecker_factored_gptq_gb300 import workloads as WL

from _gpu_helpers import TOL, MAX_FRAC, to_dev

pytestmark = pytest.mark.gpu

# Once one near-tie decision goes the other way (both are correct roundings),
# every later entry sees a different error history: the GPU's trajectory and
# the unguided oracle's are two valid GPTQ runs, and at these sizes their
# losses drift apart by more than 1e-3.  Measured with the oracle alone on the
# 14336 x 4096 workload (seed 0): perturbing W by 1e-7 and 1e-6 relative
# moved the loss by 1.7e-3 and 2.4e-3 (29% and 36% of the codes changed).
# The bound is twice the larger drift; the codes themselves are checked
# exactly against the guided oracle.
FULL_LOSS_RTOL = 5e-3

FULL = ["c4096", "mlp4096x14336", "mlp14336x4096", "c8192"]
RB = 8   # rows per block of the oracle's row-blocked traversal
EPS32 = float(np.finfo(np.float32).eps)


@pytest.fixture(scope="module", params=FULL)
def case(request):
    import torch
    from kronecker_factored_gptq_gb300 import bakron as kb
    w = WL.load(request.param, seed=0, device="cuda")
    LA, UA = O.prepare(w.A, w.damp_A)
    LB, UB = O.prepare(w.B, w.damp_B)
    UA32, UB32 = UA.astype(np.float32), UB.astype(np.float32)
    s = O.row_scale(w.W, w.qmax)
    dW, dUA, dUB, ds = to_dev(w.W, UA32, UB32, s)
    V, c, _ = kb.bakron_quantize(dW, dUA, dUB, ds, w.qmin, w.qmax)
    r = {"w": w, "s": s, "UA32": UA32, "UB32": UB32, "UA": UA, "UB": UB,
         "V": V.cpu().numpy(), "codes": c.cpu().numpy().astype(np.float64)}
    del dW, dUA, dUB, ds, V, c
    dA, dB = to_dev(w.A, w.B)
    gUA, gUB, _, _, info = kb.bakron_prepare(dA, w.damp_A, dB, w.damp_B)
    r["info"] = info
    r["gUA"], r["gUB"] = gUA.cpu().numpy(), gUB.cpu().numpy()
    del dA, dB, gUA, gUB
    torch.cuda.empty_cache()
    return r


def test_whole_solve_matches_oracle(case):
    w, s, codes, V = case["w"], case["s"], case["codes"], case["V"]
    UA = case["UA32"].astype(np.float64)
    UB = case["UB32"].astype(np.float64)
    np.testing.assert_array_equal(V, (s[:, None] * codes.astype(np.float32)).astype(np.float32))
    g = O.rowacc(w.W, UA, UB, s, w.qmin, w.qmax, guide=codes, guide_tol=TOL, rows_per_block=RB)
    diff = int(np.count_nonzero(g.codes != codes))
    assert diff == 0, "%s: %d GPU codes differ from the guided oracle (not near ties)" % (w.name, diff)
    assert g.overrides <= MAX_FRAC * w.m * w.n, (w.name, g.overrides)
    LA = O.lower_from_update(UA)
    LB = O.lower_from_update(UB)
    l_gpu = O.proxy_loss(w.W, V, LA, LB)
    if g.overrides == 0:
        # the guide changed no decision: the guided run is the oracle's own
        l_ref = l_gpu
    else:
        ref = O.rowacc(w.W, UA, UB, s, w.qmin, w.qmax, rows_per_block=RB)
        V_ref = (s[:, None] * ref.codes.astype(np.float32)).astype(np.float32)
        l_ref = O.proxy_loss(w.W, V_ref, LA, LB)
    assert abs(l_gpu - l_ref) <= FULL_LOSS_RTOL * abs(l_ref), (w.name, l_gpu, l_ref)


def _cond_estimate(Ad, U):
    """lambda_max(Ad) / lambda_min(Ad) by Lanczos: the largest eigenvalue of
    Ad, and of Ad^{-1} = U^T U (U the oracle's update factor)."""
    from scipy.sparse.linalg import LinearOperator, eigsh
    k = Ad.shape[0]
    lmax = eigsh(Ad, k=1, which="LA", tol=1e-4, return_eigenvectors=False)[0]
    inv = LinearOperator((k, k), matvec=lambda v: U.T @ (U @ v), dtype=np.float64)
    imax = eigsh(inv, k=1, which="LA", tol=1e-4, ncv=64, return_eigenvectors=False)[0]
    return float(lmax * imax)


def test_gpu_factors_match_oracle_factors(case):
    w = case["w"]
    assert case["info"] == (-1, -1)
    for X, damp, U_o, U_g in ((w.A, w.damp_A, case["UA"], case["gUA"]),
                              (w.B, w.damp_B, case["UB"], case["gUB"])):
        k = X.shape[0]
        Ad = O.damp(X.astype(np.float64), damp)
        cond = _cond_estimate(Ad, U_o)
        Ug = U_g.astype(np.float64)
        assert not np.any(np.tril(Ug, -1))
        rel = np.linalg.norm(Ug - U_o) / np.linalg.norm(U_o)
        assert rel < 10 * k * EPS32 * cond, (w.name, k, rel, cond)
