"""GPU parity on other base quantizers: column-group and asymmetric (min-max
with zero point) grids, for the two-sided solver and the one-sided path.

The oracle takes the same grid as a per-entry ``oracle.Grid`` built from the
GPU's grid parameters, which must first equal the oracle's own
(``oracle.symmetric_grid`` / ``oracle.asymmetric_grid``) bit for bit.  The
comparison rule is the one of the other parity tests: guided oracle (GPU code
taken only at the oracle's own near ties), exact codes after that, at most
0.1% guided decisions, V = s (c - z) in fp32 bit for bit, pre-rounding values
within 1e-4 grid units, the certificate, proxy loss to 1e-3.
"""

import numpy as np
import pytest

import oracle as O
from kronecker_factored_gptq_gb300 import workloads as WL

from _gpu_helpers import TOL, MAX_FRAC, LOSS_RTOL, shared_factors, to_dev

pytestmark = pytest.mark.gpu


def gpu_grid(W, bits, asym, group):
    from kronecker_factored_gptq_gb300 import bakron as kb
    (dW,) = to_dev(W)
    s, z, qmin, qmax = kb.bakron_grid_params(dW, bits, asymmetric=asym, group=group)
    return s.cpu().numpy(), z.cpu().numpy(), qmin, qmax


def oracle_grid_of(W, bits, asym, group):
    return (O.asymmetric_grid if asym else O.symmetric_grid)(W, bits, group)


def as_grid(s, z, qmin, qmax, group, n):
    g = n if (not group or group >= n) else group
    S = np.repeat(s.astype(np.float64), g, axis=1)[:, :n]
    Z = np.repeat(z.astype(np.float64), g, axis=1)[:, :n]
    return O.Grid(S, Z, qmin, qmax)


def check_grid_parity(W, UA32, UB32, grid, V, codes, pre, one_sided=False):
    UA = UA32.astype(np.float64)
    m, n = W.shape
    if one_sided:
        g = O.gptq_rows(W, UA, grid, guide=codes, guide_tol=TOL)
        ref = O.gptq_rows(W, UA, grid)
        UB = np.eye(m)
    else:
        UB = UB32.astype(np.float64)
        g = O.antidiag(W, UA, UB, grid, guide=codes, guide_tol=TOL)
        ref = O.antidiag(W, UA, UB, grid)
    diff = int(np.count_nonzero(g.codes != codes))
    assert diff == 0, "GPU codes differ from the guided oracle at %d entries" % diff
    assert g.overrides <= max(1, MAX_FRAC * m * n), g.overrides
    S32 = grid.S.astype(np.float32)
    Z32 = grid.Z.astype(np.float32)
    want_V = (S32 * (codes.astype(np.float32) - Z32)).astype(np.float32)
    np.testing.assert_array_equal(V, want_V)
    err = np.max(np.abs(pre - g.preround) / grid.S)
    assert err < TOL, err
    cert = O.certificate(W, V, codes, UA, UB, grid, tol=TOL, max_frac=MAX_FRAC)
    assert cert["ok"], (cert["mismatch"], cert["bad"])
    LA = O.lower_from_update(UA)
    LB = O.lower_from_update(UB)
    V_ref = (S32 * (ref.codes.astype(np.float32) - Z32)).astype(np.float32)
    l_gpu = O.proxy_loss(W, V, LA, LB)
    l_ref = O.proxy_loss(W, V_ref, LA, LB)
    assert abs(l_gpu - l_ref) <= LOSS_RTOL * abs(l_ref) + 1e-30


@pytest.mark.parametrize("asym", [False, True])
@pytest.mark.parametrize("bits,group", [(2, None), (3, 32), (4, 64), (7, 96), (8, None)])
def test_grid_params_bit_exact(asym, bits, group):
    rng = np.random.default_rng(bits * 10 + (group or 0))
    W = (0.03 * rng.standard_normal((37, 300)) + 0.005).astype(np.float32)
    W[4] = 0.0
    W[6, :40] = 0.0
    W[7] = np.abs(W[7])          # an all-positive row (lo = 0)
    s, z, qmin, qmax = gpu_grid(W, bits, asym, group)
    _, s_ref, z_ref = oracle_grid_of(W, bits, asym, group)
    np.testing.assert_array_equal(s, s_ref)
    np.testing.assert_array_equal(z, z_ref)
    assert (qmin, qmax) == ((0, (1 << bits) - 1) if asym else (-(1 << (bits - 1)), (1 << (bits - 1)) - 1))


@pytest.mark.parametrize("m,n,bits,asym,group", [(200, 328, 3, True, 32), (129, 384, 4, False, 128),
                                                 (300, 260, 4, True, 64), (64, 64, 2, True, None),
                                                 (130, 200, 7, True, 32)])
def test_grid_two_sided_parity(m, n, bits, asym, group):
    from kronecker_factored_gptq_gb300 import bakron as kb
    w = WL.random_problem(m, n, seed=m + n + bits, bits=bits)
    UA32, UB32 = shared_factors(w.A, w.damp_A, w.B, w.damp_B)
    s, z, qmin, qmax = gpu_grid(w.W, bits, asym, group)
    dW, dUA, dUB, ds, dz = to_dev(w.W, UA32, UB32, s, z)
    V, c, pre = kb.bakron_quantize_grid(dW, dUA, dUB, ds, dz, group, qmin, qmax, want_preround=True)
    grid = as_grid(s, z, qmin, qmax, group, n)
    check_grid_parity(w.W, UA32, UB32, grid, V.cpu().numpy(), c.cpu().numpy().astype(np.float64),
                      pre.cpu().numpy())


@pytest.mark.parametrize("m,n,bits,asym,group", [(150, 320, 3, True, 32), (257, 130, 4, False, 64)])
def test_grid_one_sided_parity(m, n, bits, asym, group):
    from kronecker_factored_gptq_gb300 import bakron as kb
    w = WL.random_problem(m, n, seed=m * 2 + n, bits=bits)
    UA32, _ = shared_factors(w.A, w.damp_A, w.B, w.damp_B)
    s, z, qmin, qmax = gpu_grid(w.W, bits, asym, group)
    dW, dUA, ds, dz = to_dev(w.W, UA32, s, z)
    V, c, pre = kb.bakron_quantize_grid(dW, dUA, None, ds, dz, group, qmin, qmax, want_preround=True)
    grid = as_grid(s, z, qmin, qmax, group, n)
    check_grid_parity(w.W, UA32, None, grid, V.cpu().numpy(), c.cpu().numpy().astype(np.float64),
                      pre.cpu().numpy(), one_sided=True)


def test_grid_rejects_bad_arguments():
    from kronecker_factored_gptq_gb300 import bakron as kb
    w = WL.random_problem(64, 96, seed=1)
    UA32, UB32 = shared_factors(w.A, w.damp_A, w.B, w.damp_B)
    dW, dUA, dUB = to_dev(w.W, UA32, UB32)
    with pytest.raises(ValueError):
        kb.bakron_grid_params(dW, 4, group=48)          # not a multiple of 32
    s, z, qmin, qmax = kb.bakron_grid_params(dW, 4, asymmetric=True, group=32)
    z[3, 1] = 20.0                                       # outside [0, 15]
    with pytest.raises(kb.BakronError) as ei:
        kb.bakron_quantize_grid(dW, dUA, dUB, s, z, 32, qmin, qmax)
    assert ei.value.status == 4
    z[3, 1] = 2.5                                        # not an integer
    with pytest.raises(kb.BakronError) as ei:
        kb.bakron_quantize_grid(dW, dUA, dUB, s, z, 32, qmin, qmax)
    assert ei.value.status == 4


def test_grid_full_size_strips():
    """4096 x 4096 workload, 4-bit asymmetric grid in groups of 128, the whole
    path on the GPU: the top 128 rows and the left 128 columns are complete
    problems for the oracle (updates only move to the bottom-right)."""
    import torch
    from kronecker_factored_gptq_gb300 import bakron as kb
    w = WL.load("c4096", seed=0, device="cuda")
    dW, dA, dB = to_dev(w.W, w.A, w.B)
    s, z, qmin, qmax = kb.bakron_grid_params(dW, 4, asymmetric=True, group=128)
    UA, UB, _, _, info = kb.bakron_prepare(dA, w.damp_A, dB, w.damp_B)
    assert info == (-1, -1)
    V, c, _ = kb.bakron_quantize_grid(dW, UA, UB, s, z, 128, qmin, qmax)
    torch.cuda.synchronize()
    s, z = s.cpu().numpy(), z.cpu().numpy()
    _, s_ref, z_ref = O.asymmetric_grid(w.W, 4, 128)
    np.testing.assert_array_equal(s, s_ref)
    np.testing.assert_array_equal(z, z_ref)
    c = c.cpu().numpy().astype(np.float64)
    grid = as_grid(s, z, qmin, qmax, 128, w.n)
    UA64 = UA.cpu().numpy().astype(np.float64)
    UB64 = UB.cpu().numpy().astype(np.float64)
    for (a, b) in ((128, w.n), (w.m, 128)):
        sub = O.Grid(grid.S[:a, :b], grid.Z[:a, :b], qmin, qmax)
        g = O.antidiag(w.W[:a, :b], UA64[:b, :b], UB64[:a, :a], sub, guide=c[:a, :b], guide_tol=TOL)
        assert np.count_nonzero(g.codes != c[:a, :b]) == 0
        assert g.overrides <= MAX_FRAC * a * b


@pytest.mark.parametrize("m,n,group,one_sided", [(40, 100, 32, False), (33, 70, 64, True),
                                                  (5, 40, 32, False)])
def test_grid_ragged_groups_and_small_shapes(m, n, group, one_sided):
    """Groups that do not divide n (the last group is short) and problems
    smaller than one tile."""
    from kronecker_factored_gptq_gb300 import bakron as kb
    w = WL.random_problem(m, n, seed=m * 11 + n, bits=4)
    UA32, UB32 = shared_factors(w.A, w.damp_A, w.B, w.damp_B)
    s, z, qmin, qmax = gpu_grid(w.W, 4, True, group)
    _, s_ref, z_ref = oracle_grid_of(w.W, 4, True, group)
    np.testing.assert_array_equal(s, s_ref)
    np.testing.assert_array_equal(z, z_ref)
    dW, dUA, dUB, ds, dz = to_dev(w.W, UA32, UB32, s, z)
    V, c, pre = kb.bakron_quantize_grid(dW, dUA, None if one_sided else dUB, ds, dz, group, qmin, qmax,
                                        want_preround=True)
    grid = as_grid(s, z, qmin, qmax, group, n)
    check_grid_parity(w.W, UA32, None if one_sided else UB32, grid, V.cpu().numpy(),
                      c.cpu().numpy().astype(np.float64), pre.cpu().numpy(), one_sided=one_sided)
