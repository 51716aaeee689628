"""Shared helpers of the GPU parity tests (CUDA path through the C ABI vs
the fp64 oracle).

Solve parity uses SHARED factors: the oracle prepares U_A, U_B in fp64, they
are rounded to fp32 once, and that fp32 pair feeds both the CUDA solver and
the oracle (upcast).  The factor preparation on the GPU is checked separately
(residuals and distance to the oracle's factors).

The comparison rule: codes may differ from the oracle only where the oracle's
pre-rounding value lies within 1e-4 grid units of a rounding boundary, for at
most 0.1% of the entries; the proxy loss ||L(B)(V-W)L(A)^T||_F^2 must agree to
1e-3 relative.  Because one flipped near-tie decision changes every entry to
its bottom-right, the oracle is re-run GUIDED by the GPU codes (at its own
near ties it takes the GPU's decision) and must then reproduce the GPU codes
exactly; the count of guided decisions is the number of near-tie
disagreements.  The certificate (teacher-forced replay) is checked as well.
"""

import numpy as np

import oracle as O

TOL = 1e-4          # grid units, near-tie window
MAX_FRAC = 1e-3     # at most 0.1% of entries may differ
LOSS_RTOL = 1e-3


def shared_factors(A, damp_A, B, damp_B):
    LA, UA = O.prepare(A, damp_A)
    LB, UB = O.prepare(B, damp_B)
    UA32 = UA.astype(np.float32)
    UB32 = UB.astype(np.float32)
    return UA32, UB32


def to_dev(*arrs):
    import torch
    return [torch.from_numpy(np.ascontiguousarray(a)).to("cuda") for a in arrs]


def gpu_quantize(W, UA32, UB32, s32, qmin, qmax, use_3xtf32, preround=True):
    from kronecker_factored_gptq_gb300 import bakron as kb
    dW, dUA, dUB, ds = to_dev(W, UA32, UB32, s32)
    opts = kb.default_opts(use_3xtf32=use_3xtf32)
    V, c, p = kb.bakron_quantize(dW, dUA, dUB, ds, qmin, qmax, want_preround=preround, opts=opts)
    return (V.cpu().numpy(), c.cpu().numpy().astype(np.float64),
            None if p is None else p.cpu().numpy())


def oracle_grid(qmin, qmax):
    from kronecker_factored_gptq_gb300 import bakron as kb
    return (None if qmin == kb.INT32_MIN else qmin, None if qmax == kb.INT32_MAX else qmax)


def check_parity(W, UA32, UB32, s32, qmin, qmax, V, codes, pre=None, variant="antidiag"):
    """Full parity check of a GPU result against the oracle (sizes where the
    oracle runs).  Returns a dict of the measured quantities."""
    UA = UA32.astype(np.float64)
    UB = UB32.astype(np.float64)
    oq = oracle_grid(qmin, qmax)
    m, n = W.shape
    solve = {"antidiag": O.antidiag, "bakron": O.bakron}[variant]
    ref = solve(W, UA, UB, s32, *oq)
    guided = solve(W, UA, UB, s32, *oq, guide=codes, guide_tol=TOL)
    diff = int(np.count_nonzero(guided.codes != codes))
    assert diff == 0, "GPU codes differ from the guided oracle at %d entries (not near ties)" % diff
    assert guided.overrides <= MAX_FRAC * m * n, "too many near-tie disagreements: %d" % guided.overrides
    np.testing.assert_array_equal(V, (s32[:, None] * codes.astype(np.float32)).astype(np.float32))
    cert = O.certificate(W, V, codes, UA, UB, s32, *oq, tol=TOL, max_frac=MAX_FRAC)
    assert cert["ok"], "certificate: %d mismatches, %d not near ties" % (cert["mismatch"], cert["bad"])
    LA = O.lower_from_update(UA)
    LB = O.lower_from_update(UB)
    l_gpu = O.proxy_loss(W, V, LA, LB)
    # V is an fp32 output on both sides: s_i * code rounded once to fp32
    V_ref = (s32[:, None] * ref.codes.astype(np.float32)).astype(np.float32)
    l_ref = O.proxy_loss(W, V_ref, LA, LB)
    assert abs(l_gpu - l_ref) <= LOSS_RTOL * abs(l_ref) + 1e-30, (l_gpu, l_ref)
    out = {"overrides": guided.overrides, "loss_gpu": l_gpu, "loss_ref": l_ref,
           "cert_mismatch": cert["mismatch"]}
    if pre is not None:
        err = np.max(np.abs(pre - guided.preround) / s32[:, None])
        out["preround_err_grid_units"] = float(err)
        assert err < TOL, "pre-rounding values off by %.3g grid units" % err
    return out


def corner_check(W, UA32, UB32, s32, qmin, qmax, codes, a, b, variant="antidiag"):
    """Exact oracle on the top-left a x b corner: its GPTQ output depends only
    on W[:a, :b] and the leading blocks of the factors (updates only move to
    the bottom-right), so it must match the full-size GPU result there."""
    oq = oracle_grid(qmin, qmax)
    Wc = W[:a, :b]
    UA = UA32[:b, :b].astype(np.float64)
    UB = UB32[:a, :a].astype(np.float64)
    solve = {"antidiag": O.antidiag, "bakron": O.bakron}[variant]
    g = solve(Wc, UA, UB, s32[:a], *oq, guide=codes[:a, :b], guide_tol=TOL)
    diff = int(np.count_nonzero(g.codes != codes[:a, :b]))
    assert diff == 0, "corner %dx%d: %d codes differ from the guided oracle" % (a, b, diff)
    assert g.overrides <= MAX_FRAC * a * b
    return g.overrides
