"""GPU parity of batched solves (bakron_quantize_batch): several problems of
different shapes, grids and factor kinds (two-sided and B = I) run
concurrently on their own stream sets; each must pass the same oracle parity
check as a single call (guided oracle, exact codes after that, V = s (c - z),
the certificate, proxy loss), and a failing problem reports its own status.
"""

import numpy as np
import pytest

import oracle as O
from kronecker_factored_gptq_gb300 import workloads as WL

from _gpu_helpers import TOL, MAX_FRAC, check_parity, shared_factors, to_dev

pytestmark = pytest.mark.gpu


def _problem(m, n, seed, one_sided=False, grid=None):
    w = WL.random_problem(m, n, seed=seed, bits=4)
    UA32, UB32 = shared_factors(w.A, w.damp_A, w.B, w.damp_B)
    if grid is None:
        s = O.row_scale(w.W, w.qmax)
        z, group, qmin, qmax = None, None, w.qmin, w.qmax
        og = None
    else:
        bits, group = grid
        og, s, z = O.asymmetric_grid(w.W, bits, group)
        qmin, qmax = og.qmin, og.qmax
    return dict(w=w, UA32=UA32, UB32=None if one_sided else UB32, s=s, z=z, group=group,
                qmin=qmin, qmax=qmax, grid=og)


def test_batch_mixed_problems():
    from kronecker_factored_gptq_gb300 import bakron as kb
    probs = [_problem(200, 328, 1), _problem(129, 384, 2, one_sided=True),
             _problem(300, 260, 3, grid=(3, 32)), _problem(64, 64, 4),
             _problem(257, 150, 5, one_sided=True, grid=(4, 64))]
    reqs = []
    for p in probs:
        dW, dUA, ds = to_dev(p["w"].W, p["UA32"], p["s"])
        req = dict(W=dW, UA=dUA, scale=ds, group=p["group"], qmin=p["qmin"], qmax=p["qmax"])
        if p["UB32"] is not None:
            req["UB"] = to_dev(p["UB32"])[0]
        if p["z"] is not None:
            req["zero"] = to_dev(p["z"])[0]
        reqs.append(req)
    outs = kb.bakron_quantize_batch(reqs)
    for p, (V, C) in zip(probs, outs):
        w = p["w"]
        V = V.cpu().numpy()
        c = C.cpu().numpy().astype(np.float64)
        UB = p["UB32"] if p["UB32"] is not None else np.eye(w.m, dtype=np.float32)
        s = p["grid"] if p["grid"] is not None else p["s"]
        if p["grid"] is None:
            check_parity(w.W, p["UA32"], UB, p["s"], p["qmin"], p["qmax"], V, c)
        else:
            g = O.antidiag(w.W, p["UA32"].astype(np.float64), UB.astype(np.float64), p["grid"],
                           guide=c, guide_tol=TOL)
            assert np.count_nonzero(g.codes != c) == 0 and g.overrides <= MAX_FRAC * c.size
            np.testing.assert_array_equal(
                V, (p["grid"].S.astype(np.float32) * (c.astype(np.float32) -
                                                      p["grid"].Z.astype(np.float32))))


def test_batch_reports_each_status():
    from kronecker_factored_gptq_gb300 import bakron as kb
    good, bad = _problem(130, 140, 6), _problem(130, 140, 7)
    reqs = []
    for k, p in enumerate((good, bad)):
        W = p["w"].W.copy()
        if k == 1:
            W[70, 90] = np.nan
        dW, dUA, dUB, ds = to_dev(W, p["UA32"], p["UB32"], p["s"])
        reqs.append(dict(W=dW, UA=dUA, UB=dUB, scale=ds, qmin=p["qmin"], qmax=p["qmax"]))
    with pytest.raises(kb.BakronError) as ei:
        kb.bakron_quantize_batch(reqs)
    assert ei.value.status == 3 and ei.value.statuses == [0, 3]


def test_batch_more_problems_than_stream_sets():
    """Eleven problems on eight stream sets (three queue behind others)."""
    from kronecker_factored_gptq_gb300 import bakron as kb
    probs = [_problem(70 + 13 * i, 90 + 7 * i, 100 + i, one_sided=(i % 3 == 2)) for i in range(11)]
    reqs = []
    for p in probs:
        dW, dUA, ds = to_dev(p["w"].W, p["UA32"], p["s"])
        req = dict(W=dW, UA=dUA, scale=ds, qmin=p["qmin"], qmax=p["qmax"])
        if p["UB32"] is not None:
            req["UB"] = to_dev(p["UB32"])[0]
        reqs.append(req)
    outs = kb.bakron_quantize_batch(reqs)
    for p, (V, C) in zip(probs, outs):
        w = p["w"]
        UB = p["UB32"] if p["UB32"] is not None else np.eye(w.m, dtype=np.float32)
        check_parity(w.W, p["UA32"], UB, p["s"], p["qmin"], p["qmax"], V.cpu().numpy(),
                     C.cpu().numpy().astype(np.float64))
