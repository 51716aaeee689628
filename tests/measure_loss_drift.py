"""Drift of the proxy loss between two valid GPTQ trajectories, measured with
the oracle alone (no GPU): the row-accumulator oracle on W and on W with a
small relative perturbation, which moves decisions inside the near-tie window;
both losses are taken against the original W.  This is the basis of the
full-size loss bound in test_gpu_fullsize_oracle.py.

    python tests/measure_loss_drift.py mlp14336x4096

(the four full-size workloads take minutes each on 8 to 16 cores).
"""
import os
import sys
import time

import numpy as np

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import oracle as O  # noqa: E402
from kronecker_factored_gptq_gb300 import workloads as WL  # noqa: E402


def main(name, seed=0, eps_list=(1e-7, 1e-6)):
    w = WL.load(name, seed=seed)
    t = time.time()
    _, UA = O.prepare(w.A, w.damp_A)
    _, UB = O.prepare(w.B, w.damp_B)
    # the factors both sides of the GPU test use: fp64 rounded once to fp32
    UA = UA.astype(np.float32).astype(np.float64)
    UB = UB.astype(np.float32).astype(np.float64)
    LA, LB = O.lower_from_update(UA), O.lower_from_update(UB)
    s = O.row_scale(w.W, w.qmax)

    def loss(codes):
        V = (s[:, None] * codes.astype(np.float32)).astype(np.float32)
        return O.proxy_loss(w.W, V, LA, LB)

    r0 = O.rowacc(w.W, UA, UB, s, w.qmin, w.qmax, rows_per_block=8)
    l0 = loss(r0.codes)
    print("%s: loss %.6f (%.0f s)" % (name, l0, time.time() - t), flush=True)
    rng = np.random.default_rng(1)
    for eps in eps_list:
        Wp = (w.W.astype(np.float64) * (1 + eps * rng.standard_normal(w.W.shape))).astype(np.float32)
        r1 = O.rowacc(Wp, UA, UB, s, w.qmin, w.qmax, rows_per_block=8)
        l1 = loss(r1.codes)
        print("  eps %g: %.1f%% of codes differ, loss %.6f, relative drift %.2e (%.0f s)"
              % (eps, 100.0 * np.count_nonzero(r1.codes != r0.codes) / r0.codes.size, l1,
                 (l1 - l0) / l0, time.time() - t), flush=True)


if __name__ == "__main__":
    main(sys.argv[1] if len(sys.argv) > 1 else "mlp14336x4096")
