"""Writes the stored oracle outputs under tests/golden/ (run from the repo
root: python tests/golden/make_golden.py).

Only the fp64 oracle (oracle/) and the seeded input generators
(kronecker_factored_gptq_gb300/workloads.py, which hold none of the method's
arithmetic) are called; nothing here touches the CUDA path.  The fixtures pin
the oracle against unintended change: tests/test_golden.py recomputes them.

Cases (summary page "FastKron: Efficient Quantization with Kronecker-Factored
Hessians", problem set-up and section 3: GPTQ on vec(W) with the Hessian
A (x) B, which every BaKron variant reproduces by its Theorem 3.2):
  tiny64   the 64 x 64 workload, seed 0, 4-bit per-row symmetric grid;
  unit6x5  a 6 x 5 problem on the unclamped unit grid (scale 1), W scaled by 100;
  asym7x9  a 7 x 9 problem with a 3-bit asymmetric grid in column groups of 4
           (the last group short), solved by the anti-diagonal oracle.
"""

import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import oracle as O  # noqa: E402
from kronecker_factored_gptq_gb300 import workloads as WL  # noqa: E402


def cases():
    """name -> dict of arrays, recomputed identically by the test."""
    out = {}
    w = WL.tiny64(seed=0)
    _, UA = O.prepare(w.A.astype(np.float64), w.damp_A)
    _, UB = O.prepare(w.B.astype(np.float64), w.damp_B)
    s = O.row_scale(w.W, w.qmax)
    r = O.bakron(w.W, UA, UB, s, w.qmin, w.qmax)
    LA, LB = O.lower_from_update(UA), O.lower_from_update(UB)
    V = s[:, None].astype(np.float64) * r.codes
    out["tiny64"] = {"codes": r.codes, "scale": s,
                     "proxy_loss": np.array([O.proxy_loss(w.W, V, LA, LB)])}

    p = WL.random_problem(6, 5, seed=11)
    _, UA = O.prepare(p.A.astype(np.float64), p.damp_A)
    _, UB = O.prepare(p.B.astype(np.float64), p.damp_B)
    W100 = 100.0 * p.W.astype(np.float64)
    r = O.bakron(W100, UA, UB, np.ones(6))
    out["unit6x5"] = {"codes": r.codes, "preround": r.preround}

    q = WL.random_problem(7, 9, seed=12, bits=3)
    _, UA = O.prepare(q.A.astype(np.float64), q.damp_A)
    _, UB = O.prepare(q.B.astype(np.float64), q.damp_B)
    grid, S, Z = O.asymmetric_grid(q.W, 3, 4)
    r = O.antidiag(q.W, UA, UB, grid)
    out["asym7x9"] = {"codes": r.codes, "S": S, "Z": Z}
    return out


def write(path, arrays, header):
    with open(path, "w") as f:
        for line in header:
            f.write("# " + line + "\n")
        for k, a in arrays.items():
            a = np.asarray(a)
            f.write("%s %s %s\n" % (k, "x".join(str(d) for d in a.shape), " ".join(repr(float(x)) for x in a.ravel())))


def read(path):
    arrays = {}
    with open(path) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            k, shape, *vals = line.split()
            dims = tuple(int(d) for d in shape.split("x")) if shape else ()
            arrays[k] = np.array([float(v) for v in vals], dtype=np.float64).reshape(dims)
    return arrays


if __name__ == "__main__":
    for name, arrays in cases().items():
        write(os.path.join(HERE, name + ".txt"), arrays,
              ["written by tests/golden/make_golden.py from the fp64 oracle (oracle/)",
               "problem: GPTQ on vec(W) with Hessian A (x) B (summary page 'FastKron: Efficient Quantization",
               "with Kronecker-Factored Hessians', problem set-up, section 3 and Theorem 3.2)",
               "case %s; see make_golden.py for the inputs" % name])
        print("wrote", name)
