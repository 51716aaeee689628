"""Plain fp64 CPU oracle for the BaKron solver (Kronecker-factored GPTQ).

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or
execute anything in this package: only ``tests/``, ``__graft_entry__.smoke()``
and ``bench.py`` (its ``cpu_baseline`` leg and its ``--impl reference`` arm)
use it.  It shares no code with the CUDA library and imports nothing from it.

What it computes, and where each piece comes from (the sources are the web
pages about "BaKron: Efficient Quantization with Kronecker-Factored Hessians",
Birnick & Saab):

* ``factors``   - damping, RevCholesky ``A = L^T L`` (L lower) and the update
  factor ``U = L^{-T}`` (summary page "FastKron: Efficient Quantization with
  Kronecker-Factored Hessians", Corollary 3.4 names ``L(A) = RevCholesky(A)``).
* ``quantizer`` - the base quantizers (per-row or per-column-group,
  symmetric or asymmetric b-bit grids) and the near-tie rule used by every
  comparison (abstract: BaKron is modular in the base quantizer).
* ``solvers``   - GPTQ on vec(W) with Hessian A (x) B written out four ways, in
  the order the summary page derives them (section 3): naive (explicit
  mn x mn Hessian), anti-diagonal, recursive (divide and conquer over the
  vec order) and BaKron (anti-diagonal parallelism + divide and conquer over
  the anti-diagonal dimension); plus textbook one-sided GPTQ (Hessian A (x) I).
  Theorem 3.2 on the summary page states the four give the same output.
* ``rowacc``    - the same GPTQ output in the row-accumulator form (every
  entry pushes its error along its row through U_A and the finished row
  accumulator down its column through U_B), written in plain C
  (``rowacc.c``, compiled by ``build_c.py``): m n (m + n) flops, so whole
  solves at the full workload sizes can be compared.
* ``hessians``  - K-FAC and one-step Shampoo Kronecker factors of a layer
  Hessian from activation and gradient samples (summary page, section on the
  Hessians).
* ``checks``    - the output certificate, the proxy loss
  ||L(B)(V-W)L(A)^T||_F^2 and the Corollary 3.4 bound 1/4 tr(A) tr(B).

Everything is fp64 except the rounding decision, which is taken in fp32
(the pages' kernel computes in float32), see ``quantizer.quantize_codes``.

Parity status: every function here is pinned by a ``-m "not gpu"`` test in
``tests/test_oracle_pins.py`` against something other than itself (closed
forms, brute force, special cases that reduce to textbook routines, the
Corollary 3.4 inequality, cross-formulation equality).
"""

from .factors import damp, rev_cholesky, update_factor, prepare, lower_from_update
from .quantizer import (row_scale, quantize_codes, near_tie, Grid, symmetric_grid,
                        asymmetric_grid)
from .solvers import (SolveResult, gptq_rows, naive_vec_gptq, antidiag,
                      recursive_vec, bakron, bakron_tiled_order_check)
from .checks import (certificate, proxy_loss, cor34_bound, cor34_tight_bound,
                     compare_codes)
from .hessians import kfac_factors, shampoo_factors
from .rowacc import rowacc

__all__ = [
    "damp", "rev_cholesky", "update_factor", "prepare", "lower_from_update",
    "row_scale", "quantize_codes", "near_tie", "Grid", "symmetric_grid", "asymmetric_grid",
    "gptq_rows", "naive_vec_gptq", "antidiag", "recursive_vec", "bakron",
    "bakron_tiled_order_check",
    "certificate", "proxy_loss", "cor34_bound", "cor34_tight_bound",
    "compare_codes", "SolveResult", "kfac_factors", "shampoo_factors", "rowacc",
]
