"""Pins of the fp64 oracle against things other than itself.

Each test ties an oracle function to a closed form, a brute-force
formulation, a textbook special case or an inequality fixed by the pages
("BaKron: Efficient Quantization with Kronecker-Factored Hessians": the summary
page's section 3, Proposition 3.1, Theorem 3.2, Corollary 3.4, and the ainews
article's statement that one-sided GPTQ is the Hessian A (x) I).  The cases
are chosen so that a dropped term, a wrong sign, a transposed factor or a
swapped A/B role fails at least one of them.
"""

import numpy as np
import pytest

import oracle as O


def spd(k, rng, over=3, shift=0.0):
    X = rng.standard_normal((k, over * k + 1))
    return X @ X.T / X.shape[1] + shift * np.eye(k)


def problem(m, n, seed, bits=4):
    rng = np.random.default_rng(seed)
    W = 0.02 * rng.standard_normal((m, n))
    A = O.damp(spd(n, rng), 0.01)
    B = O.damp(spd(m, rng), 0.01)
    LA, UA = O.prepare(A, 0.0)
    LB, UB = O.prepare(B, 0.0)
    qmax = (1 << (bits - 1)) - 1
    s = O.row_scale(W, qmax)
    return dict(W=W, A=A, B=B, LA=LA, UA=UA, LB=LB, UB=UB, s=s,
                qmin=-(qmax + 1), qmax=qmax)


# ---------------------------------------------------------------- factors

def test_rev_cholesky_2x2_closed_form():
    a, b, c = 4.0, 1.2, 2.5
    L = O.rev_cholesky(np.array([[a, b], [b, c]]))
    want = np.array([[np.sqrt(a - b * b / c), 0.0], [b / np.sqrt(c), np.sqrt(c)]])
    np.testing.assert_allclose(L, want, rtol=1e-14, atol=1e-14)


def test_rev_cholesky_reconstructs_and_is_lower():
    rng = np.random.default_rng(1)
    for k in (1, 2, 5, 17):
        A = spd(k, rng)
        L = O.rev_cholesky(A)
        assert np.allclose(np.triu(L, 1), 0.0)
        assert np.all(np.diag(L) > 0)
        np.testing.assert_allclose(L.T @ L, A, rtol=1e-12, atol=1e-12)


def test_update_factor_is_upper_cholesky_of_inverse():
    # U = L^{-T} must equal the upper Cholesky factor of A^{-1}, computed here
    # by a different route (explicit inverse, then numpy's lower Cholesky).
    rng = np.random.default_rng(2)
    for k in (1, 3, 9, 24):
        A = spd(k, rng)
        L, U = O.prepare(A, 0.0)
        U2 = np.linalg.cholesky(np.linalg.inv(A)).T
        np.testing.assert_allclose(U, U2, rtol=1e-9, atol=1e-12)
        np.testing.assert_allclose(np.diag(U), 1.0 / np.diag(L), rtol=1e-13)
        np.testing.assert_allclose(O.lower_from_update(U), L, rtol=1e-10, atol=1e-12)


def test_damp_closed_form():
    A = np.diag([1.0, 2.0, 3.0, 6.0])
    Ad = O.damp(A, 0.5)
    np.testing.assert_array_equal(np.diag(Ad), np.array([1, 2, 3, 6]) + 0.5 * 3.0)
    assert O.damp(A, 0.0) is not A


def test_rev_cholesky_rejects_indefinite():
    with pytest.raises(np.linalg.LinAlgError):
        O.rev_cholesky(np.array([[1.0, 2.0], [2.0, 1.0]]))


# -------------------------------------------------------------- quantizer

def test_row_scale_values():
    W = np.array([[0.5, -1.75, 0.0], [0.0, 0.0, 0.0], [3.0, 1.0, -3.5]], np.float32)
    s = O.row_scale(W, 7)
    assert s.dtype == np.float32
    np.testing.assert_array_equal(s, np.array([np.float32(1.75) / np.float32(7), 1.0,
                                               np.float32(3.5) / np.float32(7)], np.float32))


def test_quantize_half_even_and_clamp():
    x = np.array([0.5, 1.5, 2.5, -0.5, -2.5, 7.6, -9.0, 3.49])
    c = O.quantize_codes(x, np.ones_like(x), -8, 7)
    np.testing.assert_array_equal(c, [0, 2, 2, -0, -2, 7, -8, 3])
    cu = O.quantize_codes(x, np.ones_like(x))
    np.testing.assert_array_equal(cu, [0, 2, 2, 0, -2, 8, -9, 3])


def test_near_tie_rule():
    s = np.ones(5)
    x = np.array([0.50005, 0.5002, 7.5, -8.49995, 2.49999])
    nt = O.near_tie(x, s, -8, 7, 1e-4)
    # 7.5 separates 7 and 8 (8 is clamped away): not a decision boundary;
    # -8.5 separates -9 and -8 (-9 clamped away): not one either.
    np.testing.assert_array_equal(nt, [True, False, False, False, True])
    assert O.near_tie(np.array([7.5]), np.ones(1), None, None, 1e-4)[0]


# ------------------------------------------------------ brute-force pins

def obs_bruteforce(W, H, s, qmin, qmax, order):
    """Sequential optimal-brain-surgeon rounding, by explicit least squares.

    After rounding entry k, the still-free entries R move by the minimiser of
    the quadratic loss with entry k fixed: delta_R = H_RR^{-1} H_Rk (w_k - q_k).
    No Cholesky factor and no Kronecker structure are used.
    """
    m, n = W.shape
    x = W.reshape(-1, order="F").astype(np.float64).copy()
    free = np.ones(m * n, dtype=bool)
    codes = np.zeros(m * n)
    for k in order:
        i = k % m
        c = O.quantize_codes(x[k:k + 1], s[i:i + 1], qmin, qmax)[0]
        codes[k] = c
        free[k] = False
        R = np.nonzero(free)[0]
        if len(R):
            delta = np.linalg.solve(H[np.ix_(R, R)], H[R, k]) * (x[k] - s[i] * c)
            x[R] += delta
    return codes.reshape((m, n), order="F")


@pytest.mark.parametrize("m,n,seed", [(2, 3, 0), (3, 2, 1), (4, 4, 2), (1, 6, 3), (5, 1, 4)])
def test_naive_equals_obs_bruteforce(m, n, seed):
    p = problem(m, n, seed)
    H = np.kron(p["A"], p["B"])
    want = obs_bruteforce(p["W"], H, p["s"], p["qmin"], p["qmax"], range(m * n))
    got = O.naive_vec_gptq(p["W"], p["s"], p["qmin"], p["qmax"], A=p["A"], B=p["B"])
    np.testing.assert_array_equal(got.codes, want)


def test_1x2_closed_form_compensation():
    # GPTQ on two weights: after rounding w0, w1 moves by (w0 - q0) H01 / H11.
    A = np.array([[2.0, 0.7], [0.7, 1.3]])
    B = np.array([[1.0]])
    W = np.array([[0.26, 0.1]])
    s = np.array([0.1], np.float32)
    r = O.naive_vec_gptq(W, s, A=A, B=B)
    q0 = np.float64(s[0]) * np.rint(np.float32(0.26) / s[0])
    np.testing.assert_allclose(r.preround[0, 1], 0.1 + (0.26 - q0) * 0.7 / 1.3, rtol=1e-12)


def test_prop31_vec_identity():
    # (A (x) B) vec(X) = vec(B X A^T) with column-major vec: fixes the index map
    rng = np.random.default_rng(5)
    A = rng.standard_normal((4, 4)); B = rng.standard_normal((3, 3)); X = rng.standard_normal((3, 4))
    np.testing.assert_allclose(np.kron(A, B) @ X.reshape(-1, order="F"),
                               (B @ X @ A.T).reshape(-1, order="F"), rtol=1e-12)


# ------------------------------------------- Theorem 3.2: all variants agree

SHAPES = [(2, 3), (3, 2), (5, 7), (7, 5), (1, 9), (9, 1), (8, 8), (6, 13), (16, 12)]


@pytest.mark.parametrize("m,n", SHAPES)
def test_theorem32_variants_identical(m, n):
    p = problem(m, n, seed=m * 100 + n)
    args = (p["W"], p["UA"], p["UB"], p["s"], p["qmin"], p["qmax"])
    ref = O.naive_vec_gptq(p["W"], p["s"], p["qmin"], p["qmax"], A=p["A"], B=p["B"])
    ref_f = O.naive_vec_gptq(p["W"], p["s"], p["qmin"], p["qmax"], UA=p["UA"], UB=p["UB"])
    outs = [ref_f, O.antidiag(*args), O.recursive_vec(*args), O.bakron(*args),
            O.bakron(*args, leaf_width=3), O.bakron(*args, leaf_width=4),
            O.bakron_tiled_order_check(*args, tile=2), O.bakron_tiled_order_check(*args, tile=3)]
    for r in outs:
        np.testing.assert_array_equal(r.codes, ref.codes)
        np.testing.assert_allclose(r.preround, ref.preround, rtol=0, atol=1e-12)
        np.testing.assert_allclose(r.E, ref.E, rtol=0, atol=1e-10)


def test_theorem32_at_64x64():
    p = problem(64, 64, seed=7)
    args = (p["W"], p["UA"], p["UB"], p["s"], p["qmin"], p["qmax"])
    ref = O.naive_vec_gptq(p["W"], p["s"], p["qmin"], p["qmax"], A=p["A"], B=p["B"])
    for r in (O.antidiag(*args), O.bakron(*args), O.bakron(*args, leaf_width=16)):
        np.testing.assert_array_equal(r.codes, ref.codes)
        np.testing.assert_allclose(r.preround, ref.preround, atol=1e-11)


# ------------------------------------------------------- special cases

@pytest.mark.parametrize("m,n", [(4, 9), (7, 7), (12, 5)])
def test_b_identity_is_rowwise_gptq(m, n):
    p = problem(m, n, seed=11)
    I = np.eye(m)
    two = O.antidiag(p["W"], p["UA"], I, p["s"], p["qmin"], p["qmax"])
    one = O.gptq_rows(p["W"], p["UA"], p["s"], p["qmin"], p["qmax"])
    np.testing.assert_array_equal(two.codes, one.codes)
    np.testing.assert_allclose(two.preround, one.preround, atol=1e-14)
    full = O.bakron(p["W"], p["UA"], I, p["s"], p["qmin"], p["qmax"])
    np.testing.assert_array_equal(full.codes, one.codes)


def test_gptq_rows_guided_by_its_own_codes_is_unchanged():
    # the guide only decides near ties, and agrees with the decision there
    p = problem(9, 13, seed=12)
    one = O.gptq_rows(p["W"], p["UA"], p["s"], p["qmin"], p["qmax"])
    g = O.gptq_rows(p["W"], p["UA"], p["s"], p["qmin"], p["qmax"], guide=one.codes)
    np.testing.assert_array_equal(g.codes, one.codes)
    np.testing.assert_array_equal(g.preround, one.preround)
    assert g.overrides == 0


def test_gptq_rows_guide_takes_a_near_tie():
    # one entry placed exactly on a rounding boundary (x / s = k + 1/2 in
    # column 0, which no update reaches): round half to even takes one side,
    # a guide with the other code is followed there, and the changed error
    # then moves every later entry of that row only
    p = problem(4, 6, seed=13)
    W = p["W"].copy()
    s = p["s"]
    W[2, 0] = 0.5 * s[2]
    one = O.gptq_rows(W, p["UA"], s, p["qmin"], p["qmax"])
    assert one.codes[2, 0] == 0.0
    guide = one.codes.copy()
    guide[2, 0] = 1.0
    g = O.gptq_rows(W, p["UA"], s, p["qmin"], p["qmax"], guide=guide)
    assert g.codes[2, 0] == 1.0 and g.overrides >= 1
    np.testing.assert_array_equal(np.delete(g.codes, 2, axis=0), np.delete(one.codes, 2, axis=0))
    assert not np.allclose(g.preround[2, 1:], one.preround[2, 1:])


def test_diagonal_factors_give_rtn():
    rng = np.random.default_rng(3)
    m, n = 9, 11
    W = 0.02 * rng.standard_normal((m, n))
    UA = np.diag(rng.uniform(0.5, 2.0, n))
    UB = np.diag(rng.uniform(0.5, 2.0, m))
    s = O.row_scale(W, 3)
    r = O.bakron(W, UA, UB, s, -4, 3)
    np.testing.assert_array_equal(r.codes, O.quantize_codes(W, s[:, None], -4, 3))


def test_single_row_and_column_are_vector_gptq():
    rng = np.random.default_rng(4)
    # m = 1: GPTQ on the row with Hessian A (any B scalar)
    p = problem(1, 10, seed=4)
    r = O.bakron(p["W"], p["UA"], 3.0 * np.eye(1), p["s"], p["qmin"], p["qmax"])
    g = O.gptq_rows(p["W"], p["UA"], p["s"], p["qmin"], p["qmax"])
    np.testing.assert_array_equal(r.codes, g.codes)
    # n = 1 with unit-step unclamped grid: GPTQ down the column with Hessian B
    q = problem(10, 1, seed=5)
    ones = np.ones(10)
    r = O.bakron(q["W"] * 50, 2.0 * np.eye(1), q["UB"], ones)
    g = O.gptq_rows((q["W"] * 50).T, q["UB"], np.ones(1))
    np.testing.assert_array_equal(r.codes, g.codes.T)


def test_transpose_symmetry_unit_grid():
    # With a unit-step grid the problem (W, A, B) and (W^T, B, A) are the same
    # quadratic; by Theorem 3.2 the order does not matter, so V^T must match.
    p = problem(6, 9, seed=6)
    Wb = p["W"] * 80
    r1 = O.bakron(Wb, p["UA"], p["UB"], np.ones(6))
    r2 = O.bakron(Wb.T, p["UB"], p["UA"], np.ones(9))
    np.testing.assert_array_equal(r1.codes, r2.codes.T)


def test_scale_invariance():
    p = problem(7, 6, seed=8)
    r1 = O.bakron(p["W"], p["UA"], p["UB"], p["s"], p["qmin"], p["qmax"])
    _, UA2 = O.prepare(3.7 * p["A"], 0.0)
    _, UB2 = O.prepare(0.21 * p["B"], 0.0)
    r2 = O.bakron(p["W"], UA2, UB2, p["s"], p["qmin"], p["qmax"])
    np.testing.assert_array_equal(r1.codes, r2.codes)


# ------------------------------------------- certificate, loss, Cor 3.4

def test_certificate_accepts_and_replays():
    p = problem(12, 10, seed=9)
    r = O.bakron(p["W"], p["UA"], p["UB"], p["s"], p["qmin"], p["qmax"])
    c = O.certificate(p["W"], r.V, r.codes, p["UA"], p["UB"], p["s"], p["qmin"], p["qmax"])
    assert c["ok"] and c["mismatch"] == 0
    np.testing.assert_allclose(c["wt"], r.preround, atol=1e-12)


def test_certificate_rejects_perturbed_code():
    p = problem(12, 10, seed=10)
    r = O.bakron(p["W"], p["UA"], p["UB"], p["s"], p["qmin"], p["qmax"])
    codes = r.codes.copy()
    i, j = 5, 4
    codes[i, j] = codes[i, j] + (1 if codes[i, j] < p["qmax"] else -1)
    V = p["s"][:, None].astype(np.float64) * codes
    c = O.certificate(p["W"], V, codes, p["UA"], p["UB"], p["s"], p["qmin"], p["qmax"])
    assert not c["ok"] and c["bad"] >= 1


def test_proxy_loss_three_ways():
    p = problem(5, 8, seed=12)
    r = O.bakron(p["W"], p["UA"], p["UB"], p["s"], p["qmin"], p["qmax"])
    D = r.V - p["W"]
    l1 = O.proxy_loss(p["W"], r.V, p["LA"], p["LB"])
    l2 = np.trace(D.T @ p["B"] @ D @ p["A"])
    d = D.reshape(-1, order="F")
    l3 = d @ np.kron(p["A"], p["B"]) @ d
    np.testing.assert_allclose([l1, l1], [l2, l3], rtol=1e-10)
    np.testing.assert_allclose(l1, np.sum(r.E ** 2), rtol=1e-9)


@pytest.mark.parametrize("m,n,seed", [(8, 8, 0), (6, 11, 1), (16, 9, 2), (64, 64, 3)])
def test_corollary34_bound_unclamped(m, n, seed):
    p = problem(m, n, seed)
    Wb = 10 * p["W"]
    r = O.bakron(Wb, p["UA"], p["UB"], np.ones(m))
    loss = O.proxy_loss(Wb, r.V, p["LA"], p["LB"])
    tight = O.cor34_tight_bound(p["LA"], p["LB"])
    assert loss <= tight <= O.cor34_bound(p["A"], p["B"]) * (1 + 1e-12)


def test_compare_codes_rule():
    codes = np.zeros((2, 3))
    pre = np.array([[0.49999, 0.2, 1.1], [0.0, -0.50002, 0.3]])
    s = np.ones(2)
    other = codes.copy(); other[0, 0] = 1; other[1, 1] = -1
    r = O.compare_codes(other, codes, pre, s, -8, 7, 1e-4, max_frac=0.5)
    assert r["ok"] and r["diff"] == 2 and r["bad"] == 0
    other[0, 1] = 1
    assert not O.compare_codes(other, codes, pre, s, -8, 7, 1e-4, max_frac=0.5)["ok"]


def test_guide_only_acts_on_near_ties():
    p = problem(6, 7, seed=13)
    args = (p["W"], p["UA"], p["UB"], p["s"], p["qmin"], p["qmax"])
    r = O.antidiag(*args)
    g = O.antidiag(*args, guide=r.codes)
    assert g.overrides == 0
    np.testing.assert_array_equal(g.codes, r.codes)
    # a guide that disagrees everywhere changes nothing away from near ties
    g2 = O.antidiag(*args, guide=r.codes + 1, guide_tol=1e-9)
    np.testing.assert_array_equal(g2.codes, r.codes)


# ------------------------------------------------- Hessian factor accumulation

def _fisher_terms(X, G):
    """Per-sample Hessians vec(g a^T) vec(g a^T)^T with the column-major vec
    (entry (i, j) of the m x n gradient at index i + m j), written out."""
    N, n = X.shape
    m = G.shape[1]
    F = np.zeros((N, m * n, m * n))
    for t in range(N):
        v = np.outer(G[t], X[t]).reshape(-1, order="F")
        F[t] = np.outer(v, v)
    return F


def test_kfac_factors_brute_force_and_single_sample_kronecker():
    rng = np.random.default_rng(30)
    X = rng.standard_normal((7, 4))
    G = rng.standard_normal((7, 3))
    A, B = O.kfac_factors(X, G)
    A_bf = sum(np.outer(x, x) for x in X) / 7
    B_bf = sum(np.outer(g, g) for g in G) / 7
    np.testing.assert_allclose(A, A_bf, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(B, B_bf, rtol=1e-13, atol=1e-14)
    # one sample: the Kronecker product is the exact per-sample Hessian
    A1, B1 = O.kfac_factors(X[:1], G[:1])
    np.testing.assert_allclose(np.kron(A1, B1), _fisher_terms(X[:1], G[:1])[0], atol=1e-13)
    assert O.kfac_factors(X, None)[1] is None and O.kfac_factors(None, G)[0] is None


def test_shampoo_factors_are_partial_traces_of_the_fisher():
    # One power step from the identity: A = tr_B(E[F]) and B = tr_A(E[F]),
    # the partial traces of the explicit mn x mn expected Hessian.
    rng = np.random.default_rng(31)
    X = rng.standard_normal((6, 3))
    G = rng.standard_normal((6, 4))
    A, B = O.shampoo_factors(X, G)
    F = _fisher_terms(X, G).mean(axis=0).reshape(3, 4, 3, 4)   # [j, i, j', i']
    np.testing.assert_allclose(A, np.einsum("jiki->jk", F), rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(B, np.einsum("jijk->ik", F), rtol=1e-12, atol=1e-13)


def test_shampoo_with_equal_norms_is_scaled_kfac():
    rng = np.random.default_rng(32)
    X = rng.standard_normal((9, 5))
    G = rng.standard_normal((9, 4))
    G /= np.linalg.norm(G, axis=1, keepdims=True) / 1.5   # every |g_t| = 1.5
    A, _ = O.shampoo_factors(X, G)
    Ak, _ = O.kfac_factors(X, G)
    np.testing.assert_allclose(A, 2.25 * Ak, rtol=1e-12)
    assert np.isclose(np.trace(Ak), np.mean(np.sum(X * X, axis=1)))


# ------------------------------------------------- base quantizers (grids)

def test_symmetric_grid_per_row_is_row_scale():
    rng = np.random.default_rng(40)
    W = (0.02 * rng.standard_normal((5, 12))).astype(np.float32)
    W[2] = 0.0
    g, s, z = O.symmetric_grid(W, 4)
    np.testing.assert_array_equal(s[:, 0], O.row_scale(W, 7))
    assert np.all(z == 0) and g.qmin == -8 and g.qmax == 7
    g2, s2, _ = O.symmetric_grid(W, 4, group=4)
    assert s2.shape == (5, 3)
    np.testing.assert_array_equal(s2[:, 1], O.row_scale(W[:, 4:8], 7))


def test_asymmetric_grid_hand_example():
    W = np.array([[-0.3, 0.1, 0.5]], dtype=np.float32)
    g, s, z = O.asymmetric_grid(W, 2)
    s_want = np.float32((np.float32(0.5) - np.float32(-0.3)) / np.float32(3.0))   # fp32 span / 3
    assert s[0, 0] == s_want and z[0, 0] == 1.0
    c = O.quantize_codes(W[0], g.S[0], g.qmin, g.qmax, g.Z[0])
    np.testing.assert_array_equal(c, [0.0, 1.0, 3.0])
    np.testing.assert_allclose(g.values(c[None, :])[0], s_want * np.array([-1.0, 0.0, 2.0]))


@pytest.mark.parametrize("kind", ["sym", "asym"])
@pytest.mark.parametrize("group", [None, 3])
def test_grid_rtn_error_bounds(kind, group):
    rng = np.random.default_rng(41)
    W = (0.05 * rng.standard_normal((6, 10)) + 0.01).astype(np.float32)
    g, s, z = (O.symmetric_grid if kind == "sym" else O.asymmetric_grid)(W, 3, group)
    c = O.quantize_codes(W, g.S, g.qmin, g.qmax, g.Z)
    err = np.abs(g.values(c) - W.astype(np.float64))
    # symmetric: the data lie inside the representable range (error <= s/2);
    # asymmetric: the zero point is rounded, so the range can miss by s/2
    bound = (0.5 if kind == "sym" else 1.0) * g.S * (1 + 1e-6)
    assert np.all(err <= bound)
    assert np.all((c >= g.qmin) & (c <= g.qmax))


def test_theorem32_with_grouped_asymmetric_grid():
    p = problem(5, 7, seed=42)
    g, _, _ = O.asymmetric_grid(p["W"], 3, group=2)
    ref = O.naive_vec_gptq(p["W"], g, UA=p["UA"], UB=p["UB"])
    for r in (O.antidiag(p["W"], p["UA"], p["UB"], g), O.bakron(p["W"], p["UA"], p["UB"], g),
              O.recursive_vec(p["W"], p["UA"], p["UB"], g),
              O.bakron_tiled_order_check(p["W"], p["UA"], p["UB"], g, tile=2)):
        np.testing.assert_array_equal(r.codes, ref.codes)
        np.testing.assert_allclose(r.preround, ref.preround, atol=1e-12)
        np.testing.assert_allclose(r.V, ref.V, atol=1e-15)
    # B = I: row-wise GPTQ with the same grid
    one = O.gptq_rows(p["W"], p["UA"], g)
    two = O.antidiag(p["W"], p["UA"], np.eye(5), g)
    np.testing.assert_array_equal(one.codes, two.codes)
    # the certificate accepts the output and rejects a flipped code
    cert = O.certificate(p["W"], ref.V, ref.codes, p["UA"], p["UB"], g)
    assert cert["ok"] and cert["mismatch"] == 0


def test_grid_diagonal_factors_give_grid_rtn():
    rng = np.random.default_rng(43)
    W = 0.02 * rng.standard_normal((4, 9))
    g, _, _ = O.asymmetric_grid(W, 4, group=3)
    UA = np.diag(rng.uniform(0.5, 2.0, 9))
    UB = np.diag(rng.uniform(0.5, 2.0, 4))
    r = O.bakron(W, UA, UB, g)
    np.testing.assert_array_equal(r.codes, O.quantize_codes(W, g.S, g.qmin, g.qmax, g.Z))


# ------------------------- the C row-accumulator solver (oracle/rowacc.c)

@pytest.mark.parametrize("m,n", SHAPES + [(33, 20), (20, 33)])
def test_rowacc_equals_naive_explicit_hessian(m, n):
    """Theorem 3.2 for the row-accumulator form: the same codes as GPTQ on
    vec(W) with the explicit mn x mn Hessian, the same pre-rounding values
    and errors up to fp64 rounding (a different summation order)."""
    from oracle.rowacc import rowacc
    p = problem(m, n, seed=m * 100 + n + 7)
    ref = O.naive_vec_gptq(p["W"], p["s"], p["qmin"], p["qmax"], A=p["A"], B=p["B"])
    r = rowacc(p["W"], p["UA"], p["UB"], p["s"], p["qmin"], p["qmax"])
    np.testing.assert_array_equal(r.codes, ref.codes)
    np.testing.assert_allclose(r.preround, ref.preround, rtol=0, atol=1e-12)
    np.testing.assert_allclose(r.E, ref.E, rtol=0, atol=1e-10)
    np.testing.assert_array_equal(r.V, p["s"].astype(np.float64)[:, None] * r.codes)


def test_rowacc_unclamped_and_64x64_match_antidiag():
    from oracle.rowacc import rowacc
    p = problem(64, 64, seed=17)
    ones = np.ones(64, np.float32)
    for W, s, lo, hi in ((p["W"], p["s"], p["qmin"], p["qmax"]), (10 * p["W"], ones, None, None)):
        a = O.antidiag(W, p["UA"], p["UB"], s, lo, hi)
        r = rowacc(W, p["UA"], p["UB"], s, lo, hi)
        np.testing.assert_array_equal(r.codes, a.codes)
        np.testing.assert_allclose(r.preround, a.preround, rtol=0, atol=1e-11)


def test_rowacc_b_identity_and_diagonal_factors():
    """B = I reduces to per-row GPTQ; diagonal A and B reduce to rounding to
    nearest (no entry updates another)."""
    from oracle.rowacc import rowacc
    p = problem(7, 12, seed=19)
    I = np.eye(7)
    one = O.gptq_rows(p["W"], p["UA"], p["s"], p["qmin"], p["qmax"])
    r = rowacc(p["W"], p["UA"], I, p["s"], p["qmin"], p["qmax"])
    np.testing.assert_array_equal(r.codes, one.codes)
    np.testing.assert_allclose(r.preround, one.preround, rtol=0, atol=1e-14)
    rng = np.random.default_rng(20)
    UA = np.diag(rng.uniform(0.5, 2.0, 12))
    UB = np.diag(rng.uniform(0.5, 2.0, 7))
    d = rowacc(p["W"], UA, UB, p["s"], -4, 3)
    np.testing.assert_array_equal(d.codes, O.quantize_codes(p["W"], p["s"][:, None], -4, 3))


def test_rowacc_guide_and_transpose_symmetry():
    """A guide equal to the solver's own codes changes nothing; with a unit
    grid, (W, A, B) and (W^T, B, A) are the same problem (vec order swaps)."""
    from oracle.rowacc import rowacc
    p = problem(9, 14, seed=21)
    r = rowacc(p["W"], p["UA"], p["UB"], p["s"], p["qmin"], p["qmax"])
    g = rowacc(p["W"], p["UA"], p["UB"], p["s"], p["qmin"], p["qmax"], guide=r.codes)
    np.testing.assert_array_equal(g.codes, r.codes)
    assert g.overrides == 0
    W = 40 * p["W"]
    a = rowacc(W, p["UA"], p["UB"], np.ones(9, np.float32))
    b = rowacc(W.T.copy(), p["UB"], p["UA"], np.ones(14, np.float32))
    np.testing.assert_array_equal(a.codes, b.codes.T)
    np.testing.assert_allclose(a.preround, b.preround.T, rtol=0, atol=1e-12)


def test_rowacc_guide_takes_a_planted_near_tie():
    """An entry placed exactly on a rounding boundary (entry (0, 0), which no
    update reaches): round half to even takes one side; a guide with the other
    code is followed there and counted."""
    from oracle.rowacc import rowacc
    p = problem(5, 6, seed=22)
    W = p["W"].copy()
    W[0, 0] = 0.5 * float(p["s"][0])
    r = rowacc(W, p["UA"], p["UB"], p["s"], p["qmin"], p["qmax"])
    assert r.codes[0, 0] == 0.0
    guide = r.codes.copy()
    guide[0, 0] = 1.0
    g = rowacc(W, p["UA"], p["UB"], p["s"], p["qmin"], p["qmax"], guide=guide)
    assert g.codes[0, 0] == 1.0 and g.overrides >= 1
    ref = O.antidiag(W, p["UA"], p["UB"], p["s"], p["qmin"], p["qmax"], guide=guide)
    np.testing.assert_array_equal(g.codes, ref.codes)


@pytest.mark.parametrize("m,n,rb", [(5, 7, 3), (33, 20, 8), (37, 100, 16), (129, 77, 8)])
def test_rowacc_row_blocks_equal_antidiagonal_traversal(m, n, rb):
    """The row-blocked traversal of the C solver (the one the full-size
    comparisons use) against its anti-diagonal traversal: same codes, and the
    same pre-rounding values up to the regrouped column sums; with one row
    per block the two are the same computation, bit for bit."""
    from oracle.rowacc import rowacc
    p = problem(m, n, seed=m + 3 * n)
    a = rowacc(p["W"], p["UA"], p["UB"], p["s"], p["qmin"], p["qmax"])
    b = rowacc(p["W"], p["UA"], p["UB"], p["s"], p["qmin"], p["qmax"], rows_per_block=rb)
    np.testing.assert_array_equal(b.codes, a.codes)
    np.testing.assert_allclose(b.preround, a.preround, rtol=0, atol=1e-13)
    one = rowacc(p["W"], p["UA"], p["UB"], p["s"], p["qmin"], p["qmax"], rows_per_block=1)
    np.testing.assert_array_equal(one.preround, a.preround)
    ones = np.ones(m, np.float32)
    u = rowacc(12 * p["W"], p["UA"], p["UB"], ones, rows_per_block=rb)
    ua = O.antidiag(12 * p["W"], p["UA"], p["UB"], ones)
    np.testing.assert_array_equal(u.codes, ua.codes)
    g = rowacc(p["W"], p["UA"], p["UB"], p["s"], p["qmin"], p["qmax"], guide=a.codes, rows_per_block=rb)
    np.testing.assert_array_equal(g.codes, a.codes)
    assert g.overrides == 0
