"""Pins of the factorization oracle against things other than itself.

The oracle follows the outline of "Addition is almost all you need:
Compressing large language models with double binary factorization",
section 2 (Algoritmo de Optimización): alternating minimisation over the two
sign factors, ADMM for each step, SVID as the projection.  Each test below
checks one step against mathematics or a library routine that the oracle
does not use for that step, so that a dropped term, a wrong sign or a
transposed operand fails at least one of them.
"""

import numpy as np
import pytest

from oracle import dbf_factorize as fz


def _rng(seed):
    return np.random.default_rng(seed)


def _exact_problem(seed, N=48, M=40, k=12):
    g = _rng(seed)
    a = g.uniform(0.5, 2.0, N)
    A = fz.sign_pm1(g.standard_normal((N, k)))
    mL = g.uniform(0.5, 2.0, k)
    mR = g.uniform(0.5, 2.0, k)
    B = fz.sign_pm1(g.standard_normal((k, M)))
    b = g.uniform(0.5, 2.0, M)
    return (a, A, mL, mR, B, b), fz.reconstruct(a, A, mL, mR, B, b)


def test_sign_of_zero_is_plus_one():
    s = fz.sign_pm1(np.array([[0.0, -0.0, 1e-300, -1e-300, 3.0, -2.0]]))
    assert s.dtype == np.int8
    assert s.tolist() == [[1, 1, 1, -1, 1, -1]]


def test_svid_is_exact_and_idempotent_on_its_set():
    g = _rng(1)
    r = g.uniform(0.1, 3.0, 30)
    c = g.uniform(0.1, 3.0, 17)
    S = fz.sign_pm1(g.standard_normal((30, 17)))
    y = fz.svid_dense(r, S, c)
    r1, S1, c1 = fz.svid(y, 1)
    np.testing.assert_array_equal(S1, S)
    np.testing.assert_allclose(np.outer(r1, c1), np.outer(r, c), rtol=1e-12)
    z = fz.svid_dense(r1, S1, c1)
    r2, S2, c2 = fz.svid(z, 3)
    np.testing.assert_allclose(fz.svid_dense(r2, S2, c2), z, rtol=1e-12)


def test_svid_rank1_matches_leading_singular_pair():
    g = _rng(2)
    y = g.standard_normal((40, 25)) * g.uniform(0.2, 2.0, (40, 1))
    r, S, c = fz.svid(y, 300)
    u, s, vt = np.linalg.svd(np.abs(y))
    best = s[0] * np.outer(u[:, 0], vt[0])
    np.testing.assert_allclose(np.outer(r, c), best, rtol=1e-9, atol=1e-12)
    assert np.all(c >= 0) and np.all(r >= 0)
    np.testing.assert_allclose(np.linalg.norm(c), 1.0, rtol=1e-12)


def test_svid_zero_matrix():
    r, S, c = fz.svid(np.zeros((5, 4)), 4)
    assert np.all(r == 0) and np.all(c == 0) and np.all(S == 1)


def test_penalty_closed_forms():
    f = np.where(_rng(3).standard_normal((6, 11)) >= 0, 1.0, -1.0)
    assert fz.penalty(f, 0.5) == pytest.approx(0.5 * 11)
    assert fz.penalty(np.zeros((6, 11)), 0.25) == 0.25


def test_p_update_is_the_stacked_least_squares_solution():
    # argmin_P 1/2||T - P F||^2 + rho/2 ||P - (Z - U)||^2, row by row as an
    # ordinary least-squares problem on [F^T; sqrt(rho) I].
    g = _rng(4)
    n, p, k = 9, 14, 5
    t = g.standard_normal((n, p))
    f = g.standard_normal((k, p))
    z = g.standard_normal((n, k))
    u = g.standard_normal((n, k))
    rho = 0.7
    stacked = np.vstack([f.T, np.sqrt(rho) * np.eye(k)])
    want = np.empty((n, k))
    for i in range(n):
        rhs = np.concatenate([t[i], np.sqrt(rho) * (z[i] - u[i])])
        want[i] = np.linalg.lstsq(stacked, rhs, rcond=None)[0]
    np.testing.assert_allclose(fz.p_update(t, f, z, u, rho), want, rtol=1e-10, atol=1e-12)


@pytest.mark.parametrize("inner", [1, 3])
def test_exact_factors_are_a_fixed_point(inner):
    (a, A, mL, mR, B, b), w = _exact_problem(5)
    r, S, c = fz.admm_left(w, fz.svid_dense(mR, B, b), a, A, mL, inner, 4, 0.5)
    np.testing.assert_allclose(fz.svid_dense(r, S, c), fz.svid_dense(a, A, mL), rtol=1e-10, atol=1e-12)
    f = fz.factorize(w, (a, A, mL), (mR, B, b), 2, inner, 4, 0.5)
    assert fz.rel_error(w, *f) < 1e-12


def test_admm_from_zero_recovers_the_left_factor():
    (a, A, mL, mR, B, b), w = _exact_problem(0)
    N, k = A.shape
    start = (np.zeros(N), np.ones((N, k), np.int8), np.zeros(k))
    ps = fz.svid_dense(a, A, mL)
    r, S, c = fz.admm_left(w, fz.svid_dense(mR, B, b), *start, 50, 8, 0.01)
    assert np.abs(fz.svid_dense(r, S, c) - ps).max() / np.abs(ps).max() < 1e-3
    np.testing.assert_array_equal(S, A)


def test_planted_dual_sign_mistake_fails_recovery():
    (a, A, mL, mR, B, b), w = _exact_problem(0)
    N, k = A.shape
    start = (np.zeros(N), np.ones((N, k), np.int8), np.zeros(k))
    ps = fz.svid_dense(a, A, mL)
    r, S, c = fz.admm_left(w, fz.svid_dense(mR, B, b), *start, 50, 8, 0.01, _dual_sign=-1.0)
    assert np.abs(fz.svid_dense(r, S, c) - ps).max() / np.abs(ps).max() > 1.0


def test_b_step_is_the_a_step_of_the_transposed_problem():
    # One round from a given start equals an explicit A-step on W followed by
    # an explicit A-step on W^T with the roles of the factors exchanged.
    g = _rng(6)
    N, M, k = 20, 16, 6
    w = g.standard_normal((N, M))
    left = (np.zeros(N), np.ones((N, k), np.int8), np.zeros(k))
    right = (np.ones(k), fz.sign_pm1(g.standard_normal((k, M))), np.ones(M))
    a, A, mL, mR, B, b = fz.factorize(w, left, right, 1, 4, 5, 1.0)
    a2, A2, mL2 = fz.admm_left(w, fz.svid_dense(*right), *left, 4, 5, 1.0)
    b2, Bt2, mR2 = fz.admm_left(w.T, fz.svid_dense(a2, A2, mL2).T, right[2], right[1].T, right[0], 4, 5, 1.0)
    np.testing.assert_array_equal(A, A2)
    np.testing.assert_array_equal(B, Bt2.T)
    np.testing.assert_allclose(fz.reconstruct(a, A, mL, mR, B, b), fz.reconstruct(a2, A2, mL2, mR2, Bt2.T, b2))


def test_alternation_reduces_the_error_on_a_random_matrix():
    g = _rng(1)
    N, M, k = 256, 192, 256
    w = g.standard_normal((N, M)) * 0.02
    left = (np.zeros(N), np.ones((N, k), np.int8), np.zeros(k))
    right = (np.ones(k), fz.sign_pm1(g.standard_normal((k, M))), np.ones(M))
    e1 = fz.rel_error(w, *fz.factorize(w, left, right, 1, 10, 8, 1.0))
    e6 = fz.rel_error(w, *fz.factorize(w, left, right, 6, 10, 8, 1.0))
    r, S, c = fz.svid(w, 20)
    one_bit = np.linalg.norm(w - fz.svid_dense(r, S, c)) / np.linalg.norm(w)
    assert e6 < e1
    assert e6 < one_bit


def _weighted_case(seed, N=96, M=80, k=64):
    g = _rng(seed)
    w = g.standard_normal((N, M)) * 0.02
    left = (np.zeros(N), np.ones((N, k), np.int8), np.zeros(k))
    right = (np.ones(k), fz.sign_pm1(g.standard_normal((k, M))), np.ones(M))
    return w, left, right


def test_unit_importance_weights_change_nothing():
    w, left, right = _weighted_case(10)
    plain = fz.factorize(w, left, right, 2, 4, 5, 1.0)
    weighted = fz.factorize_weighted(w, np.ones(w.shape[0]), np.ones(w.shape[1]), left, right, 2, 4, 5, 1.0)
    for x, y in zip(plain, weighted):
        assert np.array_equal(x, y)


def test_weighted_result_is_the_scaled_problem_solved_and_unscaled():
    # The weighted error of the returned factors equals the plain error of
    # factorizing W' = diag(d_out) W diag(d_in) from the explicitly scaled
    # start; a result left in the scaled variables (a planted mistake) or
    # scaled the wrong way does not.
    w, left, right = _weighted_case(11)
    g = _rng(12)
    d_out = np.exp(0.5 * g.standard_normal(w.shape[0]))
    d_in = np.exp(0.5 * g.standard_normal(w.shape[1]))
    res = fz.factorize_weighted(w, d_out, d_in, left, right, 2, 4, 5, 1.0)
    wp = d_out[:, None] * w * d_in[None, :]
    direct = fz.factorize(wp, (left[0] * d_out, left[1], left[2]), (right[0], right[1], right[2] * d_in),
                          2, 4, 5, 1.0)
    e_direct = fz.rel_error(wp, *direct)
    assert fz.weighted_rel_error(w, d_out, d_in, *res) == pytest.approx(e_direct, rel=1e-10)
    left_scaled = (direct[0],) + tuple(res[1:])
    assert abs(fz.weighted_rel_error(w, d_out, d_in, *left_scaled) - e_direct) > 1e-2
    wrong_way = (res[0] / d_out,) + tuple(res[1:5]) + (res[5] / d_in,)
    assert abs(fz.weighted_rel_error(w, d_out, d_in, *wrong_way) - e_direct) > 1e-2


def test_weighting_input_columns_lowers_their_error():
    w, left, right = _weighted_case(13, N=128, M=96, k=96)
    heavy = np.arange(0, w.shape[1], 8)
    d_in = np.ones(w.shape[1])
    d_in[heavy] = 10.0
    plain = fz.factorize(w, left, right, 4, 8, 6, 1.0)
    weighted = fz.factorize_weighted(w, np.ones(w.shape[0]), d_in, left, right, 4, 8, 6, 1.0)

    def col_err(f):
        d = w - fz.reconstruct(*f)
        return np.sqrt(np.sum(d[:, heavy] ** 2) / np.sum(w[:, heavy] ** 2))

    assert col_err(weighted) < 0.8 * col_err(plain)


def test_scalar_step_closed_form():
    # n = 1, k = 1, p = 3, one iteration from Z = 0: rho = rho_rel |f|^2 (the
    # mean diagonal of a 1 x 1 F F^T), P = t.f / ((1 + rho_rel) |f|^2), and
    # SVID of a 1 x 1 matrix is exact: r = |P|, S = sign(P), c = 1.
    t = np.array([[0.3, -1.2, 0.5]])
    f = np.array([[2.0, 1.0, -0.5]])
    for rho_rel in (0.25, 1.0, 3.0):
        r, S, c = fz.admm_left(t, f, np.zeros(1), np.ones((1, 1), np.int8), np.zeros(1), 1, 3, rho_rel)
        tf, ff = (t @ f.T).item(), (f @ f.T).item()
        p = tf / ((1.0 + rho_rel) * ff)
        assert r[0] == pytest.approx(abs(p), rel=1e-14)
        assert S[0, 0] == (1 if p >= 0 else -1)
        assert c[0] == pytest.approx(1.0, rel=1e-15)


def test_rank_one_step_converges_to_least_squares():
    # With k = 1 every n x 1 matrix is of the SVID form (r_i = |y_i|, c = 1),
    # so the constraint is vacuous and ADMM must converge to the plain
    # least-squares factor T F^T / (F F^T).
    g = _rng(21)
    t = g.standard_normal((7, 5))
    f = g.standard_normal((1, 5))
    r, S, c = fz.admm_left(t, f, np.zeros(7), np.ones((7, 1), np.int8), np.zeros(1), 200, 2, 1.0)
    want = (t @ f.T) / (f @ f.T).item()
    np.testing.assert_allclose(fz.svid_dense(r, S, c), want, rtol=1e-10, atol=1e-14)
