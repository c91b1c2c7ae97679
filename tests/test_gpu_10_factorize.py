"""dbf_factorize (double binary factorization of a dense W) against the fp64 oracle.

The path computes in fp32 and the oracle in fp64.  The SVID step takes the
sign of Y = P + U, so where Y is within rounding of zero the two may decide
differently, and one flipped sign changes that factor entry by twice its
magnitude.  A later step whose fixed factor carries such flips sees a
perturbed problem and flips a few tenths of a percent of its own signs (an
fp32 solve through LAPACK shows the same: 99.85% agreement on B after one
round at 4096 x 4096, k = 3072).  So the comparison is:

  first step (A-step of the first round, one ADMM iteration, Y = P is a
  continuous function of the inputs): every sign agrees wherever the
  oracle's |Y| exceeds 3e-4 of its RMS (fp32 GEMM sums of <= 4096 terms
  and a solve with condition number <= k / rho_rel + 1 keep the error of Y
  far below that); the scales r = |Y| c and c, continuous in |Y|, agree
  within 1e-4 of their maximum;
  any later step: signs agree on >= 99.5% (99% after several rounds) of the
  entries and the objective ||W - W_hat|| / ||W|| within 0.5% (0.1% at
  full size) of the oracle's.
"""

import numpy as np
import pytest
import torch

from oracle import dbf_factorize as FZ
from oracle import dbf_oracle as O
from tests import gpu_util as U
from workloads import generators as G

pytestmark = pytest.mark.gpu

SHAPES = [(200, 136, 40), (97, 300, 70), (64, 64, 1), (300, 260, 130), (20, 30, 64)]


def _dev(arrs):
    return [torch.from_numpy(np.ascontiguousarray(a)).cuda() for a in arrs]


def _host(ts):
    return [t.cpu().numpy() for t in ts]


def _run(cuda_lib, w, start, outer, inner, q, rho):
    wt = torch.from_numpy(w).cuda()
    fs = _dev(start)
    cuda_lib.factorize(wt, *fs, outer=outer, inner=inner, power_iters=q, rho_rel=rho)
    st = cuda_lib.check_status()
    assert st == 0, cuda_lib.status_string(st)
    return _host(fs)


BAND = 3e-4


def _check_first_step(w, start, got, q):
    r, S, c, y = FZ.admm_left(w, FZ.svid_dense(*start[3:]), *start[:3], 1, q, 1.0, return_y=True)
    a, A, mL = got[:3]
    decided = np.abs(y) > BAND * np.sqrt(np.mean(y * y))
    wrong = int(np.sum(A[decided] != S[decided]))
    assert wrong == 0, f"{wrong} signs differ outside the rounding band ({decided.sum()} decided)"
    assert np.abs(a - r).max() <= 1e-4 * np.abs(r).max(), np.abs(a - r).max() / np.abs(r).max()
    assert np.abs(mL - c).max() <= 1e-4 * np.abs(c).max(), np.abs(mL - c).max() / np.abs(c).max()


def _check_round(w, got, want, sign_agree, obj_tol):
    a, A, mL, mR, B, b = got
    assert set(np.unique(A)) <= {-1, 1} and set(np.unique(B)) <= {-1, 1}
    assert all(np.all(np.isfinite(v)) for v in (a, mL, mR, b))
    assert np.mean(A == want[1]) >= sign_agree, np.mean(A == want[1])
    assert np.mean(B == want[4]) >= sign_agree, np.mean(B == want[4])
    eg, ew = FZ.rel_error(w, *got), FZ.rel_error(w, *want)
    assert abs(eg - ew) <= obj_tol * ew, (eg, ew)


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("sched", [(1, 1, 4), (2, 5, 6)])
def test_factorize_matches_oracle(cuda_lib, shape, sched):
    N, M, k = shape
    outer, inner, q = sched
    seed = 7000 + N + M + k
    w = G.make_dense_weight(N, M, seed)
    start = G.make_factorize_start(N, M, k, seed)
    got = _run(cuda_lib, w, start, outer, inner, q, 1.0)
    want = FZ.factorize(w, start[:3], start[3:], outer, inner, q, 1.0)
    if inner == 1:
        _check_first_step(w, start, got, q)
    _check_round(w, got, want, 0.995 if outer == 1 else 0.99, 5e-3)


def _exact(seed, N=48, M=40, k=12):
    g = np.random.default_rng(seed)
    a = g.uniform(0.5, 2.0, N).astype(np.float32)
    A = np.where(g.standard_normal((N, k)) >= 0, 1, -1).astype(np.int8)
    mL = g.uniform(0.5, 2.0, k).astype(np.float32)
    mR = g.uniform(0.5, 2.0, k).astype(np.float32)
    B = np.where(g.standard_normal((k, M)) >= 0, 1, -1).astype(np.int8)
    b = g.uniform(0.5, 2.0, M).astype(np.float32)
    p = a.astype(np.float64)[:, None] * A * mL.astype(np.float64)[None, :]
    qm = mR.astype(np.float64)[:, None] * B * b.astype(np.float64)[None, :]
    return (a, A, mL, mR, B, b), (p @ qm).astype(np.float32)


def test_exact_factors_are_a_fixed_point(cuda_lib):
    f, w = _exact(11)
    got = _run(cuda_lib, w, f, 2, 3, 4, 0.5)
    np.testing.assert_array_equal(got[1], f[1])
    np.testing.assert_array_equal(got[4], f[4])
    assert FZ.rel_error(w, *got) < 1e-5


def test_recovers_the_factors_of_an_exact_matrix(cuda_lib):
    f, w = _exact(0)
    N, k = f[1].shape
    start = (np.zeros(N, np.float32), np.ones((N, k), np.int8), np.zeros(k, np.float32)) + tuple(f[3:])
    got = _run(cuda_lib, w, start, 1, 50, 8, 0.01)
    np.testing.assert_array_equal(got[1], f[1])
    assert FZ.rel_error(w, *got) < 1e-3


def test_rerun_is_bitwise_identical_and_w_is_read_only(cuda_lib):
    N, M, k = 300, 260, 130
    w = G.make_dense_weight(N, M, 71)
    start = G.make_factorize_start(N, M, k, 71)
    wt = torch.from_numpy(w).cuda()
    outs = []
    for _ in range(2):
        fs = _dev(start)
        cuda_lib.factorize(wt, *fs, outer=2, inner=4, power_iters=5, rho_rel=1.0)
        outs.append(_host(fs))
    assert cuda_lib.check_status() == 0
    for x, y in zip(*outs):
        assert np.array_equal(x, y)
    assert np.array_equal(wt.cpu().numpy(), w)


def test_zero_rounds_leave_the_factors(cuda_lib):
    N, M, k = 50, 40, 20
    w = G.make_dense_weight(N, M, 5)
    start = list(G.make_factorize_start(N, M, k, 5))
    start[0] = np.full(N, 0.5, np.float32)
    for outer, inner in ((0, 5), (3, 0)):
        got = _run(cuda_lib, w, start, outer, inner, 4, 1.0)
        for x, y in zip(got, start):
            assert np.array_equal(x, y)
    assert cuda_lib.factorize_launch_count(N, M, k, 0, 5, 4, 1.0) == 0


def test_argument_errors(cuda_lib):
    w = torch.zeros((8, 8), dtype=torch.float32, device="cuda")
    fs = _dev(G.make_factorize_start(8, 8, 4, 1))
    with pytest.raises(ValueError):
        cuda_lib.factorize(w.half(), *fs)
    with pytest.raises(ValueError):
        cuda_lib.factorize(w, fs[0], fs[1].float(), *fs[2:])
    with pytest.raises(cuda_lib.DbfError) as e:
        cuda_lib.factorize(w, *fs, rho_rel=0.0)
    assert e.value.code == cuda_lib.DBF_ERR_INVALID_ARG
    with pytest.raises(cuda_lib.DbfError) as e:
        cuda_lib.factorize(w, *fs, workspace=torch.empty(256, dtype=torch.uint8, device="cuda"))
    assert e.value.code == cuda_lib.DBF_ERR_WORKSPACE


def test_nan_in_the_fixed_factor_reports_a_numeric_status(cuda_lib):
    # A NaN scale makes every pivot of F F^T + rho I NaN, which fails the
    # positivity check: the call still completes (no value decides an
    # address) and the status word says DBF_ERR_NUMERIC; reading it clears it.
    N, M, k = 40, 36, 8
    w = G.make_dense_weight(N, M, 9)
    start = list(G.make_factorize_start(N, M, k, 9))
    start[3] = start[3].copy()
    start[3][2] = np.nan
    fs = _dev(start)
    cuda_lib.factorize(torch.from_numpy(w).cuda(), *fs, outer=1, inner=2, power_iters=3, rho_rel=1.0)
    assert cuda_lib.check_status() == cuda_lib.DBF_ERR_NUMERIC
    assert cuda_lib.check_status() == 0
    assert cuda_lib.status_string(cuda_lib.DBF_ERR_NUMERIC) != "unknown status"


def _weights(N, M, seed):
    g = np.random.default_rng(seed)
    return (np.exp(0.5 * g.standard_normal(N)).astype(np.float32),
            np.exp(0.5 * g.standard_normal(M)).astype(np.float32))


def _run_weighted(cuda_lib, w, d_out, d_in, start, outer, inner, q, rho):
    fs = _dev(start)
    cuda_lib.factorize_weighted(torch.from_numpy(w).cuda(), torch.from_numpy(d_out).cuda(),
                                torch.from_numpy(d_in).cuda(), *fs, outer=outer, inner=inner, power_iters=q,
                                rho_rel=rho)
    st = cuda_lib.check_status()
    assert st == 0, cuda_lib.status_string(st)
    return _host(fs)


def test_unit_weights_give_the_plain_bits(cuda_lib):
    N, M, k = 200, 136, 40
    w = G.make_dense_weight(N, M, 31)
    start = G.make_factorize_start(N, M, k, 31)
    plain = _run(cuda_lib, w, start, 2, 3, 4, 1.0)
    weighted = _run_weighted(cuda_lib, w, np.ones(N, np.float32), np.ones(M, np.float32), start, 2, 3, 4, 1.0)
    for x, y in zip(plain, weighted):
        assert np.array_equal(x, y)


@pytest.mark.parametrize("shape", [(200, 136, 40), (97, 300, 70), (300, 260, 130)])
def test_weighted_factorization_matches_oracle(cuda_lib, shape):
    # Same checks as the plain rounds, on the weighted objective; the first
    # step's signs and scales are those of the scaled problem.
    N, M, k = shape
    seed = 7500 + N + k
    w = G.make_dense_weight(N, M, seed)
    d_out, d_in = _weights(N, M, seed)
    start = G.make_factorize_start(N, M, k, seed)
    got = _run_weighted(cuda_lib, w, d_out, d_in, start, 1, 1, 4, 1.0)
    wp = d_out.astype(np.float64)[:, None] * w * d_in.astype(np.float64)[None, :]
    sstart = (start[0] * d_out, start[1], start[2], start[3], start[4], start[5] * d_in)
    scaled_got = [got[0] * d_out.astype(np.float64)] + list(got[1:5]) + [got[5] * d_in.astype(np.float64)]
    _check_first_step(wp, sstart, scaled_got, 4)
    want = FZ.factorize_weighted(w, d_out, d_in, start[:3], start[3:], 1, 1, 4, 1.0)
    assert np.mean(got[1] == want[1]) >= 0.995 and np.mean(got[4] == want[4]) >= 0.995
    eg = FZ.weighted_rel_error(w, d_out, d_in, *got)
    ew = FZ.weighted_rel_error(w, d_out, d_in, *want)
    assert abs(eg - ew) <= 5e-3 * ew, (eg, ew)
    got = _run_weighted(cuda_lib, w, d_out, d_in, start, 2, 5, 6, 1.0)
    want = FZ.factorize_weighted(w, d_out, d_in, start[:3], start[3:], 2, 5, 6, 1.0)
    assert np.mean(got[1] == want[1]) >= 0.99 and np.mean(got[4] == want[4]) >= 0.99
    eg = FZ.weighted_rel_error(w, d_out, d_in, *got)
    ew = FZ.weighted_rel_error(w, d_out, d_in, *want)
    assert abs(eg - ew) <= 5e-3 * ew, (eg, ew)


def test_a_non_positive_weight_is_reported(cuda_lib):
    N, M, k = 40, 36, 8
    w = G.make_dense_weight(N, M, 8)
    d_out, d_in = _weights(N, M, 8)
    d_in[5] = 0.0
    fs = _dev(G.make_factorize_start(N, M, k, 8))
    cuda_lib.factorize_weighted(torch.from_numpy(w).cuda(), torch.from_numpy(d_out).cuda(),
                                torch.from_numpy(d_in).cuda(), *fs, outer=1, inner=1, power_iters=2)
    assert cuda_lib.check_status() == cuda_lib.DBF_ERR_DEVICE_ARG
    assert cuda_lib.check_status() == 0


def _balanced_fp16(a, m, b):
    # fp16 scales for the matmul: equalise the geometric means of alpha, beta
    # and gamma (their product per entry of W_hat is unchanged).
    ga, gm, gb = (float(np.exp(np.mean(np.log(np.abs(v) + 1e-30)))) for v in (a, m, b))
    t = (ga * gm * gb) ** (1.0 / 3.0)
    return ((a * (t / ga)).astype(np.float16)[None, :], (m * (t / gm)).astype(np.float16)[None, :],
            (b * (t / gb)).astype(np.float16)[None, :])


def test_factors_serve_through_the_matmul(cuda_lib):
    # Compress, then run the product with the packed result: y = x W_hat^T
    # exactly as for any factor set, and y approximates x W^T by the
    # factorization error.
    N, M, k, T = 256, 192, 256, 24
    w = G.make_dense_weight(N, M, 90)
    a, A, mL, mR, B, b = _run(cuda_lib, w, G.make_factorize_start(N, M, k, 90), 4, 8, 6, 1.0)
    alpha, beta, gamma = _balanced_fp16(a, mL * mR, b)
    f = G.Factors(A, B, alpha, beta, gamma)
    df = U.device_factors(f)
    xb = G.make_x(T, M, 91)
    y = cuda_lib.matmul(df, U.bits_to_bf16(xb))
    yref, _ = O.matmul(xb, f)
    U.assert_close(U.bf16_to_bits(y), yref, "factorized product")
    x64 = O.bf16_bits_to_f64(xb)
    err_w = FZ.rel_error(w, a, A, mL, mR, B, b)
    err_y = O.rel_frobenius(O.bf16_bits_to_f64(U.bf16_to_bits(y)), x64 @ w.astype(np.float64).T)
    assert err_w < 0.6
    assert abs(err_y - err_w) < 0.1


@pytest.mark.slow
def test_full_size_1p5_bit_layer(cuda_lib):
    # 4096 x 4096 at k = 3072 (1.5 bits per weight): one round of one ADMM
    # iteration per step (first-step check on every sign and scale), then one
    # round of two iterations, against the oracle on the whole result.
    N = M = 4096
    k = 3072
    w = G.make_dense_weight(N, M, 4096)
    start = G.make_factorize_start(N, M, k, 4096)
    got = _run(cuda_lib, w, start, 1, 1, 4, 1.0)
    _check_first_step(w, start, got, 4)
    _check_round(w, got, FZ.factorize(w, start[:3], start[3:], 1, 1, 4, 1.0), 0.995, 1e-3)
    got = _run(cuda_lib, w, start, 1, 2, 4, 1.0)
    _check_round(w, got, FZ.factorize(w, start[:3], start[3:], 1, 2, 4, 1.0), 0.995, 1e-3)
