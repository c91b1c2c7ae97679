"""The factorization's tensor-core GEMM (dbf_selftest_split_gemm) against fp64.

Each fp32 operand is split into hi = tf32(x) and lo = tf32(x - hi), and
A B^T is summed as A_hi B_hi^T + A_hi B_lo^T + A_lo B_hi^T on tcgen05
kind::tf32 with fp32 accumulation (the dropped lo*lo term is below
2^-22 |a||b| per product).  Measured on B300 its relative Frobenius error is
about 1e-5 at K = 1000: some 30 times numpy's fp32 matmul (blocked FMA
accumulation), and 30 times smaller than a single tf32 product's 3e-4.  The
checks: the Frobenius error is at most a sixth of that of the tf32 product
of the same operands (rounded to tf32 as the tensor cores would, summed in
fp64), which a GEMM that dropped a cross term, or did not split, misses; it
is at most 100 times numpy's fp32 matmul error; and no entry is off by more
than 2^-14 of its sum of magnitudes.
"""

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


def _case(m, n, kk, seed, scale_spread=False):
    rng = np.random.default_rng(seed)
    a = rng.standard_normal((m, kk)).astype(np.float32)
    b = rng.standard_normal((n, kk)).astype(np.float32)
    if scale_spread:  # rows over several orders of magnitude, like a weighted problem
        a *= (10.0 ** rng.uniform(-3, 3, size=(m, 1))).astype(np.float32)
        b *= (10.0 ** rng.uniform(-3, 3, size=(n, 1))).astype(np.float32)
    c = rng.standard_normal((m, n)).astype(np.float32)
    return a, b, c


def _check(got, a, b, c0, alpha, beta, rows=None, cols=None, lower=False):
    a64, b64 = a.astype(np.float64), b.astype(np.float64)
    a32, b32 = a, b
    if rows is not None:
        a64, a32 = a64[rows], a32[rows]
    if cols is not None:
        b64, b32 = b64[cols], b32[cols]
    c = c0
    if rows is not None:
        c = c[rows]
    if cols is not None:
        c = c[:, cols]
    want = alpha * (a64 @ b64.T) + beta * c.astype(np.float64)
    ref32 = (np.float32(alpha) * (a32 @ b32.T) + np.float32(beta) * c).astype(np.float64)
    mag = abs(alpha) * (np.abs(a64) @ np.abs(b64).T) + abs(beta) * np.abs(c.astype(np.float64))
    g = got.astype(np.float64)
    keep = np.ones(want.shape, bool)
    if lower:
        # tiles (128 x 256) wholly above the diagonal are left as they were
        r = np.arange(want.shape[0])[:, None] if rows is None else np.asarray(rows)[:, None]
        col = np.arange(want.shape[1])[None, :] if cols is None else np.asarray(cols)[None, :]
        above = (col // 256) * 256 >= (r // 128) * 128 + 128
        assert np.array_equal(g[above], c.astype(np.float64)[above])
        keep = ~above
    reft = alpha * (_tf32(a32).astype(np.float64) @ _tf32(b32).astype(np.float64).T) + beta * c.astype(np.float64)
    err = np.linalg.norm((g - want)[keep])
    err32 = np.linalg.norm((ref32 - want)[keep])
    errt = np.linalg.norm((reft - want)[keep])
    norm = np.linalg.norm(want[keep])
    assert err <= errt / 6 + 8 * 2.0 ** -24 * norm, (err, errt, norm)
    assert err <= 100 * err32 + 8 * 2.0 ** -24 * norm, (err, err32, norm)
    assert (np.abs(g - want)[keep] <= 2.0 ** -14 * mag[keep] + 1e-30).all()


def _tf32(x):
    """x rounded to tf32 (10 explicit mantissa bits, to nearest, ties away from zero)."""
    u = np.asarray(x, np.float32).view(np.uint32).astype(np.uint64)
    return ((u + 0x1000) & 0xFFFFE000).astype(np.uint32).view(np.float32)


@pytest.mark.parametrize("m,n,kk", [(1, 1, 1), (97, 300, 70), (300, 260, 130), (129, 257, 33), (640, 520, 1000)])
@pytest.mark.parametrize("alpha,beta", [(1.0, 0.0), (-1.0, 1.0), (0.5, -2.0)])
def test_split_gemm_matches_fp64(cuda_lib, m, n, kk, alpha, beta):
    a, b, c = _case(m, n, kk, 9000 + m + kk)
    C = torch.from_numpy(c).cuda()
    cuda_lib.selftest_split_gemm(torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda(), C, alpha, beta)
    assert cuda_lib.check_status() == 0
    _check(C.cpu().numpy(), a, b, c, alpha, beta)


@pytest.mark.parametrize("m,n,kk", [(300, 300, 96), (520, 520, 64)])
def test_split_gemm_lower_leaves_upper_tiles(cuda_lib, m, n, kk):
    a, b, c = _case(m, n, kk, 9100 + m)
    C = torch.from_numpy(c).cuda()
    cuda_lib.selftest_split_gemm(torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda(), C, 1.0, 0.0, lower=True)
    assert cuda_lib.check_status() == 0
    _check(C.cpu().numpy(), a, b, c, 1.0, 0.0, lower=True)


def test_split_gemm_wide_dynamic_range(cuda_lib):
    a, b, c = _case(256, 384, 500, 9200, scale_spread=True)
    C = torch.from_numpy(c).cuda()
    cuda_lib.selftest_split_gemm(torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda(), C, 1.0, 1.0)
    assert cuda_lib.check_status() == 0
    _check(C.cpu().numpy(), a, b, c, 1.0, 1.0)


def test_split_gemm_strided_operands(cuda_lib):
    m, n, kk = 200, 150, 90
    a, b, c = _case(m, n, kk + 7, 9300)  # row strides kk + 7, the first kk columns used
    A = torch.from_numpy(a).cuda()[:, :kk]
    B = torch.from_numpy(b).cuda()[:, :kk]
    C = torch.from_numpy(c).cuda()
    cuda_lib.selftest_split_gemm(A, B, C, 2.0, 0.0)
    assert cuda_lib.check_status() == 0
    _check(C.cpu().numpy(), a[:, :kk], b[:, :kk], c, 2.0, 0.0)


def test_split_gemm_p_update_size_sampled(cuda_lib):
    # the P-update of the 1.5-bit layer: 4096 x 3072 x 3072, beta = 1; entries sampled at the
    # tile edges (128-row and 256-column tiles) and at random
    m, n, kk = 4096, 3072, 3072
    a, b, c = _case(m, n, kk, 9400)
    C = torch.from_numpy(c).cuda()
    cuda_lib.selftest_split_gemm(torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda(), C, 1.0, 1.0)
    assert cuda_lib.check_status() == 0
    rng = np.random.default_rng(9401)
    rows = np.unique(np.concatenate([[0, 127, 128, 255, 256, m - 129, m - 128, m - 1], rng.integers(0, m, 24)]))
    cols = np.unique(np.concatenate([[0, 255, 256, 511, 512, n - 257, n - 256, n - 1], rng.integers(0, n, 24)]))
    got = C.cpu().numpy()[np.ix_(rows, cols)]
    _check(got, a, b, c, 1.0, 1.0, rows=rows, cols=cols)


def test_split_gemm_argument_errors(cuda_lib):
    L = cuda_lib._lib
    assert L.dbf_selftest_split_gemm(0, 1, 1, 1.0, 1, 1, 1, 1, 0.0, 1, 1, 0, None, 0, None) == \
        cuda_lib.DBF_ERR_INVALID_ARG
    assert L.dbf_selftest_split_gemm(1, 1, 70000, 1.0, 1, 70000, 1, 70000, 0.0, 1, 1, 0, None, 0, None) == \
        cuda_lib.DBF_ERR_UNSUPPORTED
    assert L.dbf_selftest_split_gemm(4, 4, 8, 1.0, 1, 4, 1, 8, 0.0, 1, 4, 0, None, 0, None) == \
        cuda_lib.DBF_ERR_INVALID_ARG  # lda < kk
    assert L.dbf_selftest_split_gemm(4, 4, 8, 1.0, 1, 8, 1, 8, 0.0, 1, 4, 0, None, 0, None) == \
        cuda_lib.DBF_ERR_WORKSPACE
    assert L.dbf_selftest_split_gemm_workspace_bytes(0, 4, 4) == 0
