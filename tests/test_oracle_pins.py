"""Pins for the fp64 oracle: facts fixed by the pages and by mathematics.

Every check here compares the oracle with something other than itself: a
hand-derived fixture, a closed form that holds only for special factors, a
symmetry of the product, an exact integer computation, a scalar brute-force
loop, or an independent library conversion.
"""

import json
import os

import numpy as np
import pytest

from oracle import dbf_oracle as O
from workloads import generators as G
from workloads.generators import Factors


def _factors_from_lists(c):
    return Factors(np.asarray(c["B1"], dtype=np.int8), np.asarray(c["B2"], dtype=np.int8),
                   np.asarray(c["alpha"], dtype=np.float16), np.asarray(c["beta"], dtype=np.float16),
                   np.asarray(c["gamma"], dtype=np.float16))


# ----------------------------------------------------------------- packing

def test_golden_pack_format(golden_dir):
    with open(os.path.join(golden_dir, "pack_format.json")) as fh:
        cases = json.load(fh)["cases"]
    for c in cases:
        signs = np.asarray([[1 if ch == "+" else -1 for ch in c["signs"]]], dtype=np.int8)
        assert signs.shape[1] == c["cols"]
        want = np.asarray([[int(w, 16) for w in c["words"]]], dtype=np.uint32)
        got = O.pack_signs(signs, c["ldw"])
        assert got.dtype == np.uint32
        assert np.array_equal(got, want), c["name"]
        assert np.array_equal(O.unpack_words(got, c["cols"]), signs), c["name"]


@pytest.mark.parametrize("rows,cols,extra", [(1, 1, 0), (3, 31, 0), (5, 32, 3), (7, 33, 1), (16, 257, 4), (9, 5013, 0)])
def test_pack_roundtrip_and_popcount(rows, cols, extra):
    rng = np.random.default_rng(rows * 1000 + cols)
    s = np.where(rng.random((rows, cols)) < 0.5, 1, -1).astype(np.int8)
    ldw = O.words_per_row(cols) + extra
    w = O.pack_signs(s, ldw)
    assert w.shape == (rows, ldw)
    assert np.array_equal(O.unpack_words(w, cols), s)
    # popcount of a row = number of +1 entries
    pop = np.array([sum(bin(int(v)).count("1") for v in row) for row in w])
    assert np.array_equal(pop, (s > 0).sum(axis=1))
    # bits past the last column are zero
    full = O.unpack_words(w, ldw * 32)
    assert (full[:, cols:] == -1).all()


def test_pack_maps_positive_to_one_and_zero_to_zero_bit():
    s = np.array([[3, 0, -2, 1, 127, -128]], dtype=np.int8)
    w = O.pack_signs(s)
    # bit 1 only where the entry is > 0: columns 0, 3, 4
    assert int(w[0, 0]) == (1 << 0) | (1 << 3) | (1 << 4)


# --------------------------------------------------------- bf16 rounding

def test_bf16_rounding_matches_library_conversion_on_float32_values():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(7)
    vals = np.concatenate([
        rng.standard_normal(20000).astype(np.float32),
        (rng.standard_normal(20000) * 1e-39).astype(np.float32),   # bf16 subnormals
        (rng.standard_normal(2000) * 1e38).astype(np.float32),     # near overflow
        # exact ties: 8 significant bits plus a trailing half-ulp
        np.ldexp(rng.integers(128, 256, 4000) * 2 + 1, rng.integers(-20, 20, 4000) - 9).astype(np.float32),
        np.array([0.0, -0.0, 1.0, -1.0, 65504.0, 3.3895313892515355e38], dtype=np.float32),
    ])
    got = O.round_to_bf16_bits(vals.astype(np.float64))
    want = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, want)


def test_bf16_rounding_is_single_step_from_float64():
    # 1 + 2^-8 + 2^-40 is above the tie between 1 and 1 + 2^-7; a route through
    # float32 would first drop 2^-40, land on the tie and round to even (down).
    v = np.array([1.0 + 2.0 ** -8 + 2.0 ** -40, 1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8])
    assert list(O.round_to_bf16_bits(v)) == [0x3F81, 0x3F80, 0x3F82]


# ------------------------------------------------- hand-derived products

def test_golden_small_products(golden_dir):
    with open(os.path.join(golden_dir, "small_products.json")) as fh:
        cases = json.load(fh)["cases"]
    for c in cases:
        f = _factors_from_lists(c)
        x = np.asarray(c["x"], dtype=np.float64)
        want = np.asarray(c["y"], dtype=np.float64)
        for route in (O.y_factored, O.y_dense, O.y_bruteforce):
            got = route(x, f)
            assert np.array_equal(got, want), (c["name"], route.__name__, got)


# -------------------------------------------- two pages, same product

@pytest.mark.parametrize("N,M,R,ell,seed", [(8, 8, 4, 1, 1), (37, 19, 11, 1, 2), (64, 48, 33, 2, 3), (16, 40, 7, 3, 4)])
def test_dense_route_equals_factored_route(N, M, R, ell, seed):
    f = G.make_factors(N, M, R, ell, seed)
    x = O.bf16_bits_to_f64(G.make_x(5, M, seed))
    a = O.y_dense(x, f)
    b = O.y_factored(x, f)
    assert O.rel_frobenius(a, b) < 1e-12


@pytest.mark.parametrize("ell", [1, 2])
def test_bruteforce_tiny(ell):
    f = G.make_factors(8, 8, 4, ell, 10 + ell)
    x = O.bf16_bits_to_f64(G.make_x(3, 8, 10 + ell))
    bf = O.y_bruteforce(x, f)
    assert O.rel_frobenius(O.y_factored(x, f), bf) < 1e-12
    assert O.rel_frobenius(O.y_dense(x, f), bf) < 1e-12


@pytest.mark.parametrize("ell", [1, 2])
def test_bruteforce_tiny_integer_mode_exact(ell):
    f = G.make_factors(8, 8, 4, ell, 20 + ell, unit_scales=True)
    x = O.bf16_bits_to_f64(G.make_x(4, 8, 20 + ell, integer=True))
    bf = O.y_bruteforce(x, f)
    assert np.array_equal(O.y_factored(x, f), bf)
    assert np.array_equal(O.y_dense(x, f), bf)


# --------------------------------------------------------- closed forms

@pytest.mark.parametrize("ell", [1, 2])
def test_all_ones_signs_collapse_to_rank_one(ell):
    N, M, R = 24, 40, 9
    f = G.make_factors(N, M, R, ell, 30 + ell)
    x = O.bf16_bits_to_f64(G.make_x(6, M, 30 + ell))
    a64, b64, g64 = (O.fp16_to_f64(v) for v in (f.alpha, f.beta, f.gamma))

    def closed(sign):
        y = np.zeros((x.shape[0], N))
        for i in range(ell):
            y += sign * np.outer(x @ g64[i], a64[i]) * b64[i].sum()
        return y

    ones = Factors(np.ones((N, R), np.int8), np.ones((R, M), np.int8), f.alpha, f.beta, f.gamma)
    neg = Factors(-np.ones((N, R), np.int8), -np.ones((R, M), np.int8), f.alpha, f.beta, f.gamma)
    flip1 = Factors(-np.ones((N, R), np.int8), np.ones((R, M), np.int8), f.alpha, f.beta, f.gamma)
    assert O.rel_frobenius(O.y_factored(x, ones), closed(1.0)) < 1e-13
    assert O.rel_frobenius(O.y_factored(x, neg), closed(1.0)) < 1e-13
    assert O.rel_frobenius(O.y_factored(x, flip1), closed(-1.0)) < 1e-13


def _sylvester(k):
    H = np.array([[1]], dtype=np.int64)
    for _ in range(k):
        H = np.block([[H, H], [H, -H]])
    return H


@pytest.mark.parametrize("k", [3, 5])
def test_permuted_hadamard_gives_diagonal_update(k):
    n = 2 ** k
    H = _sylvester(k)
    perm = np.random.default_rng(k).permutation(n)
    B2 = H[perm].astype(np.int8)          # P H
    B1 = B2.T.copy()                      # (P H)^T, not symmetric
    assert not np.array_equal(B1, B1.T)
    rng = np.random.default_rng(100 + k)
    alpha = (rng.integers(1, 8, (1, n)) / 4.0).astype(np.float16)
    gamma = (rng.integers(1, 8, (1, n)) / 2.0).astype(np.float16)
    beta = np.ones((1, n), dtype=np.float16)
    f = Factors(B1, B2, alpha, beta, gamma)
    x = O.bf16_bits_to_f64(G.make_x(5, n, 40 + k, integer=True))
    want = n * x * (alpha[0].astype(np.float64) * gamma[0].astype(np.float64))[None, :]
    assert np.array_equal(O.y_factored(x, f), want)
    assert np.array_equal(O.y_dense(x, f), want)


# ---------------------------------------------------------- symmetries

def test_paired_flip_leaves_output_unchanged_and_row_flip_negates():
    N, M, R, ell = 20, 30, 12, 2
    f = G.make_factors(N, M, R, ell, 50)
    x = O.bf16_bits_to_f64(G.make_x(4, M, 50))
    y = O.y_factored(x, f)
    B1 = f.B1.copy()
    B2 = f.B2.copy()
    for r in (0, 5, 11):
        B1[:, r] *= -1
        B2[r, :] *= -1
    g = Factors(B1, B2, f.alpha, f.beta, f.gamma)
    assert np.array_equal(O.y_factored(x, g), y)
    B1 = f.B1.copy()
    B1[3, :] *= -1
    h = Factors(B1, f.B2, f.alpha, f.beta, f.gamma)
    yh = O.y_factored(x, h)
    assert np.array_equal(yh[:, 3], -y[:, 3])
    assert np.array_equal(np.delete(yh, 3, axis=1), np.delete(y, 3, axis=1))


def test_linear_in_x_and_in_each_scale():
    N, M, R, ell = 16, 24, 10, 2
    f = G.make_factors(N, M, R, ell, 60)
    x1 = O.bf16_bits_to_f64(G.make_x(3, M, 61))
    x2 = O.bf16_bits_to_f64(G.make_x(3, M, 62))
    y = O.y_factored
    assert O.rel_frobenius(y(2 * x1 - 3 * x2, f), 2 * y(x1, f) - 3 * y(x2, f)) < 1e-13
    base = y(x1, f)
    # scaling term 0's alpha, beta or gamma by 2 adds exactly term 0 once more
    only0 = Factors(f.B1, f.B2, f.alpha[:1], f.beta[:1], f.gamma[:1])
    t0 = y(x1, only0)
    for name in ("alpha", "beta", "gamma"):
        s = {k: getattr(f, k).copy() for k in ("alpha", "beta", "gamma")}
        s[name][0] = (s[name][0].astype(np.float64) * 2).astype(np.float16)
        g = Factors(f.B1, f.B2, s["alpha"], s["beta"], s["gamma"])
        assert O.rel_frobenius(y(x1, g), base + t0) < 1e-13, name


# ------------------------------------------------ exact integer results

def test_integer_mode_matches_exact_integer_arithmetic():
    f = G.make_factors(256, 256, 32, 1, 0, "gauss", "tiny", unit_scales=True)
    xb = G.make_x(8, 256, 0, integer=True)
    x_int = O.bf16_bits_to_f64(xb).astype(np.int64)
    # exact integer route: u = B2 x, y = B1 u, in int64
    u = x_int @ f.B2.astype(np.int64).T
    y_int = u @ f.B1.astype(np.int64).T
    y64, bits = O.matmul(xb, f)
    assert np.array_equal(y64, y_int.astype(np.float64))
    assert np.abs(y_int).max() <= 4 * 256 * 32
    # every |y| <= 32768 whose magnitude needs <= 8 significant bits is exact in bf16
    small = np.abs(y_int) <= 256
    assert np.array_equal(O.bf16_bits_to_f64(bits)[small], y64[small])


# ------------------------------------------- sampled and segmented forms

def test_sampled_outputs_equal_full_result():
    f = G.make_factors(40, 50, 13, 2, 70)
    xb = G.make_x(9, 50, 70)
    x = O.bf16_bits_to_f64(xb)
    full = O.y_factored(x, f)
    toks, outs = [0, 4, 8], [1, 7, 39, 20]
    assert O.rel_frobenius(O.y_sampled(x, f, toks, outs), full[np.ix_(toks, outs)]) < 1e-14


def test_segmented_with_one_shared_adapter_equals_plain_call():
    f = G.make_factors(32, 48, 8, 2, 80)
    xb = G.make_x(12, 48, 80)
    off = np.array([0, 3, 3, 7, 12], dtype=np.int32)   # includes an empty segment
    ad = np.array([0, 1, 0, 1], dtype=np.int32)
    y_seg, b_seg = O.matmul_segmented(xb, [f, f], off, ad)
    y, b = O.matmul(xb, f)
    assert O.rel_frobenius(y_seg, y) < 1e-14


def test_segmented_routes_each_token_to_its_adapter():
    fa = G.make_factors(16, 24, 8, 1, 81)
    fb = G.make_factors(16, 24, 8, 1, 82)
    xb = G.make_x(6, 24, 83)
    off = np.array([0, 2, 6], dtype=np.int32)
    ad = np.array([1, 0], dtype=np.int32)
    y_seg, _ = O.matmul_segmented(xb, [fa, fb], off, ad)
    ya, _ = O.matmul(xb, fa)
    yb, _ = O.matmul(xb, fb)
    assert np.array_equal(y_seg[:2], yb[:2])
    assert np.array_equal(y_seg[2:], ya[2:])


def test_accumulate_mode_adds_before_single_rounding():
    f = G.make_factors(16, 16, 4, 1, 90)
    xb = G.make_x(2, 16, 90)
    y_in = G.make_x(2, 16, 91)
    y64, bits = O.matmul(xb, f, y_in)
    branch, _ = O.matmul(xb, f)
    assert np.array_equal(y64, branch + O.bf16_bits_to_f64(y_in))
    assert np.array_equal(bits, O.round_to_bf16_bits(y64))


# ---------------------------------------------------------- backward (dx)

def test_transpose_packed_matches_transposed_signs_and_round_trips():
    rng = np.random.default_rng(41)
    for rows, cols, extra in [(1, 1, 0), (33, 70, 1), (64, 32, 0), (5, 200, 3)]:
        s = np.where(rng.random((rows, cols)) < 0.5, 1, -1).astype(np.int8)
        w = O.pack_signs(s)
        wt = O.transpose_packed(w, cols, O.words_per_row(rows) + extra)
        assert np.array_equal(O.unpack_words(wt, rows), s.T)
        assert np.array_equal(O.transpose_packed(wt, rows, O.words_per_row(cols)), w)


def test_transpose_packed_golden_word():
    # a 32 x 32 block with only row 3 all +1: the transpose has bit 3 set in every word
    s = -np.ones((32, 32), dtype=np.int8)
    s[3, :] = 1
    wt = O.transpose_packed(O.pack_signs(s), 32)
    assert (wt[:, 0] == np.uint32(1 << 3)).all()


@pytest.mark.parametrize("N,M,R,ell,seed", [(8, 8, 4, 1, 5), (40, 24, 9, 2, 6), (17, 33, 12, 3, 7)])
def test_dx_equals_dy_times_dense_update(N, M, R, ell, seed):
    f = G.make_factors(N, M, R, ell, seed)
    dy = np.random.default_rng(seed).standard_normal((5, N))
    np.testing.assert_allclose(O.dx_factored(dy, f), dy @ O.dense_delta_w(f), rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("ell", [1, 2, 4])
def test_adjoint_identity(ell):
    # <x dW^T, dy> = <x, dy dW> for any x and dy: the backward product is the adjoint of the forward one
    f = G.make_factors(30, 20, 7, ell, 60 + ell)
    rng = np.random.default_rng(70 + ell)
    x = rng.standard_normal((6, 20))
    dy = rng.standard_normal((6, 30))
    lhs = float((O.y_factored(x, f) * dy).sum())
    rhs = float((x * O.dx_factored(dy, f)).sum())
    assert abs(lhs - rhs) <= 1e-12 * max(1.0, abs(lhs))


def test_dx_is_the_forward_product_of_the_transposed_factors():
    # the library computes dx with its forward kernels on (B2^T, B1^T, gamma, beta, alpha)
    f = G.make_factors(24, 40, 10, 2, 80)
    ft = Factors(np.ascontiguousarray(f.B2.T), np.ascontiguousarray(f.B1.T), f.gamma, f.beta, f.alpha)
    dy = np.random.default_rng(81).standard_normal((3, 24))
    np.testing.assert_allclose(O.y_factored(dy, ft), O.dx_factored(dy, f), rtol=1e-12, atol=1e-12)


def test_dx_bruteforce_tiny():
    f = G.make_factors(8, 8, 4, 2, 90)
    dy = np.random.default_rng(91).standard_normal((2, 8))
    alpha, beta, gamma = (O.fp16_to_f64(a) for a in (f.alpha, f.beta, f.gamma))
    want = np.zeros((2, 8))
    for t in range(2):
        for m in range(8):
            for i in range(2):
                for r in range(4):
                    for n in range(8):
                        want[t, m] += gamma[i, m] * f.B2[r, m] * beta[i, r] * f.B1[n, r] * alpha[i, n] * dy[t, n]
    np.testing.assert_allclose(O.dx_factored(dy, f), want, rtol=1e-12, atol=1e-12)


# ------------------------------------------------------ scale gradients

def _loss_dense(x, dy, f):
    # L = sum_t <dy_t, y_t> through the dense route (dW built explicitly)
    return float((O.y_dense(x, f) * dy).sum())


def _with(f, **kw):
    d = dict(B1=f.B1, B2=f.B2, alpha=f.alpha, beta=f.beta, gamma=f.gamma)
    d.update(kw)
    return Factors(d["B1"], d["B2"], d["alpha"], d["beta"], d["gamma"])


@pytest.mark.parametrize("N,M,R,ell,seed", [(12, 9, 5, 1, 11), (30, 20, 7, 2, 12), (17, 33, 12, 3, 13)])
def test_scale_grads_are_the_directional_derivatives(N, M, R, ell, seed):
    # y is linear in each scale vector, so for a new fp16 vector s' the change of L is exactly
    # <d, s' - s> (the difference of two fp16 numbers is exact in float64)
    f = G.make_factors(N, M, R, ell, seed)
    rng = np.random.default_rng(seed + 1)
    x = rng.standard_normal((6, M))
    dy = rng.standard_normal((6, N))
    da, db, dg = O.scale_grads_f64(x, dy, f)
    L0 = _loss_dense(x, dy, f)
    for name, d in (("alpha", da), ("beta", db), ("gamma", dg)):
        old = getattr(f, name)
        new = (rng.standard_normal(old.shape) * 0.5).astype(np.float16)
        L1 = _loss_dense(x, dy, _with(f, **{name: new}))
        pred = float((d * (new.astype(np.float64) - old.astype(np.float64))).sum())
        assert abs((L1 - L0) - pred) <= 1e-10 * max(1.0, abs(L0), abs(L1)), name


@pytest.mark.parametrize("ell", [1, 2, 4])
def test_scale_grads_euler_identity_per_term(ell):
    # L is linear in alpha_i, in beta_i and in gamma_i, so <alpha_i, dalpha_i> = <beta_i, dbeta_i>
    # = <gamma_i, dgamma_i> = the share of term i in L, computed here with term i alone
    f = G.make_factors(26, 19, 8, ell, 40 + ell)
    rng = np.random.default_rng(50 + ell)
    x = rng.standard_normal((5, 19))
    dy = rng.standard_normal((5, 26))
    da, db, dg = O.scale_grads_f64(x, dy, f)
    a, b, g = (O.fp16_to_f64(v) for v in (f.alpha, f.beta, f.gamma))
    for i in range(ell):
        fi = _with(f, alpha=f.alpha[i:i + 1], beta=f.beta[i:i + 1], gamma=f.gamma[i:i + 1])
        Li = _loss_dense(x, dy, fi)
        for v, d in ((a, da), (b, db), (g, dg)):
            assert abs(float(v[i] @ d[i]) - Li) <= 1e-11 * max(1.0, abs(Li))


def test_scale_grads_all_ones_signs_closed_form():
    # B1 = B2 = all +1: B2 (gamma . x) has every entry s = gamma . x, B1^T (alpha . dy) every entry
    # p = alpha . dy, so dalpha = sum_t dy_t * sum(beta) * s_t, dbeta = sum_t p_t s_t (same for
    # every r) and dgamma = sum_t x_t * sum(beta) * p_t
    N, M, R, ell = 9, 7, 5, 2
    f = G.make_factors(N, M, R, ell, 31)
    f = _with(f, B1=np.ones((N, R), dtype=np.int8), B2=np.ones((R, M), dtype=np.int8))
    rng = np.random.default_rng(32)
    x = rng.standard_normal((4, M))
    dy = rng.standard_normal((4, N))
    da, db, dg = O.scale_grads_f64(x, dy, f)
    a, b, g = (O.fp16_to_f64(v) for v in (f.alpha, f.beta, f.gamma))
    for i in range(ell):
        s = x @ g[i]            # [T]
        p = dy @ a[i]           # [T]
        np.testing.assert_allclose(da[i], b[i].sum() * (dy * s[:, None]).sum(0), rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(db[i], np.full(R, (p * s).sum()), rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(dg[i], b[i].sum() * (x * p[:, None]).sum(0), rtol=1e-12, atol=1e-12)


def test_scale_grad_pins_catch_a_transposed_carrier(monkeypatch):
    # plant a plausible mistake in the oracle (B2 used as if it were square-transposed: the
    # dgamma path contracts with B2 reversed along r) and check that the derivative pin sees it
    f = G.make_factors(10, 10, 10, 1, 21)
    rng = np.random.default_rng(22)
    x = rng.standard_normal((3, 10))
    dy = rng.standard_normal((3, 10))
    good = O.scale_grads_f64(x, dy, f)
    bad_f = _with(f, B2=np.ascontiguousarray(f.B2[::-1]))
    real = O.scale_grads_f64

    def planted(x64, dy64, ff):
        da, db, _ = real(x64, dy64, ff)
        _, _, dg = real(x64, dy64, bad_f)
        return da, db, dg

    monkeypatch.setattr(O, "scale_grads_f64", planted)
    da, db, dg = O.scale_grads_f64(x, dy, f)
    L0 = _loss_dense(x, dy, f)
    new = (rng.standard_normal(f.gamma.shape) * 0.5).astype(np.float16)
    L1 = _loss_dense(x, dy, _with(f, gamma=new))
    pred_bad = float((dg * (new.astype(np.float64) - f.gamma.astype(np.float64))).sum())
    pred_good = float((good[2] * (new.astype(np.float64) - f.gamma.astype(np.float64))).sum())
    assert abs((L1 - L0) - pred_good) <= 1e-10 * max(1.0, abs(L0))
    assert abs((L1 - L0) - pred_bad) > 1e-6 * max(1.0, abs(L0))


def test_scale_grads_sampled_equals_full():
    f = G.make_factors(40, 28, 11, 2, 71)
    rng = np.random.default_rng(72)
    x = rng.standard_normal((7, 28))
    dy = rng.standard_normal((7, 40))
    full = O.scale_grads_f64(x, dy, f)
    n, r, k = [0, 5, 39], [10, 3], [27, 0, 13, 14]
    part = O.scale_grads_sampled(x, dy, f, n, r, k)
    for want, got, idx in zip(full, part, (n, r, k)):
        np.testing.assert_allclose(got, want[:, idx], rtol=1e-12, atol=1e-12)


def test_grouped_is_the_list_of_independent_products():
    # a group couples nothing: each entry equals the plain call on its own problem, whatever the
    # other problems are, and reordering the group reorders the results
    shapes = [(12, 9, 5, 2), (20, 33, 17, 2), (7, 4, 30, 2)]
    fs = [G.make_factors(N, M, R, ell, 90 + k) for k, (N, M, R, ell) in enumerate(shapes)]
    xs = [G.make_x(3, f.M, 95 + k) for k, f in enumerate(fs)]
    got = O.matmul_grouped(xs, fs)
    rev = O.matmul_grouped(xs[::-1], fs[::-1])[::-1]
    for (y, bits), (y2, bits2), xb, f in zip(got, rev, xs, fs):
        yd = O.y_dense(O.bf16_bits_to_f64(xb), f)
        np.testing.assert_allclose(y, yd, rtol=1e-12, atol=1e-12)
        assert np.array_equal(bits, bits2)
