"""Backward pass dbf_backward: dx and the scale gradients dalpha, dbeta, dgamma against the oracle."""

import ctypes

import numpy as np
import pytest
import torch

from oracle import dbf_oracle as O
from tests import gpu_util as U
from workloads import configs as C
from workloads import generators as G

pytestmark = pytest.mark.gpu

# Tolerance of the fp32 scale gradients against the exact float64 ones: relative Frobenius error
# <= 2e-3 and max|err| <= 1e-2 * max|ref|.  The error comes from the fp16 intermediates (gamma*x,
# beta*h, h, alpha*dy, beta*g: at most three 2^-11 roundings on any path, RMS about 5e-4); the fp32
# accumulation over tokens adds ~1e-7 relative.
GRAD_FROB = 2e-3
GRAD_MAX = 1e-2


def _grad_close(got, want, what):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert np.isfinite(got).all(), f"{what}: non-finite"
    scale = np.abs(want).max()
    max_rel = np.abs(got - want).max() / scale if scale > 0 else np.abs(got).max()
    frob = O.rel_frobenius(got, want)
    assert frob <= GRAD_FROB and max_rel <= GRAD_MAX, f"{what}: frob={frob:.3e} max_rel={max_rel:.3e}"


def _run(cuda_lib, f, xb, dyb, want_dx=True):
    df = U.device_factors(f)
    ft = cuda_lib.TransposedFactors(df)
    dx, da, db, dg = cuda_lib.backward(df, ft, U.bits_to_bf16(xb), U.bits_to_bf16(dyb), dx=want_dx)
    st = cuda_lib.check_status()
    assert st == 0, cuda_lib.status_string(st)
    out = [None if dx is None else U.bf16_to_bits(dx)]
    out += [t.cpu().numpy().astype(np.float64) for t in (da, db, dg)]
    return out


def test_backward_integer_mode_bit_exact(cuda_lib):
    # unit scales and integer x, dy in [-4, 4]: every intermediate is an integer small enough for
    # fp16 and every partial sum stays below 2^24, so fp32 atomics in any order give the exact sums
    f = G.make_factors(128, 96, 40, 2, 2300, unit_scales=True)
    xb = G.make_x(64, 96, 2301, integer=True)
    dyb = G.make_x(64, 128, 2302, integer=True)
    dx, da, db, dg = _run(cuda_lib, f, xb, dyb)
    wa, wb, wg = O.scale_grads(xb, dyb, f)
    assert np.array_equal(da, wa) and np.array_equal(db, wb) and np.array_equal(dg, wg)
    _, want_dx = O.matmul_dx(dyb, f)
    assert np.array_equal(dx, want_dx)


@pytest.mark.parametrize("N,M,R,ell,T", [
    (300, 200, 77, 2, 300), (512, 384, 256, 1, 513), (96, 160, 40, 4, 70), (257, 130, 33, 3, 7),
    (160, 96, 40, 2, 1), (4096, 4096, 64, 1, 16), (1024, 2048, 768, 2, 40), (96, 2050, 1030, 2, 2048),
    (257, 64, 2050, 4, 3000)])
def test_backward_matches_oracle(cuda_lib, N, M, R, ell, T):
    f = G.make_factors(N, M, R, ell, 2400 + N + T)
    xb = G.make_x(T, M, 2410 + T)
    dyb = G.make_x(T, N, 2420 + T)
    dx, da, db, dg = _run(cuda_lib, f, xb, dyb)
    wa, wb, wg = O.scale_grads(xb, dyb, f)
    _grad_close(da, wa, f"dalpha {N}x{M} R={R} ell={ell} T={T}")
    _grad_close(db, wb, f"dbeta {N}x{M} R={R} ell={ell} T={T}")
    _grad_close(dg, wg, f"dgamma {N}x{M} R={R} ell={ell} T={T}")
    want_dx, _ = O.matmul_dx(dyb, f)
    U.assert_close(dx, want_dx, f"dx {N}x{M} R={R} ell={ell} T={T}")


def test_backward_without_dx_and_with_zero_tokens(cuda_lib):
    f = G.make_factors(300, 200, 77, 2, 2500)
    xb = G.make_x(50, 200, 2501)
    dyb = G.make_x(50, 300, 2502)
    dx, da, db, dg = _run(cuda_lib, f, xb, dyb, want_dx=False)
    assert dx is None
    wa, wb, wg = O.scale_grads(xb, dyb, f)
    _grad_close(da, wa, "dalpha (no dx)")
    _grad_close(db, wb, "dbeta (no dx)")
    _grad_close(dg, wg, "dgamma (no dx)")
    # T = 0: the gradients are overwritten with zeros
    df = U.device_factors(f)
    ft = cuda_lib.TransposedFactors(df)
    bufs = [torch.full((2, n), 5.0, dtype=torch.float32, device="cuda") for n in (300, 77, 200)]
    rc = cuda_lib._lib.dbf_backward(ctypes.byref(df.struct), ctypes.byref(ft.struct), None, None, 0, None,
                                    *(cuda_lib._ptr(b) for b in bufs), None, 0, None)
    assert rc == 0
    torch.cuda.synchronize()
    assert all(bool((b == 0).all()) for b in bufs)


def test_backward_writes_nothing_past_its_outputs(cuda_lib):
    N, M, R, ell, T = 257, 130, 33, 3, 20
    f = G.make_factors(N, M, R, ell, 2600)
    xb = G.make_x(T, M, 2601)
    dyb = G.make_x(T, N, 2602)
    df = U.device_factors(f)
    ft = cuda_lib.TransposedFactors(df)
    pad = 64
    sizes = (ell * N, ell * R, ell * M)
    bufs = [torch.full((n + pad,), 7.0, dtype=torch.float32, device="cuda") for n in sizes]
    dxbuf = torch.full((T * M + pad,), 7.0, dtype=torch.bfloat16, device="cuda")
    ws = cuda_lib.new_workspace(cuda_lib.backward_workspace_bytes(df, T), "cuda")
    x = U.bits_to_bf16(xb)
    dy = U.bits_to_bf16(dyb)
    rc = cuda_lib._lib.dbf_backward(ctypes.byref(df.struct), ctypes.byref(ft.struct), cuda_lib._ptr(x),
                                    cuda_lib._ptr(dy), T, cuda_lib._ptr(dxbuf),
                                    *(cuda_lib._ptr(b) for b in bufs), cuda_lib._ptr(ws), ws.numel(), None)
    assert rc == 0
    assert cuda_lib.check_status() == 0
    for b, n in zip(bufs, sizes):
        assert bool((b[n:] == 7.0).all())
    assert bool((dxbuf[T * M:] == 7.0).all())
    wa, wb, wg = O.scale_grads(xb, dyb, f)
    for b, n, w, name in zip(bufs, sizes, (wa, wb, wg), ("dalpha", "dbeta", "dgamma")):
        _grad_close(b[:n].cpu().numpy().reshape(w.shape), w, name + " (raw call)")


def test_backward_rejects_mismatched_transpose(cuda_lib):
    f = G.make_factors(96, 64, 40, 1, 2700)
    g = G.make_factors(64, 96, 40, 1, 2701)
    df = U.device_factors(f)
    dg = U.device_factors(g)
    ft_wrong = cuda_lib.TransposedFactors(dg)  # transposed descriptor of another shape (N'=96, M'=64)
    x = torch.zeros((4, 64), dtype=torch.bfloat16, device="cuda")
    dy = torch.zeros((4, 96), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(cuda_lib.DbfError):
        cuda_lib.backward(df, ft_wrong, x, dy)


def test_backward_mlp_up_projection_full_size_sampled(cuda_lib):
    p = C.DBF_MLP.projections[0]
    T = C.DBF_MLP.tokens[0]
    f = G.make_factors(p.N, p.M, p.R, p.ell, p.seed)
    xb = G.make_x(T, p.M, p.seed + 11)
    dyb = G.make_x(T, p.N, p.seed + 12)
    dx, da, db, dg = _run(cuda_lib, f, xb, dyb)
    rng = np.random.default_rng(2800)
    n_idx = np.sort(rng.choice(p.N, 64, replace=False))
    r_idx = np.sort(rng.choice(p.R, 64, replace=False))
    k_idx = np.sort(rng.choice(p.M, 64, replace=False))
    wa, wb, wg = O.scale_grads_sampled(O.bf16_bits_to_f64(xb), O.bf16_bits_to_f64(dyb), f, n_idx, r_idx, k_idx)
    _grad_close(da[:, n_idx], wa, "dalpha mlp up sampled")
    _grad_close(db[:, r_idx], wb, "dbeta mlp up sampled")
    _grad_close(dg[:, k_idx], wg, "dgamma mlp up sampled")
    toks = U.tile_boundary_tokens(T, p.ell)
    U.assert_close(dx[toks], O.dx_factored(O.bf16_bits_to_f64(dyb[toks]), f), "dx mlp up sampled rows")
