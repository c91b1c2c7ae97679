"""Decode path (T <= 16 tokens, and forced for larger T) against the fp64 oracle."""

import numpy as np
import pytest
import torch

from oracle import dbf_oracle as O
from tests import gpu_util as U
from workloads import configs as C
from workloads import generators as G

pytestmark = pytest.mark.gpu


def run(cuda_lib, f, xb, path, ldw1=None, ldw2=None, y_in=None, guard=0):
    df = U.device_factors(f, ldw1, ldw2)
    x = U.bits_to_bf16(xb)
    T, N = xb.shape[0], f.N
    ybuf = torch.full((T + guard, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    if guard:
        ybuf[T:] = 7.0
    y = ybuf[:T]
    if y_in is not None:
        y.copy_(U.bits_to_bf16(y_in))
    cuda_lib.matmul_path(df, x, y, accumulate=y_in is not None, path=path)
    assert cuda_lib.check_status() == 0
    if guard:
        assert bool((ybuf[T:] == 7.0).all()), "wrote past the output"
    return U.bf16_to_bits(y)


@pytest.mark.parametrize("T", [1, 8])
def test_tiny_integer_mode_bit_exact(cuda_lib, T):
    p = C.TINY.projections[0]
    f = G.make_factors(p.N, p.M, p.R, p.ell, p.seed, p.sign_mode, p.scale_mode, unit_scales=True)
    xb = G.make_x(T, p.M, p.seed, integer=True)
    got = run(cuda_lib, f, xb, 1)
    _, want = O.matmul(xb, f)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("T", [1, 8])
def test_tiny_random(cuda_lib, T):
    p = C.TINY.projections[0]
    f = G.make_factors(p.N, p.M, p.R, p.ell, p.seed, p.sign_mode, p.scale_mode)
    xb = G.make_x(T, p.M, p.seed)
    got = run(cuda_lib, f, xb, 0, guard=3)
    y, _ = O.matmul(xb, f)
    U.assert_close(got, y, f"tiny T={T}")


@pytest.mark.parametrize("T", [1, 4, 16])
def test_adapter_4k(cuda_lib, T):
    p = C.ADAPTER_4K.projections[0]
    f = G.make_factors(p.N, p.M, p.R, p.ell, p.seed)
    xb = G.make_x(T, p.M, p.seed)
    got = run(cuda_lib, f, xb, 0)
    y, _ = O.matmul(xb, f)
    U.assert_close(got, y, f"adapter4k T={T}")


@pytest.mark.parametrize("T", [1, 8])
def test_dbf_1p5_bits(cuda_lib, T):
    w = C.DBF_1P5
    p = w.projections[0]
    f = G.make_factors(p.N, p.M, p.R, p.ell, p.seed)
    xb = G.make_x(T, p.M, p.seed, outlier_scale=w.outlier_scale)
    got = run(cuda_lib, f, xb, 0)
    y, _ = O.matmul(xb, f)
    U.assert_close(got, y, f"dbf1p5 T={T}")


@pytest.mark.parametrize("N,M,R,ell,T,pad", [
    (257, 257, 33, 1, 3, 0), (300, 200, 77, 2, 5, 3), (130, 1000, 50, 3, 7, 0), (64, 96, 1, 4, 16, 1),
    (33, 31, 640, 1, 2, 4), (512, 4100, 96, 2, 9, 0), (16, 16, 16, 1, 1, 0),
    # cluster exchange variants of the fused kernel (rows of u past round_up(R, 32), 8-row ownership)
    (1024, 2048, 130, 2, 12, 0), (2048, 4096, 96, 2, 12, 0), (4096, 8192, 256, 1, 3, 0), (3000, 4096, 64, 1, 16, 1),
    (4096, 4096, 64, 2, 16, 0)])
def test_odd_shapes(cuda_lib, N, M, R, ell, T, pad):
    f = G.make_factors(N, M, R, ell, N + M + R)
    xb = G.make_x(T, M, N + M + R)
    ldw1 = (R + 31) // 32 + pad
    ldw2 = (M + 31) // 32 + pad
    got = run(cuda_lib, f, xb, 1, ldw1, ldw2, guard=2)
    y, _ = O.matmul(xb, f)
    U.assert_close(got, y, f"odd {N}x{M} R={R} ell={ell} T={T}")


@pytest.mark.parametrize("ell", [1, 2, 3, 4])
def test_integer_mode_each_ell_bit_exact(cuda_lib, ell):
    f = G.make_factors(96, 160, 40, ell, 300 + ell, unit_scales=True)
    xb = G.make_x(6, 160, 300 + ell, integer=True)
    got = run(cuda_lib, f, xb, 1)
    _, want = O.matmul(xb, f)
    assert np.array_equal(got, want)


def test_accumulate_mode(cuda_lib):
    f = G.make_factors(200, 300, 64, 2, 410)
    xb = G.make_x(5, 300, 410)
    y_in = G.make_x(5, 200, 411)
    got = run(cuda_lib, f, xb, 1, y_in=y_in)
    y, _ = O.matmul(xb, f, y_in)
    U.assert_close(got, y, "accumulate")


@pytest.mark.parametrize("T,ell", [(40, 2), (70, 1), (17, 4)])
def test_forced_decode_many_tokens(cuda_lib, T, ell):
    f = G.make_factors(128, 256, 64, ell, 500 + T)
    xb = G.make_x(T, 256, 500 + T)
    got = run(cuda_lib, f, xb, 1, guard=1)
    y, _ = O.matmul(xb, f)
    U.assert_close(got, y, f"forced decode T={T}")


def test_decode_is_deterministic(cuda_lib):
    p = C.DBF_1P5.projections[0]
    f = G.make_factors(1024, 2048, 768, 1, 77)
    xb = G.make_x(8, 2048, 77)
    a = run(cuda_lib, f, xb, 1)
    b = run(cuda_lib, f, xb, 1)
    assert np.array_equal(a, b)
