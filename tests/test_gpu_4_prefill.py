"""Prefill path (tcgen05 GEMMs) against the fp64 oracle."""

import numpy as np
import pytest
import torch

from oracle import dbf_oracle as O
from tests import gpu_util as U
from workloads import configs as C
from workloads import generators as G

pytestmark = pytest.mark.gpu

PREFILL = 2


def run(cuda_lib, f, xb, path=PREFILL, ldw1=None, ldw2=None, y_in=None, guard=0, df=None):
    df = df or U.device_factors(f, ldw1, ldw2)
    x = U.bits_to_bf16(xb)
    T, N = xb.shape[0], f.N
    ybuf = torch.full((T + guard, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    if guard:
        ybuf[T:] = 7.0
    y = ybuf[:T]
    if y_in is not None:
        y.copy_(U.bits_to_bf16(y_in))
    cuda_lib.matmul_path(df, x, y, accumulate=y_in is not None, path=path)
    st = cuda_lib.check_status()
    assert st == 0, cuda_lib.status_string(st)
    if guard:
        assert bool((ybuf[T:] == 7.0).all()), "wrote past the output"
    return U.bf16_to_bits(y)


def test_prefill_integer_mode_bit_exact(cuda_lib):
    f = G.make_factors(256, 256, 32, 1, 1100, "gauss", "tiny", unit_scales=True)
    xb = G.make_x(256, 256, 1100, integer=True)
    got = run(cuda_lib, f, xb)
    _, want = O.matmul(xb, f)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("ell", [1, 2, 3, 4])
def test_prefill_integer_mode_each_ell(cuda_lib, ell):
    f = G.make_factors(128, 192, 40, ell, 1200 + ell, unit_scales=True)
    xb = G.make_x(100, 192, 1200 + ell, integer=True)
    got = run(cuda_lib, f, xb, guard=2)
    _, want = O.matmul(xb, f)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("N,M,R,ell,T,pad", [
    (300, 200, 77, 2, 300, 0), (257, 130, 33, 1, 257, 1), (1000, 700, 300, 3, 100, 0),
    (200, 300, 100, 4, 70, 2), (384, 512, 256, 1, 513, 0), (128, 64, 5013, 2, 20, 0)])
def test_prefill_odd_shapes(cuda_lib, N, M, R, ell, T, pad):
    f = G.make_factors(N, M, R, ell, 1300 + N)
    xb = G.make_x(T, M, 1300 + N)
    got = run(cuda_lib, f, xb, ldw1=(R + 31) // 32 + pad, ldw2=(M + 31) // 32 + pad, guard=2)
    y, _ = O.matmul(xb, f)
    U.assert_close(got, y, f"prefill {N}x{M} R={R} ell={ell} T={T}")


# Shapes that select each tile layout of the GEMMs (the launch picks 256, 240, 224 or 192 activation
# rows per tile, one or two CTAs per SM, from the shape), as (stage-1 width, stage-2 width).
@pytest.mark.parametrize("N,M,R,ell,T", [
    (96, 2050, 2050, 1, 2048),   # 256, 240
    (96, 2050, 33, 1, 17),       # 240, 192
    (96, 2050, 1030, 2, 2048),   # 256, 192
    (96, 2050, 33, 2, 17),       # 240, 192
    (96, 2050, 33, 3, 17),       # 240, 192
    (257, 64, 2050, 4, 3000),    # 192, 256
    (96, 2050, 33, 4, 17),       # 224, 192
])
def test_prefill_each_tile_layout(cuda_lib, N, M, R, ell, T):
    f = G.make_factors(N, M, R, ell, 1600 + N + T)
    xb = G.make_x(T, M, 1600 + M + T)
    got = run(cuda_lib, f, xb, path=2, guard=2)
    y, _ = O.matmul(xb, f)
    U.assert_close(got, y, f"prefill layout {N}x{M} R={R} ell={ell} T={T}")


def test_prefill_accumulate(cuda_lib):
    f = G.make_factors(256, 320, 96, 2, 1400)
    xb = G.make_x(64, 320, 1400)
    y_in = G.make_x(64, 256, 1401)
    got = run(cuda_lib, f, xb, y_in=y_in)
    y, _ = O.matmul(xb, f, y_in)
    U.assert_close(got, y, "prefill accumulate")


def test_decode_and_prefill_agree_with_oracle_on_same_inputs(cuda_lib):
    f = G.make_factors(512, 768, 200, 2, 1500)
    xb = G.make_x(16, 768, 1500)
    df = U.device_factors(f)
    a = run(cuda_lib, f, xb, path=1, df=df)
    b = run(cuda_lib, f, xb, path=2, df=df)
    y, _ = O.matmul(xb, f)
    U.assert_close(a, y, "decode")
    U.assert_close(b, y, "prefill")


@pytest.mark.parametrize("proj", [0, 1])
def test_dbf_mlp_full_size_sampled(cuda_lib, proj):
    w = C.DBF_MLP
    p = w.projections[proj]
    T = w.tokens[0]
    f = G.make_factors(p.N, p.M, p.R, p.ell, p.seed)
    xb = G.make_x(T, p.M, p.seed)
    got = run(cuda_lib, f, xb)
    y_all = O.bf16_bits_to_f64(got)
    assert np.isfinite(y_all).all()
    toks = U.tile_boundary_tokens(T, p.ell)
    ref = O.y_sampled(O.bf16_bits_to_f64(xb), f, toks, np.arange(p.N))
    U.assert_close(got[toks], ref, f"dbf mlp {p.name} sampled rows")
