"""Grouped call dbf_matmul_grouped: independent projections of different shapes (non-uniform R) in one call."""

import ctypes

import numpy as np
import pytest
import torch

from oracle import dbf_oracle as O
from tests import gpu_util as U
from workloads import generators as G

pytestmark = pytest.mark.gpu

MIXED = [(300, 200, 77), (4096, 4096, 64), (1024, 2048, 768), (257, 130, 33), (96, 160, 3072)]


def _group(shapes, ell, seed, **kw):
    fs = [G.make_factors(N, M, R, ell, seed + 17 * k, **kw) for k, (N, M, R) in enumerate(shapes)]
    return fs, [U.device_factors(f) for f in fs]


def _check(cuda_lib, fs, ys, xbs, ybs_in=None):
    st = cuda_lib.check_status()
    assert st == 0, cuda_lib.status_string(st)
    want = O.matmul_grouped(xbs, fs, ybs_in)
    for p, (y, (yref, _)) in enumerate(zip(ys, want)):
        U.assert_close(U.bf16_to_bits(y), yref, f"problem {p} ({fs[p].N}x{fs[p].M} R={fs[p].R})")


@pytest.mark.parametrize("T", [1, 5, 16])
@pytest.mark.parametrize("ell", [1, 2])
def test_grouped_decode_mixed_shapes(cuda_lib, T, ell):
    fs, dfs = _group(MIXED, ell, 3000 + T)
    xbs = [G.make_x(T, f.M, 3100 + 7 * k + T) for k, f in enumerate(fs)]
    assert cuda_lib.grouped_launch_count(dfs, T) == 2
    ys = cuda_lib.matmul_grouped(dfs, [U.bits_to_bf16(b) for b in xbs])
    _check(cuda_lib, fs, ys, xbs)


def test_grouped_decode_accumulate(cuda_lib):
    T, ell = 8, 2
    fs, dfs = _group(MIXED[:3], ell, 3200)
    xbs = [G.make_x(T, f.M, 3210 + k) for k, f in enumerate(fs)]
    ybs = [G.make_x(T, f.N, 3220 + k) for k, f in enumerate(fs)]
    ys = [U.bits_to_bf16(b).clone() for b in ybs]
    cuda_lib.matmul_grouped(dfs, [U.bits_to_bf16(b) for b in xbs], ys, accumulate=True)
    _check(cuda_lib, fs, ys, xbs, ybs)


def test_grouped_integer_mode_bit_exact(cuda_lib):
    T = 6
    shapes = [(160, 96, 40), (64, 300, 130), (257, 64, 33)]
    fs, dfs = _group(shapes, 2, 3300, unit_scales=True)
    xbs = [G.make_x(T, f.M, 3310 + k, integer=True) for k, f in enumerate(fs)]
    ys = cuda_lib.matmul_grouped(dfs, [U.bits_to_bf16(b) for b in xbs])
    assert cuda_lib.check_status() == 0
    for y, (_, bits) in zip(ys, O.matmul_grouped(xbs, fs)):
        assert np.array_equal(U.bf16_to_bits(y), bits)


def test_grouped_prefill_runs_each_problem(cuda_lib):
    T = 40
    fs, dfs = _group(MIXED[:4], 2, 3400)
    xbs = [G.make_x(T, f.M, 3410 + k) for k, f in enumerate(fs)]
    assert cuda_lib.grouped_launch_count(dfs, T) == 3 * 4
    ys = cuda_lib.matmul_grouped(dfs, [U.bits_to_bf16(b) for b in xbs])
    _check(cuda_lib, fs, ys, xbs)


@pytest.mark.parametrize("T", [3, 33])
def test_grouped_writes_nothing_past_the_outputs(cuda_lib, T):
    fs, dfs = _group(MIXED[:3] + [(257, 130, 33)], 1, 3500 + T)
    xbs = [G.make_x(T, f.M, 3510 + k) for k, f in enumerate(fs)]
    bufs = [torch.full((T + 1, f.N), 7.0, dtype=torch.bfloat16, device="cuda") for f in fs]
    ys = [b[:T] for b in bufs]
    cuda_lib.matmul_grouped(dfs, [U.bits_to_bf16(b) for b in xbs], ys)
    _check(cuda_lib, fs, ys, xbs)
    for b in bufs:
        assert bool((b[T:] == 7.0).all())


def test_grouped_rejects_bad_arguments(cuda_lib):
    fs, dfs = _group(MIXED[:2], 1, 3600)
    f3 = U.device_factors(G.make_factors(64, 64, 16, 2, 3601))
    x = [torch.zeros((4, f.M), dtype=torch.bfloat16, device="cuda") for f in dfs]
    with pytest.raises(cuda_lib.DbfError) as e:
        cuda_lib.matmul_grouped(dfs + [f3], x + [torch.zeros((4, 64), dtype=torch.bfloat16, device="cuda")])
    assert e.value.code == -1  # mixed ell: invalid argument
    with pytest.raises(cuda_lib.DbfError) as e:
        cuda_lib.matmul_grouped([dfs[0]] * 17, [x[0]] * 17)
    assert e.value.code == -3  # more than 16 problems: unsupported
    structs = (cuda_lib.DbfFactors * 2)(dfs[0].struct, dfs[1].struct)
    assert cuda_lib._lib.dbf_matmul_grouped(structs, 0, None, None, 4, 0, None, 0, None) == -1
    # a misaligned x
    xb = torch.zeros((4 * dfs[0].M + 8,), dtype=torch.bfloat16, device="cuda")
    xp = (ctypes.c_void_p * 2)(xb.data_ptr() + 2, x[1].data_ptr())
    y = [torch.zeros((4, f.N), dtype=torch.bfloat16, device="cuda") for f in dfs]
    yp = (ctypes.c_void_p * 2)(*[t.data_ptr() for t in y])
    ws = cuda_lib.new_workspace(cuda_lib.grouped_workspace_bytes(dfs, 4), "cuda")
    assert cuda_lib._lib.dbf_matmul_grouped(structs, 2, xp, yp, 4, 0, cuda_lib._ptr(ws), ws.numel(), None) == -2


def test_grouped_qkv_full_size_sampled(cuda_lib):
    # q, k, v of a 4096-wide block with grouped-query heads, each at its own middle dimension
    T = 8
    shapes = [(4096, 4096, 3072), (1024, 4096, 1536), (1024, 4096, 2048)]
    fs, dfs = _group(shapes, 1, 3700)
    xb = G.make_x(T, 4096, 3710)
    x = U.bits_to_bf16(xb)
    ys = cuda_lib.matmul_grouped(dfs, [x, x, x])
    assert cuda_lib.check_status() == 0
    rng = np.random.default_rng(3720)
    for p, (f, y) in enumerate(zip(fs, ys)):
        outs = np.sort(rng.choice(f.N, 96, replace=False))
        ref = O.y_sampled(O.bf16_bits_to_f64(xb), f, list(range(T)), outs)
        U.assert_close(U.bf16_to_bits(y)[:, outs], ref, f"qkv problem {p} sampled")
