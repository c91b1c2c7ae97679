"""The decode path's two stages in one cooperative launch (dbf_selftest_decode_one_launch).

The comparison arm of the two-launch decode (stage 1 writes V, stage 2 reads
it): the same stage code behind a grid-wide barrier.  Checked against the fp64
oracle, bit for bit against dbf_matmul_path(DECODE) where that call takes the
two launches (R > 256), over repeated calls that reuse one barrier pair, and
for its argument errors.
"""

import ctypes

import numpy as np
import pytest
import torch

from oracle import dbf_oracle as O
from tests import gpu_util as U
from workloads import configs as C
from workloads import generators as G

pytestmark = pytest.mark.gpu


def _run(cuda_lib, f, xb, barrier, y_in=None):
    df = U.device_factors(f)
    x = U.bits_to_bf16(xb)
    T = xb.shape[0]
    ybuf = torch.full((T + 2, f.N), float("nan"), dtype=torch.bfloat16, device="cuda")
    ybuf[T:] = 7.0
    y = ybuf[:T]
    if y_in is not None:
        y.copy_(U.bits_to_bf16(y_in))
    cuda_lib.selftest_decode_one_launch(df, x, barrier, y, accumulate=y_in is not None)
    assert cuda_lib.check_status() == 0
    assert bool((ybuf[T:] == 7.0).all()), "wrote past the output"
    return U.bf16_to_bits(y), df, x


def _two_launch(cuda_lib, df, x, y_in=None):
    y = torch.empty((x.shape[0], df.N), dtype=torch.bfloat16, device="cuda")
    if y_in is not None:
        y.copy_(U.bits_to_bf16(y_in))
    cuda_lib.matmul_path(df, x, y, accumulate=y_in is not None, path=cuda_lib.PATH_DECODE)
    assert cuda_lib.check_status() == 0
    return U.bf16_to_bits(y)


@pytest.mark.parametrize("T", [1, 8, 16])
def test_one_launch_dbf_1p5_bits(cuda_lib, T):
    w = C.DBF_1P5
    p = w.projections[0]
    f = G.make_factors(p.N, p.M, p.R, p.ell, p.seed)
    xb = G.make_x(T, p.M, p.seed, outlier_scale=w.outlier_scale)
    bar = torch.zeros(2, dtype=torch.int32, device="cuda")
    got, df, x = _run(cuda_lib, f, xb, bar)
    y, _ = O.matmul(xb, f)
    U.assert_close(got, y, f"one-launch dbf1p5 T={T}")
    assert np.array_equal(got, _two_launch(cuda_lib, df, x))
    assert bar.cpu().tolist() == [1024, 0]  # one call advances the arrival counter by 1024


# plans covered: stage 2 without a K split in a cluster launch (300 x 520), stage 1 without one
# (4096 x 1000), 4 and 8 column tiles, 8-CTA clusters, a grid larger than stage 1's
@pytest.mark.parametrize("N,M,R,ell,T", [
    (300, 520, 300, 2, 5), (4096, 1000, 2000, 1, 3), (1000, 777, 1025, 3, 16), (2048, 3000, 700, 2, 12),
    (512, 8192, 1500, 1, 7)])
def test_one_launch_odd_shapes(cuda_lib, N, M, R, ell, T):
    f = G.make_factors(N, M, R, ell, N + 3 * M + R)
    xb = G.make_x(T, M, N + R)
    y_in = G.make_x(T, N, N + R + 1)
    bar = torch.zeros(2, dtype=torch.int32, device="cuda")
    try:
        got, df, x = _run(cuda_lib, f, xb, bar, y_in=y_in)
    except cuda_lib.DbfError as e:
        # a shape whose two stage plans differ in cluster size or rows per CTA has no one-launch form
        if e.code != cuda_lib.DBF_ERR_UNSUPPORTED:
            raise
        pytest.skip(f"no one-launch plan: {cuda_lib.last_cuda_error()}")
    y, _ = O.matmul(xb, f, y_in_bits=y_in)
    U.assert_close(got, y, f"one-launch {N}x{M} R={R} ell={ell} T={T}")
    assert np.array_equal(got, _two_launch(cuda_lib, df, x, y_in=y_in))


def test_one_launch_unsupported_plan(cuda_lib):
    # 257 x 4100, R = 640, ell = 4, T = 4: stage 1 splits K over 8 CTAs, stage 2 over 4
    f = G.make_factors(257, 4100, 640, 4, 11)
    bar = torch.zeros(2, dtype=torch.int32, device="cuda")
    with pytest.raises(cuda_lib.DbfError) as ei:
        _run(cuda_lib, f, G.make_x(4, 4100, 12), bar)
    assert ei.value.code == cuda_lib.DBF_ERR_UNSUPPORTED
    assert "cluster" in cuda_lib.last_cuda_error()
    assert bar.cpu().tolist() == [0, 0]


def test_one_launch_integer_mode_bit_exact(cuda_lib):
    f = G.make_factors(640, 1024, 512, 2, 77, unit_scales=True)
    xb = G.make_x(8, 1024, 78, integer=True)
    bar = torch.zeros(2, dtype=torch.int32, device="cuda")
    got, _, _ = _run(cuda_lib, f, xb, bar)
    _, want = O.matmul(xb, f)
    assert np.array_equal(got, want)


def test_one_launch_barrier_reuse(cuda_lib):
    # 24 calls on one barrier pair, streamed back to back: the same bits every call and the
    # arrival counter at 24 * 1024
    w = C.DBF_1P5
    p = w.projections[0]
    f = G.make_factors(p.N, p.M, p.R, p.ell, p.seed)
    df = U.device_factors(f)
    x = U.bits_to_bf16(G.make_x(8, p.M, p.seed + 5, outlier_scale=w.outlier_scale))
    bar = torch.zeros(2, dtype=torch.int32, device="cuda")
    ys = [torch.empty((8, p.N), dtype=torch.bfloat16, device="cuda") for _ in range(24)]
    for y in ys:
        cuda_lib.selftest_decode_one_launch(df, x, bar, y)
    torch.cuda.synchronize()
    assert cuda_lib.check_status() == 0
    assert bar.cpu().tolist() == [24 * 1024, 0]
    for y in ys[1:]:
        assert torch.equal(y.view(torch.int16), ys[0].view(torch.int16))


def test_one_launch_argument_errors(cuda_lib):
    L = cuda_lib._lib
    f = G.make_factors(300, 520, 300, 1, 5)
    df = U.device_factors(f)
    x = U.bits_to_bf16(G.make_x(4, 520, 6))
    y = torch.empty((4, 300), dtype=torch.bfloat16, device="cuda")
    ws = cuda_lib.new_workspace(cuda_lib.workspace_bytes(df, 4, cuda_lib.PATH_DECODE), "cuda")
    bar = torch.zeros(4, dtype=torch.int32, device="cuda")
    args = (ctypes.byref(df.struct), x.data_ptr(), 4, y.data_ptr(), 0, ws.data_ptr(), ws.numel())
    s = None
    assert L.dbf_selftest_decode_one_launch(*args, None, s) == cuda_lib.DBF_ERR_INVALID_ARG
    assert L.dbf_selftest_decode_one_launch(*args, bar.data_ptr() + 4, s) == cuda_lib.DBF_ERR_INVALID_ARG
    x17 = U.bits_to_bf16(G.make_x(17, 520, 7))
    y17 = torch.empty((17, 300), dtype=torch.bfloat16, device="cuda")
    ws17 = cuda_lib.new_workspace(cuda_lib.workspace_bytes(df, 17, cuda_lib.PATH_DECODE), "cuda")
    assert L.dbf_selftest_decode_one_launch(ctypes.byref(df.struct), x17.data_ptr(), 17, y17.data_ptr(), 0,
                                            ws17.data_ptr(), ws17.numel(), bar.data_ptr(), s) == \
        cuda_lib.DBF_ERR_INVALID_ARG
    assert L.dbf_selftest_decode_one_launch(*args[:5], ws.data_ptr(), 16, bar.data_ptr(), s) == \
        cuda_lib.DBF_ERR_WORKSPACE
    bad_acc = args[:4] + (2,) + args[5:]
    assert L.dbf_selftest_decode_one_launch(*bad_acc, bar.data_ptr(), s) == cuda_lib.DBF_ERR_INVALID_ARG
    # T = 0: nothing to do, not even a launch
    assert L.dbf_selftest_decode_one_launch(ctypes.byref(df.struct), x.data_ptr(), 0, y.data_ptr(), 0, None, 0,
                                            bar.data_ptr(), s) == cuda_lib.DBF_OK
    torch.cuda.synchronize()
    assert bar.cpu().tolist() == [0, 0, 0, 0]
    assert cuda_lib.check_status() == 0
