"""Host-memory entry points: dbf_matmul_hostio and the pipelined dbf_matmul_hostio_batch, against the oracle."""

import numpy as np
import pytest
import torch

from oracle import dbf_oracle as O
from tests import gpu_util as U
from workloads import generators as G

pytestmark = pytest.mark.gpu


def _host_bf16(bits, pinned=True):
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
    return t.pin_memory() if pinned else t.clone()


def _host_bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("T,pinned", [(4, True), (16, False), (40, True)])
def test_hostio_single_call(cuda_lib, T, pinned):
    f = G.make_factors(300, 200, 77, 2, 4000 + T)
    df = U.device_factors(f)
    xb = G.make_x(T, 200, 4010 + T)
    xh = _host_bf16(xb, pinned)
    yh = _host_bf16(np.zeros((T, 300), dtype=np.uint16), pinned)
    cuda_lib.matmul_hostio(df, xh, yh)
    torch.cuda.synchronize()
    assert cuda_lib.check_status() == 0
    yref, _ = O.matmul(xb, f)
    U.assert_close(_host_bits(yh), yref, f"hostio T={T}")


@pytest.mark.parametrize("T,accumulate", [(1, False), (16, True), (33, False)])
def test_hostio_batch_matches_each_call(cuda_lib, T, accumulate):
    shapes = [(300, 200, 77), (4096, 4096, 64), (257, 130, 33), (96, 160, 40), (512, 384, 256)]
    fs = [G.make_factors(N, M, R, 1, 4100 + 13 * k + T) for k, (N, M, R) in enumerate(shapes)]
    dfs = [U.device_factors(f) for f in fs]
    xbs = [G.make_x(T, f.M, 4200 + k + T) for k, f in enumerate(fs)]
    ybs = [G.make_x(T, f.N, 4300 + k + T) for k, f in enumerate(fs)]
    xs = [_host_bf16(b) for b in xbs]
    ys = [_host_bf16(b) for b in ybs]
    cuda_lib.matmul_hostio_batch(dfs, xs, ys, accumulate=accumulate)
    torch.cuda.synchronize()
    assert cuda_lib.check_status() == 0
    for k, (xb, yb, f, y) in enumerate(zip(xbs, ybs, fs, ys)):
        yref, _ = O.matmul(xb, f, yb if accumulate else None)
        U.assert_close(_host_bits(y), yref, f"batch call {k} T={T}")


def test_hostio_batch_in_a_cuda_graph(cuda_lib):
    # the pipeline forks from and joins back to the capturing stream; replays see new host inputs
    T = 8
    fs = [G.make_factors(4096, 4096, 64, 1, 4400 + k) for k in range(7)]
    dfs = [U.device_factors(f) for f in fs]
    xs = [_host_bf16(np.zeros((T, 4096), dtype=np.uint16)) for _ in fs]
    ys = [_host_bf16(np.zeros((T, 4096), dtype=np.uint16)) for _ in fs]
    ws = cuda_lib.new_workspace(cuda_lib.hostio_batch_workspace_bytes(dfs, T), "cuda")
    cuda_lib.matmul_hostio_batch(dfs, xs, ys, workspace=ws)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        cuda_lib.matmul_hostio_batch(dfs, xs, ys, workspace=ws, stream=s)
    torch.cuda.synchronize()
    for rep in range(2):
        xbs = [G.make_x(T, 4096, 4500 + 10 * rep + k) for k in range(len(fs))]
        for x, b in zip(xs, xbs):
            x.copy_(torch.from_numpy(b.view(np.int16)).view(torch.bfloat16))
        g.replay()
        torch.cuda.synchronize()
        assert cuda_lib.check_status() == 0
        for k, (xb, f, y) in enumerate(zip(xbs, fs, ys)):
            yref, _ = O.matmul(xb, f)
            U.assert_close(_host_bits(y), yref, f"graph replay {rep} call {k}")


def test_hostio_batch_empty_and_errors(cuda_lib):
    f = U.device_factors(G.make_factors(64, 64, 16, 1, 4600))
    assert cuda_lib.matmul_hostio_batch([], [], []) == []
    x = _host_bf16(np.zeros((0, 64), dtype=np.uint16))
    y = _host_bf16(np.zeros((0, 64), dtype=np.uint16))
    cuda_lib.matmul_hostio_batch([f], [x], [y])  # T = 0: nothing to do
    structs = (cuda_lib.DbfFactors * 1)(f.struct)
    assert cuda_lib._lib.dbf_matmul_hostio_batch(structs, 1, None, None, 4, 0, None, 0, None) == -1
    assert cuda_lib._lib.dbf_hostio_batch_workspace_bytes(structs, 0, 4) == 0


@pytest.mark.parametrize("accumulate", [False, True])
def test_hostio_batch_contiguous_buffers_share_copies(cuda_lib, accumulate):
    # calls whose host buffers follow one another are moved in chunks of up to 32 with one copy each
    # way over four device slots, the sizes ramping up at the start and down at the end: 140 calls
    # give chunks of 4, 8, 16, 32, 32, 24, 12, 6, 4 and 2 (the fifth and later reuse slots once their
    # read-back is done), and the shapes differ from call to call
    T = 8
    shapes = [(256, 512, 32), (512, 256, 48), (384, 384, 40)]
    fs = [G.make_factors(*shapes[k % 3], 1, 4700 + k) for k in range(140)]
    dfs = [U.device_factors(f) for f in fs]
    xbs = [G.make_x(T, f.M, 4800 + k) for k, f in enumerate(fs)]
    ybs = [G.make_x(T, f.N, 4900 + k) for k, f in enumerate(fs)]
    xall = torch.from_numpy(np.concatenate([b.ravel() for b in xbs]).view(np.int16)).view(torch.bfloat16).pin_memory()
    yall = torch.from_numpy(np.concatenate([b.ravel() for b in ybs]).view(np.int16)).view(torch.bfloat16).pin_memory()
    xs, ys, ox, oy = [], [], 0, 0
    for f in fs:
        xs.append(xall[ox:ox + T * f.M].view(T, f.M))
        ys.append(yall[oy:oy + T * f.N].view(T, f.N))
        ox += T * f.M
        oy += T * f.N
    cuda_lib.matmul_hostio_batch(dfs, xs, ys, accumulate=accumulate)
    torch.cuda.synchronize()
    assert cuda_lib.check_status() == 0
    for k, (xb, yb, f, y) in enumerate(zip(xbs, ybs, fs, ys)):
        yref, _ = O.matmul(xb, f, yb if accumulate else None)
        U.assert_close(_host_bits(y), yref, f"contiguous batch call {k}")
