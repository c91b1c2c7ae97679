"""The debug build of the library (libdbf_debug.so, -DDBF_DEBUG=1).

The debug build adds bounds checks to the index arithmetic of the kernels:
an index that falls outside the buffer it addresses records DBF_ERR_BOUNDS
in the device status word and the access is skipped.  On valid calls it must
produce the release library's bits and record nothing.  The library is
loaded beside the release one through ctypes and called with the same
device buffers.
"""

import ctypes

import numpy as np
import pytest
import torch

from tests import gpu_util as U
from workloads import generators as G

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def debug_lib(cuda_lib):
    from double_binary_rank_packed_b300 import build
    lib = ctypes.CDLL(build.build(debug=True))
    lib.dbf_matmul_path.restype = ctypes.c_int
    lib.dbf_matmul_path.argtypes = [ctypes.POINTER(cuda_lib.DbfFactors), ctypes.c_void_p, ctypes.c_int64,
                                    ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t,
                                    ctypes.c_void_p, ctypes.c_int]
    lib.dbf_check_status.restype = ctypes.c_int
    lib.dbf_check_status.argtypes = [ctypes.c_void_p]
    lib.dbf_selftest_decode_one_launch.restype = ctypes.c_int
    lib.dbf_selftest_decode_one_launch.argtypes = [ctypes.POINTER(cuda_lib.DbfFactors), ctypes.c_void_p,
                                                   ctypes.c_int64, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p,
                                                   ctypes.c_size_t, ctypes.c_void_p, ctypes.c_void_p]
    return lib


# (N, M, R, ell, T, path): reduce-scatter decode kernel, accumulate; all-to-all fused kernel (ell = 3);
# two-stage decode (R > 256); prefill GEMMs with ragged tiles; prefill whose second GEMM takes
# 160-row tiles
CASES = [(4096, 4096, 64, 1, 16, 1), (300, 200, 77, 2, 5, 1), (257, 130, 96, 4, 9, 1), (200, 300, 100, 3, 7, 1),
         (1024, 2048, 768, 2, 8, 1), (300, 200, 77, 2, 300, 2), (384, 512, 256, 1, 513, 2),
         (4096, 1024, 1000, 2, 2048, 2)]


@pytest.mark.parametrize("N,M,R,ell,T,path", CASES)
@pytest.mark.parametrize("accumulate", [0, 1])
def test_debug_build_matches_release_and_records_nothing(cuda_lib, debug_lib, N, M, R, ell, T, path, accumulate):
    f = G.make_factors(N, M, R, ell, 3300 + N + R)
    df = U.device_factors(f)
    x = U.bits_to_bf16(G.make_x(T, M, 3300 + N + R))
    y0 = U.bits_to_bf16(G.make_x(T, N, 3301 + N))
    want = y0.clone()
    cuda_lib.matmul_path(df, x, want, accumulate=bool(accumulate), path=path)
    assert cuda_lib.check_status() == 0
    ws = cuda_lib.new_workspace(cuda_lib.workspace_bytes(df, T, path), "cuda")
    got = y0.clone()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = debug_lib.dbf_matmul_path(ctypes.byref(df.struct), ctypes.c_void_p(x.data_ptr()), T,
                                   ctypes.c_void_p(got.data_ptr()), accumulate, ctypes.c_void_p(ws.data_ptr()),
                                   ws.numel(), stream, path)
    assert rc == cuda_lib.DBF_OK
    assert debug_lib.dbf_check_status(stream) == cuda_lib.DBF_OK
    assert np.array_equal(U.bf16_to_bits(got), U.bf16_to_bits(want))


@pytest.mark.parametrize("N,M,R,ell,T", [(640, 1024, 512, 2, 8), (4096, 4096, 3072, 1, 8), (300, 520, 300, 2, 5)])
def test_debug_build_one_launch(cuda_lib, debug_lib, N, M, R, ell, T):
    # both decode stages in one cooperative launch, debug build: the release two-launch bits, no
    # bounds error, and the arrival counter advanced by one call
    f = G.make_factors(N, M, R, ell, 3500 + N + R)
    df = U.device_factors(f)
    x = U.bits_to_bf16(G.make_x(T, M, 3500 + R))
    want = torch.empty((T, N), dtype=torch.bfloat16, device="cuda")
    cuda_lib.matmul_path(df, x, want, path=cuda_lib.PATH_DECODE)
    assert cuda_lib.check_status() == 0
    ws = cuda_lib.new_workspace(cuda_lib.workspace_bytes(df, T, cuda_lib.PATH_DECODE), "cuda")
    bar = torch.zeros(2, dtype=torch.int32, device="cuda")
    got = torch.empty((T, N), dtype=torch.bfloat16, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = debug_lib.dbf_selftest_decode_one_launch(ctypes.byref(df.struct), ctypes.c_void_p(x.data_ptr()), T,
                                                  ctypes.c_void_p(got.data_ptr()), 0,
                                                  ctypes.c_void_p(ws.data_ptr()), ws.numel(),
                                                  ctypes.c_void_p(bar.data_ptr()), stream)
    assert rc == cuda_lib.DBF_OK
    assert debug_lib.dbf_check_status(stream) == cuda_lib.DBF_OK
    assert np.array_equal(U.bf16_to_bits(got), U.bf16_to_bits(want))
    assert bar.cpu().tolist() == [1024, 0]
