"""dbf_matmul_decode_noalloc: the decode path for callers that cannot allocate.

Callers recording a CUDA graph, serving loops that must avoid cudaMalloc's
device synchronisation, and runtimes with a fixed pre-planned memory arena
cannot hand the library a workspace.  This entry point keeps the decode
scratch in a 2 MiB static device array instead.  The test calls it through
the C ABI twice in a row (different shapes, so the second call reuses the
array after the first left its contents there) and checks each result
against the ordinary dbf_matmul decode path, within the tolerance the other
GPU tests use.  It also checks that a call needing more than 2 MiB of
scratch is refused before any device work.
"""

import ctypes

import numpy as np
import pytest
import torch

from tests import gpu_util as U
from workloads import generators as G

pytestmark = pytest.mark.gpu


def _noalloc(lib, f, x, y, accumulate=0):
    fn = lib._lib.dbf_matmul_decode_noalloc
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.POINTER(lib.DbfFactors), ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p,
                   ctypes.c_int, ctypes.c_void_p]
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return fn(ctypes.byref(f.struct), ctypes.c_void_p(x.data_ptr()), x.shape[0], ctypes.c_void_p(y.data_ptr()),
              accumulate, stream)


@pytest.mark.parametrize("order", ["small_then_large", "large_then_small"])
def test_noalloc_matches_workspace_path_on_two_calls_in_a_row(cuda_lib, order):
    cases = [(4096, 4096, 64, 1, 16, 2000), (1024, 2048, 768, 2, 8, 2100)]
    if order == "large_then_small":
        cases = cases[::-1]
    for (N, M, R, ell, T, seed) in cases:
        f = G.make_factors(N, M, R, ell, seed)
        df = U.device_factors(f)
        x = U.bits_to_bf16(G.make_x(T, M, seed))
        y_ref = cuda_lib.matmul_path(df, x, path=cuda_lib.PATH_DECODE)
        y = torch.full((T, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        assert _noalloc(cuda_lib, df, x, y) == cuda_lib.DBF_OK
        torch.cuda.synchronize()
        assert cuda_lib.check_status() == 0
        U.assert_close(U.bf16_to_bits(y), _as_f64(y_ref), f"noalloc {N}x{M} R={R}")


def _as_f64(t):
    from oracle import dbf_oracle as O
    return O.bf16_bits_to_f64(U.bf16_to_bits(t))


def test_noalloc_refuses_scratch_beyond_the_static_array(cuda_lib):
    # ell * T * round_up(R, 64) * 2 bytes > 2 MiB: 4 * 64 * 4160 * 2 = 2.1 MB
    f = G.make_factors(64, 64, 4150, 4, 2200)
    df = U.device_factors(f)
    x = torch.zeros((64, 64), dtype=torch.bfloat16, device="cuda")
    y = torch.zeros((64, 64), dtype=torch.bfloat16, device="cuda")
    assert _noalloc(cuda_lib, df, x, y) == cuda_lib.DBF_ERR_WORKSPACE
    assert "2 MiB" in cuda_lib.last_cuda_error()
