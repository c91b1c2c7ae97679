"""dbf_matmul_decode_noalloc: the decode path for callers that cannot allocate.

Some callers cannot give the library a device workspace: serving loops that
must never take cudaMalloc's implicit device synchronisation on the token
path, runtimes whose device memory is one arena planned at start-up, and
plug-in hosts that hand a library only its inputs and outputs.  This entry
point keeps the decode scratch in a 2 MiB static device array inside the
library instead.

The tests call it through the C ABI twice in a row on different shapes (so
the second call finds the first call's contents in the shared array) and
check every result bit for bit against the ordinary entry point
dbf_matmul_path with the decode path, and against the fp64 oracle within the
tolerance the other GPU tests use.  The shapes cover the one-launch fused
kernel (no scratch) and the two-stage kernels (V in the static array).  A
call that would need more than 2 MiB of scratch is refused before any device
work.  This file is collected last, so a run that stops at the first failure
has run every other test before it.
"""

import ctypes

import numpy as np
import pytest
import torch

from oracle import dbf_oracle as O
from tests import gpu_util as U
from workloads import generators as G

pytestmark = pytest.mark.gpu

# (N, M, R, ell, T, seed): fused kernel; two-stage kernels (R > 256) twice, at two scratch sizes
CASES = [(4096, 4096, 64, 1, 16, 2000), (1024, 2048, 768, 2, 8, 2100), (4096, 4096, 3072, 1, 8, 3000)]


def _noalloc(lib, f, x, y, accumulate=0):
    fn = lib._lib.dbf_matmul_decode_noalloc
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.POINTER(lib.DbfFactors), ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p,
                   ctypes.c_int, ctypes.c_void_p]
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return fn(ctypes.byref(f.struct), ctypes.c_void_p(x.data_ptr()), x.shape[0], ctypes.c_void_p(y.data_ptr()),
              accumulate, stream)


@pytest.mark.parametrize("accumulate", [0, 1])
@pytest.mark.parametrize("order", ["as_listed", "reversed"])
def test_noalloc_matches_decode_path_and_oracle_on_calls_in_a_row(cuda_lib, order, accumulate):
    cases = CASES if order == "as_listed" else CASES[::-1]
    for (N, M, R, ell, T, seed) in cases:
        f = G.make_factors(N, M, R, ell, seed)
        df = U.device_factors(f)
        xb = G.make_x(T, M, seed)
        x = U.bits_to_bf16(xb)
        y_in = G.make_x(T, N, seed + 1) if accumulate else None
        y_ref = torch.empty((T, N), dtype=torch.bfloat16, device="cuda")
        y = torch.full((T, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        if accumulate:
            y_ref.copy_(U.bits_to_bf16(y_in))
            y.copy_(U.bits_to_bf16(y_in))
        cuda_lib.matmul_path(df, x, y_ref, accumulate=bool(accumulate), path=cuda_lib.PATH_DECODE)
        assert _noalloc(cuda_lib, df, x, y, accumulate) == cuda_lib.DBF_OK
        torch.cuda.synchronize()
        assert cuda_lib.check_status() == 0
        got = U.bf16_to_bits(y)
        assert np.array_equal(got, U.bf16_to_bits(y_ref)), f"noalloc {N}x{M} R={R}: differs from the decode path"
        want, _ = O.matmul(xb, f, y_in)
        U.assert_close(got, want, f"noalloc {N}x{M} R={R} ell={ell} T={T} acc={accumulate}")


def test_noalloc_refuses_scratch_beyond_the_static_array(cuda_lib):
    # ell * T * round_up(R, 64) * 2 bytes > 2 MiB: 4 * 64 * 4160 * 2 = 2.1 MB
    f = G.make_factors(64, 64, 4150, 4, 2200)
    df = U.device_factors(f)
    x = torch.zeros((64, 64), dtype=torch.bfloat16, device="cuda")
    y = torch.full((64, 64), 3.0, dtype=torch.bfloat16, device="cuda")
    assert _noalloc(cuda_lib, df, x, y) == cuda_lib.DBF_ERR_WORKSPACE
    assert "2 MiB" in cuda_lib.last_cuda_error()
    torch.cuda.synchronize()
    assert bool((y == 3.0).all()), "a refused call wrote its output"
