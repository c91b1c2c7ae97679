"""Calls on a caller-chosen stream that is not torch's current stream.

The binding allocates the workspace (and any contiguous copy of an input)
itself when the caller passes none.  Those tensors must be allocated on the
stream the kernels run on, so that the caching allocator cannot hand their
memory to other work while the kernels still use it.  The tests run a call on
a side stream, then immediately allocate and overwrite memory on the current
stream, and compare the result with the same call made on the current stream.
"""

import numpy as np
import pytest
import torch

from tests import gpu_util as U
from workloads import generators as G

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("N,M,R,ell,T", [(1024, 2048, 768, 2, 8), (512, 768, 200, 2, 300)])
def test_matmul_on_a_side_stream_with_library_allocated_workspace(cuda_lib, N, M, R, ell, T):
    f = G.make_factors(N, M, R, ell, 3100 + T)
    df = U.device_factors(f)
    x_full = U.bits_to_bf16(G.make_x(T, 2 * M, 3100 + T))
    x = x_full[:, ::2]  # not contiguous: the binding makes a copy
    want = cuda_lib.matmul(df, x.contiguous())
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    for _ in range(3):
        y = cuda_lib.matmul(df, x, stream=side)
        # new allocations on the current stream, written at once, while the side stream may still run
        junk = [torch.full((1 << 20,), 7.0, device="cuda") for _ in range(8)]
        del junk
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        assert cuda_lib.check_status() == 0
        assert np.array_equal(U.bf16_to_bits(y), U.bf16_to_bits(want))
