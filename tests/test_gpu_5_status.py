"""Failure path on the GPU without a fault: a bounded wait that runs out."""

import numpy as np
import pytest

from oracle import dbf_oracle as O
from tests import gpu_util as U
from workloads import generators as G

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_context_stays_usable(cuda_lib):
    assert cuda_lib.check_status() == 0
    assert cuda_lib.selftest_bounded_wait(20000) == 0       # 20 ms limit
    assert cuda_lib.check_status() == cuda_lib.DBF_ERR_TIMEOUT
    assert cuda_lib.check_status() == 0                      # cleared
    # the context still runs kernels correctly afterwards
    f = G.make_factors(64, 64, 32, 1, 1600, unit_scales=True)
    xb = G.make_x(4, 64, 1600, integer=True)
    y = cuda_lib.matmul(U.device_factors(f), U.bits_to_bf16(xb))
    assert cuda_lib.check_status() == 0
    _, want = O.matmul(xb, f)
    assert np.array_equal(U.bf16_to_bits(y), want)
