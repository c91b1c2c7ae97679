"""Multi-adapter routed batches (dbf_matmul_segmented) against the oracle."""

import numpy as np
import pytest
import torch

from oracle import dbf_oracle as O
from tests import gpu_util as U
from workloads import configs as C
from workloads import generators as G

pytestmark = pytest.mark.gpu


def run_segmented(cuda_lib, adapters, N, M, R, ell, xb, off, ad, y_in=None):
    dev = [U.device_factors(f) for f in adapters]
    table = cuda_lib.adapter_table(dev, "cuda")
    x = U.bits_to_bf16(xb)
    T = xb.shape[0]
    if y_in is None:
        y = torch.zeros((T, N), dtype=torch.bfloat16, device="cuda")
    else:
        y = U.bits_to_bf16(y_in).clone()
    offs = torch.from_numpy(np.asarray(off, dtype=np.int32)).cuda()
    ads = torch.from_numpy(np.asarray(ad, dtype=np.int32)).cuda()
    cuda_lib.matmul_segmented(table, len(dev), N, M, R, ell, x, offs, ads, y, accumulate=y_in is not None)
    st = cuda_lib.check_status()
    return U.bf16_to_bits(y), st


def test_multi_adapter_serving_workload(cuda_lib):
    w = C.MULTI_ADAPTER
    T = w.tokens[0]
    adapters = [G.make_factors(p.N, p.M, p.R, p.ell, p.seed) for p in w.projections]
    off, ad, _ = G.make_routing(T, w.n_adapters, w.routing_seed)
    xb = G.make_x(T, 4096, w.routing_seed)
    got, st = run_segmented(cuda_lib, adapters, 4096, 4096, 32, 2, xb, off, ad)
    assert st == 0
    y, _ = O.matmul_segmented(xb, adapters, off, ad)
    U.assert_close(got, y, "multi-adapter")


def test_segments_edge_cases(cuda_lib):
    N, M, R, ell = 160, 224, 48, 2
    adapters = [G.make_factors(N, M, R, ell, 900 + a) for a in range(3)]
    T = 60
    xb = G.make_x(T, M, 901)
    # empty segments, a long segment (several column chunks), single-token segments
    off = [0, 0, 1, 41, 41, 42, 60]
    ad = [2, 1, 0, 2, 1, 2]
    got, st = run_segmented(cuda_lib, adapters, N, M, R, ell, xb, off, ad)
    assert st == 0
    y, _ = O.matmul_segmented(xb, adapters, off, ad)
    U.assert_close(got, y, "segment edge cases")


def test_segmented_accumulate_and_uncovered_rows(cuda_lib):
    N, M, R, ell = 96, 128, 32, 1
    adapters = [G.make_factors(N, M, R, ell, 950 + a) for a in range(2)]
    T = 12
    xb = G.make_x(T, M, 951)
    y_in = G.make_x(T, N, 952)
    off = [2, 5, 10]   # tokens 0,1 and 10,11 belong to no segment: left as y_in
    ad = [1, 0]
    got, st = run_segmented(cuda_lib, adapters, N, M, R, ell, xb, off, ad, y_in=y_in)
    assert st == 0
    y, _ = O.matmul_segmented(xb, adapters, off, ad, y_in)
    U.assert_close(got, y, "segmented accumulate")
    assert np.array_equal(got[:2], y_in[:2]) and np.array_equal(got[10:], y_in[10:])


def test_bad_segment_entry_is_reported_and_skipped(cuda_lib):
    N, M, R, ell = 64, 64, 32, 1
    adapters = [G.make_factors(N, M, R, ell, 970)]
    T = 8
    xb = G.make_x(T, M, 971)
    off = [0, 4, 8]
    ad = [0, 5]        # adapter 5 does not exist
    got, st = run_segmented(cuda_lib, adapters, N, M, R, ell, xb, off, ad)
    assert st == cuda_lib.DBF_ERR_DEVICE_ARG
    assert cuda_lib.check_status() == 0  # cleared by the first read
    y, _ = O.matmul_segmented(xb, adapters, [0, 4], [0])
    U.assert_close(got[:4], y[:4], "valid segment")
    assert (got[4:] == 0).all()


def test_chunk_clusters_match_segment_clusters(cuda_lib):
    # The same routing twice: compact (S <= 1024: a cluster per chunk, found by a scan
    # on the device) and padded with empty segments past 1024 (a cluster per segment,
    # chunks in turn).  The two are planned for different segment lengths (their tile
    # plans, and so their summation orders, may differ): each is held to the oracle.
    N, M, R, ell = 160, 224, 48, 2
    adapters = [G.make_factors(N, M, R, ell, 990 + a) for a in range(3)]
    T = 70
    xb = G.make_x(T, M, 991)
    off = [0, 1, 37, 38, 45, 70]      # segments of 1, 36, 1, 7 and 25 tokens
    ad = [2, 0, 1, 2, 0]
    compact, st = run_segmented(cuda_lib, adapters, N, M, R, ell, xb, off, ad)
    assert st == 0
    pad_off, pad_ad = [0], []
    for s in range(len(ad)):
        for _ in range(230):          # 230 empty segments before each real one
            pad_off.append(off[s])
            pad_ad.append(1)
        pad_off.append(off[s + 1])
        pad_ad.append(ad[s])
    assert len(pad_ad) > 1024
    padded, st = run_segmented(cuda_lib, adapters, N, M, R, ell, xb, pad_off, pad_ad)
    assert st == 0
    y, _ = O.matmul_segmented(xb, adapters, off, ad)
    U.assert_close(compact, y, "chunk clusters")
    U.assert_close(padded, y, "segment clusters")


def test_bad_entry_of_an_empty_segment_is_reported(cuda_lib):
    N, M, R, ell = 64, 96, 32, 1
    adapters = [G.make_factors(N, M, R, ell, 975)]
    T = 8
    xb = G.make_x(T, M, 976)
    off = [0, 4, 4, 8]
    ad = [0, 9, 0]     # the empty middle segment names a missing adapter
    got, st = run_segmented(cuda_lib, adapters, N, M, R, ell, xb, off, ad)
    assert st == cuda_lib.DBF_ERR_DEVICE_ARG
    y, _ = O.matmul_segmented(xb, adapters, [0, 4, 8], [0, 0])
    U.assert_close(got, y, "segments around the bad entry")


def test_large_adapter_table(cuda_lib):
    # 160 adapters (a table larger than the shared-memory copy takes), four of them used
    N, M, R, ell = 96, 128, 32, 1
    base = [G.make_factors(N, M, R, ell, 1000 + a) for a in range(4)]
    adapters = [base[a % 4] for a in range(160)]
    T = 20
    xb = G.make_x(T, M, 1001)
    off = [0, 3, 11, 12, 20]
    ad = [159, 2, 80, 41]
    got, st = run_segmented(cuda_lib, adapters, N, M, R, ell, xb, off, ad)
    assert st == 0
    y, _ = O.matmul_segmented(xb, adapters, off, ad)
    U.assert_close(got, y, "large adapter table")
