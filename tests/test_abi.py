"""The C ABI without a GPU: the library builds, loads, exports every function
include/dbf.h declares, and rejects bad arguments on the host before any
device work (fake pointers are never dereferenced)."""

import ctypes
import os
import re

import pytest

from tests.conftest import ROOT


@pytest.fixture(scope="module")
def lib():
    from double_binary_rank_packed_b300 import build
    build.build()
    from double_binary_rank_packed_b300 import dbf
    return dbf


def declared_functions():
    with open(os.path.join(ROOT, "include", "dbf.h")) as fh:
        text = fh.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(dbf_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_boundary_calls():
    names = declared_functions()
    for must in ("dbf_pack", "dbf_matmul", "dbf_matmul_segmented", "dbf_check_status", "dbf_workspace_bytes"):
        assert must in names


def test_every_declared_function_is_exported(lib):
    cdll = ctypes.CDLL(lib.LIB_PATH)
    missing = [n for n in declared_functions() if not hasattr(cdll, n)]
    assert not missing, missing
    assert set(lib.EXPORTED) <= set(declared_functions())


def test_struct_layout_matches_header(lib):
    assert ctypes.sizeof(lib.DbfFactors) == 64
    assert lib.DbfFactors.B1.offset == 24


def test_status_strings(lib):
    for code in range(0, -10, -1):
        assert lib.status_string(code) != "unknown status"
    assert lib.status_string(5) == "unknown status"


FAKE = 0x10000000  # 256-byte aligned, never dereferenced by the checks below


def _factors(lib, N=64, M=64, R=32, ell=1, ldw1=None, ldw2=None, base=FAKE):
    return lib.DbfFactors(N, M, R, ell, ldw1 if ldw1 is not None else (R + 31) // 32,
                          ldw2 if ldw2 is not None else (M + 31) // 32,
                          base, base + 0x1000, base + 0x2000, base + 0x3000, base + 0x4000)


def _call(lib, f, x=FAKE + 0x5000, T=4, y=FAKE + 0x6000, ws=FAKE + 0x7000, ws_bytes=1 << 30, acc=0, path=0):
    fp = ctypes.byref(f) if f is not None else None
    return lib._lib.dbf_matmul_path(fp, ctypes.c_void_p(x), T, ctypes.c_void_p(y), acc, ctypes.c_void_p(ws),
                                    ws_bytes, None, path)


def test_host_side_argument_checks(lib):
    assert _call(lib, None) == lib.DBF_ERR_INVALID_ARG
    assert _call(lib, _factors(lib, ell=0)) == lib.DBF_ERR_INVALID_ARG
    assert _call(lib, _factors(lib, ell=5)) == lib.DBF_ERR_INVALID_ARG
    assert _call(lib, _factors(lib, N=0)) == lib.DBF_ERR_INVALID_ARG
    assert _call(lib, _factors(lib, ldw2=1)) == lib.DBF_ERR_INVALID_ARG       # M=64 needs 2 words
    assert _call(lib, _factors(lib, ldw1=0)) == lib.DBF_ERR_INVALID_ARG
    assert _call(lib, _factors(lib, base=FAKE + 4)) == lib.DBF_ERR_ALIGNMENT
    assert _call(lib, _factors(lib), x=FAKE + 2) == lib.DBF_ERR_ALIGNMENT
    assert _call(lib, _factors(lib), y=0) == lib.DBF_ERR_INVALID_ARG
    assert _call(lib, _factors(lib), T=-1) == lib.DBF_ERR_INVALID_ARG
    assert _call(lib, _factors(lib), acc=2) == lib.DBF_ERR_INVALID_ARG
    assert _call(lib, _factors(lib), path=7) == lib.DBF_ERR_INVALID_ARG
    assert _call(lib, _factors(lib), ws_bytes=16) == lib.DBF_ERR_WORKSPACE
    assert _call(lib, _factors(lib), ws=0) == lib.DBF_ERR_WORKSPACE
    assert _call(lib, _factors(lib), ws=FAKE + 0x7010) == lib.DBF_ERR_ALIGNMENT
    # T = 0 is a no-op and needs nothing else
    assert _call(lib, _factors(lib), T=0, x=0, y=0, ws=0, ws_bytes=0) == lib.DBF_OK


def test_workspace_sizes(lib):
    f = _factors(lib, N=4096, M=4096, R=3072, ell=1, ldw1=96, ldw2=128)
    dec = lib._lib.dbf_workspace_bytes_path(ctypes.byref(f), 8, lib.PATH_DECODE)
    pre = lib._lib.dbf_workspace_bytes_path(ctypes.byref(f), 8, lib.PATH_PREFILL)
    assert dec >= 8 * 3072 * 2 and dec % 256 == 0
    assert pre >= 8 * (4096 + 3072) * 2
    assert lib._lib.dbf_workspace_bytes(ctypes.byref(f), 8) == dec  # T <= 16 goes to decode
    assert lib._lib.dbf_workspace_bytes(ctypes.byref(f), 2048) == \
        lib._lib.dbf_workspace_bytes_path(ctypes.byref(f), 2048, lib.PATH_PREFILL)
    assert lib._lib.dbf_workspace_bytes(None, 8) == 0


def test_pack_and_segmented_host_checks(lib):
    L = lib._lib
    assert L.dbf_pack(ctypes.c_void_p(FAKE), 4, 40, ctypes.c_void_p(FAKE), 1, None) == lib.DBF_ERR_INVALID_ARG
    assert L.dbf_pack(ctypes.c_void_p(FAKE), 4, 40, ctypes.c_void_p(FAKE + 2), 2, None) == lib.DBF_ERR_ALIGNMENT
    assert L.dbf_pack(None, 0, 40, None, 2, None) == lib.DBF_OK
    assert L.dbf_matmul_segmented(None, 1, 64, 64, 32, 1, None, 0, None, None, None, 1, 0, None, 0, None) == lib.DBF_OK
    assert L.dbf_matmul_segmented(None, 1, 64, 64, 32, 5, None, 8, None, None, None, 1, 0, None, 0, None) \
        == lib.DBF_ERR_INVALID_ARG
    assert L.dbf_matmul_segmented(None, 1, 64, 64, 32, 1, ctypes.c_void_p(FAKE), 8, ctypes.c_void_p(FAKE), None,
                                  None, 1, 0, None, 0, None) == lib.DBF_ERR_INVALID_ARG
    assert L.dbf_selftest_bounded_wait(0, None) == lib.DBF_ERR_INVALID_ARG


def _fz_call(lib, N=64, M=48, k=16, prm=(2, 3, 4, 1.0), W=FAKE, ws=FAKE + 0x8000, ws_bytes=1 << 30, scale=FAKE):
    p = lib.DbfFactorizeParams(*prm) if prm is not None else None
    vp = ctypes.c_void_p
    return lib._lib.dbf_factorize(vp(W), N, M, k, ctypes.byref(p) if p is not None else None,
                                  vp(scale), vp(FAKE + 0x1000), vp(FAKE + 0x2000), vp(FAKE + 0x3000),
                                  vp(FAKE + 0x4000), vp(FAKE + 0x5000), vp(ws), ws_bytes, None)


def test_factorize_host_checks(lib):
    assert _fz_call(lib, prm=None) == lib.DBF_ERR_INVALID_ARG
    assert _fz_call(lib, N=0) == lib.DBF_ERR_INVALID_ARG
    assert _fz_call(lib, k=0) == lib.DBF_ERR_INVALID_ARG
    assert _fz_call(lib, prm=(-1, 3, 4, 1.0)) == lib.DBF_ERR_INVALID_ARG
    assert _fz_call(lib, prm=(1, 3, 4, 0.0)) == lib.DBF_ERR_INVALID_ARG
    assert _fz_call(lib, prm=(1, 3, 4, float("nan"))) == lib.DBF_ERR_INVALID_ARG
    assert _fz_call(lib, N=65536) == lib.DBF_ERR_UNSUPPORTED
    assert _fz_call(lib, k=16385) == lib.DBF_ERR_UNSUPPORTED
    assert _fz_call(lib, W=0) == lib.DBF_ERR_INVALID_ARG
    assert _fz_call(lib, ws_bytes=16) == lib.DBF_ERR_WORKSPACE
    assert _fz_call(lib, ws=FAKE + 0x8010) == lib.DBF_ERR_ALIGNMENT
    assert _fz_call(lib, scale=FAKE + 2) == lib.DBF_ERR_ALIGNMENT


def test_factorize_sizes_and_launch_counts(lib):
    ws = lib.factorize_workspace_bytes(4096, 4096, 1024)
    # W^T, F, four k x k, two n x k, the split forms ([hi | lo], twice the size) of W, W^T, F,
    # the inverse and the right-hand side, the sign transpose, small vectors
    assert ws >= 4 * (5 * 4096 * 4096 + 3 * 1024 * 4096 + 6 * 1024 * 1024 + 4 * 4096 * 1024) + 4096 * 1024
    assert ws % 256 == 0
    assert lib.factorize_workspace_bytes(0, 4, 4) == 0
    assert lib.factorize_workspace_bytes(4, 4, 16385) == 0
    # per call: transposes of W and B, split forms of W and W^T, the rounds, transpose of B out.
    # per step: F and its split form, F F^T, ridge; 2 per 32-column Cholesky block less 1 (diagonal
    # and panel, trailing update); the blocked L^-1 (zero fill and one leaf of 128 rows at k = 70);
    # inverse, its mirror and its split form, T F^T, first dual; per iteration 1 GEMM + 3q + 1 SVID
    # passes, dual between iterations
    k, inner, q = 70, 4, 5
    step = 4 + (2 * 3 - 1) + 2 + 5 + inner * (1 + 3 * q + 1) + (inner - 1)
    assert lib.factorize_launch_count(100, 80, k, 3, inner, q, 1.0) == 4 + 3 * 2 * step + 1
    step0 = 4 + (2 * 3 - 1) + 2 + 5 + inner * (1 + 1 + 1) + (inner - 1)   # power_iters = 0: fill + rows
    assert lib.factorize_launch_count(100, 80, k, 1, inner, 0, 1.0) == 4 + 2 * step0 + 1
    assert lib.factorize_launch_count(100, 80, k, 0, inner, q, 1.0) == 0
    assert lib.factorize_launch_count(100, 80, k, 1, 0, q, 1.0) == 0
    assert lib.factorize_launch_count(100, 80, 0, 1, 1, q, 1.0) == -1


def test_factorize_weighted_host_checks(lib):
    vp = ctypes.c_void_p
    p = lib.DbfFactorizeParams(1, 2, 3, 1.0)

    def call(d_out=FAKE + 0x9000, d_in=FAKE + 0xA000, ws_bytes=1 << 30, N=64, M=48, k=16):
        return lib._lib.dbf_factorize_weighted(vp(FAKE), N, M, k, ctypes.byref(p), vp(d_out), vp(d_in),
                                               vp(FAKE + 0x1000), vp(FAKE + 0x2000), vp(FAKE + 0x3000),
                                               vp(FAKE + 0x4000), vp(FAKE + 0x5000), vp(FAKE + 0x6000),
                                               vp(FAKE + 0x8000), ws_bytes, None)

    assert call(d_out=0) == lib.DBF_ERR_INVALID_ARG
    assert call(d_in=0) == lib.DBF_ERR_INVALID_ARG
    assert call(d_in=FAKE + 0xA002) == lib.DBF_ERR_ALIGNMENT
    assert call(N=70000) == lib.DBF_ERR_UNSUPPORTED
    plain = lib.factorize_workspace_bytes(64, 48, 16)
    weighted = lib.factorize_weighted_workspace_bytes(64, 48, 16)
    assert weighted >= plain + 4 * 64 * 48 and weighted % 256 == 0
    assert call(ws_bytes=plain) == lib.DBF_ERR_WORKSPACE
    assert lib.factorize_weighted_launch_count(64, 48, 16, 2, 3, 4, 1.0) == \
        lib.factorize_launch_count(64, 48, 16, 2, 3, 4, 1.0) + 5
    assert lib.factorize_weighted_launch_count(64, 48, 16, 0, 3, 4, 1.0) == 0


def test_noalloc_host_checks_match_the_workspace_entry_point(lib):
    """dbf_matmul_decode_noalloc rejects what dbf_matmul_path rejects, with the same codes,
    before any device work (shape limits included)."""
    fn = lib._lib.dbf_matmul_decode_noalloc
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.POINTER(lib.DbfFactors), ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p,
                   ctypes.c_int, ctypes.c_void_p]

    def call(f, x=FAKE + 0x5000, T=4, y=FAKE + 0x6000, acc=0):
        return fn(ctypes.byref(f) if f is not None else None, ctypes.c_void_p(x), T, ctypes.c_void_p(y), acc, None)

    for f, kw in [(None, {}), (_factors(lib, ell=0), {}), (_factors(lib, N=0), {}), (_factors(lib, ldw2=1), {}),
                  (_factors(lib, base=FAKE + 4), {}), (_factors(lib), {"x": FAKE + 2}), (_factors(lib), {"y": 0}),
                  (_factors(lib), {"T": -1}), (_factors(lib), {"acc": 2}),
                  (_factors(lib, N=(1 << 24) + 1), {}), (_factors(lib, M=(1 << 24) + 1), {}),
                  (_factors(lib, R=(1 << 20) + 1), {})]:
        want = _call(lib, f, path=lib.PATH_DECODE, **kw)
        assert want != lib.DBF_OK
        assert call(f, **kw) == want
    assert call(_factors(lib, N=(1 << 24) + 1)) == lib.DBF_ERR_UNSUPPORTED
    assert call(_factors(lib), T=0, x=0, y=0) == lib.DBF_OK
    # more than the 2 MiB static array: ell * T * round_up(R, 64) * 2 = 4 * 64 * 4160 * 2 bytes
    assert call(_factors(lib, N=64, M=64, R=4150, ell=4), T=64) == lib.DBF_ERR_WORKSPACE
    assert "2 MiB" in lib.last_cuda_error()
