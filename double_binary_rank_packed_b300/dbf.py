"""ctypes binding of libdbf.so (packed double-binary matmul, sm_103a).

Argument marshalling only: every step of the computation runs in the CUDA
library.  PyTorch supplies device memory and the current stream.  Importing
this module loads libdbf.so and fails loudly when it is missing; there is no
fallback implementation.

Names follow the C ABI in include/dbf.h (dbf_<name>): pack, unpack,
transpose_packed; matmul, matmul_path, matmul_decode_noalloc, matmul_hostio,
matmul_hostio_batch, matmul_segmented, matmul_grouped; backward; factorize,
factorize_weighted; the matching *_workspace_bytes and *_launch_count calls;
check_status, status_string, last_cuda_error, selftest_bounded_wait.
"""

from __future__ import annotations

import ctypes
import functools
import inspect
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdbf.so")

DBF_OK = 0
DBF_ERR_INVALID_ARG = -1
DBF_ERR_ALIGNMENT = -2
DBF_ERR_UNSUPPORTED = -3
DBF_ERR_WORKSPACE = -4
DBF_ERR_CUDA = -5
DBF_ERR_TIMEOUT = -6
DBF_ERR_DEVICE_ARG = -7
DBF_ERR_NUMERIC = -8
DBF_ERR_BOUNDS = -9

PATH_AUTO = 0
PATH_DECODE = 1
PATH_PREFILL = 2

EXPORTED = (
    "dbf_pack", "dbf_unpack", "dbf_workspace_bytes", "dbf_workspace_bytes_path",
    "dbf_decode_max_tokens", "dbf_matmul", "dbf_matmul_path", "dbf_hostio_workspace_bytes",
    "dbf_matmul_hostio", "dbf_segmented_workspace_bytes", "dbf_matmul_segmented",
    "dbf_check_status", "dbf_selftest_bounded_wait", "dbf_status_string", "dbf_last_cuda_error",
    "dbf_launch_count", "dbf_segmented_launch_count", "dbf_transpose_packed", "dbf_factors_transposed",
    "dbf_backward", "dbf_backward_workspace_bytes", "dbf_matmul_grouped", "dbf_grouped_workspace_bytes",
    "dbf_grouped_launch_count", "dbf_matmul_hostio_batch", "dbf_hostio_batch_workspace_bytes",
    "dbf_factorize", "dbf_factorize_workspace_bytes", "dbf_factorize_launch_count",
    "dbf_factorize_weighted", "dbf_factorize_weighted_workspace_bytes", "dbf_factorize_weighted_launch_count",
    "dbf_selftest_split_gemm", "dbf_selftest_split_gemm_workspace_bytes", "dbf_selftest_decode_one_launch",
)


class DbfFactors(ctypes.Structure):
    """Mirror of struct dbf_factors (include/dbf.h)."""

    _fields_ = [
        ("N", ctypes.c_int32), ("M", ctypes.c_int32), ("R", ctypes.c_int32), ("ell", ctypes.c_int32),
        ("ldw1", ctypes.c_int32), ("ldw2", ctypes.c_int32),
        ("B1", ctypes.c_void_p), ("B2", ctypes.c_void_p),
        ("alpha", ctypes.c_void_p), ("beta", ctypes.c_void_p), ("gamma", ctypes.c_void_p),
    ]


class DbfFactorizeParams(ctypes.Structure):
    """Mirror of struct dbf_factorize_params (include/dbf.h)."""

    _fields_ = [("outer", ctypes.c_int32), ("inner", ctypes.c_int32), ("power_iters", ctypes.c_int32),
                ("rho_rel", ctypes.c_float)]


class DbfError(RuntimeError):
    def __init__(self, code: int, what: str):
        msg = f"{what}: {status_string(code)} ({code})"
        if code == DBF_ERR_CUDA:
            msg += f" [{last_cuda_error()}]"
        super().__init__(msg)
        self.code = code


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"libdbf.so not found at {LIB_PATH}; build it with "
            "`python -m double_binary_rank_packed_b300.build` (no CPU fallback exists)")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i64, i32, sz, ci = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_size_t, ctypes.c_int
    fp = ctypes.POINTER(DbfFactors)
    sig = {
        "dbf_pack": (ci, [vp, i64, i64, vp, i64, vp]),
        "dbf_unpack": (ci, [vp, i64, i64, i64, vp, vp]),
        "dbf_workspace_bytes": (sz, [fp, i64]),
        "dbf_workspace_bytes_path": (sz, [fp, i64, ci]),
        "dbf_decode_max_tokens": (ci, []),
        "dbf_matmul": (ci, [fp, vp, i64, vp, ci, vp, sz, vp]),
        "dbf_matmul_path": (ci, [fp, vp, i64, vp, ci, vp, sz, vp, ci]),
        "dbf_hostio_workspace_bytes": (sz, [fp, i64]),
        "dbf_matmul_hostio": (ci, [fp, vp, i64, vp, ci, vp, sz, vp]),
        "dbf_segmented_workspace_bytes": (sz, [i32, i32, i32, i32, i64, i32]),
        "dbf_matmul_segmented": (ci, [vp, i32, i32, i32, i32, i32, vp, i64, vp, vp, vp, i32, ci, vp, sz, vp]),
        "dbf_check_status": (ci, [vp]),
        "dbf_selftest_bounded_wait": (ci, [i64, vp]),
        "dbf_selftest_split_gemm_workspace_bytes": (sz, [i32, i32, i32]),
        "dbf_selftest_split_gemm": (ci, [i32, i32, i32, ctypes.c_float, vp, i64, vp, i64, ctypes.c_float, vp, i64,
                                         ci, vp, sz, vp]),
        "dbf_selftest_decode_one_launch": (ci, [fp, vp, i64, vp, ci, vp, sz, vp, vp]),
        "dbf_status_string": (ctypes.c_char_p, [ci]),
        "dbf_last_cuda_error": (ctypes.c_char_p, []),
        "dbf_launch_count": (ci, [fp, i64, ci]),
        "dbf_transpose_packed": (ci, [vp, i64, i64, i64, vp, i64, vp]),
        "dbf_factors_transposed": (ci, [fp, vp, i32, vp, i32, fp]),
        "dbf_segmented_launch_count": (ci, [i32, i32, i32, i32, i64, i32]),
        "dbf_backward": (ci, [fp, fp, vp, vp, i64, vp, vp, vp, vp, vp, sz, vp]),
        "dbf_backward_workspace_bytes": (sz, [fp, i64]),
        "dbf_matmul_grouped": (ci, [fp, i32, vp, vp, i64, ci, vp, sz, vp]),
        "dbf_grouped_workspace_bytes": (sz, [fp, i32, i64]),
        "dbf_grouped_launch_count": (ci, [fp, i32, i64]),
        "dbf_matmul_hostio_batch": (ci, [fp, i32, vp, vp, i64, ci, vp, sz, vp]),
        "dbf_hostio_batch_workspace_bytes": (sz, [fp, i32, i64]),
        "dbf_factorize": (ci, [vp, i64, i64, i64, ctypes.POINTER(DbfFactorizeParams),
                               vp, vp, vp, vp, vp, vp, vp, sz, vp]),
        "dbf_factorize_workspace_bytes": (sz, [i64, i64, i64]),
        "dbf_factorize_launch_count": (ci, [i64, i64, i64, ctypes.POINTER(DbfFactorizeParams)]),
        "dbf_factorize_weighted": (ci, [vp, i64, i64, i64, ctypes.POINTER(DbfFactorizeParams),
                                        vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]),
        "dbf_factorize_weighted_workspace_bytes": (sz, [i64, i64, i64]),
        "dbf_factorize_weighted_launch_count": (ci, [i64, i64, i64, ctypes.POINTER(DbfFactorizeParams)]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


_lib = _load()


def status_string(code: int) -> str:
    return _lib.dbf_status_string(int(code)).decode()


def last_cuda_error() -> str:
    return _lib.dbf_last_cuda_error().decode()


def _check(code: int, what: str):
    if code != DBF_OK:
        raise DbfError(code, what)


def _stream_handle(stream=None):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _on_stream(fn):
    """Run a wrapper with the caller's `stream` as torch's current stream.

    The tensors a wrapper makes itself (workspace, contiguous copies, outputs)
    are then allocated, filled and released on the stream the library works
    on, so the caching allocator cannot hand their memory to other work while
    the kernels may still use it, and copies are ordered before the kernels.
    """
    sig = inspect.signature(fn)

    @functools.wraps(fn)
    def wrapped(*args, **kwargs):
        stream = sig.bind(*args, **kwargs).arguments.get("stream")
        if stream is None:
            return fn(*args, **kwargs)
        with torch.cuda.stream(stream):
            return fn(*args, **kwargs)

    return wrapped


def _ptr(t) -> ctypes.c_void_p:
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def words_per_row(cols: int) -> int:
    return (cols + 31) // 32


# ------------------------------------------------------------------ packing

@_on_stream
def pack(signs: torch.Tensor, ldw: int | None = None, stream=None) -> torch.Tensor:
    """Pack a device int8 sign matrix [rows, cols] into uint32 words [rows, ldw] (dbf_pack)."""
    if signs.dtype != torch.int8 or signs.dim() != 2 or not signs.is_cuda:
        raise ValueError("signs must be a 2-D int8 CUDA tensor")
    signs = signs.contiguous()
    rows, cols = signs.shape
    if ldw is None:
        ldw = words_per_row(cols)
    words = torch.empty((rows, ldw), dtype=torch.int32, device=signs.device)
    _check(_lib.dbf_pack(_ptr(signs), rows, cols, _ptr(words), ldw, _stream_handle(stream)), "dbf_pack")
    return words


@_on_stream
def unpack(words: torch.Tensor, cols: int, stream=None) -> torch.Tensor:
    """Inverse of pack: int8 +1/-1 [rows, cols] (dbf_unpack)."""
    rows, ldw = words.shape
    signs = torch.empty((rows, cols), dtype=torch.int8, device=words.device)
    _check(_lib.dbf_unpack(_ptr(words), rows, cols, ldw, _ptr(signs), _stream_handle(stream)), "dbf_unpack")
    return signs


@_on_stream
def transpose_packed(words: torch.Tensor, cols: int, ldw_t: int | None = None, stream=None) -> torch.Tensor:
    """Packed transpose of a rows x cols packed sign matrix (dbf_transpose_packed)."""
    rows, ldw = words.shape
    if ldw_t is None:
        ldw_t = words_per_row(rows)
    out = torch.empty((cols, ldw_t), dtype=torch.int32, device=words.device)
    _check(_lib.dbf_transpose_packed(_ptr(words), rows, cols, ldw, _ptr(out), ldw_t, _stream_handle(stream)),
           "dbf_transpose_packed")
    return out


# ------------------------------------------------------------------ factors

class PackedFactors:
    """Device tensors of one factor set: packed B1, B2 and fp16 scales.

    B1w int32 [N, ldw1], B2w int32 [R, ldw2], alpha [ell, N], beta [ell, R],
    gamma [ell, M] (torch.float16).  Keeps the tensors alive for as long as
    the struct handed to the library may be used.
    """

    def __init__(self, B1w, B2w, alpha, beta, gamma, N, M, R):
        self.B1w, self.B2w = B1w, B2w
        self.alpha, self.beta, self.gamma = alpha.contiguous(), beta.contiguous(), gamma.contiguous()
        self.N, self.M, self.R = int(N), int(M), int(R)
        self.ell = int(alpha.shape[0])
        self._struct = DbfFactors(self.N, self.M, self.R, self.ell, int(B1w.shape[1]), int(B2w.shape[1]),
                                  B1w.data_ptr(), B2w.data_ptr(), self.alpha.data_ptr(),
                                  self.beta.data_ptr(), self.gamma.data_ptr())

    @classmethod
    def from_signs(cls, B1, B2, alpha, beta, gamma, ldw1=None, ldw2=None, stream=None):
        """Pack device int8 sign matrices with dbf_pack and wrap them."""
        N, R = B1.shape
        _, M = B2.shape
        return cls(pack(B1, ldw1, stream), pack(B2, ldw2, stream), alpha, beta, gamma, N, M, R)

    @property
    def struct(self) -> DbfFactors:
        return self._struct

    def struct_bytes(self) -> bytes:
        return ctypes.string_at(ctypes.addressof(self._struct), ctypes.sizeof(DbfFactors))


class TransposedFactors(PackedFactors):
    """Factors of the backward product dx = dy dW (dbf_factors_transposed).

    Holds the packed transposes of B1 and B2 (made once with
    dbf_transpose_packed) and shares the scale tensors of `f`; use it with
    matmul / matmul_path: matmul(TransposedFactors(f), dy) is dx.
    """

    def __init__(self, f: PackedFactors, stream=None):
        self.source = f
        self.B1w = transpose_packed(f.B2w, f.M, stream=stream)  # B2^T: [M][ceil(R/32)]
        self.B2w = transpose_packed(f.B1w, f.R, stream=stream)  # B1^T: [R][ceil(N/32)]
        self.alpha, self.beta, self.gamma = f.gamma, f.beta, f.alpha
        self.N, self.M, self.R, self.ell = f.M, f.N, f.R, f.ell
        self._struct = DbfFactors()
        _check(_lib.dbf_factors_transposed(ctypes.byref(f.struct), _ptr(self.B1w), int(self.B1w.shape[1]),
                                           _ptr(self.B2w), int(self.B2w.shape[1]), ctypes.byref(self._struct)),
               "dbf_factors_transposed")


def workspace_bytes(f: PackedFactors, T: int, path: int = PATH_AUTO) -> int:
    return int(_lib.dbf_workspace_bytes_path(ctypes.byref(f.struct), T, path))


def launch_count(f: PackedFactors, T: int, path: int = PATH_AUTO) -> int:
    """Kernel launches of one matmul_path call (dbf_launch_count)."""
    return int(_lib.dbf_launch_count(ctypes.byref(f.struct), T, path))


def segmented_launch_count(N, M, R, ell, T, S) -> int:
    """Kernel launches of one matmul_segmented call (dbf_segmented_launch_count)."""
    return int(_lib.dbf_segmented_launch_count(N, M, R, ell, T, S))


def decode_max_tokens() -> int:
    return int(_lib.dbf_decode_max_tokens())


def new_workspace(nbytes: int, device) -> torch.Tensor:
    # torch's caching allocator returns blocks aligned to at least 512 bytes
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


# ------------------------------------------------------------------ matmul

@_on_stream
def matmul_path(f: PackedFactors, x: torch.Tensor, y: torch.Tensor | None = None, accumulate: bool = False,
                workspace: torch.Tensor | None = None, path: int = PATH_AUTO, stream=None) -> torch.Tensor:
    """y = sum_i alpha_i . B1 (beta_i . (B2 (gamma_i . x))) for x bf16 [T, M] (dbf_matmul_path)."""
    if x.dtype != torch.bfloat16 or x.dim() != 2 or x.shape[1] != f.M:
        raise ValueError("x must be bf16 [T, M]")
    x = x.contiguous()
    T = x.shape[0]
    if y is None:
        if accumulate:
            raise ValueError("accumulate needs y")
        y = torch.empty((T, f.N), dtype=torch.bfloat16, device=x.device)
    need = workspace_bytes(f, T, path)
    if workspace is None:
        workspace = new_workspace(need, x.device)
    rc = _lib.dbf_matmul_path(ctypes.byref(f.struct), _ptr(x), T, _ptr(y), int(bool(accumulate)),
                              _ptr(workspace), workspace.numel(), _stream_handle(stream), int(path))
    _check(rc, "dbf_matmul")
    return y


def matmul(f: PackedFactors, x: torch.Tensor, y: torch.Tensor | None = None, accumulate: bool = False,
           workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    return matmul_path(f, x, y, accumulate, workspace, PATH_AUTO, stream)


def backward_workspace_bytes(f: PackedFactors, T: int) -> int:
    return int(_lib.dbf_backward_workspace_bytes(ctypes.byref(f.struct), T))


@_on_stream
def backward(f: PackedFactors, ft: "TransposedFactors", x: torch.Tensor, dy: torch.Tensor, dx: bool = True,
             workspace: torch.Tensor | None = None, stream=None, out=None):
    """dx, dalpha, dbeta, dgamma of L = sum_t <dy_t, y_t> (dbf_backward).

    x bf16 [T, M], dy bf16 [T, N]; returns (dx bf16 [T, M] or None, dalpha fp32 [ell, N],
    dbeta fp32 [ell, R], dgamma fp32 [ell, M]).  `out` may hold those four tensors
    (dx may be None) to write into instead of new ones.
    """
    if x.dtype != torch.bfloat16 or x.dim() != 2 or x.shape[1] != f.M:
        raise ValueError("x must be bf16 [T, M]")
    if dy.dtype != torch.bfloat16 or dy.dim() != 2 or dy.shape != (x.shape[0], f.N):
        raise ValueError("dy must be bf16 [T, N]")
    x = x.contiguous()
    dy = dy.contiguous()
    T = x.shape[0]
    ell = f.alpha.shape[0]
    dev = x.device
    if out is not None:
        dxt, da, db, dg = out
        shapes = ((ell, f.N), (ell, f.R), (ell, f.M))
        if any(t.dtype != torch.float32 or tuple(t.shape) != sh or not t.is_contiguous()
               for t, sh in zip((da, db, dg), shapes)):
            raise ValueError("out: dalpha, dbeta, dgamma must be contiguous fp32 [ell, N], [ell, R], [ell, M]")
        if dxt is not None and (dxt.dtype != torch.bfloat16 or tuple(dxt.shape) != (T, f.M)
                                or not dxt.is_contiguous()):
            raise ValueError("out: dx must be contiguous bf16 [T, M]")
    else:
        dxt = torch.empty((T, f.M), dtype=torch.bfloat16, device=dev) if dx else None
        da = torch.empty((ell, f.N), dtype=torch.float32, device=dev)
        db = torch.empty((ell, f.R), dtype=torch.float32, device=dev)
        dg = torch.empty((ell, f.M), dtype=torch.float32, device=dev)
    need = backward_workspace_bytes(f, T)
    if workspace is None:
        workspace = new_workspace(need, dev)
    rc = _lib.dbf_backward(ctypes.byref(f.struct), ctypes.byref(ft.struct), _ptr(x), _ptr(dy), T,
                           _ptr(dxt) if dxt is not None else None, _ptr(da), _ptr(db), _ptr(dg),
                           _ptr(workspace), workspace.numel(), _stream_handle(stream))
    _check(rc, "dbf_backward")
    return dxt, da, db, dg


def _group_structs(fs):
    arr = (DbfFactors * len(fs))()
    for k, f in enumerate(fs):
        arr[k] = f.struct
    return arr


def grouped_workspace_bytes(fs, T: int) -> int:
    return int(_lib.dbf_grouped_workspace_bytes(_group_structs(fs), len(fs), T))


def grouped_launch_count(fs, T: int) -> int:
    return int(_lib.dbf_grouped_launch_count(_group_structs(fs), len(fs), T))


@_on_stream
def matmul_grouped(fs, xs, ys=None, accumulate: bool = False, workspace: torch.Tensor | None = None, stream=None):
    """ys[p] = product of fs[p] applied to xs[p] for G independent projections (dbf_matmul_grouped).

    fs: list of PackedFactors (one ell); xs: list of bf16 [T, M_p]; ys: list of bf16 [T, N_p] or None.
    """
    G = len(fs)
    if G == 0 or len(xs) != G or (ys is not None and len(ys) != G):
        raise ValueError("fs, xs (and ys) must have the same non-zero length")
    xs = [x.contiguous() for x in xs]
    T = xs[0].shape[0]
    for f, x in zip(fs, xs):
        if x.dtype != torch.bfloat16 or x.dim() != 2 or x.shape != (T, f.M):
            raise ValueError("every x must be bf16 [T, M_p] with one T")
    if ys is None:
        if accumulate:
            raise ValueError("accumulate needs ys")
        ys = [torch.empty((T, f.N), dtype=torch.bfloat16, device=xs[0].device) for f in fs]
    structs = _group_structs(fs)
    need = int(_lib.dbf_grouped_workspace_bytes(structs, G, T))
    if workspace is None:
        workspace = new_workspace(need, xs[0].device)
    xp = (ctypes.c_void_p * G)(*[x.data_ptr() for x in xs])
    yp = (ctypes.c_void_p * G)(*[y.data_ptr() for y in ys])
    rc = _lib.dbf_matmul_grouped(structs, G, xp, yp, T, int(bool(accumulate)), _ptr(workspace),
                                 workspace.numel(), _stream_handle(stream))
    _check(rc, "dbf_matmul_grouped")
    return ys


def hostio_workspace_bytes(f: PackedFactors, T: int) -> int:
    return int(_lib.dbf_hostio_workspace_bytes(ctypes.byref(f.struct), T))


@_on_stream
def matmul_hostio(f: PackedFactors, x_host: torch.Tensor, y_host: torch.Tensor, accumulate: bool = False,
                  workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Host (pinned) bf16 x [T, M] in, host bf16 y [T, N] out (dbf_matmul_hostio); asynchronous."""
    T = x_host.shape[0]
    if workspace is None:
        workspace = new_workspace(hostio_workspace_bytes(f, T), torch.device("cuda"))
    rc = _lib.dbf_matmul_hostio(ctypes.byref(f.struct), _ptr(x_host), T, _ptr(y_host), int(bool(accumulate)),
                                _ptr(workspace), workspace.numel(), _stream_handle(stream))
    _check(rc, "dbf_matmul_hostio")
    return y_host


def hostio_batch_workspace_bytes(fs, T: int) -> int:
    return int(_lib.dbf_hostio_batch_workspace_bytes(_group_structs(fs), len(fs), T))


@_on_stream
def matmul_hostio_batch(fs, xs_host, ys_host, accumulate: bool = False, workspace: torch.Tensor | None = None,
                        stream=None):
    """L independent host-io calls, copies overlapped with the kernels (dbf_matmul_hostio_batch).

    fs: list of PackedFactors; xs_host, ys_host: lists of CPU bf16 tensors [T, M_l] and [T, N_l]
    (pinned for overlap).  Returns ys_host.
    """
    L = len(fs)
    if L == 0:
        return ys_host
    if len(xs_host) != L or len(ys_host) != L:
        raise ValueError("fs, xs_host and ys_host must have the same length")
    T = xs_host[0].shape[0]
    for f, x, y in zip(fs, xs_host, ys_host):
        if x.device.type != "cpu" or y.device.type != "cpu" or not x.is_contiguous() or not y.is_contiguous():
            raise ValueError("host tensors must be contiguous CPU tensors")
        if x.dtype != torch.bfloat16 or x.shape != (T, f.M) or y.dtype != torch.bfloat16 or y.shape != (T, f.N):
            raise ValueError("x_host bf16 [T, M_l] and y_host bf16 [T, N_l] with one T")
    structs = _group_structs(fs)
    need = int(_lib.dbf_hostio_batch_workspace_bytes(structs, L, T))
    if workspace is None:
        workspace = new_workspace(need, "cuda")
    xp = (ctypes.c_void_p * L)(*[x.data_ptr() for x in xs_host])
    yp = (ctypes.c_void_p * L)(*[y.data_ptr() for y in ys_host])
    rc = _lib.dbf_matmul_hostio_batch(structs, L, xp, yp, T, int(bool(accumulate)), _ptr(workspace),
                                      workspace.numel(), _stream_handle(stream))
    _check(rc, "dbf_matmul_hostio_batch")
    return ys_host


def adapter_table(adapters, device) -> torch.Tensor:
    """Device array of dbf_factors structs for matmul_segmented."""
    raw = b"".join(a.struct_bytes() for a in adapters)
    host = torch.frombuffer(bytearray(raw), dtype=torch.uint8)
    return host.to(device)


def segmented_workspace_bytes(N, M, R, ell, T, S) -> int:
    return int(_lib.dbf_segmented_workspace_bytes(N, M, R, ell, T, S))


@_on_stream
def matmul_segmented(table: torch.Tensor, n_adapters: int, N: int, M: int, R: int, ell: int, x: torch.Tensor,
                     seg_offsets: torch.Tensor, seg_adapter: torch.Tensor, y: torch.Tensor | None = None,
                     accumulate: bool = False, workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Routed multi-adapter call (dbf_matmul_segmented); offsets/adapters are device int32."""
    T = x.shape[0]
    S = seg_adapter.shape[0]
    if y is None:
        y = torch.zeros((T, N), dtype=torch.bfloat16, device=x.device)
    if workspace is None:
        workspace = new_workspace(segmented_workspace_bytes(N, M, R, ell, T, S), x.device)
    rc = _lib.dbf_matmul_segmented(_ptr(table), n_adapters, N, M, R, ell, _ptr(x), T, _ptr(y),
                                   _ptr(seg_offsets), _ptr(seg_adapter), S, int(bool(accumulate)),
                                   _ptr(workspace), workspace.numel(), _stream_handle(stream))
    _check(rc, "dbf_matmul_segmented")
    return y


def factorize_workspace_bytes(N: int, M: int, k: int) -> int:
    return int(_lib.dbf_factorize_workspace_bytes(N, M, k))


def factorize_launch_count(N: int, M: int, k: int, outer: int, inner: int, power_iters: int,
                           rho_rel: float) -> int:
    prm = DbfFactorizeParams(outer, inner, power_iters, rho_rel)
    return int(_lib.dbf_factorize_launch_count(N, M, k, ctypes.byref(prm)))


def _check_factor_tensors(W, a, A, m_left, m_right, B, b):
    if W.dtype != torch.float32 or W.dim() != 2:
        raise ValueError("W must be fp32 [N, M]")
    N, M = W.shape
    k = A.shape[1] if A.dim() == 2 else -1
    want = ((a, torch.float32, (N,)), (A, torch.int8, (N, k)), (m_left, torch.float32, (k,)),
            (m_right, torch.float32, (k,)), (B, torch.int8, (k, M)), (b, torch.float32, (M,)))
    for t, dt, sh in want:
        if t.dtype != dt or tuple(t.shape) != sh or not t.is_contiguous() or t.device != W.device:
            raise ValueError("factors: a fp32 [N], A int8 [N, k], m_left fp32 [k], m_right fp32 [k], "
                             "B int8 [k, M], b fp32 [M], contiguous, on W's device")
    return N, M, k


def factorize_weighted_workspace_bytes(N: int, M: int, k: int) -> int:
    return int(_lib.dbf_factorize_weighted_workspace_bytes(N, M, k))


def factorize_weighted_launch_count(N: int, M: int, k: int, outer: int, inner: int, power_iters: int,
                                    rho_rel: float) -> int:
    prm = DbfFactorizeParams(outer, inner, power_iters, rho_rel)
    return int(_lib.dbf_factorize_weighted_launch_count(N, M, k, ctypes.byref(prm)))


@_on_stream
def factorize_weighted(W: torch.Tensor, d_out: torch.Tensor, d_in: torch.Tensor, a: torch.Tensor,
                       A: torch.Tensor, m_left: torch.Tensor, m_right: torch.Tensor, B: torch.Tensor,
                       b: torch.Tensor, outer: int = 6, inner: int = 10, power_iters: int = 8,
                       rho_rel: float = 1.0, workspace: torch.Tensor | None = None, stream=None):
    """factorize with importance weights d_out fp32 [N], d_in fp32 [M] (dbf_factorize_weighted):
    the error ||diag(d_out)(W - W_hat)diag(d_in)|| is minimised.  Factors updated in place."""
    N, M, k = _check_factor_tensors(W, a, A, m_left, m_right, B, b)
    for t, n in ((d_out, N), (d_in, M)):
        if t.dtype != torch.float32 or tuple(t.shape) != (n,) or not t.is_contiguous() or t.device != W.device:
            raise ValueError("d_out, d_in: contiguous fp32 [N], [M] on W's device")
    W = W.contiguous()
    prm = DbfFactorizeParams(outer, inner, power_iters, rho_rel)
    if workspace is None:
        workspace = new_workspace(max(factorize_weighted_workspace_bytes(N, M, k), 256), W.device)
    rc = _lib.dbf_factorize_weighted(_ptr(W), N, M, k, ctypes.byref(prm), _ptr(d_out), _ptr(d_in), _ptr(a),
                                     _ptr(A), _ptr(m_left), _ptr(m_right), _ptr(B), _ptr(b), _ptr(workspace),
                                     workspace.numel(), _stream_handle(stream))
    _check(rc, "dbf_factorize_weighted")
    return a, A, m_left, m_right, B, b


@_on_stream
def factorize(W: torch.Tensor, a: torch.Tensor, A: torch.Tensor, m_left: torch.Tensor, m_right: torch.Tensor,
              B: torch.Tensor, b: torch.Tensor, outer: int = 6, inner: int = 10, power_iters: int = 8,
              rho_rel: float = 1.0, workspace: torch.Tensor | None = None, stream=None):
    """Double binary factorization W ~ (a . A . m^T)(B . b^T), m = m_left . m_right (dbf_factorize).

    W fp32 [N, M]; the left factor a fp32 [N], A int8 [N, k], m_left fp32 [k] and the
    right factor m_right fp32 [k], B int8 [k, M], b fp32 [M] are device tensors updated
    in place (the left factor is the start of the first step; the right one is fixed
    in it).  Returns (a, A, m_left, m_right, B, b).
    """
    N, M, k = _check_factor_tensors(W, a, A, m_left, m_right, B, b)
    W = W.contiguous()
    prm = DbfFactorizeParams(outer, inner, power_iters, rho_rel)
    need = factorize_workspace_bytes(N, M, k)
    if workspace is None:
        workspace = new_workspace(max(need, 256), W.device)
    rc = _lib.dbf_factorize(_ptr(W), N, M, k, ctypes.byref(prm), _ptr(a), _ptr(A), _ptr(m_left), _ptr(m_right),
                            _ptr(B), _ptr(b), _ptr(workspace), workspace.numel(), _stream_handle(stream))
    _check(rc, "dbf_factorize")
    return a, A, m_left, m_right, B, b


def check_status(stream=None) -> int:
    """Synchronise the stream, return and clear the device status word (dbf_check_status)."""
    return int(_lib.dbf_check_status(_stream_handle(stream)))


def selftest_bounded_wait(limit_us: int, stream=None) -> int:
    return int(_lib.dbf_selftest_bounded_wait(limit_us, _stream_handle(stream)))


@_on_stream
def selftest_split_gemm(A: torch.Tensor, B: torch.Tensor, C: torch.Tensor, alpha: float = 1.0, beta: float = 0.0,
                        lower: bool = False, stream=None) -> torch.Tensor:
    """C = alpha A B^T + beta C on the factorization's split-tf32 tensor-core GEMM
    (dbf_selftest_split_gemm); A [m, kk], B [n, kk], C [m, n], fp32 CUDA tensors, rows contiguous."""
    for t in (A, B, C):
        if t.dtype != torch.float32 or t.dim() != 2 or not t.is_cuda or t.stride(1) != 1:
            raise ValueError("A, B and C must be 2-D fp32 CUDA tensors with contiguous rows")
    m, kk = A.shape
    n = B.shape[0]
    if B.shape[1] != kk or tuple(C.shape) != (m, n):
        raise ValueError("shapes must be A [m, kk], B [n, kk], C [m, n]")
    ws = new_workspace(int(_lib.dbf_selftest_split_gemm_workspace_bytes(m, n, kk)), A.device)
    _check(_lib.dbf_selftest_split_gemm(m, n, kk, alpha, _ptr(A), A.stride(0), _ptr(B), B.stride(0), beta, _ptr(C),
                                        C.stride(0), int(lower), _ptr(ws), ws.numel(), _stream_handle(stream)),
           "dbf_selftest_split_gemm")
    return C


@_on_stream
def selftest_decode_one_launch(f: PackedFactors, x: torch.Tensor, barrier: torch.Tensor,
                               y: torch.Tensor | None = None, accumulate: bool = False,
                               workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """The decode path's two stages in one cooperative launch (dbf_selftest_decode_one_launch).
    barrier: int32 CUDA tensor of >= 2 elements, zero before the first call, one per concurrent stream."""
    if x.dtype != torch.bfloat16 or x.dim() != 2 or x.shape[1] != f.M:
        raise ValueError("x must be bf16 [T, M]")
    if barrier.dtype != torch.int32 or not barrier.is_cuda or barrier.numel() < 2:
        raise ValueError("barrier must be an int32 CUDA tensor of at least 2 elements")
    x = x.contiguous()
    T = x.shape[0]
    if y is None:
        if accumulate:
            raise ValueError("accumulate needs y")
        y = torch.empty((T, f.N), dtype=torch.bfloat16, device=x.device)
    if workspace is None:
        workspace = new_workspace(workspace_bytes(f, T, PATH_DECODE), x.device)
    rc = _lib.dbf_selftest_decode_one_launch(ctypes.byref(f.struct), _ptr(x), T, _ptr(y), int(bool(accumulate)),
                                             _ptr(workspace), workspace.numel(), _ptr(barrier),
                                             _stream_handle(stream))
    _check(rc, "dbf_selftest_decode_one_launch")
    return y


# ------------------------------------------------------- no-allocation variant

_lib.dbf_matmul_decode_noalloc.restype = ctypes.c_int
_lib.dbf_matmul_decode_noalloc.argtypes = [ctypes.POINTER(DbfFactors), ctypes.c_void_p, ctypes.c_int64,
                                           ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p]


@_on_stream
def matmul_decode_noalloc(f: PackedFactors, x: torch.Tensor, y: torch.Tensor | None = None,
                          accumulate: bool = False, stream=None) -> torch.Tensor:
    """Decode-path product with the library's static scratch (dbf_matmul_decode_noalloc).

    For callers that cannot allocate device memory; needs no workspace.  The
    output tensor is allocated here only when y is None.
    """
    if x.dtype != torch.bfloat16 or x.dim() != 2 or x.shape[1] != f.M:
        raise ValueError("x must be bf16 [T, M]")
    x = x.contiguous()
    T = x.shape[0]
    if y is None:
        y = torch.empty((T, f.N), dtype=torch.bfloat16, device=x.device)
    rc = _lib.dbf_matmul_decode_noalloc(ctypes.byref(f.struct), _ptr(x), T, _ptr(y), int(bool(accumulate)),
                                        _stream_handle(stream))
    _check(rc, "dbf_matmul_decode_noalloc")
    return y
