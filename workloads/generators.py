"""Seeded synthetic inputs for the packed double-binary matmul.

This module only draws random numbers and rounds them to the storage types
(int8 signs, fp16 scales, bf16 activations).  It holds none of the method's
arithmetic, so both the fp64 oracle and the CUDA path can take their inputs
from here without sharing any computation.

Storage conventions (all numpy, host side):
  signs   int8, values exactly +1 or -1
  fp16    numpy.float16 arrays (the bit pattern is what the library reads)
  bf16    numpy.uint16 arrays holding bf16 bit patterns (numpy has no bf16)

Draw recipe (fixed so that every run and every machine sees the same data):
  factors:  rng = default_rng(seed);  B1 [N,R], then B2 [R,M], then alpha
            [ell,N], beta [ell,R], gamma [ell,M]
  x:        rng = default_rng(seed + 500); x [T,M] row-major, so the first T'
            rows of a T-row draw equal a T'-row draw
  integer x: rng = default_rng(seed + 501), uniform integers in [-4, 4]
  outlier columns: rng = default_rng(seed + 502), chosen without replacement
  dense W:  rng = default_rng(seed + 600); W [N,M] = N(0,1) * 0.02 times a
            per-row factor exp(N(0, 0.25)) (rows of unequal norm), float32
  factorization start: rng = default_rng(seed + 601); B [k,M] signs; the
            other parts are constants (a = 0, A = +1, m_left = 0,
            m_right = 1, b = 1)
"""

from __future__ import annotations

import numpy as np


def f32_to_bf16_bits(a) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest, ties to even); return bits.

    Input values must be finite.  The input is first taken to float32 (numpy's
    correctly rounded float64 -> float32 conversion), then the low 16 bits are
    rounded away.
    """
    f = np.ascontiguousarray(np.asarray(a, dtype=np.float32))
    bits = f.view(np.uint32).astype(np.uint64)
    lsb = (bits >> 16) & 1
    rounded = (bits + 0x7FFF + lsb) >> 16
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(bits) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32)


def draw_signs(rng: np.random.Generator, shape, mode: str) -> np.ndarray:
    """Draw a +-1 int8 matrix.

    mode "bernoulli": +1 where rng.random() < 0.5 (i.i.d. p = 0.5)
    mode "gauss":     the sign of an N(0,1) draw, with sign(0) taken as +1
    """
    if mode == "bernoulli":
        u = rng.random(shape)
        return np.where(u < 0.5, 1, -1).astype(np.int8)
    if mode == "gauss":
        g = rng.standard_normal(shape)
        return np.where(g >= 0.0, 1, -1).astype(np.int8)
    raise ValueError(f"unknown sign mode {mode!r}")


def draw_scales(rng: np.random.Generator, ell: int, n: int, mode: str, R: int) -> np.ndarray:
    """Draw an [ell, n] fp16 scale array.

    mode "abs005":   |N(0, 0.05)| + 1e-3          (tiny workload)
    mode "abs002":   |N(0, 0.02)|                 (alpha and gamma elsewhere)
    mode "beta":     |N(0, 1)| / sqrt(R)          (beta elsewhere)
    mode "ones":     exactly 1                    (integer mode)
    Values are formed in float64 and rounded once to fp16 (numpy's
    float64 -> float16 conversion rounds to nearest even; subnormals kept).
    """
    if mode == "ones":
        return np.ones((ell, n), dtype=np.float16)
    g = rng.standard_normal((ell, n))
    if mode == "abs005":
        v = np.abs(g) * 0.05 + 1e-3
    elif mode == "abs002":
        v = np.abs(g) * 0.02
    elif mode == "beta":
        v = np.abs(g) / np.sqrt(float(R))
    else:
        raise ValueError(f"unknown scale mode {mode!r}")
    return v.astype(np.float16)


class Factors:
    """One set of double-binary factors in host memory (unpacked signs)."""

    def __init__(self, B1, B2, alpha, beta, gamma):
        self.B1 = B1          # int8 [N, R]
        self.B2 = B2          # int8 [R, M]
        self.alpha = alpha    # fp16 [ell, N]
        self.beta = beta      # fp16 [ell, R]
        self.gamma = gamma    # fp16 [ell, M]

    @property
    def N(self):
        return self.B1.shape[0]

    @property
    def R(self):
        return self.B1.shape[1]

    @property
    def M(self):
        return self.B2.shape[1]

    @property
    def ell(self):
        return self.alpha.shape[0]


def make_factors(N: int, M: int, R: int, ell: int, seed: int,
                 sign_mode: str = "bernoulli", scale_mode: str = "lordba",
                 unit_scales: bool = False) -> Factors:
    """Draw B1, B2, alpha, beta, gamma for one projection.

    scale_mode "tiny":   alpha, beta, gamma all |N(0,0.05)| + 1e-3
    scale_mode "lordba": alpha, gamma |N(0,0.02)|; beta |N(0,1)|/sqrt(R)
    unit_scales=True replaces every scale by exactly 1 (integer mode).
    """
    rng = np.random.default_rng(seed)
    B1 = draw_signs(rng, (N, R), sign_mode)
    B2 = draw_signs(rng, (R, M), sign_mode)
    if unit_scales:
        modes = ("ones", "ones", "ones")
    elif scale_mode == "tiny":
        modes = ("abs005", "abs005", "abs005")
    elif scale_mode == "lordba":
        modes = ("abs002", "beta", "abs002")
    else:
        raise ValueError(f"unknown scale mode {scale_mode!r}")
    alpha = draw_scales(rng, ell, N, modes[0], R)
    beta = draw_scales(rng, ell, R, modes[1], R)
    gamma = draw_scales(rng, ell, M, modes[2], R)
    return Factors(B1, B2, alpha, beta, gamma)


def outlier_columns(M: int, seed: int, frac: float = 0.01) -> np.ndarray:
    """round(frac*M) distinct input columns, drawn from default_rng(seed+502)."""
    k = int(round(frac * M))
    rng = np.random.default_rng(seed + 502)
    return np.sort(rng.choice(M, size=k, replace=False))


def make_x(T: int, M: int, seed: int, outlier_scale: float = 0.0,
           integer: bool = False) -> np.ndarray:
    """Draw activations x [T, M] as bf16 bits (numpy uint16).

    Normal mode: N(0,1) in float64; when outlier_scale > 0 the 1% outlier
    columns are multiplied by it; then rounded to bf16.
    Integer mode: uniform integers in [-4, 4] (exact in bf16).
    """
    if integer:
        rng = np.random.default_rng(seed + 501)
        v = rng.integers(-4, 5, size=(T, M)).astype(np.float64)
        return f32_to_bf16_bits(v)
    rng = np.random.default_rng(seed + 500)
    v = rng.standard_normal((T, M))
    if outlier_scale > 0.0:
        cols = outlier_columns(M, seed)
        v[:, cols] *= outlier_scale
    return f32_to_bf16_bits(v)


def make_routing(T: int, n_adapters: int, seed: int):
    """Assign each of T tokens uniformly to an adapter, sorted by adapter.

    Returns (seg_offsets int32 [S+1], seg_adapter int32 [S], token_adapter
    int32 [T]) where segment s covers tokens [off[s], off[s+1]) and every
    segment is non-empty.  Drawn from default_rng(seed).
    """
    rng = np.random.default_rng(seed)
    a = np.sort(rng.integers(0, n_adapters, size=T)).astype(np.int32)
    offsets = [0]
    adapters = []
    for t in range(T):
        if t == 0 or a[t] != a[t - 1]:
            if t > 0:
                offsets.append(t)
            adapters.append(int(a[t]))
    offsets.append(T)
    return (np.asarray(offsets, dtype=np.int32),
            np.asarray(adapters, dtype=np.int32), a)


def make_dense_weight(N: int, M: int, seed: int) -> np.ndarray:
    """A dense float32 weight W [N, M] to factorize: N(0, 0.02^2) entries with
    log-normal row norms (sigma 0.25), drawn from default_rng(seed + 600)."""
    rng = np.random.default_rng(seed + 600)
    w = rng.standard_normal((N, M)) * 0.02
    w *= np.exp(0.25 * rng.standard_normal((N, 1)))
    return w.astype(np.float32)


def make_factorize_start(N: int, M: int, k: int, seed: int):
    """Starting factors of a factorization: a zero left factor (a = 0, A = +1,
    m_left = 0) and a right factor of random signs with unit scales.
    Returns (a, A, m_left, m_right, B, b) as float32 / int8 numpy arrays."""
    rng = np.random.default_rng(seed + 601)
    B = draw_signs(rng, (k, M), "bernoulli")
    return (np.zeros(N, np.float32), np.ones((N, k), np.int8), np.zeros(k, np.float32),
            np.ones(k, np.float32), B, np.ones(M, np.float32))
