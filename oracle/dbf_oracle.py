"""fp64 CPU oracle for the packed double-binary matmul.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import or call
this module: only the tests, the smoke check and the CPU-baseline leg of the
benchmark use it.  It shares no code with the CUDA library.

What it computes (plain definitions, evaluated in float64):

  LoRDBA - "Adaptación Binaria Doble de Bajo Rango", section 2
  (Metodología, Arquitectura Central): the adapter update is
      dW = sum_{i=1..ell} diag(alpha_i) B1 diag(beta_i) B2 diag(gamma_i)
  with B1 in {+1,-1}^{N x R}, B2 in {+1,-1}^{R x M}, 1 bit per sign entry
  and fp16 per-channel scale vectors.  Only the scales carry the index i;
  B1 and B2 are shared by the ell terms.

  "Addition is almost all you need: Compressing large language models with
  double binary factorization", section 2 (Formulación Matemática, Cálculo
  en la inferencia): a linear layer X W^T with W ~ (a . A . m^T)(B . b^T)
  is evaluated as ((((X . b^T) B^T) . m^T) A^T) . a^T.  This is the ell = 1
  case of the update above with a = alpha, A = B1, m = beta, B = B2,
  b = gamma, and it fixes the orientation y = x dW^T with x [T, M] and
  y [T, N].

Two independent routes are provided: the dense route (build dW, then x dW^T)
and the factored route (gamma, B2, beta, B1, alpha in that order).  A third,
scalar brute-force loop exists for tiny sizes.  The result is exact up to
floating-point rounding: the method is not an approximation of anything once
the factors are given.

Readings where the pages are silent:
  * output rounding: the final y is rounded once to bf16, round to nearest
    even, from the exact (float64) value; the pages give no output type.
  * accumulate mode: y = bf16(y_in + branch) with a single rounding, the
    unmerged adapter branch added onto a base output.
  * bit order: bit j of word w of row r holds the sign of column 32w + j
    (least significant bit first), 1 means +1, words are row-major with a
    row stride of ldw words, and bits past the last column are 0.  The pages
    fix only "1 bit per entry".
  * sign(0) is taken as +1 when packing; any entry > 0 packs to bit 1.

Pins (tests/test_oracle_pins.py): closed forms (all-ones signs collapse to a
rank-1 product; a permuted Sylvester-Hadamard pair gives a diagonal dW),
symmetries (paired sign flips, row flips, linearity), dense route = factored
route, brute force on N=M=8, R=4, exact integer results, bf16 rounding
against an independent library conversion, and hand-derived golden fixtures.
"""

from __future__ import annotations

import numpy as np


# --------------------------------------------------------------------------
# storage format (bits, fp16, bf16)
# --------------------------------------------------------------------------

def words_per_row(cols: int) -> int:
    """Smallest row stride in 32-bit words that holds `cols` sign bits."""
    return (cols + 31) // 32


def pack_signs(signs: np.ndarray, ldw: int | None = None) -> np.ndarray:
    """Pack a sign matrix into LSB-first uint32 words, row-major.

    Bit j of word w in row r is 1 exactly when signs[r, 32*w + j] > 0.
    Bits past the last column and words past ceil(cols/32) are 0.
    """
    s = np.asarray(signs)
    rows, cols = s.shape
    if ldw is None:
        ldw = words_per_row(cols)
    if ldw < words_per_row(cols):
        raise ValueError("ldw too small for cols")
    bits = np.zeros((rows, ldw * 32), dtype=np.uint64)
    bits[:, :cols] = (s > 0).astype(np.uint64)
    bits = bits.reshape(rows, ldw, 32)
    weights = np.left_shift(np.uint64(1), np.arange(32, dtype=np.uint64))
    words = (bits * weights).sum(axis=2)
    return words.astype(np.uint32)


def unpack_words(words: np.ndarray, cols: int) -> np.ndarray:
    """Inverse of pack_signs: int8 +1 where the bit is 1, -1 where it is 0."""
    w = np.asarray(words, dtype=np.uint32)
    rows, ldw = w.shape
    if ldw * 32 < cols:
        raise ValueError("not enough words for cols")
    shifts = np.arange(32, dtype=np.uint32)
    bits = (w[:, :, None] >> shifts[None, None, :]) & np.uint32(1)
    bits = bits.reshape(rows, ldw * 32)[:, :cols]
    return np.where(bits == 1, 1, -1).astype(np.int8)


def fp16_to_f64(a) -> np.ndarray:
    """Exact widening of numpy float16 values to float64."""
    return np.asarray(a, dtype=np.float16).astype(np.float64)


def bf16_bits_to_f64(bits) -> np.ndarray:
    """Exact widening of bf16 bit patterns (uint16) to float64."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def round_to_bf16_bits(v) -> np.ndarray:
    """Round float64 values to bf16 (nearest, ties to even) in one step.

    bf16 keeps 8 significant bits.  A value with frexp exponent e (v = f*2^e,
    0.5 <= |f| < 1) sits on a grid of spacing 2^(e-8); below the smallest
    normal 2^-126 the grid spacing stays 2^-133.  Rounding to that grid with
    ties to even, then reading the (now exactly representable) value as
    float32, gives the bf16 bits.  Values past the largest bf16 become inf.
    """
    v = np.asarray(v, dtype=np.float64)
    _, e = np.frexp(v)
    e_eff = np.maximum(e, -125)
    q = np.rint(np.ldexp(v, 8 - e_eff))
    r = np.ldexp(q, e_eff - 8)
    with np.errstate(over="ignore"):
        r32 = r.astype(np.float32)
    return (r32.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


# --------------------------------------------------------------------------
# the product, three ways
# --------------------------------------------------------------------------

def _scales(f):
    return fp16_to_f64(f.alpha), fp16_to_f64(f.beta), fp16_to_f64(f.gamma)


def dense_delta_w(f) -> np.ndarray:
    """dW [N, M] = sum_i diag(alpha_i) B1 diag(beta_i) B2 diag(gamma_i).

    LoRDBA page, section 2 (Arquitectura Central).  Each term is formed as a
    product of the five matrices exactly as written, in float64.
    """
    alpha, beta, gamma = _scales(f)
    B1 = np.asarray(f.B1, dtype=np.float64)
    B2 = np.asarray(f.B2, dtype=np.float64)
    dW = np.zeros((B1.shape[0], B2.shape[1]), dtype=np.float64)
    for i in range(alpha.shape[0]):
        dW += np.diag(alpha[i]) @ B1 @ np.diag(beta[i]) @ B2 @ np.diag(gamma[i])
    return dW


def y_dense(x64: np.ndarray, f) -> np.ndarray:
    """y [T, N] = x dW^T through the dense update (DBF page: X W^T)."""
    return np.asarray(x64, dtype=np.float64) @ dense_delta_w(f).T


def y_factored(x64: np.ndarray, f) -> np.ndarray:
    """y [T, N] through the factored route, one envelope term at a time.

    DBF page, section 2 (Cálculo en la inferencia): scale the input by
    gamma_i, contract with B2 (over M), scale by beta_i, contract with B1
    (over R), scale by alpha_i; the LoRDBA sum over i adds the terms.
    """
    alpha, beta, gamma = _scales(f)
    x = np.asarray(x64, dtype=np.float64)
    B1 = np.asarray(f.B1, dtype=np.float64)
    B2 = np.asarray(f.B2, dtype=np.float64)
    y = np.zeros((x.shape[0], B1.shape[0]), dtype=np.float64)
    for i in range(alpha.shape[0]):
        xs = x * gamma[i][None, :]          # X . gamma_i^T        [T, M]
        u = xs @ B2.T                       # (.) B2^T              [T, R]
        v = u * beta[i][None, :]            # (.) . beta_i^T        [T, R]
        w = v @ B1.T                        # (.) B1^T              [T, N]
        y += w * alpha[i][None, :]          # (.) . alpha_i^T       [T, N]
    return y


def y_bruteforce(x64: np.ndarray, f) -> np.ndarray:
    """Scalar loop over (t, n, i, r, m); only for tiny shapes."""
    alpha, beta, gamma = _scales(f)
    x = np.asarray(x64, dtype=np.float64)
    T, M = x.shape
    N, R = f.B1.shape
    y = np.zeros((T, N), dtype=np.float64)
    for t in range(T):
        for n in range(N):
            acc = 0.0
            for i in range(alpha.shape[0]):
                for r in range(R):
                    for m in range(M):
                        acc += (alpha[i, n] * float(f.B1[n, r]) * beta[i, r]
                                * float(f.B2[r, m]) * gamma[i, m] * x[t, m])
            y[t, n] = acc
    return y


def y_sampled(x64: np.ndarray, f, tokens, outputs) -> np.ndarray:
    """y[t, n] for the listed tokens t and output channels n only.

    Same factored route, restricted: u_i is formed for the chosen tokens
    over all R, then each requested output is one dot product over R.
    Returns an array [len(tokens), len(outputs)].
    """
    alpha, beta, gamma = _scales(f)
    x = np.asarray(x64, dtype=np.float64)[np.asarray(tokens)]
    B1 = np.asarray(f.B1[np.asarray(outputs)], dtype=np.float64)   # [n', R]
    B2 = np.asarray(f.B2, dtype=np.float64)
    out = np.zeros((x.shape[0], B1.shape[0]), dtype=np.float64)
    for i in range(alpha.shape[0]):
        u = (x * gamma[i][None, :]) @ B2.T
        v = u * beta[i][None, :]
        out += (v @ B1.T) * alpha[i][np.asarray(outputs)][None, :]
    return out


def transpose_packed(words: np.ndarray, cols: int, ldw_t: int | None = None) -> np.ndarray:
    """Packed words of the transposed sign matrix.

    `words` holds a rows x cols sign matrix (see pack_signs); the result holds
    its cols x rows transpose in the same format, row stride ldw_t words.
    """
    signs = unpack_words(words, cols)
    return pack_signs(signs.T, ldw_t)


def dx_factored(dy64: np.ndarray, f) -> np.ndarray:
    """Input gradient of y = x dW^T for the output gradient dy [T, N]: dx [T, M].

    dx = dy dW = sum_i gamma_i . B2^T (beta_i . (B1^T (alpha_i . dy))), the
    backward pass of the sign-factor product that training through it needs
    (LoRDBA page, section 2, Pipeline de Entrenamiento: the carriers and scales
    are trained jointly, so the gradient flows back through both sign
    matrices).  Term by term, in this order: scale dy by alpha_i, contract
    with B1 over N, scale by beta_i, contract with B2 over R, scale by gamma_i.
    """
    alpha, beta, gamma = _scales(f)
    dy = np.asarray(dy64, dtype=np.float64)
    B1 = np.asarray(f.B1, dtype=np.float64)
    B2 = np.asarray(f.B2, dtype=np.float64)
    dx = np.zeros((dy.shape[0], B2.shape[1]), dtype=np.float64)
    for i in range(alpha.shape[0]):
        g = (dy * alpha[i][None, :]) @ B1      # B1^T (alpha_i . dy)   [T, R]
        h = (g * beta[i][None, :]) @ B2        # B2^T (beta_i . g)     [T, M]
        dx += h * gamma[i][None, :]
    return dx


def scale_grads_f64(x64: np.ndarray, dy64: np.ndarray, f):
    """Gradients of L = sum_t <dy_t, y_t> with respect to the scale vectors.

    Training through the product updates the scales together with the sign
    carriers (LoRDBA page, section 2, Pipeline de Entrenamiento), so besides
    dx it needs, for each envelope term i and the output gradient dy [T, N]:
      dalpha_i[n] = sum_t dy_t[n] * (B1 (beta_i . B2 (gamma_i . x_t)))[n]
      dbeta_i[r]  = sum_t (B1^T (alpha_i . dy_t))[r] * (B2 (gamma_i . x_t))[r]
      dgamma_i[k] = sum_t x_t[k] * (B2^T (beta_i . B1^T (alpha_i . dy_t)))[k]
    (y is linear in each of alpha_i, beta_i, gamma_i, so these are the
    coefficients of that linear dependence).  The intermediates are formed
    term by term in the order of the forward and backward products.
    Returns (dalpha [ell, N], dbeta [ell, R], dgamma [ell, M]) in float64.
    """
    alpha, beta, gamma = _scales(f)
    x = np.asarray(x64, dtype=np.float64)
    dy = np.asarray(dy64, dtype=np.float64)
    B1 = np.asarray(f.B1, dtype=np.float64)
    B2 = np.asarray(f.B2, dtype=np.float64)
    ell = alpha.shape[0]
    dalpha = np.zeros((ell, B1.shape[0]))
    dbeta = np.zeros((ell, B1.shape[1]))
    dgamma = np.zeros((ell, B2.shape[1]))
    for i in range(ell):
        h = (x * gamma[i][None, :]) @ B2.T      # B2 (gamma_i . x_t)        [T, R]
        u = (h * beta[i][None, :]) @ B1.T       # B1 (beta_i . h_t)         [T, N]
        g = (dy * alpha[i][None, :]) @ B1       # B1^T (alpha_i . dy_t)     [T, R]
        w = (g * beta[i][None, :]) @ B2         # B2^T (beta_i . g_t)       [T, M]
        dalpha[i] = (dy * u).sum(axis=0)
        dbeta[i] = (g * h).sum(axis=0)
        dgamma[i] = (x * w).sum(axis=0)
    return dalpha, dbeta, dgamma


def scale_grads_sampled(x64: np.ndarray, dy64: np.ndarray, f, n_idx, r_idx, k_idx):
    """scale_grads_f64 restricted to the listed output channels n, middle
    channels r and input channels k (same definitions; only the columns of
    the intermediates those entries need are formed, except g, which dgamma
    needs whole).  Returns (dalpha [ell, len(n_idx)], dbeta [ell, len(r_idx)],
    dgamma [ell, len(k_idx)]).
    """
    alpha, beta, gamma = _scales(f)
    x = np.asarray(x64, dtype=np.float64)
    dy = np.asarray(dy64, dtype=np.float64)
    n_idx, r_idx, k_idx = (np.asarray(v) for v in (n_idx, r_idx, k_idx))
    B1 = np.asarray(f.B1, dtype=np.float64)
    B2 = np.asarray(f.B2, dtype=np.float64)
    ell = alpha.shape[0]
    da = np.zeros((ell, n_idx.size))
    db = np.zeros((ell, r_idx.size))
    dg = np.zeros((ell, k_idx.size))
    for i in range(ell):
        h = (x * gamma[i][None, :]) @ B2.T                       # [T, R]
        u_n = (h * beta[i][None, :]) @ B1[n_idx].T               # [T, n']
        g = (dy * alpha[i][None, :]) @ B1                        # [T, R]
        w_k = (g * beta[i][None, :]) @ B2[:, k_idx]              # [T, k']
        da[i] = (dy[:, n_idx] * u_n).sum(axis=0)
        db[i] = (g[:, r_idx] * h[:, r_idx]).sum(axis=0)
        dg[i] = (x[:, k_idx] * w_k).sum(axis=0)
    return da, db, dg


def scale_grads(x_bits: np.ndarray, dy_bits: np.ndarray, f):
    """Reference for the backward call's scale gradients from bf16 x and dy."""
    return scale_grads_f64(bf16_bits_to_f64(x_bits), bf16_bits_to_f64(dy_bits), f)


def matmul_dx(dy_bits: np.ndarray, f):
    """Reference for the backward call: (exact float64 dx, expected bf16 bits)."""
    dx = dx_factored(bf16_bits_to_f64(dy_bits), f)
    return dx, round_to_bf16_bits(dx)


# --------------------------------------------------------------------------
# what the library call must return
# --------------------------------------------------------------------------

def matmul(x_bits: np.ndarray, f, y_in_bits: np.ndarray | None = None):
    """Reference for one call: (exact float64 y, expected bf16 bits of y).

    x_bits: bf16 bits [T, M].  With y_in_bits the branch is added to the
    widened y_in before the single rounding (accumulate mode).
    """
    y = y_factored(bf16_bits_to_f64(x_bits), f)
    if y_in_bits is not None:
        y = y + bf16_bits_to_f64(y_in_bits)
    return y, round_to_bf16_bits(y)


def matmul_grouped(x_bits_list, factor_list, y_in_bits_list=None):
    """Reference for a grouped call: [(exact y, expected bf16 bits)] per problem.

    Independent products with their own factors, e.g. layers whose middle
    dimension differs (DBF page, section 2, Control Granular de Compresión:
    the ratio is set per layer through k).  Each entry is `matmul` of its
    own problem; nothing couples them.
    """
    out = []
    for p, (xb, f) in enumerate(zip(x_bits_list, factor_list)):
        y_in = None if y_in_bits_list is None else y_in_bits_list[p]
        out.append(matmul(xb, f, y_in))
    return out


def matmul_segmented(x_bits: np.ndarray, adapters, seg_offsets, seg_adapter,
                     y_in_bits: np.ndarray | None = None):
    """Reference for a routed batch: tokens [off[s], off[s+1]) use adapter seg_adapter[s].

    Multi-adapter serving as on the LoRDBA page (section 1, S-LoRA / Punica
    style batches of unmerged adapters): each segment of the sorted token
    batch is one ordinary call with its own factors.  Tokens outside every
    segment are left as y_in (or 0 when y_in is absent).
    """
    x = bf16_bits_to_f64(x_bits)
    T = x.shape[0]
    N = adapters[0].B1.shape[0]
    y = np.zeros((T, N), dtype=np.float64) if y_in_bits is None else bf16_bits_to_f64(y_in_bits).copy()
    off = np.asarray(seg_offsets)
    for s, a in enumerate(np.asarray(seg_adapter)):
        t0, t1 = int(off[s]), int(off[s + 1])
        if t1 > t0:
            y[t0:t1] += y_factored(x[t0:t1], adapters[int(a)])
    return y, round_to_bf16_bits(y)


def rel_frobenius(a, b) -> float:
    """||a - b||_F / ||b||_F in float64 (0 when both are 0)."""
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    nb = np.linalg.norm(b)
    if nb == 0.0:
        return float(np.linalg.norm(a))
    return float(np.linalg.norm(a - b) / nb)
