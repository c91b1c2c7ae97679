"""fp64 CPU oracle for the double binary factorization of a dense matrix.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import or call
this module: only the tests, the smoke check and the CPU legs of the
benchmark use it.  It shares no code with the CUDA library.

What it computes.  "Addition is almost all you need: Compressing large
language models with double binary factorization", section 2 (Formulación
Matemática): a dense W [N x M] is approximated by

    W ~ (a . A . m^T)(B . b^T),   A in {+1,-1}^{N x k},  B in {+1,-1}^{k x M},

with scale vectors a [N], m [k], b [M].  Section 2 (Algoritmo de
Optimización) outlines how the factors are found: the problem is NP-hard, so
A and B are optimised in turn with the other held fixed (alternating
minimisation); each subproblem is solved by ADMM, whose projection onto the
set of matrices of the form a . S . m^T (S a sign matrix) is the SVID step:
the sign of the matrix times a rank-1 approximation of its magnitude.

Written out (the pages give the steps, not the equations; the readings below
fill them in):

  left factor P = diag(a) A diag(mL) [N x k], right factor
  Q = diag(mR) B diag(b) [k x M], so W ~ P Q and m = mL . mR.

  A-step: min_P 1/2 ||W - P Q||_F^2  subject to P = diag(r) S diag(c).
  B-step: the same problem for W^T ~ Q^T P^T (the left factor of the
          transposed problem is Q^T = diag(b) B^T diag(mR)).

  ADMM (scaled form) for one step with target T [n x p] and fixed F [k x p]:
      P <- (T F^T + rho (Z - U)) (F F^T + rho I)^-1
      Z <- SVID(P + U)
      U <- U + P - Z
  starting from Z = the current left factor, U = 0; the result is the last Z.

  SVID(Y): S = sign(Y); |Y| ~ r c^T by power iteration from the all-ones
  direction: v = 1/sqrt(k); q times {u = |Y| v; v = |Y|^T u; v = v/||v||};
  then c = v and r = |Y| c (the least-squares row scale for that c).

Readings where the pages are silent (each stated once here):
  * scaled-form ADMM with the 1/2 in the objective (the P-update above);
  * rho = rho_rel * mean(diag(F F^T)), fixed during a step; if F is zero,
    rho = rho_rel (no penalty schedule is given);
  * fixed iteration counts: `outer` alternations (A-step then B-step),
    `inner` ADMM iterations per step, `power_iters` power iterations per
    SVID; the pages give no stopping rule;
  * warm start: each step starts from the factor it replaces (a zero factor
    starts the first step at Z = 0); the initial factors are inputs;
  * sign(0) = +1, as when packing signs;
  * the middle scale of the result is m = mL . mR (each step owns one side);
  * importance (same section: input activation norms and output gradient
    norms weight the approximation error): the objective becomes
    ||diag(d_out) (W - W_hat) diag(d_in)||_F with positive weights d_out [N],
    d_in [M].  Since diag(d_out) P and Q diag(d_in) are again of the
    factored form (the weights fold into a and b), this is the unweighted
    problem for W' = diag(d_out) W diag(d_in): factorize W' from the start
    (d_out . a, A, mL; mR, B, b . d_in), then divide d_out out of a and d_in
    out of b.  The weights themselves are inputs (no calibration data here).

Pins (tests/test_oracle_factorize_pins.py): SVID is exact and idempotent on its set;
its rank-1 part converges to the leading singular pair of |Y| (library SVD);
the P-update equals the ridge least-squares solution of a stacked system
(library least squares); the exact factors of an exactly representable W
are a fixed point of both ADMM steps; ADMM started from zero recovers the
left factor of such a W; a planted dual-sign mistake fails that recovery;
unit importance weights change nothing; the weighted error of the result is
the plain error of the scaled problem; weighting a set of input columns
lowers their error.
"""

from __future__ import annotations

import numpy as np


def sign_pm1(y: np.ndarray) -> np.ndarray:
    """Entrywise sign with sign(0) = +1, as int8."""
    return np.where(np.asarray(y) >= 0, 1, -1).astype(np.int8)


def svid_dense(r: np.ndarray, s: np.ndarray, c: np.ndarray) -> np.ndarray:
    """diag(r) S diag(c) in float64."""
    return np.asarray(r, np.float64)[:, None] * np.asarray(s, np.float64) * np.asarray(c, np.float64)[None, :]


def svid(y: np.ndarray, power_iters: int):
    """SVID projection of y [n x k] (DBF page, section 2, Proyección SVID).

    Returns (r [n], S [n x k] int8, c [k]) with y ~ diag(r) S diag(c):
    S = sign(y) and r c^T a rank-1 approximation of |y| from `power_iters`
    power iterations started at the all-ones direction.
    """
    y = np.asarray(y, np.float64)
    mag = np.abs(y)
    k = y.shape[1]
    v = np.full(k, 1.0 / np.sqrt(k)) if k else np.zeros(0)
    for _ in range(power_iters):
        u = mag @ v
        v = mag.T @ u
        nv = np.sqrt(np.dot(v, v))
        if nv > 0:
            v = v / nv
    r = mag @ v
    return r, sign_pm1(y), v


def penalty(f: np.ndarray, rho_rel: float) -> float:
    """rho = rho_rel * mean(diag(F F^T)); rho_rel when F is zero."""
    f = np.asarray(f, np.float64)
    k = f.shape[0]
    mean_diag = float(np.sum(f * f)) / k if k else 0.0
    return rho_rel * mean_diag if mean_diag > 0 else float(rho_rel)


def p_update(t: np.ndarray, f: np.ndarray, z: np.ndarray, u: np.ndarray, rho: float) -> np.ndarray:
    """ADMM P-update: (T F^T + rho (Z - U)) (F F^T + rho I)^-1, by a library solve."""
    t = np.asarray(t, np.float64)
    f = np.asarray(f, np.float64)
    g = f @ f.T + rho * np.eye(f.shape[0])
    rhs = t @ f.T + rho * (z - u)
    return np.linalg.solve(g, rhs.T).T


def admm_left(t, f, r0, s0, c0, inner: int, power_iters: int, rho_rel: float, _dual_sign: float = 1.0,
              return_y: bool = False):
    """One alternating step: ADMM for min_P 1/2||T - P F||^2, P in the SVID set.

    t [n x p] target, f [k x p] fixed factor, (r0, s0, c0) the current left
    factor (warm start).  Returns the new left factor (r, S, c), and with
    return_y also the matrix P + U that the last SVID projected (None when
    inner = 0): its entries near zero are where a sign is decided by rounding.
    `_dual_sign` exists only so that a test can plant a wrong dual update.
    """
    t = np.asarray(t, np.float64)
    f = np.asarray(f, np.float64)
    rho = penalty(f, rho_rel)
    r, s, c = np.asarray(r0, np.float64), np.asarray(s0, np.int8), np.asarray(c0, np.float64)
    z = svid_dense(r, s, c)
    u = np.zeros_like(z)
    y = None
    for _ in range(inner):
        p = p_update(t, f, z, u, rho)
        y = p + u
        r, s, c = svid(y, power_iters)
        z = svid_dense(r, s, c)
        u = u + _dual_sign * (p - z)
    return (r, s, c, y) if return_y else (r, s, c)


def factorize(w, left, right, outer: int, inner: int, power_iters: int, rho_rel: float):
    """Alternating minimisation (DBF page, section 2, Algoritmo de Optimización).

    w [N x M]; left = (a [N], A [N x k], mL [k]); right = (mR [k], B [k x M],
    b [M]).  Each of `outer` rounds runs the A-step, then the B-step on the
    transposed problem.  Returns (a, A, mL, mR, B, b).
    """
    w = np.asarray(w, np.float64)
    a, A, mL = (np.asarray(left[0], np.float64), np.asarray(left[1], np.int8), np.asarray(left[2], np.float64))
    mR, B, b = (np.asarray(right[0], np.float64), np.asarray(right[1], np.int8), np.asarray(right[2], np.float64))
    for _ in range(outer):
        q = svid_dense(mR, B, b)                       # k x M
        a, A, mL = admm_left(w, q, a, A, mL, inner, power_iters, rho_rel)
        pt = svid_dense(a, A, mL).T                    # k x N
        b, bt, mR = admm_left(w.T, pt, b, B.T, mR, inner, power_iters, rho_rel)
        B = np.ascontiguousarray(bt.T)
    return a, A, mL, mR, B, b


def factorize_weighted(w, d_out, d_in, left, right, outer: int, inner: int, power_iters: int, rho_rel: float):
    """Importance-weighted factorization (DBF page, section 2, Importancia de
    Entradas y Salidas): minimise ||diag(d_out)(W - W_hat)diag(d_in)|| by the
    same alternating steps on W' = diag(d_out) W diag(d_in) in the variables
    a' = d_out . a, b' = b . d_in.  Returns (a, A, mL, mR, B, b)."""
    w = np.asarray(w, np.float64)
    d_out = np.asarray(d_out, np.float64)
    d_in = np.asarray(d_in, np.float64)
    wp = d_out[:, None] * w * d_in[None, :]
    lp = (np.asarray(left[0], np.float64) * d_out, left[1], left[2])
    rp = (right[0], right[1], np.asarray(right[2], np.float64) * d_in)
    a, A, mL, mR, B, b = factorize(wp, lp, rp, outer, inner, power_iters, rho_rel)
    return a / d_out, A, mL, mR, B, b / d_in


def weighted_rel_error(w, d_out, d_in, a, A, mL, mR, B, b) -> float:
    """||diag(d_out)(W - W_hat)diag(d_in)||_F / ||diag(d_out) W diag(d_in)||_F."""
    w = np.asarray(w, np.float64)
    d_out = np.asarray(d_out, np.float64)[:, None]
    d_in = np.asarray(d_in, np.float64)[None, :]
    d = d_out * (w - reconstruct(a, A, mL, mR, B, b)) * d_in
    ref = d_out * w * d_in
    return float(np.sqrt(np.sum(d * d) / np.sum(ref * ref)))


def reconstruct(a, A, mL, mR, B, b) -> np.ndarray:
    """(a . A . m^T)(B . b^T) with m = mL . mR, in float64."""
    return svid_dense(a, A, mL) @ svid_dense(mR, B, b)


def rel_error(w, a, A, mL, mR, B, b) -> float:
    """||W - W_hat||_F / ||W||_F."""
    w = np.asarray(w, np.float64)
    d = w - reconstruct(a, A, mL, mR, B, b)
    return float(np.sqrt(np.sum(d * d) / np.sum(w * w)))
