"""Marshalling between the seeded host inputs and the CUDA library, for tests.

Inputs come from workloads.generators; expected values come from the fp64
oracle; this module only moves arrays between numpy and torch and measures
the difference.
"""

import numpy as np
import torch

from oracle import dbf_oracle as O

# Tolerances for bf16 outputs of random floating-point inputs (stated for
# this product): max|y - y_ref| <= 1e-2 * max|y_ref| and relative Frobenius
# error <= 2e-3, y_ref the exact (float64) result.
#
# Every output of at least SMALL_OUTPUT elements is held to those two bounds
# as stated.  The exactly rounded bf16 result alone carries a relative
# Frobenius error of about 1.6e-3 (half an ulp of an 8-bit significand, RMS),
# and on outputs of only a few dozen elements that figure scatters above 2e-3
# by itself (a 33 x 2 output: 2.36e-3 for the correctly rounded result).  Only
# below SMALL_OUTPUT elements is the Frobenius bound max(2e-3, floor + 5e-4),
# floor = the error of the exactly rounded result, 5e-4 = the budget of the
# two fp16 intermediates (2^-11 relative each, RMS 2.8e-4, added linearly).
MAX_REL_TOL = 1e-2
FROB_TOL = 2e-3
INTERMEDIATE_BUDGET = 5e-4
SMALL_OUTPUT = 1000


# Activation rows per tile that the prefill GEMMs can be launched with (the
# launch picks one per GEMM from the shape); activation row t*ell + i holds
# token t, term i, so a tile of BN rows spans BN / ell tokens.
PREFILL_TILE_ROWS = (160, 176, 192, 224, 240, 256)


def tile_boundary_tokens(T, ell):
    """Token rows on both sides of every token-tile boundary of every prefill
    tile layout, plus the first two and last two rows (sorted, unique)."""
    rows = {0, 1, T - 2, T - 1}
    for bn in PREFILL_TILE_ROWS:
        if bn % ell:
            continue
        step = bn // ell
        for b in range(step, T, step):
            rows.update((b - 1, b))
    return sorted(r for r in rows if 0 <= r < T)


def dbf():
    from double_binary_rank_packed_b300 import dbf as _dbf
    return _dbf


def device_factors(f, ldw1=None, ldw2=None, device="cuda"):
    """Upload one host factor set and pack its signs with the library's dbf_pack."""
    d = dbf()
    B1 = torch.from_numpy(np.ascontiguousarray(f.B1)).to(device)
    B2 = torch.from_numpy(np.ascontiguousarray(f.B2)).to(device)
    alpha = torch.from_numpy(np.ascontiguousarray(f.alpha)).to(device)
    beta = torch.from_numpy(np.ascontiguousarray(f.beta)).to(device)
    gamma = torch.from_numpy(np.ascontiguousarray(f.gamma)).to(device)
    return d.PackedFactors.from_signs(B1, B2, alpha, beta, gamma, ldw1, ldw2)


def bits_to_bf16(bits, device="cuda"):
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device)
    return t.view(torch.bfloat16)


def bf16_to_bits(t):
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def errors(y_bits, y_ref):
    """(max|dy| / max|y_ref|, relative Frobenius error) of bf16 bits vs float64 reference."""
    y = O.bf16_bits_to_f64(y_bits)
    ref = np.asarray(y_ref, dtype=np.float64)
    scale = np.abs(ref).max()
    max_rel = float(np.abs(y - ref).max() / scale) if scale > 0 else float(np.abs(y).max())
    return max_rel, O.rel_frobenius(y, ref)


def frob_tolerance(y_ref):
    if np.asarray(y_ref).size >= SMALL_OUTPUT:
        return FROB_TOL
    floor = O.rel_frobenius(O.bf16_bits_to_f64(O.round_to_bf16_bits(y_ref)), y_ref)
    return max(FROB_TOL, floor + INTERMEDIATE_BUDGET)


def assert_close(y_bits, y_ref, what=""):
    assert np.isfinite(O.bf16_bits_to_f64(y_bits)).all(), f"{what}: non-finite output"
    max_rel, frob = errors(y_bits, y_ref)
    tol = frob_tolerance(y_ref)
    # achieved errors go to the test log (pytest -s, or the captured output of a failure)
    print(f"[parity] {what}: n={np.asarray(y_ref).size} max_rel={max_rel:.3e} frob={frob:.3e} "
          f"(tol {MAX_REL_TOL:.0e} / {tol:.3e})")
    assert max_rel <= MAX_REL_TOL and frob <= tol, \
        f"{what}: max_rel={max_rel:.3e} frob={frob:.3e} (frob tol {tol:.3e})"
    return max_rel, frob
