"""Parity rules between the CUDA path and the CPU oracle.

* Codes: bit-exact, except where the oracle's pre-rounding value lies within
  1e-3 of a decision boundary j + 1/2 (j = 0, 1, 2); the rate of such allowed
  mismatches over all codes must be <= 1e-5.  The oracle decides a code as
  round_half_even((x - z) / s) in float64 from its own stored parameters.
* Scales, zeros and norms (float32): |x_gpu - x_ref| <= 1e-6 |x_ref|; exact
  when x_ref == 0.
* Decode outputs (bf16): |o_gpu - o_ref| <= 2e-3 + ulp_bf16(o_ref) / 2, where
  the half ulp accounts for the final rounding of the output to bf16.
"""
from __future__ import annotations

import numpy as np

BOUNDARY_WINDOW = 1e-3
MAX_BOUNDARY_RATE = 1e-5
META_REL = 1e-6
DECODE_ABS = 2e-3


def near_boundary(pre: np.ndarray) -> np.ndarray:
    """Where the oracle's pre-rounding value lies within 1e-3 of j + 1/2."""
    p = np.asarray(pre, np.float64)
    return np.min(np.abs(p[..., None] - np.array([0.5, 1.5, 2.5])), axis=-1) < BOUNDARY_WINDOW


def code_mismatches(gpu: np.ndarray, ref: np.ndarray, pre: np.ndarray, excused=None):
    """Return (n_mismatch, n_outside_window, n_total).  `excused` (a boolean
    mask broadcastable to the codes, optional) marks codes decided against
    parameters that legitimately differ between the two sides; mismatches
    there are not counted."""
    gpu = np.asarray(gpu)
    ref = np.asarray(ref)
    bad = gpu != ref
    if excused is not None:
        bad &= ~np.broadcast_to(excused, bad.shape)
    n_bad = int(bad.sum())
    if n_bad == 0:
        return 0, 0, gpu.size
    near = near_boundary(np.asarray(pre)[bad])
    return n_bad, int((~near).sum()), gpu.size


def assert_codes(gpu, ref, pre, what="", excused=None):
    n_bad, n_out, n = code_mismatches(gpu, ref, pre, excused)
    assert n_out == 0, f"{what}: {n_out} code mismatches outside the boundary window"
    assert n_bad <= MAX_BOUNDARY_RATE * n, \
        f"{what}: boundary mismatch rate {n_bad}/{n} > {MAX_BOUNDARY_RATE}"
    return n_bad, n


def meta_rel_err(gpu, ref):
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    zero = ref == 0
    if np.any(gpu[zero] != 0):
        return np.inf
    nz = ~zero
    if not np.any(nz):
        return 0.0
    return float(np.max(np.abs(gpu[nz] - ref[nz]) / np.abs(ref[nz])))


def assert_meta(gpu, ref, what=""):
    e = meta_rel_err(gpu, ref)
    assert e <= META_REL, f"{what}: relative error {e:.3e} > {META_REL}"
    return e


def bf16_half_ulp(x: np.ndarray) -> np.ndarray:
    x = np.abs(np.asarray(x, np.float64))
    e = np.floor(np.log2(np.maximum(x, 2.0 ** -126)))
    return 0.5 * 2.0 ** (e - 7)


def decode_err(gpu, ref):
    """Return (max |gpu - ref|, max of |gpu - ref| - tolerance)."""
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    d = np.abs(gpu - ref)
    return float(d.max()), float((d - (DECODE_ABS + bf16_half_ulp(ref))).max())


def assert_decode(gpu, ref, what=""):
    mx, over = decode_err(gpu, ref)
    assert np.all(np.isfinite(gpu)), f"{what}: non-finite outputs"
    assert over <= 0, f"{what}: max |diff| {mx:.3e} exceeds 2e-3 + half bf16 ulp by {over:.3e}"
    return mx


def bf16_ulp_err(gpu, ref) -> float:
    """max |gpu - ref| in units of the bf16 ulp at ref: <= 0.5 means the
    output is ref correctly rounded to bf16; the excess is kernel error."""
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    return float((np.abs(gpu - ref) / (2 * bf16_half_ulp(ref))).max())
