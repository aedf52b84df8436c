"""Comparison helpers for GPU-vs-oracle parity tests.

The tolerances are the ones the workload fixes, with these readings:
  * Hessian: relative Frobenius error <= 1e-5.
  * U: row-normwise  max_i ||U_gpu[i] - U_ref[i]||_inf / ||U_ref[i]||_inf <= 1e-4.
  * codes: a rounding *decision* may differ only at a near-tie: the two codes are adjacent
    and the oracle's pre-rounding value lies within 1e-3 grid steps of the .5 boundary
    between them; >= 99.99 % of decisions must agree.  A flipped near-tie changes that
    row's later working weights, so the later codes of the row are checked against the
    oracle re-run that takes the GPU's branch at each such near-tie (both are valid GPTQ
    runs); after that every code of the row must agree.
  * layer reconstruction error within 0.1 % of the oracle's.
"""

from __future__ import annotations

import numpy as np

from oracle import gptq_oracle as O

TOL_H = 1e-5
TOL_U = 1e-4
TOL_TIE = 1e-3
MIN_AGREE = 0.9999
TOL_RECON = 1e-3


def rel_fro(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def u_rowwise_err(Ug, Ur):
    Ug = np.asarray(Ug, np.float64)
    Ur = np.asarray(Ur, np.float64)
    num = np.max(np.abs(Ug - Ur), axis=1)
    den = np.maximum(np.max(np.abs(Ur), axis=1), 1e-300)
    return float(np.max(num / den))


def forced_row_sweep(w_row, U, s, z, maxq, dead, gpu_codes_row, tol=TOL_TIE):
    """Re-run the oracle's sweep on one row, taking the GPU's code at near-ties.

    Returns ``(n_forced, n_hard)``: decisions where the GPU took the other side of a
    near-tie, and decisions where it differed otherwise (must be 0).
    """
    d = w_row.shape[0]
    Wk = np.array(w_row, dtype=np.float64)[None, :].copy()
    if dead is not None:
        Wk[:, np.asarray(dead, bool)] = 0.0
    s32 = np.float32(s)
    n_forced = n_hard = 0
    sarr = np.array([s32], np.float32)
    zarr = np.array([z], np.int32)
    for j in range(d):
        c, q = O.quantize_to_grid(Wk[:, j], sarr, zarr, maxq)
        g = int(gpu_codes_row[j])
        if g != int(c[0]):
            x = float(np.float32(np.float32(Wk[0, j]) / s32))
            boundary = min(g, int(c[0])) - int(z) + 0.5
            if abs(g - int(c[0])) == 1 and abs(x - boundary) <= tol:
                n_forced += 1
                q = np.array([float(s32) * (g - int(z))])
            else:
                n_hard += 1
                q = np.array([float(s32) * (g - int(z))])
        err = (Wk[0, j] - q[0]) / U[j, j]
        Wk[0, j + 1:] -= err * U[j, j + 1:]
    return n_forced, n_hard


def check_codes(gpu_codes, W, U, scale, zero, bits, block, dead, rows=None):
    """Compare GPU codes with the oracle on the same inputs; returns a stats dict and
    raises AssertionError when the reading above is violated.  ``rows`` restricts the
    comparison to a row sample (the oracle then sweeps only those rows)."""
    W = np.asarray(W)
    if rows is not None:
        W = W[rows]
        scale = np.asarray(scale)[rows]
        zero = np.asarray(zero)[rows]
        gpu_codes = np.asarray(gpu_codes)[rows]
    oc, _ = O.gptq_quantize(W, U, scale, zero, bits, block=block, dead=dead)
    mism = gpu_codes != oc
    stats = {"entries": int(oc.size), "identical": int(oc.size - mism.sum()),
             "rows_differing": int(mism.any(axis=1).sum()), "forced": 0, "hard": 0}
    maxq = 2 ** bits - 1
    for r in np.flatnonzero(mism.any(axis=1)):
        f, h = forced_row_sweep(W[r], U, scale[r], zero[r], maxq, dead, gpu_codes[r])
        stats["forced"] += f
        stats["hard"] += h
    assert stats["hard"] == 0, f"code mismatches that are not near-ties: {stats}"
    assert stats["forced"] <= (1 - MIN_AGREE) * oc.size, f"too many near-tie flips: {stats}"
    return stats
