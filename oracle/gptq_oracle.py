"""Plain fp64 CPU oracle of GPTQ's per-layer second-order weight quantization.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports, calls or links this
module: only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline /
reference arm of ``bench.py`` may use it.  It shares no code, table or helper with the
CUDA library, and it never receives a value produced by the CUDA library.

Every function follows one passage of three web pages on GPTQ, cited by page title and
section:

  [MDU] "GPTQ › Mathematical Details of the Update" (the inverse-Hessian downdate and
        the Cholesky shortcut).
  [TGM] "tm_gptq_math", sections "Post-training quantization and the per-layer
        objective", "The reconstruction objective, written out", "Why it is
        second-order: the Hessian", "Greedy quantization with error compensation",
        "A worked two-weight example", "GPTQ's speedups: fixed order and lazy batches",
        "The Cholesky trick for the inverse Hessian".
  [GH]  "GPTQ Hessian", excerpt of "GPTQ: Block Structure in Quantization".

Where the pages leave a step open (the grid, rounding ties, what "skipping" a dead
column means, where the damping mean is taken, the code packing) the oracle takes the
readings listed in the design notes; each such function says which reading it uses.

Layout conventions: X is token-major ``[n_tok, d_in]`` (row t is one calibration input
x_t), W is ``[d_out, d_in]`` (row i is one output feature), so the pages' ``X`` of shape
``[d_in, N]`` is ``X.T`` here and ``H = 2 X X^T`` of the pages is ``2 * X.T @ X``.

All floating point is float64, except the quantization grid and the rounding decision,
which the pages do not fix and which are taken in float32 -- the precision in which the
GPU kernels take the same integer decisions -- so that both sides decide in the same
precision.
"""

from __future__ import annotations

import numpy as np

__all__ = [
    "NotPositiveDefinite",
    "hessian",
    "hessian_block",
    "hessian_diagonal",
    "damp_hessian",
    "damp_principal_block",
    "inverse_cholesky_upper",
    "inverse_cholesky_upper_reversed",
    "row_grid",
    "quantize_to_grid",
    "gptq_quantize",
    "obs_quantize_schur",
    "rtn_quantize",
    "pack_codes",
    "unpack_codes",
    "packed_words_per_row",
    "reconstruction_error",
    "reconstruction_error_direct",
    "gptq_layer",
]


class NotPositiveDefinite(np.linalg.LinAlgError):
    """The damped Hessian (or its inverse) has no Cholesky factor."""


# ---------------------------------------------------------------------------------------
# Step 1: the layer Hessian
# ---------------------------------------------------------------------------------------

def hessian(X, H=None):
    """Return ``H + 2 * X^T X`` (or ``2 * X^T X`` when ``H`` is None) in float64.

    [TGM "Why it is second-order: the Hessian"]: the per-row error is quadratic in the
    weights, so its Hessian is the constant ``2 X X^T`` (pages' column-per-token X); the
    factor 2 is kept.  [GH]: every row shares this one matrix.  Calling this once per
    token chunk and summing gives the Hessian of the concatenated calibration set.
    """
    X64 = np.asarray(X, dtype=np.float64)
    if X64.ndim != 2:
        raise ValueError("X must be [n_tok, d_in]")
    G = 2.0 * (X64.T @ X64)
    if H is None:
        return G
    return np.asarray(H, dtype=np.float64) + G


def hessian_block(X, rows, cols):
    """The block ``H[rows][:, cols]`` of ``2 X^T X`` without forming the rest of H."""
    X = np.asarray(X)
    return 2.0 * (X[:, rows].astype(np.float64).T @ X[:, cols].astype(np.float64))


def hessian_diagonal(X, chunk=8192):
    """The diagonal of ``2 X^T X``: twice each channel's sum of squares (token chunks)."""
    X = np.asarray(X)
    out = np.zeros(X.shape[1], dtype=np.float64)
    for t0 in range(0, X.shape[0], chunk):
        Xc = X[t0:t0 + chunk].astype(np.float64)
        out += np.einsum("ti,ti->i", Xc, Xc)
    return 2.0 * out


# ---------------------------------------------------------------------------------------
# Step 2: dead columns and damping
# ---------------------------------------------------------------------------------------

def damp_principal_block(H_block, diag_full, idx, damp=0.01):
    """Dead-column fix and damping of the principal block ``H[idx][:, idx]`` of a Hessian
    whose full diagonal is ``diag_full``; returns ``(H_block_damped, dead_full, lam)``.

    Same rule as :func:`damp_hessian` (lam from the mean of the whole dead-fixed diagonal),
    restricted to the rows and columns ``idx``.
    """
    diag_full = np.asarray(diag_full, dtype=np.float64)
    dead = diag_full == 0.0
    lam = float(damp) * float(np.mean(np.where(dead, 1.0, diag_full)))
    Hb = np.array(H_block, dtype=np.float64, copy=True)
    idx = np.asarray(idx)
    sub_dead = np.flatnonzero(dead[idx])
    Hb[sub_dead, sub_dead] = 1.0
    Hb[np.diag_indices_from(Hb)] += lam
    return Hb, dead, lam


def damp_hessian(H, damp=0.01):
    """Dead-column fix and diagonal damping; returns ``(H_damped, dead, lam)``.

    [TGM "The Cholesky trick for the inverse Hessian"]: channels the calibration data
    never excited have a zero diagonal and are skipped; a damping term ``lam * I`` with
    ``lam`` about one percent of the mean diagonal is added before inverting.  [GH] writes
    the damped Hessian as ``2 X X^T + lam I``.

    Readings taken: a dead column is one with ``H_ii == 0`` exactly; its diagonal is set
    to 1 (its off-diagonals are already 0 because the channel is identically zero); the
    mean is taken over all ``d`` diagonal entries *after* that fix; ``lam = damp * mean``.
    """
    Hd = np.array(H, dtype=np.float64, copy=True)
    if Hd.ndim != 2 or Hd.shape[0] != Hd.shape[1]:
        raise ValueError("H must be square")
    diag = np.diag(Hd).copy()
    dead = diag == 0.0
    idx = np.flatnonzero(dead)
    Hd[idx, idx] = 1.0
    lam = float(damp) * float(np.mean(np.diag(Hd)))
    Hd[np.diag_indices_from(Hd)] += lam
    return Hd, dead, lam


# ---------------------------------------------------------------------------------------
# Step 3: the inverse-Hessian Cholesky factor
# ---------------------------------------------------------------------------------------

def inverse_cholesky_upper(Hd):
    """Upper-triangular ``U`` with ``U^T U = Hd^{-1}``, by inverting then factoring.

    [GH]: U is the upper triangular Cholesky factor of the inverse Hessian.  [TGM "The
    Cholesky trick for the inverse Hessian"]: the factorization is computed once, up
    front, with a stable library routine; [MDU] writes the same factor as ``L = U^T``.
    """
    try:
        Hinv = np.linalg.inv(np.asarray(Hd, dtype=np.float64))
        L = np.linalg.cholesky(Hinv)
    except np.linalg.LinAlgError as exc:
        raise NotPositiveDefinite(str(exc)) from exc
    return np.ascontiguousarray(L.T)


def inverse_cholesky_upper_reversed(Hd):
    """The same ``U`` as :func:`inverse_cholesky_upper`, without inverting ``Hd`` first.

    For host-side checks at widths where the pages' route (invert, then factor) is too slow:
    with ``P`` the index reversal, factor ``P Hd P = L L^T`` (lower Cholesky, LAPACK), invert
    the triangle (LAPACK), and reverse back: ``U = P L^-1 P`` is upper triangular with a
    positive diagonal and ``U^T U = P (L L^T)^-1 P = Hd^-1``, so by uniqueness of the
    Cholesky factor it is the matrix [GH] names.  Costs ``2 d^3 / 3`` flops instead of
    ``7 d^3 / 3``.  Overwrites nothing it is given.
    """
    import scipy.linalg as sla
    from scipy.linalg import lapack
    A = np.array(np.asarray(Hd, dtype=np.float64)[::-1, ::-1], order="F", copy=True)
    try:
        L = sla.cholesky(A, lower=True, overwrite_a=True, check_finite=False)
    except np.linalg.LinAlgError as exc:
        raise NotPositiveDefinite(str(exc)) from exc
    del A
    Linv, info = lapack.dtrtri(L, lower=1, overwrite_c=1)
    if info != 0:
        raise NotPositiveDefinite(f"triangular inverse failed (info={info})")
    del L
    # the factor's strict upper triangle is zero (cleared by the factorization, untouched
    # by the triangular inverse), so the reversal is upper triangular as it stands
    return np.ascontiguousarray(Linv[::-1, ::-1])


# ---------------------------------------------------------------------------------------
# The quantization grid (not defined on the pages; reading: per-row asymmetric min-max)
# ---------------------------------------------------------------------------------------

def row_grid(W, bits):
    """Per-row asymmetric min-max grid ``(scale[d_out] float32, zero[d_out] int32)``.

    The pages only say weights go to a few-bit integer grid ([TGM "Post-training
    quantization and the per-layer objective"], [GH]) and use a grid of step 0.5 in the
    worked example.  Reading: per output row, the range ``[min(0, min_j W_ij),
    max(0, max_j W_ij)]`` is split into ``2^bits - 1`` steps (0 always lies inside, so a
    zeroed dead column is exactly representable); an all-zero row gets ``scale = 1``;
    ``zero = rint(-x_min / scale)``.  Taken in float32 (IEEE subtraction and division).
    """
    W32 = np.asarray(W, dtype=np.float32)
    maxq = np.float32(2 ** int(bits) - 1)
    xmin = np.minimum(W32.min(axis=1), np.float32(0.0))
    xmax = np.maximum(W32.max(axis=1), np.float32(0.0))
    width = (xmax - xmin).astype(np.float32)
    scale = np.where(width == 0, np.float32(1.0), width / maxq).astype(np.float32)
    zero = np.rint((-xmin) / scale).astype(np.float32)
    return scale, zero.astype(np.int32)


def quantize_to_grid(w, scale, zero, maxq):
    """Round one column of working weights to the grid; returns ``(codes, q)``.

    ``code = clamp(rint(w / scale) + zero, 0, maxq)`` and ``q = scale * (code - zero)``
    (``maxq=None`` disables the clamp, as in the worked example's unbounded grid).  The
    rounding decision is taken in float32 (``w`` rounded to float32, IEEE division by the
    float32 scale, round-half-to-even); ``q`` is returned in float64.
    """
    w32 = np.asarray(w, dtype=np.float64).astype(np.float32)
    s32 = np.asarray(scale, dtype=np.float32)
    x = (w32 / s32).astype(np.float32)
    c = np.rint(x).astype(np.int64) + np.asarray(zero, dtype=np.int64)
    if maxq is not None:
        c = np.clip(c, 0, int(maxq))
    q = s32.astype(np.float64) * (c - np.asarray(zero, dtype=np.int64)).astype(np.float64)
    return c, q


# ---------------------------------------------------------------------------------------
# Step 4 + 5: the fixed-order sweep with in-block compensation and lazy trailing update
# ---------------------------------------------------------------------------------------

def gptq_quantize(W, U, scale, zero, bits, block=128, dead=None, maxq="bits",
                  stop_after=None):
    """GPTQ column sweep driven by the rows of ``U``; returns ``(codes, W_hat)``.

    [TGM "GPTQ's speedups: fixed order and lazy batches"] and [GH]: columns are quantized
    left to right, the same order for every row, in blocks of ``block`` columns.  Inside
    a block every later column of the block is corrected immediately; the correction of
    the columns after the block is deferred and applied once per block as one product.

    The per-column correction is the OBS update of [TGM "Greedy quantization with error
    compensation"] written with the Cholesky factor: for the free weights ``F = {j..}``
    the restricted inverse Hessian is ``U[j:, j:]^T U[j:, j:]`` (the Schur-complement
    downdate of [MDU] applied column after column), whose row ``j`` is
    ``U_jj * U[j, j:]`` and pivot ``U_jj^2``, so the update becomes
    ``W[:, k] -= ((W[:, j] - q_j) / U_jj) * U[j, k]`` for the not-yet-quantized ``k``
    ([MDU]: read off the next row of the factor instead of updating the whole inverse).

    ``dead`` (bool mask) columns are set to zero before the sweep (reading of "skipped":
    their code is the zero-point, their error 0).  ``maxq="bits"`` clamps to
    ``[0, 2^bits - 1]``; ``maxq=None`` does not clamp.  ``stop_after=j`` returns the
    working matrix right after column ``j`` has been quantized and compensated (used
    by the conditional-minimiser check), with all deferred updates applied.
    """
    Wk = np.array(W, dtype=np.float64, copy=True)
    U = np.asarray(U, dtype=np.float64)
    m, d = Wk.shape
    if U.shape != (d, d):
        raise ValueError("U must be [d_in, d_in]")
    if maxq == "bits":
        maxq = 2 ** int(bits) - 1
    if dead is not None:
        Wk[:, np.asarray(dead, dtype=bool)] = 0.0
    block = max(1, int(block))
    codes = np.zeros((m, d), dtype=np.int64)
    W_hat = np.zeros((m, d), dtype=np.float64)
    for b0 in range(0, d, block):
        b1 = min(b0 + block, d)
        E = np.zeros((m, b1 - b0), dtype=np.float64)
        for j in range(b0, b1):
            c, q = quantize_to_grid(Wk[:, j], scale, zero, maxq)
            codes[:, j] = c
            W_hat[:, j] = q
            err = (Wk[:, j] - q) / U[j, j]
            E[:, j - b0] = err
            Wk[:, j + 1:b1] -= np.outer(err, U[j, j + 1:b1])
            if stop_after is not None and j == stop_after:
                Wk[:, : j + 1] = W_hat[:, : j + 1]
                Wk[:, b1:] -= E[:, : j - b0 + 1] @ U[b0:j + 1, b1:]
                return Wk
        Wk[:, b1:] -= E @ U[b0:b1, b1:]
    return codes, W_hat


def obs_quantize_schur(W, Hd, scale, zero, bits, dead=None, maxq="bits"):
    """Column-at-a-time OBS sweep with an explicit, shrinking inverse Hessian.

    The slow route the Cholesky factor replaces: [TGM "Greedy quantization with error
    compensation"] gives the correction ``delta = -(e_q / [H^-1]_qq) H^-1[:, q]`` of the
    free weights after quantizing weight ``q``; [MDU] gives the rank-one Schur-complement
    downdate ``H^-1 <- H^-1 - H^-1[:, q] H^-1[q, :] / [H^-1]_qq`` that removes ``q`` from
    the free set.  Columns go left to right (fixed order, [TGM "GPTQ's speedups"]).
    Costs O(d^2) per column; only for small checks.
    """
    Wk = np.array(W, dtype=np.float64, copy=True)
    m, d = Wk.shape
    if maxq == "bits":
        maxq = 2 ** int(bits) - 1
    if dead is not None:
        Wk[:, np.asarray(dead, dtype=bool)] = 0.0
    Hinv = np.linalg.inv(np.asarray(Hd, dtype=np.float64))
    codes = np.zeros((m, d), dtype=np.int64)
    W_hat = np.zeros((m, d), dtype=np.float64)
    for q in range(d):
        c, qv = quantize_to_grid(Wk[:, q], scale, zero, maxq)
        codes[:, q] = c
        W_hat[:, q] = qv
        e = Wk[:, q] - qv
        Wk[:, q + 1:] -= np.outer(e / Hinv[q, q], Hinv[q, q + 1:])
        Wk[:, q] = qv
        Hinv = Hinv - np.outer(Hinv[:, q], Hinv[q, :]) / Hinv[q, q]
    return codes, W_hat


def obq_greedy(W, Hd, scale, zero, bits, dead=None, forced=None, tie_tol=1e-3):
    """OBQ: greedy per-row order with an explicit Schur downdate.

    [TGM "Greedy quantization with error compensation"]: with F the free weights of a row
    and H_F^-1 their inverse Hessian, quantizing weight q costs
    ``(w_q - quant(w_q))^2 / [H_F^-1]_qq`` and the best correction of the others is
    ``delta_F = -((w_q - quant(w_q)) / [H_F^-1]_qq) H_F^-1[:, q]``; OBQ quantizes the weight
    of least cost first, row by row.  [MDU]: removing q from F is the rank-one downdate
    ``H_F^-1 <- H_F^-1 - H_F^-1[:, q] H_F^-1[q, :] / [H_F^-1]_qq``.  Ties go to the lowest
    index; codes as ``quantize_to_grid``.

    ``forced = (order, codes)`` replays another implementation's decisions, row by row:
    each forced column must be a least-cost column here up to ``slack`` (the cost gap
    relative to the largest current cost, reported as ``max_slack``), and each forced code
    must equal this rounding unless the pre-rounding value ``w/scale`` lies within
    ``tie_tol`` of a rounding boundary (counted in ``tie_flips``; other differences in
    ``bad_codes``).  Returns ``(codes, W_hat, order, info)``.
    """
    W = np.asarray(W, dtype=np.float64)
    m, d = W.shape
    maxq = 2 ** int(bits) - 1
    Hinv0 = np.linalg.inv(np.asarray(Hd, dtype=np.float64))
    s32 = np.asarray(scale, dtype=np.float32)
    zr = np.asarray(zero, dtype=np.int64)
    codes = np.zeros((m, d), dtype=np.int64)
    W_hat = np.zeros((m, d), dtype=np.float64)
    order = np.zeros((m, d), dtype=np.int64)
    info = {"max_slack": 0.0, "tie_flips": 0, "bad_codes": 0, "bad_order": 0}
    deadm = np.zeros(d, dtype=bool) if dead is None else np.asarray(dead, dtype=bool)
    for i in range(m):
        w = W[i].copy()
        w[deadm] = 0.0
        Hinv = Hinv0.copy()
        free = np.ones(d, dtype=bool)
        si, zi = s32[i:i + 1], zr[i:i + 1]
        for step in range(d):
            idx = np.flatnonzero(free)
            c_all, q_all = quantize_to_grid(w[idx], np.repeat(si, idx.size),
                                            np.repeat(zi, idx.size), maxq)
            cost = (w[idx] - q_all) ** 2 / np.diag(Hinv)[idx]
            k = int(np.argmin(cost))              # first minimum: lowest index
            if forced is not None:
                fq = int(forced[0][i, step])
                pos = np.flatnonzero(idx == fq)
                if pos.size != 1:
                    info["bad_order"] += 1
                    break
                k = int(pos[0])
                gap = (cost[k] - cost.min()) / max(cost.max(), 1e-300)
                info["max_slack"] = max(info["max_slack"], float(gap))
            q = int(idx[k])
            c, qv = int(c_all[k]), float(q_all[k])
            if forced is not None:
                fc = int(forced[1][i, q])
                if fc != c:
                    x = float(np.float32(np.float32(w[q]) / si[0]))
                    near = abs(abs(x - np.floor(x)) - 0.5) <= tie_tol
                    if near and abs(fc - c) == 1:
                        info["tie_flips"] += 1
                    else:
                        info["bad_codes"] += 1
                    c = fc
                    qv = float(si[0]) * float(c - zi[0])
            e = (w[q] - qv) / Hinv[q, q]
            w[free] -= e * Hinv[free, q]
            w[q] = qv
            codes[i, q], W_hat[i, q], order[i, step] = c, qv, q
            Hinv = Hinv - np.outer(Hinv[:, q], Hinv[q, :]) / Hinv[q, q]
            free[q] = False
    return codes, W_hat, order, info


def rtn_quantize(W, scale, zero, bits, dead=None):
    """Round-to-nearest on the same grid, every weight independently, no compensation.

    The baseline GPTQ improves on ([TGM "Post-training quantization and the per-layer
    objective"], [TGM "A worked two-weight example"]).
    """
    Wk = np.array(W, dtype=np.float64, copy=True)
    if dead is not None:
        Wk[:, np.asarray(dead, dtype=bool)] = 0.0
    maxq = 2 ** int(bits) - 1
    codes = np.zeros(Wk.shape, dtype=np.int64)
    W_hat = np.zeros(Wk.shape, dtype=np.float64)
    for j in range(Wk.shape[1]):
        codes[:, j], W_hat[:, j] = quantize_to_grid(Wk[:, j], scale, zero, maxq)
    return codes, W_hat


# ---------------------------------------------------------------------------------------
# Code packing (not on the pages; the layout is this project's)
# ---------------------------------------------------------------------------------------

def packed_words_per_row(d_in, bits):
    """uint32 words per packed row: rows are padded to a multiple of 32 columns."""
    return ((int(d_in) + 31) // 32) * int(bits)


def pack_codes(codes, bits):
    """Pack integer codes row by row into a little-endian bitstream of uint32 words.

    The code of column ``c`` occupies bits ``[c*bits, (c+1)*bits)`` of its row's stream
    (bit ``b`` of the stream is bit ``b % 32`` of word ``b // 32``); for 4 bits that is
    nibble ``c % 8`` of word ``c // 8``, for 3 bits every 32 columns fill 3 words.
    """
    codes = np.asarray(codes, dtype=np.int64)
    m, d = codes.shape
    bits = int(bits)
    out = np.zeros((m, packed_words_per_row(d, bits)), dtype=np.uint64)
    for c in range(d):
        pos = c * bits
        w, o = divmod(pos, 32)
        v = codes[:, c].astype(np.uint64)
        out[:, w] |= (v << np.uint64(o)) & np.uint64(0xFFFFFFFF)
        if o + bits > 32:
            out[:, w + 1] |= v >> np.uint64(32 - o)
    return out.astype(np.uint32)


def unpack_codes(packed, bits, d_in):
    """Inverse of :func:`pack_codes`."""
    packed = np.asarray(packed, dtype=np.uint64)
    m = packed.shape[0]
    bits = int(bits)
    mask = np.uint64((1 << bits) - 1)
    codes = np.zeros((m, int(d_in)), dtype=np.int64)
    for c in range(int(d_in)):
        pos = c * bits
        w, o = divmod(pos, 32)
        v = packed[:, w] >> np.uint64(o)
        if o + bits > 32:
            v |= packed[:, w + 1] << np.uint64(32 - o)
        codes[:, c] = (v & mask).astype(np.int64)
    return codes


# ---------------------------------------------------------------------------------------
# Quality metric
# ---------------------------------------------------------------------------------------

def reconstruction_error(W, W_hat, H0):
    """Layer output error ``||(W - W_hat) X^T||_F^2`` evaluated through the Hessian.

    [TGM "The reconstruction objective, written out"]: the rows decouple and each row's
    error is the quadratic form ``delta (X X^T) delta^T``; with the undamped
    ``H0 = 2 X^T X`` the total is ``1/2 * sum_i delta_i H0 delta_i^T``.
    """
    D = np.asarray(W, dtype=np.float64) - np.asarray(W_hat, dtype=np.float64)
    return 0.5 * float(np.einsum("ij,ij->", D @ np.asarray(H0, dtype=np.float64), D))


def reconstruction_error_direct(W, W_hat, X):
    """``||W X^T - W_hat X^T||_F^2`` computed from the activations themselves."""
    D = np.asarray(W, dtype=np.float64) - np.asarray(W_hat, dtype=np.float64)
    Y = D @ np.asarray(X, dtype=np.float64).T
    return float(np.sum(Y * Y))


def reconstruction_error_rows(W, W_hat, X):
    """Per-row terms of ``||W X^T - W_hat X^T||_F^2``: ``err_i = sum_t ((W_i - W_hat_i) . x_t)^2``.

    [TGM "The reconstruction objective, written out"]: the objective is a sum of independent
    per-row output errors over the calibration tokens.  X may be given as a list of token
    chunks (summed in order).
    """
    D = np.asarray(W, dtype=np.float64) - np.asarray(W_hat, dtype=np.float64)
    chunks = X if isinstance(X, (list, tuple)) else [X]
    err = np.zeros(D.shape[0])
    for Xc in chunks:
        Y = D @ np.asarray(Xc, dtype=np.float64).T
        err += np.sum(Y * Y, axis=1)
    return err


# ---------------------------------------------------------------------------------------
# The whole per-layer path
# ---------------------------------------------------------------------------------------

def gptq_layer(X_chunks, W, bits, block=128, damp=0.01):
    """Quantize one linear layer from its calibration activations; returns a dict.

    Steps in the pages' order: Hessian over the calibration chunks, dead-column fix and
    damping, Cholesky factor of the inverse, per-row grid, fixed-order blocked sweep,
    packing.
    """
    if isinstance(X_chunks, np.ndarray):
        X_chunks = [X_chunks]
    H = None
    for Xc in X_chunks:
        H = hessian(Xc, H)
    Hd, dead, lam = damp_hessian(H, damp)
    U = inverse_cholesky_upper(Hd)
    scale, zero = row_grid(W, bits)
    codes, W_hat = gptq_quantize(W, U, scale, zero, bits, block=block, dead=dead)
    return {
        "H": H, "H_damped": Hd, "dead": dead, "lam": lam, "U": U,
        "scale": scale, "zero": zero, "codes": codes, "W_hat": W_hat,
        "packed": pack_codes(codes, bits),
    }
