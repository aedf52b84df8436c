"""Pins of the fp64 oracle against what the pages and the mathematics fix.

Each test checks the oracle against something other than itself: a value printed on a
page, a closed form, a textbook special case, an independent algorithm (a different
factorization route, the explicit inverse-Hessian downdate, a constrained least-squares
solve, exact integer arithmetic) or an invariant of the method.
"""

import math
import os

import numpy as np
import pytest
import scipy.linalg as sla

from oracle import gptq_oracle as O
from tests.conftest import ROOT, read_golden


def correlated_problem(m, d, n, seed, dead=(), bits=4):
    rng = np.random.default_rng(seed)
    A = np.eye(d) + rng.standard_normal((d, d)) / math.sqrt(d)
    X = (A @ rng.standard_normal((d, n))).T
    X[:, list(dead)] = 0.0
    W = (rng.standard_normal((m, d)) * 0.02).astype(np.float32)
    return X, W


# ---------------------------------------------------------------------------------------
# P1: the worked two-weight example ("tm_gptq_math", "A worked two-weight example")
# ---------------------------------------------------------------------------------------

def test_worked_example_closed_form_factor():
    g = read_golden("worked_example.txt")
    H = np.array(g["H"]).reshape(2, 2)
    U = O.inverse_cholesky_upper(H)
    # H^-1 = [[3/8, -1/4], [-1/4, 1/2]] by the 2x2 adjugate; its Cholesky factor by hand
    U_hand = np.array([[math.sqrt(3 / 8), -1 / math.sqrt(6)], [0.0, 1 / math.sqrt(3)]])
    np.testing.assert_allclose(U, U_hand, rtol=0, atol=1e-15)


def test_worked_example_values():
    g = read_golden("worked_example.txt")
    w = np.array([g["w"]])
    H = np.array(g["H"]).reshape(2, 2)
    U = O.inverse_cholesky_upper(H)
    scale = np.array([g["step"]], dtype=np.float32)
    zero = np.array([0], dtype=np.int32)
    # quantize w_1 on the unbounded step-0.5 grid and compensate w_2
    Wk = O.gptq_quantize(w, U, scale, zero, bits=None, block=2, maxq=None, stop_after=0)
    assert Wk[0, 0] == pytest.approx(g["q1"], abs=1e-15)
    delta = Wk[0] - w[0]
    assert delta[0] == pytest.approx(g["delta1"], abs=1e-15)
    assert delta[1] == pytest.approx(g["delta2"], abs=1e-15)
    assert Wk[0, 1] == pytest.approx(g["w2_after"], abs=1e-15)
    err_comp = float(delta @ H @ delta)
    d_nocomp = np.array([delta[0], 0.0])
    err_nocomp = float(d_nocomp @ H @ d_nocomp)
    assert err_nocomp == pytest.approx(g["err_uncompensated"], abs=1e-15)
    assert err_comp == pytest.approx(g["err_compensated"], abs=1e-15)
    assert round(100 * (1 - err_comp / err_nocomp)) == g["reduction_percent"]
    # the Schur-downdate route gives the same correction
    codes, W_hat = O.obs_quantize_schur(w, H, scale, zero, bits=None, maxq=None)
    codes2, W_hat2 = O.gptq_quantize(w, U, scale, zero, bits=None, block=128, maxq=None)
    np.testing.assert_array_equal(codes, codes2)
    np.testing.assert_allclose(W_hat, [[0.5, 0.5]], atol=1e-15)
    np.testing.assert_allclose(W_hat2, [[0.5, 0.5]], atol=1e-15)


# ---------------------------------------------------------------------------------------
# P2: U^T U = H^-1, and an independent factorization route gives the same U
# ---------------------------------------------------------------------------------------

@pytest.mark.parametrize("d,seed", [(7, 0), (64, 1), (200, 2)])
def test_inverse_factor_identity_and_reversed_route(d, seed):
    X, _ = correlated_problem(4, d, 3 * d, seed)
    Hd, _, _ = O.damp_hessian(O.hessian(X))
    U = O.inverse_cholesky_upper(Hd)
    assert np.all(np.tril(U, -1) == 0)
    assert np.all(np.diag(U) > 0)
    cond = np.linalg.cond(Hd)
    np.testing.assert_allclose(U.T @ U @ Hd, np.eye(d), atol=50 * cond * 1e-16)
    # Route 2: Cholesky of the index-reversed H (lower), reverse back to an upper R with
    # H = R R^T, then U = R^{-1} by triangular solve (no explicit inverse of H).
    P = np.arange(d)[::-1]
    Lr = sla.cholesky(Hd[np.ix_(P, P)], lower=True)
    R = Lr[np.ix_(P, P)]
    assert np.allclose(np.tril(R, -1), 0)
    U2 = sla.solve_triangular(R, np.eye(d), lower=False)
    np.testing.assert_allclose(U, U2, rtol=0, atol=50 * cond * 1e-16 * np.abs(U).max())
    # the oracle's own reversed route (used where inverting first is too slow on the host)
    U3 = O.inverse_cholesky_upper_reversed(Hd)
    assert np.all(np.tril(U3, -1) == 0)
    np.testing.assert_allclose(U, U3, rtol=0, atol=50 * cond * 1e-16 * np.abs(U).max())


def test_not_positive_definite_raises():
    H = np.array([[1.0, 2.0], [2.0, 1.0]])  # eigenvalues 3 and -1
    with pytest.raises(O.NotPositiveDefinite):
        O.inverse_cholesky_upper(H)
    with pytest.raises(O.NotPositiveDefinite):
        O.inverse_cholesky_upper_reversed(H)


def test_reversed_route_worked_example_factor():
    # the 2 x 2 factor of the worked example by hand: U = [[sqrt(3/8), -1/sqrt(6)],
    # [0, 1/sqrt(3)]] ("tm_gptq_math", "A worked two-weight example")
    U = O.inverse_cholesky_upper_reversed(np.array([[4.0, 2.0], [2.0, 3.0]]))
    np.testing.assert_allclose(U, [[np.sqrt(3 / 8), -1 / np.sqrt(6)], [0.0, 1 / np.sqrt(3)]],
                               rtol=0, atol=1e-15)


# ---------------------------------------------------------------------------------------
# P3: Cholesky-row route == explicit inverse with Schur downdates
# ---------------------------------------------------------------------------------------

@pytest.mark.parametrize("m,d,seed,dead", [(5, 9, 3, ()), (16, 40, 4, (3, 17)),
                                           (8, 130, 5, (0, 129))])
def test_cholesky_route_equals_schur_downdate_route(m, d, seed, dead):
    X, W = correlated_problem(m, d, 2 * d, seed, dead)
    Hd, deadm, _ = O.damp_hessian(O.hessian(X))
    assert list(np.flatnonzero(deadm)) == list(dead)
    U = O.inverse_cholesky_upper(Hd)
    scale, zero = O.row_grid(W, 4)
    c1, q1 = O.gptq_quantize(W, U, scale, zero, 4, block=128, dead=deadm)
    c2, q2 = O.obs_quantize_schur(W, Hd, scale, zero, 4, dead=deadm)
    np.testing.assert_array_equal(c1, c2)
    np.testing.assert_allclose(q1, q2, atol=1e-12)


# ---------------------------------------------------------------------------------------
# P4: lazy batches are the same math as eager column updates
# ---------------------------------------------------------------------------------------

def test_lazy_batches_equal_eager_updates():
    X, W = correlated_problem(32, 300, 600, 6, dead=(5,))
    Hd, dead, _ = O.damp_hessian(O.hessian(X))
    U = O.inverse_cholesky_upper(Hd)
    scale, zero = O.row_grid(W, 3)
    ref_c, ref_q = O.gptq_quantize(W, U, scale, zero, 3, block=1, dead=dead)
    for B in (3, 32, 128, 300, 1000):
        c, q = O.gptq_quantize(W, U, scale, zero, 3, block=B, dead=dead)
        np.testing.assert_array_equal(c, ref_c)
        np.testing.assert_allclose(q, ref_q, atol=1e-12)


# ---------------------------------------------------------------------------------------
# P5: each compensation step is the conditional minimiser of the quadratic
# ---------------------------------------------------------------------------------------

@pytest.mark.parametrize("B", [1, 3, 8])
def test_compensation_is_conditional_minimiser(B):
    X, W = correlated_problem(6, 8, 20, 7)
    Hd, dead, _ = O.damp_hessian(O.hessian(X))
    U = O.inverse_cholesky_upper(Hd)
    scale, zero = O.row_grid(W, 4)
    w0 = W.astype(np.float64)
    for j in range(7):
        Wk = O.gptq_quantize(W, U, scale, zero, 4, block=B, stop_after=j)
        fx = np.arange(j + 1)
        fr = np.arange(j + 1, 8)
        # argmin_v (v - w) H (v - w)^T with v_fixed pinned to the quantized values
        rhs = Hd[np.ix_(fr, fx)] @ (Wk[:, fx] - w0[:, fx]).T
        v_free = w0[:, fr] - np.linalg.solve(Hd[np.ix_(fr, fr)], rhs).T
        np.testing.assert_allclose(Wk[:, fr], v_free, atol=1e-12)


# ---------------------------------------------------------------------------------------
# P6: a diagonal Hessian leaves nothing to compensate -> GPTQ == round-to-nearest
# ---------------------------------------------------------------------------------------

def test_diagonal_hessian_reduces_to_rtn():
    rng = np.random.default_rng(8)
    d = 50
    H = np.diag(rng.uniform(0.5, 5.0, d))
    W = (rng.standard_normal((20, d)) * 0.02).astype(np.float32)
    U = O.inverse_cholesky_upper(H)
    np.testing.assert_allclose(U, np.diag(1 / np.sqrt(np.diag(H))), rtol=1e-15)
    scale, zero = O.row_grid(W, 4)
    c, q = O.gptq_quantize(W, U, scale, zero, 4, block=16)
    cr, qr = O.rtn_quantize(W, scale, zero, 4)
    np.testing.assert_array_equal(c, cr)
    np.testing.assert_array_equal(q, qr)


def test_single_column_closed_form():
    H = np.array([[2.5]])
    U = O.inverse_cholesky_upper(H)
    assert U[0, 0] == pytest.approx(1 / math.sqrt(2.5), rel=1e-15)


# ---------------------------------------------------------------------------------------
# P7: GPTQ does not lose to round-to-nearest on correlated inputs (sanity gate)
# ---------------------------------------------------------------------------------------

@pytest.mark.parametrize("bits", [3, 4])
def test_gptq_beats_rtn_on_correlated_layer(bits):
    X, W = correlated_problem(256, 256, 512, 9)
    out = O.gptq_layer(X, W, bits)
    _, q_rtn = O.rtn_quantize(W, out["scale"], out["zero"], bits, dead=out["dead"])
    e_gptq = O.reconstruction_error(W, out["W_hat"], out["H"])
    e_rtn = O.reconstruction_error(W, q_rtn, out["H"])
    assert e_gptq < 0.8 * e_rtn


def test_reconstruction_error_two_routes_agree():
    X, W = correlated_problem(16, 24, 80, 10)
    out = O.gptq_layer(X, W, 4)
    e1 = O.reconstruction_error(W, out["W_hat"], out["H"])
    e2 = O.reconstruction_error_direct(W, out["W_hat"], X)
    assert e1 == pytest.approx(e2, rel=1e-10)


def test_reconstruction_error_rows_match_the_hessian_quadratic_forms():
    # per row: sum_t (delta . x_t)^2 equals 1/2 delta H0 delta^T with H0 = 2 X^T X, over
    # token chunks; one planted row with a single nonzero delta k reduces to 2 H0_kk / 2
    X, W = correlated_problem(12, 20, 90, 3)
    out = O.gptq_layer(X, W, 3)
    rows = O.reconstruction_error_rows(W, out["W_hat"], [X[:40], X[40:]])
    D = W.astype(np.float64) - out["W_hat"]
    quad = 0.5 * np.einsum("ij,jk,ik->i", D, O.hessian(X), D)
    np.testing.assert_allclose(rows, quad, rtol=1e-12)
    assert rows.sum() == pytest.approx(O.reconstruction_error_direct(W, out["W_hat"], X),
                                       rel=1e-12)
    Wp = np.zeros((1, 20))
    Wp[0, 7] = 0.5
    one = O.reconstruction_error_rows(Wp, np.zeros((1, 20)), X)
    assert one[0] == pytest.approx(0.25 * float(np.sum(X[:, 7].astype(np.float64) ** 2)),
                                   rel=1e-13)


# ---------------------------------------------------------------------------------------
# P8: rows decouple ("GPTQ Hessian": every row has the same H); dead-column invariance
# ---------------------------------------------------------------------------------------

def test_row_permutation_and_subset_invariance():
    X, W = correlated_problem(40, 70, 150, 11, dead=(2,))
    out = O.gptq_layer(X, W, 4, block=32)
    perm = np.random.default_rng(0).permutation(40)
    outp = O.gptq_layer(X, W[perm], 4, block=32)
    np.testing.assert_array_equal(outp["codes"], out["codes"][perm])
    sub = np.array([3, 17, 39])
    outs = O.gptq_layer(X, W[sub], 4, block=32)
    np.testing.assert_array_equal(outs["codes"], out["codes"][sub])


def test_dead_columns_are_skipped():
    dead = (4, 9)
    X, W = correlated_problem(12, 16, 40, 12, dead=dead)
    out = O.gptq_layer(X, W, 4, block=8)
    assert np.flatnonzero(out["dead"]).tolist() == list(dead)
    # a dead column quantizes to the zero point, i.e. exactly 0
    np.testing.assert_array_equal(out["codes"][:, list(dead)],
                                  np.repeat(out["zero"][:, None], 2, axis=1))
    assert np.all(out["W_hat"][:, list(dead)] == 0.0)
    # changing the dead weights without changing any row's min/max (so the grid stays
    # the same): swap the two dead columns -> no code anywhere changes
    W2 = W.copy()
    W2[:, [dead[0], dead[1]]] = W[:, [dead[1], dead[0]]]
    assert not np.array_equal(W2, W)
    out2 = O.gptq_layer(X, W2, 4, block=8)
    np.testing.assert_array_equal(out2["scale"], out["scale"])
    np.testing.assert_array_equal(out2["codes"], out["codes"])


def test_damping_mean_taken_after_dead_fix():
    H = np.diag([0.0, 4.0, 2.0])
    Hd, dead, lam = O.damp_hessian(H, 0.01)
    assert dead.tolist() == [True, False, False]
    assert lam == pytest.approx(0.01 * (1.0 + 4.0 + 2.0) / 3)
    np.testing.assert_allclose(np.diag(Hd), [1 + lam, 4 + lam, 2 + lam])


# ---------------------------------------------------------------------------------------
# P9: the high-bit limit
# ---------------------------------------------------------------------------------------

def test_high_bit_limit():
    X, W = correlated_problem(32, 64, 128, 13)
    out16 = O.gptq_layer(X, W, 16)
    out4 = O.gptq_layer(X, W, 4)
    e16 = O.reconstruction_error(W, out16["W_hat"], out16["H"])
    e4 = O.reconstruction_error(W, out4["W_hat"], out4["H"])
    assert e16 < 1e-6 * e4


# ---------------------------------------------------------------------------------------
# P10: the Hessian is exact for half-precision inputs (integer arithmetic)
# ---------------------------------------------------------------------------------------

def test_hessian_exact_against_integer_arithmetic():
    rng = np.random.default_rng(14)
    n, d = 37, 9
    ints = rng.integers(-2048, 2048, size=(n, d))
    X = (ints.astype(np.float64) * 2.0 ** -7).astype(np.float16)  # exact in fp16
    H = O.hessian(X)
    exact = 2 * (ints.T @ ints)                                       # exact integers
    np.testing.assert_array_equal(H, exact.astype(np.float64) * 2.0 ** -14)
    # chunked accumulation = whole
    H2 = O.hessian(X[20:], O.hessian(X[:20]))
    np.testing.assert_array_equal(H2, H)


# ---------------------------------------------------------------------------------------
# Grid and packing
# ---------------------------------------------------------------------------------------

def test_grid_hand_examples():
    W = np.array([[-0.3, 0.1, 0.6], [0.2, 0.4, 0.0], [0.0, 0.0, 0.0]], dtype=np.float32)
    scale, zero = O.row_grid(W, 4)
    np.testing.assert_allclose(scale, [0.9 / 15, 0.4 / 15, 1.0], rtol=1e-6)
    assert zero.tolist() == [5, 0, 0]
    codes, q = O.rtn_quantize(W, scale, zero, 4)
    assert codes[0].tolist() == [0, 7, 15]
    assert codes[1].tolist() == [8, 15, 0]
    assert codes[2].tolist() == [0, 0, 0]


def _pack_cases():
    cases = []
    with open(os.path.join(ROOT, "tests", "golden", "pack_examples.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            b, d, codes, words = [t.strip() for t in line.split("|")]
            cases.append((int(b), int(d), [int(t) for t in codes.split()],
                          [int(t, 16) for t in words.split()]))
    return cases


@pytest.mark.parametrize("bits,d,codes,words", _pack_cases())
def test_pack_hand_examples(bits, d, codes, words):
    packed = O.pack_codes(np.array([codes]), bits)
    assert packed.shape == (1, O.packed_words_per_row(d, bits))
    assert packed[0].tolist() == words
    assert O.unpack_codes(packed, bits, d)[0].tolist() == codes


@pytest.mark.parametrize("bits", [2, 3, 4, 8])
def test_pack_roundtrip_random(bits):
    rng = np.random.default_rng(bits)
    codes = rng.integers(0, 2 ** bits, size=(7, 101))
    np.testing.assert_array_equal(O.unpack_codes(O.pack_codes(codes, bits), bits, 101), codes)


# ---------------------------------------------------------------------------------------
# Block helpers used by the full-size GPU checks
# ---------------------------------------------------------------------------------------

def test_hessian_block_and_diagonal_match_full():
    rng = np.random.default_rng(15)
    ints = rng.integers(-512, 512, size=(300, 40))
    ints[:, 7] = 0                                   # a dead channel
    X = (ints * 2.0 ** -6).astype(np.float16)
    H = O.hessian(X)
    rows, cols = np.array([3, 7, 39]), np.arange(20, 40)
    np.testing.assert_array_equal(O.hessian_block(X, rows, cols), H[np.ix_(rows, cols)])
    np.testing.assert_array_equal(O.hessian_diagonal(X, chunk=64), np.diag(H))
    # exact against integers
    np.testing.assert_array_equal(O.hessian_diagonal(X), 2.0 * (ints ** 2).sum(0) * 2.0 ** -12)


def test_damped_principal_block_matches_full_damping():
    X, _ = correlated_problem(4, 30, 60, 16, dead=(2, 25))
    H = O.hessian(X)
    Hd, dead, lam = O.damp_hessian(H, 0.01)
    idx = np.arange(20, 30)
    Hb, dead_b, lam_b = O.damp_principal_block(H[np.ix_(idx, idx)], np.diag(H), idx, 0.01)
    assert lam_b == lam and np.array_equal(dead_b, dead)
    np.testing.assert_array_equal(Hb, Hd[np.ix_(idx, idx)])


@pytest.mark.parametrize("t", [1, 5, 17])
def test_trailing_block_of_u_depends_only_on_trailing_block_of_h(t):
    # H^-1 = U^T U with U upper  =>  H = R R^T, R = U^-1 upper  =>  H[t:, t:] = R22 R22^T,
    # so U[t:, t:] is the factor of H[t:, t:] alone: this lets a full-size GPU factor be
    # checked on a trailing block the oracle can afford.
    X, _ = correlated_problem(4, 24, 50, 17, dead=(20,))
    Hd, _, _ = O.damp_hessian(O.hessian(X))
    U = O.inverse_cholesky_upper(Hd)
    Ut = O.inverse_cholesky_upper(Hd[t:, t:])
    np.testing.assert_allclose(U[t:, t:], Ut, rtol=0, atol=1e-12 * np.abs(U).max())


# ---------------------------------------------------------------------------------------
# OBQ greedy order (explicit Schur downdates)
# ---------------------------------------------------------------------------------------

def _obq_case(d=7, m=4, seed=5, bits=3):
    X, W = correlated_problem(m, d, 60, seed)
    Hd, dead, _ = O.damp_hessian(O.hessian(X))
    s, z = O.row_grid(W, bits)
    return W, Hd, s, z, dead


def test_obq_first_choice_is_brute_force_least_increase():
    # for every candidate q: fix w_q to its grid value, re-solve the other weights exactly,
    # and measure the increase of 1/2 (v - w) H (v - w)^T; the least one is OBQ's first pick
    W, Hd, s, z, _ = _obq_case()
    bits, d = 3, W.shape[1]
    codes, _, order, _ = O.obq_greedy(W, Hd, s, z, bits)
    Hinv = np.linalg.inv(Hd)
    for i in range(W.shape[0]):
        inc = []
        for q in range(d):
            _, qv = O.quantize_to_grid(W[i, q:q + 1], s[i:i + 1], z[i:i + 1], 2 ** bits - 1)
            F = [k for k in range(d) if k != q]
            # v_F minimises (v - w) H (v - w)^T with v_q = qv
            dq = qv[0] - W[i, q]
            vF = W[i, F] - np.linalg.solve(Hd[np.ix_(F, F)], Hd[F, q] * dq)
            v = W[i].astype(np.float64).copy()
            v[q], v[F] = qv[0], vF
            inc.append(0.5 * (v - W[i]) @ Hd @ (v - W[i]))
            assert inc[-1] == pytest.approx(0.5 * dq * dq / Hinv[q, q], rel=1e-9)
        assert order[i, 0] == int(np.argmin(inc))


def test_obq_with_diagonal_hessian_is_rtn():
    W, _, s, z, _ = _obq_case()
    Hd = np.diag(np.linspace(0.5, 3.0, W.shape[1]))
    codes, W_hat, _, _ = O.obq_greedy(W, Hd, s, z, 3)
    c_rtn, q_rtn = O.rtn_quantize(W, s, z, 3)
    assert np.array_equal(codes, c_rtn)
    np.testing.assert_allclose(W_hat, q_rtn, rtol=0, atol=0)


def test_obq_forced_left_to_right_is_the_fixed_order_sweep():
    W, Hd, s, z, dead = _obq_case(d=9, m=5, seed=8, bits=4)
    d = W.shape[1]
    c_fix, q_fix = O.obs_quantize_schur(W, Hd, s, z, 4, dead=dead)
    order = np.tile(np.arange(d), (W.shape[0], 1))
    c, q, _, info = O.obq_greedy(W, Hd, s, z, 4, dead=dead, forced=(order, c_fix))
    assert info["bad_codes"] == 0 and info["tie_flips"] == 0 and info["bad_order"] == 0
    assert np.array_equal(c, c_fix)
    np.testing.assert_allclose(q, q_fix, rtol=0, atol=1e-15)


def test_obq_is_column_permutation_equivariant():
    W, Hd, s, z, _ = _obq_case(d=8, m=3, seed=11)
    p = np.random.default_rng(2).permutation(W.shape[1])
    c, _, order, _ = O.obq_greedy(W, Hd, s, z, 3)
    cp, _, order_p, _ = O.obq_greedy(W[:, p], Hd[np.ix_(p, p)], s, z, 3)
    assert np.array_equal(cp, c[:, p])
    assert np.array_equal(p[order_p], order)


def test_obq_beats_rtn_on_correlated_inputs():
    W, Hd, s, z, _ = _obq_case(d=10, m=6, seed=13, bits=3)
    _, W_hat, order, _ = O.obq_greedy(W, Hd, s, z, 3)
    _, q_rtn = O.rtn_quantize(W, s, z, 3)
    for i in range(W.shape[0]):
        assert sorted(order[i]) == list(range(W.shape[1]))
    assert O.reconstruction_error(W, W_hat, Hd) < O.reconstruction_error(W, q_rtn, Hd)
