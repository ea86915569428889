"""Pins of the decomposition oracle (oracle/decomposition.py) against what the pages and
the mathematics fix, and planted mistakes that at least one pin must catch.

Each pin reaches its expected value by another route than the oracle's: eigenvalues of
residᵀ·resid for the Eckart-Young error, a planted decomposition whose parts are known,
closed forms for bands of scalar multiples, the passthrough case the pages describe, and,
for the randomized SVD, exact recovery of low-rank matrices and the published error bound.
"""
import numpy as np
import pytest

import oracle
from oracle import reconstruction


def _rng(seed):
    return np.random.default_rng(seed)


# ----------------------------------------------------------------------------------
# pins, each taking the function under test
# ----------------------------------------------------------------------------------
def pin_eckart_young(truncated_svd):
    """The rank-r truncation misses exactly the energy of the smallest singular values:
    ‖R − U·Vᵀ‖_F² = Σ_{j>r} σ_j², with σ_j² the eigenvalues of Rᵀ·R (Eckart-Young)."""
    rng = _rng(11)
    R = rng.standard_normal((9, 13))
    lam = np.sort(np.linalg.eigvalsh(R.T @ R))[::-1][:9]   # the 9 nonzero ones, descending
    for r in (1, 3, 8):
        U, V = truncated_svd(R, r)
        err = np.sum((R - U @ V.T) ** 2)
        if not np.isclose(err, np.sum(lam[r:]), rtol=1e-9, atol=1e-12):
            return False
    return True


def pin_factor_structure(truncated_svd):
    """U absorbs the singular values ("U = U_svd · S"): V has orthonormal columns and
    UᵀU is diagonal with the top r eigenvalues of RᵀR, largest first."""
    rng = _rng(12)
    R = rng.standard_normal((11, 7))
    r = 4
    U, V = truncated_svd(R, r)
    if U.shape != (11, r) or V.shape != (7, r):
        return False
    lam = np.sort(np.linalg.eigvalsh(R.T @ R))[::-1][:r]
    return np.allclose(V.T @ V, np.eye(r), atol=1e-12) and np.allclose(U.T @ U, np.diag(lam), rtol=1e-10,
                                                                        atol=1e-10)


def pin_planted(decompose):
    """weight = diag(c)·W0 + A·Bᵀ with the columns of B in the null space of W0 (so every
    row of A·Bᵀ is orthogonal to the same row of W0): the least-squares scale is c exactly,
    the residual is A·Bᵀ, and rank 2 recovers it."""
    rng = _rng(13)
    out, inp, k = 6, 10, 2
    W0 = rng.standard_normal((out, inp))
    null = np.linalg.svd(W0)[2][out:].T                      # [inp, inp - out], W0 @ null = 0
    B = null @ rng.standard_normal((inp - out, k))
    A = rng.standard_normal((out, k))
    c = rng.uniform(0.5, 1.5, size=out)
    weight = c[:, None] * W0 + A @ B.T
    s, U, V = decompose(weight, W0, k)
    return np.allclose(s, c, rtol=1e-12) and np.allclose(U @ V.T, A @ B.T, atol=1e-10) and \
        np.allclose(s[:, None] * W0 + U @ V.T, weight, atol=1e-10)


def pin_full_rank_is_exact(decompose):
    """At r = min(out, in) the decomposition reproduces the weight."""
    rng = _rng(14)
    weight, W0 = rng.standard_normal((5, 8)), rng.standard_normal((5, 8))
    s, U, V = decompose(weight, W0, 5)
    return np.allclose(s[:, None] * W0 + U @ V.T, weight, atol=1e-12)


def pin_rank_zero(decompose):
    """r = 0: U and V are empty ("When r = 0, U and V are empty")."""
    rng = _rng(15)
    weight, W0 = rng.standard_normal((4, 6)), rng.standard_normal((4, 6))
    _, U, V = decompose(weight, W0, 0)
    return U.shape == (4, 0) and V.shape == (6, 0)


def pin_scalar_bands(decompose_stack):
    """Weights that are scalar multiples a_l·W: each band's W0 is the mean multiple times W,
    s of layer l is a_l over its band's mean on every row, and nothing is left for U·Vᵀ."""
    rng = _rng(16)
    W = rng.standard_normal((5, 7))
    a = np.array([0.5, 1.0, 1.5, 2.0, 3.0, 4.0])
    W0s, layers = decompose_stack([ai * W for ai in a], 2, 2)
    means = [a[:3].mean(), a[3:].mean()]
    if not all(np.allclose(W0s[b], means[b] * W, rtol=1e-13) for b in range(2)):
        return False
    for l, (band, s, U, V) in enumerate(layers):
        if band != (0 if l < 3 else 1) or not np.allclose(s, a[l] / means[band], rtol=1e-12):
            return False
        if not np.allclose(U @ V.T, 0.0, atol=1e-12):
            return False
    return True


def pin_passthrough(decompose_stack):
    """G = L ("The passthrough operating point"): each layer is its own band, its W0 is its
    weight, s = 1, the residual is zero and the weight is reconstructed exactly."""
    rng = _rng(17)
    weights = [rng.standard_normal((4, 9)) for _ in range(3)]
    W0s, layers = decompose_stack(weights, 3, 2)
    for l, (band, s, U, V) in enumerate(layers):
        if band != l or not np.array_equal(W0s[band], weights[l]):
            return False
        if not np.allclose(s, 1.0, rtol=1e-14) or not np.allclose(U @ V.T, 0.0, atol=1e-12):
            return False
    return True


def _orthonormal(rng, n, k):
    return np.linalg.qr(rng.standard_normal((n, k)))[0]


def pin_rsvd_fallback(rsvd):
    """The pages' fallback: min(m, n) <= 256, or a probe of k >= min(m, n) columns, gives
    the exact truncation."""
    rng = _rng(21)
    small = rng.standard_normal((40, 60))
    U, V = rsvd(small, 5, rng.standard_normal((60, 15)))
    U0, V0 = oracle.truncated_svd(small, 5)
    wide = rng.standard_normal((300, 280))
    U1, V1 = rsvd(wide, 4, rng.standard_normal((280, 280)))
    U2, V2 = oracle.truncated_svd(wide, 4)
    return np.allclose(U @ V.T, U0 @ V0.T, atol=1e-12) and np.allclose(U1 @ V1.T, U2 @ V2.T, atol=1e-10)


def pin_rsvd_exact_low_rank(rsvd):
    """A matrix of rank r is recovered exactly: a Gaussian probe of r + p columns spans its
    range with probability one."""
    rng = _rng(22)
    A = rng.standard_normal((300, 6)) @ rng.standard_normal((6, 400))
    U, V = rsvd(A, 6, rng.standard_normal((400, 16)))
    return np.allclose(U @ V.T, A, rtol=0, atol=1e-9 * np.abs(A).max())


def pin_rsvd_spectral_gap(rsvd):
    """Four singular values far above the rest, oversampling p = 10. Without power
    iterations the squared error stays within Halko, Martinsson and Tropp's expected-error
    factor 1 + r/(p - 1) of the optimum, the energy of the tail. With power iterations,
    which sharpen a gap of 10^4 to the rounding level, it is the optimum."""
    rng = _rng(23)
    m, n, r, p = 300, 320, 4, 10
    sig = np.concatenate([[100.0, 60.0, 30.0, 10.0], 1e-3 * rng.uniform(0.5, 1.0, size=m - 4)])
    A = (_orthonormal(rng, m, m) * sig[None, :]) @ _orthonormal(rng, n, m).T
    tail = np.sum(sig[r:] ** 2)
    for q, bound in ((0, 1 + r / (p - 1)), (1, 1 + 1e-6), (2, 1 + 1e-6)):
        U, V = rsvd(A, r, rng.standard_normal((n, r + p)), q)
        if np.sum((A - U @ V.T) ** 2) > bound * tail:
            return False
    return True


def pin_rsvd_structure(rsvd):
    """As for the exact truncation: V orthonormal, UᵀU diagonal and non-increasing."""
    rng = _rng(24)
    A = rng.standard_normal((270, 300))
    U, V = rsvd(A, 5, rng.standard_normal((300, 15)), 1)
    d = np.diag(U.T @ U)
    return np.allclose(V.T @ V, np.eye(5), atol=1e-10) and np.allclose(U.T @ U, np.diag(d), atol=1e-8 * d.max()) \
        and np.all(np.diff(d) <= 1e-9 * d.max())


RSVD_PINS = (pin_rsvd_fallback, pin_rsvd_exact_low_rank, pin_rsvd_spectral_gap, pin_rsvd_structure)


@pytest.mark.parametrize("pin", RSVD_PINS, ids=lambda p: p.__name__)
def test_randomized_svd_pins(pin):
    assert pin(oracle.randomized_svd)


def rsvd_unorthonormalised(A, r, omega, power_iters=0):   # Y used as the basis, never orthonormalised
    A = np.asarray(A, float)
    if min(A.shape) <= 256 or omega.shape[1] >= min(A.shape):
        return oracle.truncated_svd(A, r)
    Y = A @ omega
    ub, sv, vt = np.linalg.svd(Y.T @ A, full_matrices=False)
    return (Y @ ub[:, :r]) * sv[None, :r], vt[:r].T


def rsvd_without_singular_values(A, r, omega, power_iters=0):   # U = Q·Ũ, S dropped
    A = np.asarray(A, float)
    if min(A.shape) <= 256 or omega.shape[1] >= min(A.shape):
        return oracle.truncated_svd(A, r)
    Q = np.linalg.qr(A @ omega)[0]
    ub, sv, vt = np.linalg.svd(Q.T @ A, full_matrices=False)
    return Q @ ub[:, :r], vt[:r].T


def rsvd_never_falls_back(A, r, omega, power_iters=0):   # the randomized path on small matrices too
    A = np.asarray(A, float)
    Q = np.linalg.qr(A @ omega[:, : min(omega.shape[1], min(A.shape) - 1)])[0]
    ub, sv, vt = np.linalg.svd(Q.T @ A, full_matrices=False)
    return (Q @ ub[:, :r]) * sv[None, :r], vt[:r].T


@pytest.mark.parametrize("mutant", [rsvd_unorthonormalised, rsvd_without_singular_values, rsvd_never_falls_back],
                         ids=lambda m: m.__name__)
def test_pins_catch_randomized_svd_mutants(mutant):
    assert not all(pin(mutant) for pin in RSVD_PINS)


SVD_PINS = (pin_eckart_young, pin_factor_structure)
DECOMPOSE_PINS = (pin_planted, pin_full_rank_is_exact, pin_rank_zero)
STACK_PINS = (pin_scalar_bands, pin_passthrough)


@pytest.mark.parametrize("pin", SVD_PINS, ids=lambda p: p.__name__)
def test_truncated_svd_pins(pin):
    assert pin(oracle.truncated_svd)


@pytest.mark.parametrize("pin", DECOMPOSE_PINS, ids=lambda p: p.__name__)
def test_decompose_pins(pin):
    assert pin(oracle.decompose)


@pytest.mark.parametrize("pin", STACK_PINS, ids=lambda p: p.__name__)
def test_decompose_stack_pins(pin):
    assert pin(oracle.decompose_stack)


def test_decomposition_feeds_the_reconstruction_identity():
    """The factors plug into the linear the rest of the oracle computes: y through
    (W0, s, U, V) equals y through the rank-r weight diag(s)·W0 + U·Vᵀ."""
    rng = _rng(18)
    weight, W0 = rng.standard_normal((12, 16)), rng.standard_normal((12, 16))
    s, U, V = oracle.decompose(weight, W0, 3)
    x = rng.standard_normal((5, 16))
    y = oracle.linear(W0, s, U, V, x)
    assert np.allclose(y, x @ (s[:, None] * W0 + U @ V.T).T, rtol=1e-12, atol=1e-12)


# ----------------------------------------------------------------------------------
# planted mistakes: each must fail at least one pin
# ----------------------------------------------------------------------------------
def _svd_parts(R):
    u, sv, vt = np.linalg.svd(np.asarray(R, dtype=np.float64), full_matrices=False)
    return u, sv, vt


def svd_without_singular_values(R, r):        # U = U_svd, S dropped
    u, sv, vt = _svd_parts(R)
    return u[:, :r], vt[:r].T


def svd_values_on_v(R, r):                    # S absorbed by V instead of U
    u, sv, vt = _svd_parts(R)
    return u[:, :r], vt[:r].T * sv[None, :r]


def svd_smallest_values(R, r):                # keeps the r smallest singular triples
    u, sv, vt = _svd_parts(R)
    k = len(sv)
    return u[:, k - r:] * sv[None, k - r:], vt[k - r:].T


def decompose_column_scale(weight, W0, r):    # s fitted per input column
    weight, W0 = np.asarray(weight, float), np.asarray(W0, float)
    s_col = np.einsum("oi,oi->i", weight, W0) / np.einsum("oi,oi->i", W0, W0)
    resid = weight - W0 * s_col[None, :]
    U, V = oracle.truncated_svd(resid, r)
    return np.ones(weight.shape[0]), U, V


def decompose_unscaled_residual(weight, W0, r):   # resid = weight − W0 (s not applied)
    s = reconstruction.ls_scale(weight, W0)
    U, V = oracle.truncated_svd(np.asarray(weight, float) - np.asarray(W0, float), r)
    return s, U, V


def stack_first_layer_as_w0(weights, num_blocks, r):   # W0 = the band's first layer
    L = len(weights)
    bands = [reconstruction.band_of_layer(l, L, num_blocks) for l in range(L)]
    W0s = [np.asarray(weights[bands.index(b)], float) for b in range(num_blocks)]
    return W0s, [(bands[l], *oracle.decompose(weights[l], W0s[bands[l]], r)) for l in range(L)]


def stack_interleaved_bands(weights, num_blocks, r):   # band = l mod G
    L = len(weights)
    bands = [l % num_blocks for l in range(L)]
    W0s = [oracle.band_mean([weights[l] for l in range(L) if bands[l] == b]) for b in range(num_blocks)]
    return W0s, [(bands[l], *oracle.decompose(weights[l], W0s[bands[l]], r)) for l in range(L)]


@pytest.mark.parametrize("mutant", [svd_without_singular_values, svd_values_on_v, svd_smallest_values],
                         ids=lambda m: m.__name__)
def test_pins_catch_svd_mutants(mutant):
    assert not all(pin(mutant) for pin in SVD_PINS)


@pytest.mark.parametrize("mutant", [decompose_column_scale, decompose_unscaled_residual], ids=lambda m: m.__name__)
def test_pins_catch_decompose_mutants(mutant):
    assert not all(pin(mutant) for pin in DECOMPOSE_PINS)


@pytest.mark.parametrize("mutant", [stack_first_layer_as_w0, stack_interleaved_bands], ids=lambda m: m.__name__)
def test_pins_catch_stack_mutants(mutant):
    assert not all(pin(mutant) for pin in STACK_PINS)


def test_stored_scale_residual_pins():
    """The residual of the stored (bf16) scale differs from the exact least-squares residual by
    exactly (s − RN_bf16(s))·W0 row by row, and the stored scale is the bf16 rounding of the
    exact one (closed forms); with a W0 row of zeros the scale is 1 and the residual the weight."""
    rng = np.random.default_rng(11)
    W0 = oracle.round_to_bf16(rng.normal(0, 0.02, (24, 40)))
    W0[5] = 0.0
    w = oracle.round_to_bf16(W0 * rng.uniform(0.9, 1.1, (24, 1)) + rng.normal(0, 0.005, (24, 40)))
    s_b, resid = oracle.ls_residual_stored(w, W0)
    s = oracle.ls_scale(w, W0)
    np.testing.assert_array_equal(s_b, oracle.round_to_bf16(s))
    np.testing.assert_allclose(resid - oracle.ls_residual(w, W0), (s - s_b)[:, None] * W0, rtol=0, atol=1e-15)
    assert s_b[5] == 1.0 and np.array_equal(resid[5], w[5])
    # a planted mistake: the residual of the unrounded scale is not the stored one's
    assert np.max(np.abs(oracle.ls_residual(w, W0) - resid)) > 0
