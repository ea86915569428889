"""Pins of the decomposition oracle (oracle/decomposition.py) against what the pages and
the mathematics fix, and planted mistakes that at least one pin must catch.

Each pin reaches its expected value by another route than the oracle's: eigenvalues of
residᵀ·resid for the Eckart-Young error, a planted decomposition whose parts are known,
closed forms for bands of scalar multiples, and the passthrough case the pages describe.
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
