"""fp64 CPU oracle for the decomposition that produces W0, s, U and V.

TEST INFRASTRUCTURE ONLY, like the rest of this package: the library never imports it,
and it shares no code with the library. It is the reference a GPU decomposition will be
checked against, so it is the plain definition in float64 with numpy's SVD as its only
library primitive.

Sources (page title, then section):
* "How attnquant works", "How the decomposition produces s, U, and V":
  - W0 is the mean of the projection weights over the layers that share it;
  - s[o] = (weight[o] · W0[o]) / (W0[o] · W0[o]), one least-squares scale per output row;
  - resid = weight − diag(s)·W0, factored by a truncated SVD of rank r with U absorbing
    the singular values (U = U_svd·S), so that U·Vᵀ ≈ resid;
  - r = 0 leaves U and V empty.
* "How attnquant works", "The passthrough operating point": with one W0 per layer the
  residual is zero and the reconstructed weight is the original.
* "Banded sharing" (named on the concepts page): layers are grouped into G bands that
  share one W0.

Readings (each also listed in the design notes):
* The truncated SVD here is exact (the full SVD, cut at r). The pages run a randomized
  SVD for large matrices, which approximates this, so a GPU decomposition is compared
  with it through the product U·Vᵀ within that method's error bound. The factors are
  compared only up to the sign and order freedom of an SVD.
* Bands are contiguous: layer l of L belongs to band floor(l·G/L) (reconstruction.py).
"""
from __future__ import annotations

import numpy as np

from .reconstruction import band_of_layer, ls_scale


def band_mean(weights) -> np.ndarray:
    """W0 of one band: the element-wise mean of the band's projection weights, each [out, in]."""
    stack = np.asarray([np.asarray(w, dtype=np.float64) for w in weights])
    if stack.ndim != 3 or stack.shape[0] == 0:
        raise ValueError("band_mean needs one or more [out, in] weights")
    return stack.mean(axis=0)


def truncated_svd(resid, r: int):
    """The best rank-r factors of resid [out, in]: U [out, r] = U_svd[:, :r]·diag(S[:r]) and
    V [in, r] = Vt_svd[:r, :]ᵀ, so U·Vᵀ is the rank-r truncation of resid. r = 0 gives empty
    factors."""
    resid = np.asarray(resid, dtype=np.float64)
    out, inp = resid.shape
    if r < 0 or r > min(out, inp):
        raise ValueError(f"rank {r} outside 0..{min(out, inp)}")
    if r == 0:
        return np.zeros((out, 0)), np.zeros((inp, 0))
    u, sv, vt = np.linalg.svd(resid, full_matrices=False)
    return u[:, :r] * sv[None, :r], vt[:r, :].T


def randomized_svd(A, r: int, omega, power_iters: int = 0):
    """Rank-r factors of A [m, n] by the randomized SVD the pages name (Halko, Martinsson and
    Tropp, 2009: the randomized range finder, with q power iterations, then the SVD of the
    small projected matrix):
        Y = A·Ω,  Q = orth(Y),  [q times: Q = orth(A·orth(Aᵀ·Q))],  B = Qᵀ·A = Ũ·S·Vᵀ,
        U = Q·Ũ[:, :r]·diag(S[:r]),  V = V[:, :r].
    Ω [n, k] is the random test matrix, k = r + oversampling. It is an input, so that two
    implementations can be compared on the same draws. The pages' fallback applies: when
    min(m, n) <= 256, or when the probe would capture the whole matrix (k >= min(m, n)),
    the factors are the exact truncation (truncated_svd)."""
    A = np.asarray(A, dtype=np.float64)
    omega = np.asarray(omega, dtype=np.float64)
    m, n = A.shape
    k = omega.shape[1]
    if omega.shape[0] != n or k < r:
        raise ValueError(f"the test matrix must be [{n}, >= {r}], got {omega.shape}")
    if min(m, n) <= 256 or k >= min(m, n):
        return truncated_svd(A, r)
    if r == 0:
        return np.zeros((m, 0)), np.zeros((n, 0))
    Q = np.linalg.qr(A @ omega)[0]
    for _ in range(power_iters):
        Z = np.linalg.qr(A.T @ Q)[0]
        Q = np.linalg.qr(A @ Z)[0]
    ub, sv, vt = np.linalg.svd(Q.T @ A, full_matrices=False)
    return (Q @ ub[:, :r]) * sv[None, :r], vt[:r].T


def ls_residual_stored(weight, W0):
    """The scale as the bundle stores it and the residual left for U·Vᵀ: s_b = RN_bf16(s) with s
    the least-squares scale of ``ls_scale``, and resid = weight − diag(s_b)·W0. The bundle holds
    s in bfloat16 ("The theta bundle": every piece stored like the weights), so the rank-r factors
    must represent the residual of the stored scale, not of the exact one."""
    from .reconstruction import round_to_bf16
    weight = np.asarray(weight, dtype=np.float64)
    W0 = np.asarray(W0, dtype=np.float64)
    s_b = round_to_bf16(ls_scale(weight, W0))
    return s_b, weight - s_b[:, None] * W0


def decompose(weight, W0, r: int):
    """One projection weight [out, in] against its band's W0: (s, U, V) with
    weight ≈ diag(s)·W0 + U·Vᵀ."""
    weight = np.asarray(weight, dtype=np.float64)
    W0 = np.asarray(W0, dtype=np.float64)
    s = ls_scale(weight, W0)
    resid = weight - s[:, None] * W0
    U, V = truncated_svd(resid, r)
    return s, U, V


def decompose_stack(weights, num_blocks: int, r: int):
    """A stack of L layer weights of one projection family with G = num_blocks bands:
    the band W0s, and for every layer (band, s, U, V)."""
    L = len(weights)
    bands = [band_of_layer(l, L, num_blocks) for l in range(L)]
    W0s = [band_mean([weights[l] for l in range(L) if bands[l] == b]) for b in range(num_blocks)]
    layers = [(bands[l], *decompose(weights[l], W0s[bands[l]], r)) for l in range(L)]
    return W0s, layers
