"""fp64 CPU oracle for the theta-bundle reconstruction linear.

TEST INFRASTRUCTURE ONLY. This module is the independent reference the CUDA path is
checked against. Only the tests, the smoke check (``__graft_entry__.smoke``) and the
benchmark's CPU-baseline leg may import it; the library never does, and it shares no
code with the library (inputs arrive as plain float64 arrays holding bf16 values).

Everything here is the plain definition from the pages, written out in float64 with
numpy's matmul as the only library primitive; there is no blocking, fusion or
reordering beyond what the definitions state.

Sources (page title, then section):
* "How attnquant works", "The theta bundle": W0 is one dense [out, in] block per
  projection family; s is a per-output-row scale; U, V are rank-r factors.
* "How attnquant works", "The reconstruction identity": the weight is
  diag(s)·W0 + U·Vᵀ and the projection output is y = s·(W0 x) + U(Vᵀ x).
* "Execution paths", "The GEMM formulation": y = s[None, :]·(x @ W0.T) + (x @ V) @ U.T,
  which fixes the orientation: x [M, in], y [M, out], W0 [out, in], V [in, r],
  U [out, r], and s indexes the output axis.
* "Execution paths", "Precompute-outside: the production path": W_eff = s·W0 + U·Vᵀ
  built once per layer; the stacked Q/K/V layer concatenates the three projections.
* "How attnquant works", "How the decomposition produces s, U, and V": the per-row
  least-squares scale s[o] = (weight[o]·W0[o]) / (W0[o]·W0[o]) and r = 0 meaning
  empty U, V.

Readings where the pages are silent (each also listed in the design notes):
* W_eff is rounded once to bfloat16, round-to-nearest-even ("W_eff rounding").
* A W0 row that is all zero gets s = 1 in the least-squares fit (the formula divides
  by zero there).
* Layer l of L belongs to band floor(l·G/L) when L layers share G blocks.

Parity status: every function below is pinned by the CPU tests in
``tests/test_oracle_pins.py`` (closed forms, special cases, invariants, brute force
and bf16 rounding golden values); none is "parity unpinned".
"""
from __future__ import annotations

import numpy as np


def _f64(a) -> np.ndarray:
    return np.asarray(a, dtype=np.float64)


def linear(W0, s, U, V, x) -> np.ndarray:
    """y[m, o] = s[o]·Σ_i W0[o,i]·x[m,i] + Σ_k U[o,k]·(Σ_i V[i,k]·x[m,i]), in float64.

    "How attnquant works", "The reconstruction identity" (y = s·(W0 x) + U(Vᵀ x)),
    with the axes of "Execution paths", "The GEMM formulation".
    W0 [out, in], s [out], U [out, r], V [in, r], x [M, in]  ->  y [M, out].
    r = 0 (U, V of width 0) leaves the scaled shared block alone.
    """
    W0, s, U, V, x = map(_f64, (W0, s, U, V, x))
    z = x @ W0.T                  # shared-block term W0 x, one column per token
    t = x @ V                     # down-projection Vᵀ x
    return s[None, :] * z + t @ U.T


def linear_qkv(thetas, x) -> list[np.ndarray]:
    """The three attention projections of one layer applied to the same x.

    "Execution paths", "Precompute-outside: the production path" and "The GEMM
    formulation" batch q/k/v over one input; each family keeps its own W0, s, U, V,
    so the result is the three identities side by side.
    ``thetas`` is a sequence of three (W0, s, U, V) tuples.
    """
    return [linear(W0, s, U, V, x) for (W0, s, U, V) in thetas]


def effective_weight(W0, s, U, V) -> np.ndarray:
    """W_eff = diag(s)·W0 + U·Vᵀ in float64 (exact for bf16 inputs up to the final
    sum's rounding in double).

    "Execution paths", "Precompute-outside: the production path" (W_eff = s·W0 + U·Vᵀ)
    and "How attnquant works", "The reconstruction identity" (diag(s)·W0 + U·Vᵀ).
    """
    W0, s, U, V = map(_f64, (W0, s, U, V))
    return s[:, None] * W0 + U @ V.T


def round_to_bf16(v) -> np.ndarray:
    """Nearest bfloat16 value of each double, ties to even, returned as float64.

    bfloat16 keeps 8 significant bits and fp32's 8-bit exponent: a value v with
    2**(e-1) <= |v| < 2**e is rounded to a multiple of 2**(e-8), with the spacing
    never finer than 2**-133 (subnormals); magnitudes that round to 2**128 or more
    become infinities.
    """
    v = _f64(v)
    out = np.empty_like(v)
    finite = np.isfinite(v) & (v != 0)
    out[~finite] = v[~finite]
    a = np.abs(v[finite])
    e = np.floor(np.log2(a)).astype(np.int64) + 1
    # log2 may be off by one right at powers of two: fix e so 2**(e-1) <= a < 2**e
    e = np.where(np.ldexp(1.0, e - 1) > a, e - 1, e)
    e = np.where(np.ldexp(1.0, e) <= a, e + 1, e)
    step = np.maximum(e - 8, -133)
    q = np.ldexp(1.0, step)
    k = a / q                                 # exact: scaling by a power of two
    fl = np.floor(k)
    frac = k - fl
    up = (frac > 0.5) | ((frac == 0.5) & (np.fmod(fl, 2.0) == 1.0))
    mag = (fl + up) * q
    mag = np.where(mag >= 2.0 ** 128, np.inf, mag)
    out[finite] = np.sign(v[finite]) * mag
    return out


def effective_weight_bf16(W0, s, U, V) -> np.ndarray:
    """RN_bf16(W_eff): the load-time weight as a bf16 tensor would hold it
    (values returned as float64). Rounding point: one rounding of the exact sum."""
    return round_to_bf16(effective_weight(W0, s, U, V))


def ls_scale(weight, W0) -> np.ndarray:
    """Per-output-row least-squares scale of W0 toward a target weight.

    "How attnquant works", "How the decomposition produces s, U, and V":
    s[o] = (weight[o]·W0[o]) / (W0[o]·W0[o]). An all-zero W0 row gets s = 1.
    """
    weight, W0 = _f64(weight), _f64(W0)
    num = np.einsum("oi,oi->o", weight, W0)
    den = np.einsum("oi,oi->o", W0, W0)
    safe = np.where(den == 0.0, 1.0, den)
    return np.where(den == 0.0, 1.0, num / safe)


def ls_residual(weight, W0) -> np.ndarray:
    """resid = weight − diag(s)·W0 with the least-squares s above (same section)."""
    weight, W0 = _f64(weight), _f64(W0)
    return weight - ls_scale(weight, W0)[:, None] * W0


def band_of_layer(layer: int, num_layers: int, num_blocks: int) -> int:
    """Band (index of the shared W0) of a layer when num_layers share num_blocks
    blocks in contiguous bands ("How attnquant works", "How the decomposition
    produces s, U, and V": W0 is shared by the layers of a band; G = num_layers is
    one block per layer, G = 1 one block for the stack)."""
    if not (0 <= layer < num_layers) or not (1 <= num_blocks <= num_layers):
        raise ValueError("layer/band arguments out of range")
    return (layer * num_blocks) // num_layers


# ----------------------------------------------------------------------------------
# Acceptance measures (the tolerances the parity tests apply)
# ----------------------------------------------------------------------------------
def error_stats(y, y_ref) -> dict:
    """max |y − y_ref|, max |y_ref| and relative L2 error, all in float64."""
    y, y_ref = _f64(y), _f64(y_ref)
    d = y - y_ref
    nref = float(np.linalg.norm(y_ref))
    return {
        "max_abs_err": float(np.max(np.abs(d))) if d.size else 0.0,
        "max_abs_ref": float(np.max(np.abs(y_ref))) if y_ref.size else 0.0,
        "rel_l2": float(np.linalg.norm(d) / nref) if nref > 0 else float(np.linalg.norm(d)),
    }


def within_tolerance(y, y_ref, elem_tol: float = 1e-2, l2_tol: float = 2e-3) -> bool:
    """Elementwise |Δ| <= elem_tol·max|y_ref| and relative L2 <= l2_tol."""
    st = error_stats(y, y_ref)
    return st["max_abs_err"] <= elem_tol * st["max_abs_ref"] and st["rel_l2"] <= l2_tol


def linear_error_bound(W0, s, U, V, x, unit_roundoff: float = 2.0 ** -23) -> np.ndarray:
    """Element-wise bound on |y − y_ref| for a bf16 result of the identity computed with fp32
    accumulation, t held in bf16 between the down- and the up-projection, and one final
    rounding to bf16 (the rounding points read from "Execution paths", "The GEMM
    formulation" and "The custom op": bf16 storage, fp32 accumulation).

    Three terms, each from the classical analysis of floating-point sums (Higham, "Accuracy
    and Stability of Numerical Algorithms", sec. 3.1, |fl(Σ a_i) − Σ a_i| <= γ_n Σ |a_i| with
    γ_n = n·u / (1 − n·u), taken with u = 2^-23 so that truncating accumulation is covered):
      acc   = γ_n·( |s|·(|W0|·|x|) + |U|·(|V|·|x|) ),  n = in + r + 2 (the longest chain of
              roundings: a dot product over `in`, one over r, the scale and the sum);
      t_rd  = 2^-8·|U|·|t|: t rounded to bf16 (relative error at most 2^-8) before U·t;
      out   = 2^-8·(|y_ref| + acc + t_rd): the final rounding of the fp32 value to bf16.
    Returns acc + t_rd + out (+ 2^-133 for bf16's subnormal spacing). Where an output has so
    few elements that the relative-L2 bar of ``within_tolerance`` is out of reach even for
    the exactly rounded RN_bf16(y_ref), this bound is the bar each element is held to.
    """
    W0, s, U, V, x = map(_f64, (W0, s, U, V, x))
    ax = np.abs(x)
    n = W0.shape[1] + U.shape[1] + 2
    gamma = n * unit_roundoff / (1.0 - n * unit_roundoff)
    acc = gamma * (np.abs(s)[None, :] * (ax @ np.abs(W0).T) + (ax @ np.abs(V)) @ np.abs(U).T)
    t_rd = 2.0 ** -8 * (np.abs(x @ V) @ np.abs(U).T)
    y = linear(W0, s, U, V, x)
    return acc + t_rd + 2.0 ** -8 * (np.abs(y) + acc + t_rd) + 2.0 ** -133


def within_error_bound(y, W0, s, U, V, x) -> bool:
    """Every element of y within ``linear_error_bound`` of the fp64 identity."""
    y_ref = linear(W0, s, U, V, x)
    return bool(np.all(np.abs(_f64(y) - y_ref) <= linear_error_bound(W0, s, U, V, x)))


def bf16_ordinal(bits) -> np.ndarray:
    """Monotone integer image of bf16 bit patterns (+0 and −0 both map to 0), so that
    adjacent representable values differ by exactly 1."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.int64)
    mag = b & 0x7FFF
    return np.where(b & 0x8000, -mag, mag)


def weight_acceptance(got_bits, W0, s, U, V, unit_roundoff: float = 2.0 ** -23) -> dict:
    """Element-wise acceptance of a bf16 W_eff computed with fp32 accumulation.

    Bar: within 1 bf16 ulp of RN_bf16(W_eff). Where that ulp is smaller than what any
    fp32 evaluation can guarantee -- elements where s·W0 and U·Vᵀ nearly cancel -- the
    element is held instead to the classical error bound of a floating-point dot
    product of n = r + 1 terms (Higham, "Accuracy and Stability of Numerical
    Algorithms", sec. 3.1: |fl(Σ a_i) − Σ a_i| <= γ_n Σ |a_i|, γ_n = n·u / (1 − n·u)),
    taken with u = 2^-23 so that truncating accumulation is covered too, plus half a
    bf16 ulp for the final rounding. Returns counts and the largest ulp distance.
    """
    W0, s, U, V = map(_f64, (W0, s, U, V))
    exact = effective_weight(W0, s, U, V)
    ref_bits = bf16_bits_of_value(round_to_bf16(exact))
    got_bits = np.asarray(got_bits, dtype=np.uint16)
    ulp = np.abs(bf16_ordinal(got_bits) - bf16_ordinal(ref_bits))
    got = (got_bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    n = U.shape[1] + 1
    gamma = n * unit_roundoff / (1.0 - n * unit_roundoff)
    terms = np.abs(s[:, None] * W0) + np.abs(U) @ np.abs(V).T
    bound = gamma * terms + np.abs(got) * 2.0 ** -8 + 2.0 ** -133
    ok = (ulp <= 1) | (np.abs(got - exact) <= bound)
    return {"elements": int(ulp.size), "within_1ulp": int(np.count_nonzero(ulp <= 1)),
            "max_ulp": int(ulp.max()) if ulp.size else 0, "all_ok": bool(np.all(ok)),
            "outside_bound": int(np.count_nonzero(~ok))}


def bf16_bits_of_value(v) -> np.ndarray:
    """Bit patterns of doubles that are exactly representable in bf16 (e.g. the
    output of ``round_to_bf16``)."""
    v = _f64(v)
    f = v.astype(np.float32)
    if not np.array_equal(f.astype(np.float64), v, equal_nan=True):
        raise ValueError("value not representable in bf16")
    bits = f.view(np.uint32)
    if np.any(bits & np.uint32(0xFFFF)):
        raise ValueError("value not representable in bf16")
    return (bits >> np.uint32(16)).astype(np.uint16)
