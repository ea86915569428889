"""Pins of the fp64 oracle against what the pages and the mathematics fix.

None of these re-types the oracle's formula: each checks a closed form, a special
case with a known answer, an invariant, or golden values of the bf16 format. The
mutation tests at the end plant plausible mistakes in copies of the oracle (on the
CPU) and check that at least one pin catches each of them.
"""
import os

import numpy as np
import pytest

import oracle
from rank_weight_reconstruction_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ----------------------------------------------------------------------------------
# pins, parameterised by the functions under test so mutants can be run through them
# ----------------------------------------------------------------------------------
def _rng(seed):
    return np.random.default_rng(seed)


def pin_permutation_scale(linear):
    """W0 = permutation matrix P (P[o, π(o)] = 1), r = 0: y[m, o] = s[o]·x[m, π(o)].
    Fixes the axis s scales ("a per-output-row scale", "How attnquant works",
    "The theta bundle") and the orientation of W0 ("x @ W0.T", "Execution paths",
    "The GEMM formulation")."""
    rng = _rng(1)
    n, M = 7, 3
    perm = rng.permutation(n)
    W0 = np.zeros((n, n))
    W0[np.arange(n), perm] = 1.0
    s = np.arange(1, n + 1) * 0.25
    x = rng.integers(-5, 6, size=(M, n)).astype(float)
    y = linear(W0, s, np.zeros((n, 0)), np.zeros((n, 0)), x)
    return np.array_equal(y, s[None, :] * x[:, perm])


def pin_single_entry_delta(linear):
    """W0 = 0, U = c·e_a, V = e_b: the delta U·Vᵀ is c at (a, b), so y[m, a] = c·x[m, b]
    and every other output is 0 ("The reconstruction identity": U(Vᵀ x))."""
    out, inp, M = 5, 6, 4
    a, b, c = 3, 1, 2.5
    U = np.zeros((out, 1)); U[a, 0] = c
    V = np.zeros((inp, 1)); V[b, 0] = 1.0
    x = _rng(2).integers(-4, 5, size=(M, inp)).astype(float)
    y = linear(np.zeros((out, inp)), np.full(out, 3.0), U, V, x)
    want = np.zeros((M, out)); want[:, a] = c * x[:, b]
    return np.array_equal(y, want)


def pin_two_term_delta(linear):
    """Rank 2 with disjoint single entries: y[m, a1] = c1·x[m, b1], y[m, a2] = c2·x[m, b2];
    checks the sum over k pairs U's and V's columns with the same k."""
    out, inp, M = 6, 5, 3
    (a1, b1, c1), (a2, b2, c2) = (0, 4, 1.5), (5, 2, -3.0)
    U = np.zeros((out, 2)); U[a1, 0] = c1; U[a2, 1] = c2
    V = np.zeros((inp, 2)); V[b1, 0] = 1.0; V[b2, 1] = 1.0
    x = _rng(3).integers(-4, 5, size=(M, inp)).astype(float)
    y = linear(np.zeros((out, inp)), np.ones(out), U, V, x)
    want = np.zeros((M, out)); want[:, a1] = c1 * x[:, b1]; want[:, a2] = c2 * x[:, b2]
    return np.array_equal(y, want)


def pin_scaled_prefix_sum(linear):
    """r = 0 leaves the scaled shared block ("How attnquant works", "How the
    decomposition produces s, U, and V": U, V empty). With W0 lower-triangular ones,
    W0 x is the running sum of x, so y = s ⊙ cumsum(x)."""
    n, M = 9, 4
    W0 = np.tril(np.ones((n, n)))
    s = np.linspace(0.5, 2.0, n)
    x = _rng(4).integers(-6, 7, size=(M, n)).astype(float)
    y = linear(W0, s, np.zeros((n, 0)), np.zeros((n, 0)), x)
    return np.allclose(y, s[None, :] * np.cumsum(x, axis=1), rtol=0, atol=1e-12)


def pin_passthrough(linear):
    """Passthrough operating point (s = 1, U = V = 0, "The passthrough operating
    point"): the bundle is the weight itself; with W0 = tril(ones) y = cumsum(x)."""
    n, M, r = 8, 3, 4
    W0 = np.tril(np.ones((n, n)))
    x = _rng(5).integers(-6, 7, size=(M, n)).astype(float)
    y = linear(W0, np.ones(n), np.zeros((n, r)), np.zeros((n, r)), x)
    return np.array_equal(y, np.cumsum(x, axis=1))


def pin_linear_in_x(linear):
    """The projection is linear in x: y(a·x1 + b·x2) = a·y(x1) + b·y(x2)."""
    rng = _rng(6)
    out, inp, r, M = 11, 13, 3, 2
    W0, U, V = rng.normal(size=(out, inp)), rng.normal(size=(out, r)), rng.normal(size=(inp, r))
    s = rng.uniform(0.5, 1.5, out)
    x1, x2 = rng.normal(size=(M, inp)), rng.normal(size=(M, inp))
    lhs = linear(W0, s, U, V, 2.0 * x1 - 3.0 * x2)
    rhs = 2.0 * linear(W0, s, U, V, x1) - 3.0 * linear(W0, s, U, V, x2)
    return np.allclose(lhs, rhs, rtol=1e-12, atol=1e-12)


def pin_weight_consistency(linear, effective_weight):
    """"The reconstruction identity": applying weight = diag(s)·W0 + U·Vᵀ to x gives
    s·(W0 x) + U(Vᵀ x); the factorised and the materialised forms agree in fp64."""
    rng = _rng(7)
    out, inp, r, M = 17, 23, 5, 6
    W0, U, V = rng.normal(size=(out, inp)), rng.normal(size=(out, r)), rng.normal(size=(inp, r))
    s = rng.uniform(0.5, 1.5, out)
    x = rng.normal(size=(M, inp))
    y1 = linear(W0, s, U, V, x)
    y2 = x @ effective_weight(W0, s, U, V).T
    return np.max(np.abs(y1 - y2)) <= 1e-12 * np.max(np.abs(y2))


def pin_weight_single_entry(effective_weight):
    """W_eff for U = c·e_a, V = e_b is diag(s)·W0 plus c at (a, b) ("Precompute-outside:
    the production path": W_eff = s·W0 + U·Vᵀ)."""
    rng = _rng(8)
    out, inp = 6, 6                      # square, so a transposed delta would still run
    W0 = rng.integers(-3, 4, size=(out, inp)).astype(float)
    s = np.array([0.5, 1.0, 2.0, 4.0, 0.25, 8.0])
    a, b, c = 2, 5, 7.0
    U = np.zeros((out, 1)); U[a, 0] = c
    V = np.zeros((inp, 1)); V[b, 0] = 1.0
    want = W0 * s[:, None]
    want[a, b] += c
    return np.array_equal(effective_weight(W0, s, U, V), want)


ALL_LINEAR_PINS = [pin_permutation_scale, pin_single_entry_delta, pin_two_term_delta,
                   pin_scaled_prefix_sum, pin_passthrough, pin_linear_in_x]


# ----------------------------------------------------------------------------------
# the oracle passes every pin
# ----------------------------------------------------------------------------------
@pytest.mark.parametrize("pin", ALL_LINEAR_PINS, ids=lambda f: f.__name__)
def test_linear_pins(pin):
    assert pin(oracle.linear)


def test_weight_consistency():
    assert pin_weight_consistency(oracle.linear, oracle.effective_weight)


def test_weight_single_entry():
    assert pin_weight_single_entry(oracle.effective_weight)


def test_weight_passthrough_is_w0_bitwise():
    """Passthrough: the rebuilt weight equals the original exactly, bit for bit after
    rounding to bf16 ("The passthrough operating point")."""
    th = synth.passthrough_theta(("pin", "pt"), 33, 40, 8)
    W0, s, U, V = th.f64()
    W = oracle.effective_weight_bf16(W0, s, U, V)
    assert np.array_equal(oracle.bf16_bits_of_value(W), th.W0[:, :40])


def test_weight_rank0_is_rounded_scaled_block():
    """r = 0: W_eff = RN(s·W0); for s = 2^k the product is exact so RN is the identity."""
    th = synth.make_theta(("pin", "r0"), 16, 24, 0)
    W0, _, U, V = th.f64()
    s = np.ldexp(1.0, np.arange(16) % 5 - 2)
    W = oracle.effective_weight_bf16(W0, s, U, V)
    assert np.array_equal(W, s[:, None] * W0)


def _golden_rows():
    rows = []
    with open(os.path.join(GOLDEN, "bf16_rounding.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            v, bits = line.split()[:2]
            rows.append((float.fromhex(v), int(bits, 16)))
    return rows


def test_bf16_rounding_golden():
    rows = _golden_rows()
    vals = np.array([v for v, _ in rows])
    want = np.array([b for _, b in rows], dtype=np.uint16)
    got_oracle = oracle.round_to_bf16(vals)
    got_bits = np.array([(np.float32(g).view(np.uint32) >> 16) for g in got_oracle], dtype=np.uint16)
    assert np.array_equal(got_bits, want)
    # the input generator's own rounding is pinned by the same table
    assert np.array_equal(synth.bf16_bits_from_f64(vals), want)


def test_bf16_rounding_matches_generator_on_random_doubles():
    """Two independent roundings (oracle: floor/tie logic; generator: numpy's
    half-even round) agree on a million random doubles of mixed magnitudes."""
    rng = _rng(9)
    v = rng.normal(size=1_000_000) * np.ldexp(1.0, rng.integers(-140, 120, size=1_000_000))
    a = oracle.bf16_bits_of_value(oracle.round_to_bf16(v))
    b = synth.bf16_bits_from_f64(v)
    assert np.array_equal(a, b)


def test_bf16_ordinal():
    bits = np.array([0x0000, 0x8000, 0x0001, 0x8001, 0x3F80, 0x3F81, 0xBF80], dtype=np.uint16)
    assert list(oracle.bf16_ordinal(bits)) == [0, 0, 1, -1, 0x3F80, 0x3F81, -0x3F80]


def test_ls_scale_orthogonal_residual():
    """Least squares ("How the decomposition produces s, U, and V"): the residual rows
    are orthogonal to the W0 rows."""
    rng = _rng(10)
    w, W0 = rng.normal(size=(40, 64)), rng.normal(size=(40, 64))
    resid = oracle.ls_residual(w, W0)
    dots = np.einsum("oi,oi->o", resid, W0)
    bound = 1e-12 * np.linalg.norm(resid, axis=1) * np.linalg.norm(W0, axis=1) + 1e-300
    assert np.all(np.abs(dots) <= bound * 10)


def test_ls_scale_recovers_known_scale():
    """weight = diag(c)·W0 + N with N ⟂ W0 row-wise has least-squares scale c."""
    rng = _rng(11)
    W0 = rng.normal(size=(12, 30))
    c = rng.uniform(0.5, 2.0, 12)
    G = rng.normal(size=(12, 30))
    N = G - (np.einsum("oi,oi->o", G, W0) / np.einsum("oi,oi->o", W0, W0))[:, None] * W0
    s = oracle.ls_scale(c[:, None] * W0 + N, W0)
    assert np.allclose(s, c, rtol=1e-12, atol=0)
    z = W0.copy(); z[3] = 0.0
    assert oracle.ls_scale(rng.normal(size=(12, 30)), z)[3] == 1.0


def test_band_of_layer():
    assert [oracle.band_of_layer(l, 26, 1) for l in range(26)] == [0] * 26
    assert [oracle.band_of_layer(l, 26, 26) for l in range(26)] == list(range(26))
    bands = [oracle.band_of_layer(l, 60, 4) for l in range(60)]
    assert bands == sorted(bands) and all(bands.count(b) == 15 for b in range(4))
    odd = [oracle.band_of_layer(l, 10, 3) for l in range(10)]
    assert odd == sorted(odd) and {odd.count(b) for b in range(3)} <= {3, 4}
    with pytest.raises(ValueError):
        oracle.band_of_layer(26, 26, 1)


def test_brute_force_tiny():
    """Tiny sizes against explicitly expanded sums over Python floats."""
    rng = _rng(12)
    for out, inp, r, M in [(1, 1, 0, 1), (3, 2, 1, 2), (8, 8, 2, 3), (5, 7, 2, 1)]:
        W0 = rng.integers(-3, 4, size=(out, inp)).astype(float)
        U = rng.integers(-3, 4, size=(out, r)).astype(float)
        V = rng.integers(-3, 4, size=(inp, r)).astype(float)
        s = rng.choice([0.5, 1.0, 2.0], size=out)
        x = rng.integers(-3, 4, size=(M, inp)).astype(float)
        want = np.zeros((M, out))
        for m in range(M):
            for o in range(out):
                acc = 0.0
                for i in range(inp):
                    acc += s[o] * W0[o][i] * x[m][i]
                for k in range(r):
                    tk = 0.0
                    for i in range(inp):
                        tk += V[i][k] * x[m][i]
                    acc += U[o][k] * tk
                want[m][o] = acc
        assert np.array_equal(oracle.linear(W0, s, U, V, x), want)


def test_linear_qkv_is_three_projections():
    rng = _rng(13)
    x = rng.normal(size=(3, 10))
    ths = [(rng.normal(size=(o, 10)), rng.uniform(0.9, 1.1, o), rng.normal(size=(o, 2)),
            rng.normal(size=(10, 2))) for o in (8, 4, 4)]
    ys = oracle.linear_qkv(ths, x)
    assert [y.shape for y in ys] == [(3, 8), (3, 4), (3, 4)]
    for y, th in zip(ys, ths):
        assert np.array_equal(y, oracle.linear(*th, x))


def test_tolerance_measures():
    y_ref = np.array([[1.0, -2.0, 4.0]])
    assert oracle.within_tolerance(y_ref, y_ref)
    assert not oracle.within_tolerance(y_ref + np.array([[0.0, 0.0, 0.05]]), y_ref)
    st = oracle.error_stats(y_ref * (1 + 1e-3), y_ref)
    assert abs(st["rel_l2"] - 1e-3) < 1e-12


# ----------------------------------------------------------------------------------
# mutation tests: plausible mistakes planted in copies of the oracle must be caught
# ----------------------------------------------------------------------------------
def _m_drop_delta(W0, s, U, V, x):
    return s[None, :] * (x @ W0.T)


def _m_scale_input_axis(W0, s, U, V, x):
    if W0.shape[0] != W0.shape[1]:
        return np.zeros((x.shape[0], W0.shape[0]))   # would not even run on such shapes
    return (x * s[None, :]) @ W0.T + (x @ V) @ U.T


def _m_transposed_w0(W0, s, U, V, x):
    if W0.shape[0] != W0.shape[1]:
        return np.zeros((x.shape[0], W0.shape[0]))
    return s[None, :] * (x @ W0) + (x @ V) @ U.T


def _m_swapped_factors(W0, s, U, V, x):
    if U.shape[0] != V.shape[0]:
        return np.zeros((x.shape[0], W0.shape[0]))
    return s[None, :] * (x @ W0.T) + (x @ U) @ V.T


def _m_scale_on_delta(W0, s, U, V, x):
    return s[None, :] * (x @ W0.T + (x @ V) @ U.T)


def _m_no_scale(W0, s, U, V, x):
    return x @ W0.T + (x @ V) @ U.T


def _m_reversed_rank(W0, s, U, V, x):
    return s[None, :] * (x @ W0.T) + (x @ V) @ U[:, ::-1].T


def _m_squared_t(W0, s, U, V, x):
    t = x @ V
    return s[None, :] * (x @ W0.T) + (t * np.abs(t)) @ U.T


LINEAR_MUTANTS = [_m_drop_delta, _m_scale_input_axis, _m_transposed_w0, _m_swapped_factors,
                  _m_scale_on_delta, _m_no_scale, _m_reversed_rank, _m_squared_t]


@pytest.mark.parametrize("mutant", LINEAR_MUTANTS, ids=lambda f: f.__name__)
def test_pins_catch_linear_mutants(mutant):
    results = [pin(mutant) for pin in ALL_LINEAR_PINS]
    assert not all(results), f"{mutant.__name__} passed every pin"


def _w_scale_columns(W0, s, U, V):
    return W0 * np.resize(s, W0.shape[1])[None, :] + U @ V.T


def _w_transposed_delta(W0, s, U, V):
    d = V @ U.T
    return s[:, None] * W0 + (d.T if d.shape != W0.shape else d)


def _w_drop_scale(W0, s, U, V):
    return W0 + U @ V.T


@pytest.mark.parametrize("mutant", [_w_scale_columns, _w_transposed_delta, _w_drop_scale],
                         ids=lambda f: f.__name__)
def test_pins_catch_weight_mutants(mutant):
    ok_single = pin_weight_single_entry(mutant)
    ok_cons = pin_weight_consistency(oracle.linear, mutant)
    assert not (ok_single and ok_cons)


@pytest.mark.parametrize("mutant", [_m_drop_delta, _m_scale_input_axis, _m_no_scale,
                                    _m_swapped_factors],
                         ids=lambda f: f.__name__)
def test_parity_tolerance_rejects_mutants_at_tiny_config(mutant):
    """The parity bar (|Δ| <= 1e-2·max|y_ref|, rel L2 <= 2e-3) is tight enough that the
    same mistakes made by a kernel would fail on the 256x256, r=8, M=1 workload.
    (Scaling the delta by s as well is too small to see at s ~ U(0.9, 1.1); the
    integer-valued GPU cases, compared bit for bit, catch that one.)"""
    th = synth.make_theta(("pin", "tol"), 256, 256, 8)
    x = synth.bf16_bits_to_f64(synth.make_x(("pin", "tol"), 1, 256))[:, :256]
    W0, s, U, V = th.f64()
    y_ref = oracle.linear(W0, s, U, V, x)
    assert not oracle.within_tolerance(mutant(W0, s, U, V, x), y_ref)


# ----------------------------------------------------------------------------------
# the W_eff acceptance measure
# ----------------------------------------------------------------------------------
def _fp32_weight(W0, s, U, V, drop_chunk=None):
    """A plain fp32 evaluation: products summed one k at a time in fp32, then one
    rounding of s*W0 + D (the product s*W0 of two bf16 values is exact in fp32)."""
    D = np.zeros((W0.shape[0], V.shape[0]), np.float32)
    for k in range(U.shape[1]):
        if drop_chunk is not None and drop_chunk[0] <= k < drop_chunk[1]:
            continue
        D = (D + np.outer(U[:, k].astype(np.float32), V[:, k].astype(np.float32))).astype(np.float32)
    w32 = (s[:, None] * W0 + D.astype(np.float64)).astype(np.float32)
    return synth.bf16_bits_from_f64(w32.astype(np.float64))


def test_one_ulp_is_unreachable_in_fp32_near_cancellation():
    """Where s*W0 and U*V^T nearly cancel, even a careful fp32 evaluation misses 1 bf16
    ulp of the exact result; the acceptance measure holds such elements to the fp32
    dot-product error bound instead, and everything else to 1 ulp."""
    th = synth.make_theta(("pre", 520, 384, 256), 520, 384, 256)
    W0, s, U, V = th.f64()
    got = _fp32_weight(W0, s, U, V)
    acc = oracle.weight_acceptance(got, W0, s, U, V)
    assert acc["max_ulp"] > 1            # 1 ulp alone would reject a correct fp32 result
    assert acc["all_ok"] and acc["within_1ulp"] >= acc["elements"] - 4


def test_weight_acceptance_rejects_a_missing_chunk():
    th = synth.make_theta(("pre", 200, 136, 130), 200, 136, 130)
    W0, s, U, V = th.f64()
    assert oracle.weight_acceptance(_fp32_weight(W0, s, U, V), W0, s, U, V)["all_ok"]
    bad = _fp32_weight(W0, s, U, V, drop_chunk=(64, 128))
    acc = oracle.weight_acceptance(bad, W0, s, U, V)
    assert not acc["all_ok"] and acc["outside_bound"] > 1000


# ----------------------------------------------------------------------------------
# the element-wise error bound of the linear (the bar for outputs too small for the
# relative-L2 bar)
# ----------------------------------------------------------------------------------
def _fp32_linear(W0, s, U, V, x, t_bf16=True):
    """A plain fp32 evaluation: W0 x and t = V^T x summed one index at a time in fp32, t
    rounded to bf16 when t_bf16, the combine in fp32, one final rounding to bf16."""
    f = np.float32
    z = np.zeros((x.shape[0], W0.shape[0]), f)
    for i in range(W0.shape[1]):
        z = (z + np.outer(x[:, i], W0[:, i]).astype(f)).astype(f)
    t = np.zeros((x.shape[0], V.shape[1]), f)
    for i in range(V.shape[0]):
        t = (t + np.outer(x[:, i], V[i, :]).astype(f)).astype(f)
    if t_bf16:
        t = oracle.round_to_bf16(t.astype(np.float64)).astype(f)
    lr = np.zeros_like(z)
    for k in range(U.shape[1]):
        lr = (lr + np.outer(t[:, k], U[:, k]).astype(f)).astype(f)
    y32 = (s[None, :].astype(f) * z + lr).astype(f)
    return oracle.round_to_bf16(y32.astype(np.float64))


def _tiny_cases():
    for out, inp, r, M in ((8, 8, 0, 1), (8, 16, 1, 3), (24, 64, 16, 2), (64, 40, 3, 5), (16, 1152, 16, 4)):
        th = synth.make_theta(("bound", out, inp, r), out, inp, r)
        x = synth.bf16_bits_to_f64(synth.make_x(("bound", M, inp), M, inp))[:, :inp]
        yield th.f64(), x


def test_error_bound_admits_exact_rounding_and_fp32_evaluations():
    for (W0, s, U, V), x in _tiny_cases():
        y_ref = oracle.linear(W0, s, U, V, x)
        assert oracle.within_error_bound(oracle.round_to_bf16(y_ref), W0, s, U, V, x)
        assert oracle.within_error_bound(_fp32_linear(W0, s, U, V, x), W0, s, U, V, x)
        assert oracle.within_error_bound(_fp32_linear(W0, s, U, V, x, t_bf16=False), W0, s, U, V, x)


def test_error_bound_admits_fp32_near_cancellation():
    """s·W0 x and U t of opposite sign and almost equal size: the fp32 result is far from
    the exact one in relative terms, and the bound (absolute, from the terms' magnitudes)
    still admits it."""
    rng = np.random.default_rng(7)
    W0 = oracle.round_to_bf16(rng.normal(0, 0.02, (32, 64)))
    x = oracle.round_to_bf16(rng.normal(0, 1, (3, 64)))
    U = oracle.round_to_bf16(rng.normal(0, 0.5, (32, 1)))
    V = oracle.round_to_bf16(rng.normal(0, 0.02, (64, 1)))
    # choose s so that s·(W0 x) nearly cancels U t for token 0
    z, lr = x @ W0.T, (x @ V) @ U.T
    s = oracle.round_to_bf16(-lr[0] / z[0])
    y_ref = oracle.linear(W0, s, U, V, x)
    assert np.min(np.abs(y_ref[0]) / (np.abs(s * z[0]) + np.abs(lr[0]))) < 1e-2
    assert oracle.within_error_bound(_fp32_linear(W0, s, U, V, x), W0, s, U, V, x)


@pytest.mark.parametrize("mutant", [_m_drop_delta, _m_no_scale, _m_reversed_rank, _m_squared_t],
                         ids=lambda f: f.__name__)
def test_error_bound_rejects_mutants_on_tiny_outputs(mutant):
    """The same planted mistakes, made by a kernel, fail the bound on tiny outputs: on every
    tiny case where the mistake changes the result (a rank-r part; two ranks or more for the
    reversed rank order), at least one element leaves its bound. (Scaling the delta by s as
    well moves y by about (s - 1)·U t, below the output's own rounding at s ~ U(0.9, 1.1); the
    integer-valued GPU cases, compared bit for bit, catch that one.)"""
    caught = 0
    cases = 0
    for (W0, s, U, V), x in _tiny_cases():
        r = U.shape[1]
        if (r == 0 and mutant is not _m_no_scale) or (r < 2 and mutant is _m_reversed_rank):
            continue
        cases += 1
        got = oracle.round_to_bf16(mutant(W0, s, U, V, x))
        caught += not oracle.within_error_bound(got, W0, s, U, V, x)
    assert cases > 0 and caught == cases, (caught, cases)
