"""Pins of the fused-MLP oracle (CPU): properties the definitions fix, not a retyped formula."""
import numpy as np
import pytest

import oracle
from rank_weight_reconstruction_gb300 import synth


@pytest.mark.parametrize("act", [oracle.GELU_TANH, oracle.SILU])
def test_activation_odd_part_is_the_identity(act):
    """Both activations are v·w(v) with w(v) + w(−v) = 1 (tanh and the logistic function are
    odd about 1/2), so act(v) − act(−v) = v exactly in real arithmetic."""
    v = np.linspace(-8, 8, 1001)
    np.testing.assert_allclose(oracle.activation(v, act) - oracle.activation(-v, act), v, rtol=0, atol=1e-12)


@pytest.mark.parametrize("act", [oracle.GELU_TANH, oracle.SILU])
def test_activation_limits_and_zero(act):
    assert oracle.activation(np.array([0.0]), act)[0] == 0.0
    big = np.array([30.0, 60.0])
    np.testing.assert_allclose(oracle.activation(big, act), big, rtol=1e-12)
    np.testing.assert_allclose(oracle.activation(-big, act), 0.0, atol=1e-10)


def test_gelu_tanh_and_silu_differ():
    """The two readings are different functions (a swapped activation would be caught)."""
    v = np.array([1.0])
    assert abs(oracle.gelu_tanh(v)[0] - oracle.silu(v)[0]) > 0.05


def _identity_bundle(n):
    return np.eye(n), np.ones(n), np.zeros((n, 0)), np.zeros((n, 0))


@pytest.mark.parametrize("act", [oracle.GELU_TANH, oracle.SILU])
def test_mlp_with_identity_projections_is_the_gated_activation(act):
    """gate = up = down = I (s = 1, r = 0): y = RN(act(RN(x))·RN(x)) (the rounding points)."""
    n = 16
    x = synth.bf16_bits_to_f64(synth.make_x(("mlp-pin",), 3, n))[:, :n]
    I = _identity_bundle(n)
    y = oracle.mlp(I, I, I, x, act)
    xb = oracle.round_to_bf16(x)
    np.testing.assert_array_equal(y, oracle.round_to_bf16(oracle.activation(xb, act) * xb))


def test_mlp_down_is_applied_after_the_gate():
    """A permutation as the down projection permutes the gated activations (down acts on h, not
    on x), and a zero up projection gives y = 0."""
    n = 8
    x = synth.bf16_bits_to_f64(synth.make_x(("mlp-pin2",), 2, n))[:, :n]
    I = _identity_bundle(n)
    P = np.eye(n)[::-1]
    down = (P, np.ones(n), np.zeros((n, 0)), np.zeros((n, 0)))
    h = oracle.mlp(I, I, I, x)
    np.testing.assert_array_equal(oracle.mlp(I, I, down, x), h[:, ::-1])
    zero = (np.zeros((n, n)), np.ones(n), np.zeros((n, 0)), np.zeros((n, 0)))
    assert not np.any(oracle.mlp(I, zero, I, x))
