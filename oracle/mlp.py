"""fp64 CPU oracle of the fused MLP built from three theta bundles.

TEST INFRASTRUCTURE ONLY, like the rest of this package: the library never imports it.

Source: "Execution paths", "The custom op": one dispatch runs a layer's gate, up, activation and
down projections, each a reconstruction linear y = s·(W0 x) + U(Vᵀ x) ("How attnquant works",
"The reconstruction identity").

Readings (the pages are silent on both; each also listed in the design notes):
* The activation is not named. The benchmark's shapes are Gemma-3-1B's, whose MLP applies the
  tanh approximation of GELU to the gate projection and multiplies by the up projection:
  gelu_tanh(v) = v/2·(1 + tanh(√(2/π)·(v + 0.044715·v³))). SiLU, v/(1 + e^(−v)), is the other
  common choice and is offered too.
* Rounding points: the gate and up outputs are bf16 tensors (they are reconstruction linears),
  and the gated product h = act(g)·u enters the down projection as a bf16 operand.
"""
from __future__ import annotations

import numpy as np

from .reconstruction import linear, round_to_bf16

GELU_TANH = 0
SILU = 1


def gelu_tanh(v) -> np.ndarray:
    v = np.asarray(v, dtype=np.float64)
    return 0.5 * v * (1.0 + np.tanh(np.sqrt(2.0 / np.pi) * (v + 0.044715 * v ** 3)))


def silu(v) -> np.ndarray:
    v = np.asarray(v, dtype=np.float64)
    return v / (1.0 + np.exp(-v))


def activation(v, act: int) -> np.ndarray:
    if act == GELU_TANH:
        return gelu_tanh(v)
    if act == SILU:
        return silu(v)
    raise ValueError(f"unknown activation {act}")


def mlp(gate, up, down, x, act: int = GELU_TANH) -> np.ndarray:
    """y = down( RN_bf16( act(g) · u ) ), g = RN_bf16(gate(x)), u = RN_bf16(up(x)); each of
    gate, up, down a (W0, s, U, V) tuple of float64 arrays holding bf16 values."""
    g = round_to_bf16(linear(*gate, x))
    u = round_to_bf16(linear(*up, x))
    h = round_to_bf16(activation(g, act) * u)
    return linear(*down, h)
