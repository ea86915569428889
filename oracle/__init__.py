"""Independent fp64 oracle of the theta-bundle reconstruction linear.

TEST INFRASTRUCTURE ONLY: imported by the tests, the smoke check and the benchmark's
CPU-baseline leg, never by the library.
"""
from .reconstruction import (  # noqa: F401
    band_of_layer,
    bf16_bits_of_value,
    bf16_ordinal,
    effective_weight,
    effective_weight_bf16,
    error_stats,
    linear,
    linear_error_bound,
    linear_qkv,
    ls_residual,
    ls_scale,
    round_to_bf16,
    weight_acceptance,
    within_error_bound,
    within_tolerance,
)
from .decomposition import (  # noqa: F401
    band_mean,
    decompose,
    decompose_stack,
    ls_residual_stored,
    randomized_svd,
    truncated_svd,
)
from .mlp import GELU_TANH, SILU, activation, gelu_tanh, mlp, silu  # noqa: F401
from . import nvfp4  # noqa: F401
