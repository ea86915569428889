"""Theta-bundle reconstruction linear for GB300 (sm_103a).

y = s * (W0 x) + U (V^T x) and W_eff = diag(s) W0 + U V^T as hand-written CUDA kernels
behind a C ABI (include/aq.h); this package holds the in-tree build, the ctypes
binding, the banded-stack bookkeeping and the seeded input generator.
"""
from .binding import (  # noqa: F401
    AQ_ACT_GELU_TANH,
    AQ_ACT_SILU,
    AQ_ERR_TIMEOUT,
    AQ_MAX_FAMILIES,
    AQ_MAX_RANK,
    AQ_OK,
    AQ_PATH_AUTO,
    AQ_PATH_DECODE,
    AQ_PATH_MIDM,
    AQ_PATH_PREFILL,
    AQ_SF_128X4,
    AQ_SF_LINEAR,
    AqError,
    Theta,
    aq_band_mean,
    aq_decode_max_m,
    aq_device_status,
    aq_last_launch_count,
    aq_last_path,
    aq_linear,
    aq_linear_multi,
    aq_linear_qkv,
    aq_linear_workspace_bytes,
    aq_mlp,
    aq_mlp_workspace_bytes,
    aq_ls_residual,
    aq_precompute,
    aq_precompute_nvfp4,
    aq_randomized_svd,
    aq_selftest_bounded_wait,
    aq_set_path,
    load,
    new_workspace,
    nvfp4_scale_bytes,
)
from .stack import StackMismatchError, ThetaStack, band_of  # noqa: F401
