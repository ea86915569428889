"""The chunked full-output comparison used by the large GPU parity cases gives exactly the
statistics and verdict of the oracle's whole-tensor acceptance (CPU only)."""
import numpy as np

import oracle
from rank_weight_reconstruction_gb300 import synth

from helpers import close_over_rows, x_f64


def test_chunked_stats_equal_whole_tensor_stats():
    th = synth.make_theta(("chunk",), 96, 72, 5)
    xb = synth.make_x(("chunk",), 37, 72)
    W0, s, U, V = th.f64()
    xf = x_f64(xb, 72)
    ref = oracle.linear(W0, s, U, V, xf)
    # a perturbed "result": bf16 rounding plus a planted error in one element of the last chunk
    y = oracle.round_to_bf16(ref)
    y[36, 5] += 0.5 * np.max(np.abs(ref)) * 1e-2
    st, ok = close_over_rows(y, W0, s, U, V, xf, chunk=8)
    whole = oracle.error_stats(y, ref)
    for k in whole:
        assert abs(st[k] - whole[k]) <= 1e-12 * max(1.0, abs(whole[k])), (k, st, whole)
    assert ok == oracle.within_tolerance(y, ref)
    # an error above the elementwise bar in a middle chunk fails
    y[17, 3] += 2e-2 * np.max(np.abs(ref))
    st, ok = close_over_rows(y, W0, s, U, V, xf, chunk=8)
    assert not ok and not oracle.within_tolerance(y, ref)
