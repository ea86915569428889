"""Brute-force sweep of tiny shapes with every path forced.

out and in take every multiple of 8 from 8 to 64, r every value of {0, 1, 2, 3, 4, 8, 16},
M every value of 1..20 and 31, 32, 33, 129: the token counts cross the 8/16/32-token tiles
of the decode kernel, the decode limit, the 16-token N granularity of the mid-M GEMM and the
128-token tiles of the prefill GEMM; out < 16 leaves the decode kernel's 16-row slabs, the
mid-M GEMM's 128 accumulator lanes and the prefill GEMM's 64-column output chunks mostly empty,
and r below 8 or 16 leaves the padded rank columns of every path. Each path is forced with
aq_set_path (the decode kernel only up to its token limit). Integer-valued inputs, for which
every intermediate is exact, must give the oracle's result bit for bit. Random values are
held element by element to the oracle's error bound of a bf16 result computed with fp32
accumulation (oracle.linear_error_bound), and to the elementwise bar |Δ| <= 1e-2·max|y_ref|:
on outputs of a few dozen elements the relative-L2 bar of the larger cases is out of reach
even for the exactly rounded result, whose own rounding error can exceed 2e-3.
"""
import numpy as np
import pytest
import torch

import oracle
import rank_weight_reconstruction_gb300 as aq
from rank_weight_reconstruction_gb300 import synth

from helpers import dev, dev_theta, host_f64, x_f64

pytestmark = pytest.mark.gpu

SIZES = tuple(range(8, 65, 8))
RANKS = (0, 1, 2, 3, 4, 8, 16)
MS = tuple(range(1, 21)) + (31, 32, 33, 129)
PATHS = {"decode": aq.AQ_PATH_DECODE, "midm": aq.AQ_PATH_MIDM, "prefill": aq.AQ_PATH_PREFILL}


@pytest.fixture(autouse=True)
def _restore_path():
    yield
    aq.aq_set_path(aq.AQ_PATH_AUTO)


def _cases(path):
    for out in SIZES:
        for r in RANKS:
            for M in MS:
                if path == aq.AQ_PATH_DECODE and M > aq.aq_decode_max_m():
                    continue
                yield out, r, M


@pytest.mark.parametrize("inp", SIZES)
@pytest.mark.parametrize("pname", list(PATHS))
def test_tiny_random(pname, inp):
    path = PATHS[pname]
    aq.aq_set_path(path)
    xs = {M: synth.make_x(("tiny-sweep", inp, M), M, inp) for M in MS}
    failures = []
    for out, r, M in _cases(path):
        th = synth.make_theta(("tiny-sweep", out, inp, r), out, inp, r)
        xb = xs[M]
        y = aq.aq_linear(dev_theta(th), dev(xb)[:, :inp])
        torch.cuda.synchronize()
        assert aq.aq_last_path() == path
        got = host_f64(y)
        W0, s, U, V = th.f64()
        xf = x_f64(xb, inp)
        ref = oracle.linear(W0, s, U, V, xf)
        st = oracle.error_stats(got, ref)
        if not (oracle.within_error_bound(got, W0, s, U, V, xf) and st["max_abs_err"] <= 1e-2 * st["max_abs_ref"]):
            excess = float(np.max(np.abs(got - ref) / oracle.linear_error_bound(W0, s, U, V, xf)))
            failures.append(((out, inp, r, M), st, f"max |Δ| / bound = {excess:.3g}"))
    assert not failures, failures[:10]
    assert aq.aq_device_status() == aq.AQ_OK


@pytest.mark.parametrize("inp", SIZES)
@pytest.mark.parametrize("pname", list(PATHS))
def test_tiny_integer_bit_exact(pname, inp):
    path = PATHS[pname]
    aq.aq_set_path(path)
    xs = {M: synth.sparse_int_x(("tiny-int", inp, M), M, inp) for M in MS}
    failures = []
    for out, r, M in _cases(path):
        th = synth.sparse_int_theta(("tiny-int", out, inp, r), out, inp, r)
        xb = xs[M]
        W0, s, U, V = th.f64()
        xf = x_f64(xb, inp)
        ref = oracle.linear(W0, s, U, V, xf)
        # exactness preconditions: t (held in bf16 on the prefill path) and y are bf16 values
        assert np.array_equal(oracle.round_to_bf16(xf @ V), xf @ V)
        assert np.array_equal(oracle.round_to_bf16(ref), ref)
        y = aq.aq_linear(dev_theta(th), dev(xb)[:, :inp])
        torch.cuda.synchronize()
        got = host_f64(y)
        if not np.array_equal(got, ref):
            bad = np.argwhere(got != ref)
            failures.append(((out, inp, r, M), len(bad), bad[:4].tolist()))
    assert not failures, failures[:10]
    assert aq.aq_device_status() == aq.AQ_OK
