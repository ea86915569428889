"""aq_linear_noalloc: the reconstruction linear for callers that may not allocate.

Some callers cannot hand the library a workspace -- a plugin inside a runtime that owns
all device memory and passes plugins only their inputs and outputs, or a serving loop
that forbids allocation once it runs. aq_linear_noalloc serves them from a scratch array
built into the library. These tests call it through the C ABI and compare it with
aq_linear (which gets a caller-allocated workspace) on two calls in a row, the second
with different shapes so that stale scratch from the first would show. This file is
named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from rank_weight_reconstruction_gb300 import binding, build_lib, synth

from helpers import dev, dev_theta, host_f64


@pytest.fixture(scope="module")
def lib():
    build_lib.build()
    return binding.load()


def _noalloc(lib, theta, x, y):
    th = theta.c()
    st = lib.aq_linear_noalloc(ctypes.byref(th), x.data_ptr(), x.size(0), binding._ld(x), y.data_ptr(),
                               binding._ld(y), torch.cuda.current_stream().cuda_stream)
    return st


@pytest.mark.gpu
def test_noalloc_matches_aq_linear_on_two_calls_in_a_row(lib):
    binding.aq_set_path(binding.AQ_PATH_AUTO)
    # first a decode-sized call (scratch holds t), then a prefill-sized one (scratch holds
    # t and a transposed V) over different shapes and values
    cases = [((300, 264, 24), 5), ((1000, 520, 40), 200)]
    for (out, inp, r), M in cases:
        th = synth.make_theta(("noalloc", out, inp, r), out, inp, r)
        xb = synth.make_x(("noalloc", M, inp), M, inp)
        theta = dev_theta(th)
        x = dev(xb)[:, :inp]
        y_ref = binding.aq_linear(theta, x)                 # caller-provided workspace
        y = torch.full((M, (out + 7) // 8 * 8), float("nan"), dtype=torch.bfloat16, device="cuda")[:, :out]
        assert _noalloc(lib, theta, x, y) == binding.AQ_OK, binding.aq_last_error()
        torch.cuda.synchronize()
        got, ref = host_f64(y), host_f64(y_ref)
        assert np.all(np.isfinite(got))
        assert oracle.within_tolerance(got, ref), oracle.error_stats(got, ref)
    assert binding.aq_device_status() == binding.AQ_OK


def test_noalloc_rejects_calls_beyond_its_scratch(lib):
    """M = 16384 tokens at r = 256 needs more than the built-in scratch: refused with a
    message before anything reaches the GPU (runs without a GPU)."""
    out, inp, r, M = 1024, 5376, 256, 16384
    th = binding.c_theta(W0=0x100000, ld_w0=inp, s=0x200000, U=0x300000, ld_u=r, V=0x400000, ld_v=r,
                         out=out, in_=inp, r=r)
    need = lib.aq_linear_workspace_bytes(ctypes.byref(th), 1, M)
    assert need > binding.AQ_NOALLOC_WORKSPACE_BYTES
    st = lib.aq_linear_noalloc(ctypes.byref(th), 0x1000000, M, inp, 0x9000000, out, None)
    assert st == binding.AQ_ERR_WORKSPACE
    assert "scratch" in binding.aq_last_error()
    assert lib.aq_linear_noalloc(None, 0, 1, 8, 0, 8, None) == binding.AQ_ERR_INVALID_ARG
