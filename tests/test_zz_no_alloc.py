"""aq_linear_noalloc: the reconstruction linear for callers that may not allocate.

Some callers cannot hand the library a workspace -- a plugin inside a runtime that owns
all device memory and passes plugins only their inputs and outputs, or a serving loop
that forbids allocation once it runs. aq_linear_noalloc serves them from a scratch array
built into the library. These tests call it through the C ABI, several times in a row over
different shapes, paths and ranks so that stale scratch from one call would show in the
next, and check every result against the fp64 oracle and against aq_linear (which gets a
caller-allocated workspace). This file is named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from rank_weight_reconstruction_gb300 import binding, build_lib, synth

from helpers import dev, dev_theta, host_f64, x_f64


@pytest.fixture(scope="module")
def lib():
    build_lib.build()
    return binding.load()


def _noalloc(lib, theta, x, y):
    th = theta.c()
    st = lib.aq_linear_noalloc(ctypes.byref(th), x.data_ptr(), x.size(0), binding._ld(x), y.data_ptr(),
                               binding._ld(y), torch.cuda.current_stream().cuda_stream)
    return st


def _sync_part_of_scratch(lib):
    """The first AQ_WORKSPACE_SYNC_BYTES of the built-in scratch array, copied out."""
    out = torch.full((binding.AQ_WORKSPACE_SYNC_BYTES,), 0x5A, dtype=torch.uint8, device="cuda")
    st = lib.aq_noalloc_scratch_read(out.data_ptr(), 0, out.numel(), torch.cuda.current_stream().cuda_stream)
    assert st == binding.AQ_OK, binding.aq_last_error()
    return out


# (out, in, r), M. The decode calls at in = 1152, r = 32 have a V of 72 KB, too large for
# every W0-streaming CTA to stage, so a few CTAs compute t = V^T x and publish it through
# the array's sync part (its counters and fp32 accumulator); the call at 200 tokens takes
# the tcgen05 GEMM, whose scratch holds t and a transposed V past the sync part.
CASES = [((300, 264, 24), 5), ((2048, 1152, 32), 1), ((1000, 520, 40), 200), ((2048, 1152, 32), 16),
         ((2048, 1152, 32), 1)]


@pytest.mark.gpu
def test_noalloc_matches_oracle_and_aq_linear_on_calls_in_a_row(lib):
    binding.aq_set_path(binding.AQ_PATH_AUTO)
    assert int(_sync_part_of_scratch(lib).count_nonzero()) == 0
    for (out, inp, r), M in CASES:
        th = synth.make_theta(("noalloc", out, inp, r), out, inp, r)
        xb = synth.make_x(("noalloc", M, inp), M, inp)
        theta = dev_theta(th)
        x = dev(xb)[:, :inp]
        y = torch.full((M, (out + 7) // 8 * 8), float("nan"), dtype=torch.bfloat16, device="cuda")[:, :out]
        assert _noalloc(lib, theta, x, y) == binding.AQ_OK, binding.aq_last_error()
        torch.cuda.synchronize()
        got = host_f64(y)
        assert np.all(np.isfinite(got))
        ref = oracle.linear(*th.f64(), x_f64(xb, inp))
        assert oracle.within_tolerance(got, ref), ((out, inp, r, M), oracle.error_stats(got, ref))
        y_ws = host_f64(binding.aq_linear(theta, x))          # caller-provided workspace
        assert oracle.within_tolerance(got, y_ws), ((out, inp, r, M), oracle.error_stats(got, y_ws))
        # every completed call leaves the shared array's sync part zero for the next one
        assert int(_sync_part_of_scratch(lib).count_nonzero()) == 0, (out, inp, r, M)
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
    # the read-out hook refuses ranges outside the array without touching the GPU
    buf = ctypes.create_string_buffer(16)
    assert lib.aq_noalloc_scratch_read(buf, binding.AQ_NOALLOC_WORKSPACE_BYTES - 8, 16, None) == \
        binding.AQ_ERR_INVALID_ARG
    assert lib.aq_noalloc_scratch_read(None, 0, 16, None) == binding.AQ_ERR_INVALID_ARG
