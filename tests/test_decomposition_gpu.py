"""The decomposition on the GPU against the fp64 oracle ("How attnquant works", "How the
decomposition produces s, U, and V").

* band mean: bit for bit (both sum the band's bf16 values exactly in float64, divide once and
  round once to bf16);
* least-squares scale: the stored bf16 scale equal to the oracle's (within 1 bf16 ulp, where the
  two fp64 dot products in different orders could straddle a rounding boundary), the residual
  exactly weight - s * W0 with the stored s;
* randomized SVD: the factors are unique only up to the sign of each column pair, so the GPU's
  U V^T (bf16 factors) is compared with the product of the oracle's factors rounded to bf16 on
  the same test matrix Omega, and its truncation error with the pinned Eckart-Young energy.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import rank_weight_reconstruction_gb300 as aq
from rank_weight_reconstruction_gb300 import binding, synth

from helpers import bits, dev, host_f64


def _omega(key, n, k):
    return synth.normal_f64(synth.stream_seed("omega", *key), n * k).reshape(n, k)


def _rel_fro(a, b):
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


@pytest.mark.gpu
@pytest.mark.parametrize("L", [1, 4, 15])
@pytest.mark.parametrize("shape", [(300, 264), (1152, 1024)])
def test_band_mean_bit_exact(shape, L):
    out, inp = shape
    ws = [synth.make_w0(("band", out, inp, l), out, inp) for l in range(L)]
    W0 = aq.aq_band_mean([dev(w)[:, :inp] for w in ws])
    torch.cuda.synchronize()
    ref = oracle.round_to_bf16(oracle.band_mean([synth.bf16_bits_to_f64(w)[:, :inp] for w in ws]))
    np.testing.assert_array_equal(bits(W0), oracle.bf16_bits_of_value(ref))


def _layer(key, out, inp, W0_bits):
    """A synthetic layer weight around a band W0: a per-row scale, a low-rank part and noise."""
    W0 = synth.bf16_bits_to_f64(W0_bits)[:, :inp]
    a = synth.uniform_f64(synth.stream_seed("ls", *key, "a"), out, 0.9, 1.1)
    P = synth.normal_f64(synth.stream_seed("ls", *key, "P"), out * 8, 0.02).reshape(out, 8)
    Q = synth.normal_f64(synth.stream_seed("ls", *key, "Q"), inp * 8, 0.02).reshape(inp, 8)
    N = synth.normal_f64(synth.stream_seed("ls", *key, "N"), out * inp, 0.002).reshape(out, inp)
    return synth.bf16_bits_from_f64((a[:, None] * W0 + P @ Q.T + N).reshape(-1)).reshape(out, inp)


@pytest.mark.gpu
@pytest.mark.parametrize("shape", [(300, 264), (1152, 1024)])
def test_ls_residual(shape):
    out, inp = shape
    W0b = synth.make_w0(("lsr", out, inp), out, inp)
    W0b[7, :] = 0   # a W0 row of zeros keeps s = 1
    wb = _layer(("lsr", out, inp), out, inp, W0b)
    s, resid = aq.aq_ls_residual(dev(wb), dev(W0b)[:, :inp])
    torch.cuda.synchronize()
    w, W0 = synth.bf16_bits_to_f64(wb), synth.bf16_bits_to_f64(W0b)[:, :inp]
    s_ref, _ = oracle.ls_residual_stored(w, W0)
    s_gpu = host_f64(s)
    ulp = np.abs(oracle.bf16_ordinal(bits(s)) - oracle.bf16_ordinal(oracle.bf16_bits_of_value(s_ref)))
    assert ulp.max() <= 1 and np.count_nonzero(ulp) <= max(1, out // 1000), ulp.max()
    assert s_gpu[7] == 1.0
    # the residual of the stored scale, exact in float64 (bf16 x bf16 products and their
    # differences from bf16 values are representable)
    np.testing.assert_array_equal(resid.cpu().numpy(), w - s_gpu[:, None] * W0)


def _svd_case(out, inp, r, k, key, q=0):
    W0b = synth.make_w0((key, "W0"), out, inp)
    wb = _layer((key, "w"), out, inp, W0b)
    _, resid = aq.aq_ls_residual(dev(wb), dev(W0b)[:, :inp])
    A = resid.cpu().numpy()
    om = _omega((key, out, inp, k), inp, k)
    U, V = aq.aq_randomized_svd(resid, r, torch.from_numpy(om).cuda(), power_iters=q)
    torch.cuda.synchronize()
    return A, om, host_f64(U), host_f64(V)


@pytest.mark.gpu
@pytest.mark.parametrize("q", [0, 1])
@pytest.mark.parametrize("shape", [(1152, 1024), (1024, 1152), (600, 2000)])
def test_randomized_svd_matches_oracle(shape, q):
    out, inp = shape
    r, k = 16, 24
    A, om, Ug, Vg = _svd_case(out, inp, r, k, ("rsvd", q), q)
    Uo, Vo = oracle.randomized_svd(A, r, om, power_iters=q)
    ref = oracle.round_to_bf16(Uo) @ oracle.round_to_bf16(Vo).T
    # same draws, same method: the products of the bf16 factors agree far inside the factors'
    # own rounding (2^-8 relative per element)
    assert _rel_fro(Ug @ Vg.T, ref) <= 1e-4
    # the truncation error is the randomized method's, within its expected-error factor
    sv = np.linalg.svd(A, compute_uv=False)
    tail = float(np.sum(sv[r:] ** 2))
    err = float(np.linalg.norm(A - Ug @ Vg.T) ** 2)
    assert err <= (1 + r / (k - r - 1)) * tail * (1 + 1e-2)


@pytest.mark.gpu
def test_randomized_svd_exact_when_the_probe_spans_the_range():
    """k = min(m, n) <= 256 (the pages' fallback regime): the range finder captures the whole
    range and the factors are the exact rank-r truncation."""
    out, inp, r = 256, 1152, 16
    A, om, Ug, Vg = _svd_case(out, inp, r, 256, ("fallback",))
    Uo, Vo = oracle.truncated_svd(A, r)
    ref = oracle.round_to_bf16(Uo) @ oracle.round_to_bf16(Vo).T
    assert _rel_fro(Ug @ Vg.T, ref) <= 1e-4


@pytest.mark.gpu
def test_decomposition_feeds_the_reconstruction_linear():
    """A band of four layers decomposed on the GPU (band mean, stored scale, residual, rank-r
    factors) gives bundles whose reconstruction linear, run by aq_linear, matches the oracle's
    identity on the oracle's own decomposition (same Omega) within the parity tolerance."""
    out, inp, r, k, L = 1152, 1024, 16, 24, 4
    W0t = synth.make_w0(("feed", "W0"), out, inp)
    ws = [_layer(("feed", l), out, inp, W0t) for l in range(L)]
    W0 = aq.aq_band_mean([dev(w) for w in ws])
    W0_ref = oracle.round_to_bf16(oracle.band_mean([synth.bf16_bits_to_f64(w) for w in ws]))
    xb = synth.make_x(("feed", "x"), 8, inp)
    xf = synth.bf16_bits_to_f64(xb)[:, :inp]
    for l in (0, 3):
        s, resid = aq.aq_ls_residual(dev(ws[l]), W0)
        om = _omega(("feed", l), inp, k)
        U, V = aq.aq_randomized_svd(resid, r, torch.from_numpy(om).cuda())
        y = aq.aq_linear(aq.Theta(W0=W0, s=s.view(-1), U=U, V=V), dev(xb)[:, :inp])
        torch.cuda.synchronize()
        s_ref, resid_ref = oracle.ls_residual_stored(synth.bf16_bits_to_f64(ws[l]), W0_ref)
        Uo, Vo = oracle.randomized_svd(resid_ref, r, om)
        y_ref = oracle.linear(W0_ref, s_ref, oracle.round_to_bf16(Uo), oracle.round_to_bf16(Vo), xf)
        assert oracle.within_tolerance(host_f64(y), y_ref), oracle.error_stats(host_f64(y), y_ref)


def test_randomized_svd_argument_checks():
    """Refused before any device work (runs without a GPU)."""
    from rank_weight_reconstruction_gb300 import build_lib
    build_lib.build()
    lib = binding.load()
    assert lib.aq_randomized_svd_workspace_bytes(100, 100, 300, 8) == ctypes.c_size_t(-1).value
    assert lib.aq_randomized_svd_workspace_bytes(100, 100, 24, 30) == ctypes.c_size_t(-1).value
    st = lib.aq_randomized_svd(0x1000, 64, 64, 64, 8, 0x2000, 300, 300, 0, 0x3000, 8, 0x4000, 8, 0x5000, 1 << 20, None)
    assert st == binding.AQ_ERR_SHAPE
    assert lib.aq_band_mean(None, 1, 8, 8, 8, None, 8, None) == binding.AQ_ERR_INVALID_ARG
