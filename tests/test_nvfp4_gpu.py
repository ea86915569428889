"""The fused NVFP4 precompute (aq_precompute_nvfp4) against the oracle ("Execution paths",
"Precompute-outside: the production path"; "Internals and extension", "Nvfp4Spec").

* exact inputs (small integers: every fp32 evaluation of W_eff is exact): codes, scales and
  the global scale bit for bit, both scale layouts, given and computed global scale;
* the hand-worked row of tests/golden/nvfp4_row.txt as a weight: the GPU's bytes are the
  hand-derived ones;
* the synthetic Gemma-3-1B shapes (fp32 evaluation not exact): bit for bit wherever the
  decision is unique under the fp32 evaluation bound, and only near-boundary flips elsewhere;
* the 31B-class wide projection at full size: the global scale and sampled rows.
"""
import ctypes
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import nvfp4
import rank_weight_reconstruction_gb300 as aq
from rank_weight_reconstruction_gb300 import binding, synth

from helpers import dev_theta

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
LAYOUTS = [aq.AQ_SF_LINEAR, aq.AQ_SF_128X4]


def _sf_linear(sf, layout, out, inp):
    """The GPU's scales as an [out, in/16] array whatever their layout, the 128x4 padding
    checked to be zero on the way."""
    sf = sf.cpu().numpy().reshape(-1)
    if layout == aq.AQ_SF_LINEAR:
        return sf.reshape(out, inp // 16)
    KB = inp // 16
    KBP, NP = -(-KB // 4) * 4, -(-out // 128) * 128
    lin = np.zeros((NP, KBP), dtype=np.uint8)
    r = np.arange(NP)[:, None]
    c = np.arange(KBP)[None, :]
    idx = ((r // 128) * (KBP // 4) + c // 4) * 512 + 16 * (r % 32) + 4 * ((r % 128) // 32) + c % 4
    lin[:, :] = sf[idx]
    assert not lin[out:, :].any() and not lin[:, KB:].any(), "128x4 padding must be zero"
    return lin[:out, :KB]


def _run(th, layout, g=None):
    gs = None if g is None else torch.tensor([g], dtype=torch.float32, device="cuda")
    q, sf, gout = aq.aq_precompute_nvfp4(dev_theta(th), sf_layout=layout, global_scale=gs)
    torch.cuda.synchronize()
    assert aq.aq_last_launch_count() == (1 if g is not None else 2)
    assert aq.aq_device_status() == aq.AQ_OK
    codes = nvfp4.unpack(q.cpu().numpy())[:, : th.inp]
    return codes, _sf_linear(sf, layout, th.out, th.inp), np.float32(gout.item())


@pytest.mark.gpu
@pytest.mark.parametrize("layout", LAYOUTS, ids=["linear", "128x4"])
@pytest.mark.parametrize("given", [False, True], ids=["from_amax", "given"])
@pytest.mark.parametrize("shape", [(300, 272, 8), (128, 64, 0), (1152, 1024, 16), (129, 4096, 3)])
def test_exact_inputs_bit_exact(shape, given, layout):
    out, inp, r = shape
    th = synth.small_int_theta(("nvfp4", out, inp, r), out, inp, r)
    x = nvfp4.weff_f32(*th.f64())
    g = nvfp4.global_scale(np.max(np.abs(x))) if not given else np.float32(0.0117)
    codes, sf, g_gpu = _run(th, layout, None if not given else float(g))
    assert g_gpu == g
    codes_ref, sf_ref = nvfp4.quantize(x, g)
    np.testing.assert_array_equal(sf, sf_ref)
    np.testing.assert_array_equal(codes, codes_ref)


@pytest.mark.gpu
@pytest.mark.parametrize("given", [False, True], ids=["from_amax", "given"])
def test_exact_inputs_full_size_repeated(given):
    """The 31B-class square projection (5376 x 5376, r = 128) on exact integer inputs, every
    code and scale compared bit for bit, three launches in a row (the tile buffers are
    recycled hundreds of times per CTA: a buffer freed too early would show here)."""
    out, inp, r = 5376, 5376, 128
    th = synth.small_int_theta(("nvfp4-full", out, inp, r), out, inp, r)
    x = nvfp4.weff_f32(*th.f64())
    g = nvfp4.global_scale(np.max(np.abs(x))) if not given else np.float32(0.0117)
    codes_ref, sf_ref = nvfp4.quantize(x, g)
    del x
    for _ in range(3):
        codes, sf, g_gpu = _run(th, aq.AQ_SF_128X4, float(g) if given else None)
        assert g_gpu == g
        np.testing.assert_array_equal(sf, sf_ref)
        np.testing.assert_array_equal(codes, codes_ref)


@pytest.mark.gpu
@pytest.mark.parametrize("layout", LAYOUTS, ids=["linear", "128x4"])
def test_hand_worked_row_on_the_gpu(layout):
    """The golden row (ties, a subnormal scale, saturation, negative zero) as row 1 of a
    passthrough weight (s = 1, r = 0): the GPU writes the hand-derived bytes."""
    from test_nvfp4_pins import _golden_row
    x, g, packed, scales = _golden_row()
    out, inp = 3, x.shape[1]
    W = np.zeros((out, inp))
    W[1] = x[0]
    th = synth.Theta(W0=synth.bf16_bits_from_f64(W.reshape(-1)).reshape(out, inp),
                     s=synth.bf16_bits_from_f64(np.ones(out)), U=None, V=None, out=out, inp=inp, r=0)
    assert np.array_equal(synth.bf16_bits_to_f64(th.W0)[1], x[0].astype(np.float64))
    q, sf, _ = aq.aq_precompute_nvfp4(dev_theta(th), sf_layout=layout,
                                      global_scale=torch.tensor([g], dtype=torch.float32, device="cuda"))
    torch.cuda.synchronize()
    np.testing.assert_array_equal(q.cpu().numpy()[1], packed)
    assert not q.cpu().numpy()[[0, 2]].any()
    np.testing.assert_array_equal(_sf_linear(sf, layout, out, inp)[1], scales)


def _compare_flagged(codes, sf, x, bound, g, g_rel=0.0):
    """Bit-exact where the decision is unique; elsewhere a flip to a neighbouring code (or a
    neighbouring scale) only. Returns the number of flagged values that differ."""
    ele, blk = nvfp4.ambiguous(x, bound, g, g_rel)
    codes_ref, sf_ref = nvfp4.quantize(x.astype(np.float32), g)
    bad_blk = sf != sf_ref
    assert not np.any(bad_blk & ~blk), f"{np.count_nonzero(bad_blk & ~blk)} unflagged scale mismatches"
    sfd = np.abs(nvfp4.e4m3_value(sf[bad_blk]) - nvfp4.e4m3_value(sf_ref[bad_blk]))
    assert np.all(sfd <= np.abs(nvfp4.e4m3_value(sf_ref[bad_blk])) * 2.0 ** -3 + 2.0 ** -9)
    N, K = codes.shape
    blk_e = np.repeat(blk | bad_blk, 16, axis=1)
    diff = (codes != codes_ref) & ~blk_e
    assert not np.any(diff & ~ele), f"{np.count_nonzero(diff & ~ele)} unflagged code mismatches"
    # a flipped code is the neighbour on the number line (or the other zero)
    v, vr = nvfp4.e2m1_value(codes[diff]), nvfp4.e2m1_value(codes_ref[diff])
    mags = np.abs(np.stack([v, vr]))
    step = np.where(mags.max(axis=0) <= 2, 0.5, np.where(mags.max(axis=0) <= 4, 1.0, 2.0))
    assert np.all(np.abs(v - vr) <= step)
    return int(np.count_nonzero(diff)), int(np.count_nonzero(bad_blk))


@pytest.mark.gpu
@pytest.mark.parametrize("given", [False, True], ids=["from_amax", "given"])
@pytest.mark.parametrize("shape", [(1152, 1024), (6912, 1152), (1024, 1152), (256, 6912)])
def test_synthetic_gemma_shapes(shape, given):
    out, inp = shape
    r = 16
    th = synth.make_theta(("nvfp4s", out, inp), out, inp, r)
    W0, s, U, V = th.f64()
    x = oracle.effective_weight(W0, s, U, V)
    bound = nvfp4.weff_error_bound(W0, s, U, V)
    amax = np.max(np.abs(x))
    g_ref = nvfp4.global_scale(amax)
    codes, sf, g_gpu = _run(th, aq.AQ_SF_128X4, float(g_ref) if given else None)
    g_rel = 0.0
    if not given:
        # the GPU's amax is an fp32 evaluation of some |W_eff| near the largest: within the
        # largest evaluation bound of it
        rel = (float(bound.max()) + amax * 2.0 ** -24) / amax + 2.0 ** -23
        assert abs(float(g_gpu) - float(g_ref)) <= float(g_ref) * rel * 1.01
        g_rel = rel
    n_codes, n_scales = _compare_flagged(codes, sf, x, bound, g_ref, g_rel)
    assert n_codes <= max(4, out * inp // 200000) and n_scales <= 4, (n_codes, n_scales)


@pytest.mark.gpu
def test_wide_projection_full_size_sampled_rows():
    """The 31B-class wide projection (21504 x 5376, r = 128) at full size, in the launch the
    benchmark times (computed global scale, 128x4 scales): the global scale against the
    oracle's max|W_eff| over the whole weight, then 48 sampled rows (the first and last row
    tiles among them) decision by decision."""
    out, inp, r = 21504, 5376, 128
    th = synth.make_theta(("nvfp4w", out, inp), out, inp, r)
    W0, s, U, V = th.f64()
    q, sf, g = aq.aq_precompute_nvfp4(dev_theta(th), sf_layout=aq.AQ_SF_128X4)
    torch.cuda.synchronize()
    assert aq.aq_device_status() == aq.AQ_OK
    amax, amax_bound = 0.0, 0.0
    for o0 in range(0, out, 2048):
        sl = slice(o0, o0 + 2048)
        amax = max(amax, float(np.max(np.abs(oracle.effective_weight(W0[sl], s[sl], U[sl], V)))))
        amax_bound = max(amax_bound, float(nvfp4.weff_error_bound(W0[sl], s[sl], U[sl], V).max()))
    g_ref = nvfp4.global_scale(amax)
    rel = (amax_bound + amax * 2.0 ** -24) / amax + 2.0 ** -23
    assert abs(g.item() - float(g_ref)) <= float(g_ref) * rel * 1.01
    rows = np.unique(np.concatenate([np.arange(0, 8), np.arange(out - 8, out),
                                     np.random.default_rng(0).integers(0, out, 32)]))
    x = oracle.effective_weight(W0[rows], s[rows], U[rows], V)
    bound = nvfp4.weff_error_bound(W0[rows], s[rows], U[rows], V)
    codes = nvfp4.unpack(q[torch.from_numpy(rows).cuda()].cpu().numpy())
    sf_all = _sf_linear(sf, aq.AQ_SF_128X4, out, inp)
    n_codes, n_scales = _compare_flagged(codes, sf_all[rows], x, bound, g_ref, rel)
    assert n_codes <= 8 and n_scales <= 2, (n_codes, n_scales)


def test_argument_checks():
    """Refused before any device work (runs without a GPU)."""
    from rank_weight_reconstruction_gb300 import build_lib
    build_lib.build()
    lib = binding.load()
    assert lib.aq_precompute_nvfp4_workspace_bytes() >= 152 * 4
    W0, s, U, V = 0x100000, 0x200000, 0x300000, 0x400000

    def call(inp=1024, ldq=512, q=0x1000000, sf=0x2000000, layout=0, gs=0x3000000, mode=0,
             ws=0x4000000, wsb=1 << 16):
        th = binding.c_theta(W0=W0, s=s, U=U, V=V, ld_w0=inp, ld_u=16, ld_v=16, out=256, in_=inp, r=16)
        return lib.aq_precompute_nvfp4(ctypes.byref(th), q, ldq, sf, layout, gs, mode, ws, wsb, None)

    assert call(inp=1000, ldq=500) == binding.AQ_ERR_SHAPE
    assert call(ldq=500) == binding.AQ_ERR_SHAPE
    assert call(layout=2) == binding.AQ_ERR_INVALID_ARG
    assert call(mode=5) == binding.AQ_ERR_INVALID_ARG
    assert call(ldq=516) == binding.AQ_ERR_ALIGNMENT
    assert call(sf=0x2000008) == binding.AQ_ERR_ALIGNMENT
    assert call(ws=None) == binding.AQ_ERR_INVALID_ARG
    assert call(wsb=16) == binding.AQ_ERR_WORKSPACE
    assert call(q=W0) == binding.AQ_ERR_OVERLAP
    assert call(sf=0x1000000 + 1024) == binding.AQ_ERR_OVERLAP
