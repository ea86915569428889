"""Parity of the CUDA path (called through the C ABI) with the fp64 oracle.

Bars (fixed before any kernel was written):
* reconstruction linear: max |y - y_ref| <= 1e-2 * max |y_ref| and relative L2 <= 2e-3
  over the whole output, at every size (large outputs are compared in row chunks);
* integer-valued inputs: every intermediate is exact in fp32 and bf16, so the result
  must equal the oracle bit for bit on every path;
* W_eff: every element within 1 bf16 ulp of RN_bf16(oracle); passthrough and r = 0 with
  power-of-two scales exactly.
"""
import numpy as np
import pytest
import torch

import oracle
import rank_weight_reconstruction_gb300 as aq
from rank_weight_reconstruction_gb300 import synth

from helpers import bits, close_over_rows, dev, dev_theta, host_f64, x_f64

pytestmark = pytest.mark.gpu

PATHS = [aq.AQ_PATH_DECODE, aq.AQ_PATH_MIDM, aq.AQ_PATH_PREFILL]
PATH_IDS = {aq.AQ_PATH_AUTO: "auto", aq.AQ_PATH_DECODE: "decode", aq.AQ_PATH_MIDM: "midm",
            aq.AQ_PATH_PREFILL: "prefill"}


@pytest.fixture(autouse=True)
def _restore_path():
    yield
    aq.aq_set_path(aq.AQ_PATH_AUTO)


def assert_close(y, y_ref, what=""):
    st = oracle.error_stats(y, y_ref)
    assert oracle.within_tolerance(y, y_ref), f"{what}: {st}"
    return st


def run_linear(th, xb, path=aq.AQ_PATH_AUTO, M=None):
    aq.aq_set_path(path)
    x = dev(xb)[:, : th.inp]
    y = aq.aq_linear(dev_theta(th), x)
    torch.cuda.synchronize()
    return y


def decode_refused(th, xb, path):
    """The decode kernel takes at most aq_decode_max_m() tokens; forcing it beyond that
    is refused before anything is launched."""
    if path != aq.AQ_PATH_DECODE or xb.shape[0] <= aq.aq_decode_max_m():
        return False
    with pytest.raises(aq.AqError) as e:
        run_linear(th, xb, path)
    assert e.value.status == aq.binding.AQ_ERR_UNSUPPORTED
    return True


def test_bounded_wait_reports_timeout():
    assert aq.aq_device_status() == aq.AQ_OK
    aq.aq_selftest_bounded_wait(2000)
    assert aq.aq_device_status() == aq.AQ_ERR_TIMEOUT
    assert aq.aq_device_status() == aq.AQ_OK     # reading clears it
    # the context is still usable
    th = synth.make_theta(("bw",), 64, 64, 4)
    xb = synth.make_x(("bw",), 2, 64)
    y = run_linear(th, xb)
    assert_close(host_f64(y), oracle.linear(*th.f64(), x_f64(xb, 64)))
    assert aq.aq_device_status() == aq.AQ_OK


def test_prefill_gemm_abort_path():
    """A real kernel's bounded wait running out: the prefill GEMM (unpaired, one token tile,
    r = 32 so that K is not split) waits for a t-flag count no tile reaches, with a 1 ms limit.
    The call reports AQ_ERR_TIMEOUT through aq_device_status, the kernel frees its tensor memory
    and returns the workspace's sync region to zero, and the same workspace then serves a normal
    call whose output matches the oracle."""
    from rank_weight_reconstruction_gb300 import binding
    assert aq.aq_device_status() == aq.AQ_OK
    th = synth.make_theta(("abort",), 6912, 1152, 32)
    xb = synth.make_x(("abort",), 64, 1152)
    T = dev_theta(th)
    x = dev(xb)[:, :1152]
    ws = aq.new_workspace(aq.aq_linear_workspace_bytes(T, 64), x.device)
    binding.aq_selftest_prefill_timeout(T, x, 1000, workspace=ws)
    assert aq.aq_device_status() == aq.AQ_ERR_TIMEOUT
    sync = ws[: aq.binding.AQ_WORKSPACE_SYNC_BYTES].cpu()
    assert not sync.any(), "the aborted launch left the sync region dirty"
    aq.aq_set_path(aq.AQ_PATH_PREFILL)
    try:
        y = aq.aq_linear(T, x, workspace=ws)
        torch.cuda.synchronize()
    finally:
        aq.aq_set_path(aq.AQ_PATH_AUTO)
    assert aq.aq_device_status() == aq.AQ_OK
    assert_close(host_f64(y), oracle.linear(*th.f64(), x_f64(xb, 1152)))


# ----------------------------------------------------------------------------------
# integer-valued cases: bit-exact on every path
# ----------------------------------------------------------------------------------
INT_SHAPES = [  # out, in, r, M
    (8, 16, 1, 1), (16, 64, 0, 3), (40, 64, 3, 5), (130, 200, 17, 33), (257, 72, 65, 17),
    (300, 136, 64, 130), (96, 1152, 16, 16), (1000, 96, 8, 1), (64, 264, 128, 200),
    (200, 64, 256, 65), (17, 8, 2, 300),
]


@pytest.mark.parametrize("path", PATHS, ids=lambda p: PATH_IDS[p])
@pytest.mark.parametrize("shape", INT_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_integer_bit_exact(shape, path):
    out, inp, r, M = shape
    th = synth.sparse_int_theta(("int", *shape), out, inp, r)
    xb = synth.sparse_int_x(("int", *shape), M, inp)
    W0, s, U, V = th.f64()
    xf = x_f64(xb, inp)
    y_ref = oracle.linear(W0, s, U, V, xf)
    t_ref = xf @ V
    # preconditions of exactness: t (held in bf16 between kernels) and y representable
    assert np.array_equal(oracle.round_to_bf16(t_ref), t_ref)
    assert np.array_equal(oracle.round_to_bf16(y_ref), y_ref)
    if decode_refused(th, xb, path):
        return
    y = run_linear(th, xb, path)
    assert aq.aq_last_path() == path
    np.testing.assert_array_equal(host_f64(y), y_ref)


# ----------------------------------------------------------------------------------
# tiny configuration: 256 x 256, r = 8, M = 1 (+ r = 0 and passthrough)
# ----------------------------------------------------------------------------------
@pytest.mark.parametrize("path", [aq.AQ_PATH_AUTO] + PATHS, ids=lambda p: PATH_IDS[p])
@pytest.mark.parametrize("variant", ["r8", "r0", "passthrough"])
def test_tiny_config(variant, path):
    if variant == "r8":
        th = synth.make_theta(("cfg1",), 256, 256, 8)
    elif variant == "r0":
        th = synth.make_theta(("cfg1", "r0"), 256, 256, 0)
    else:
        th = synth.passthrough_theta(("cfg1", "pt"), 256, 256, 8)
    xb = synth.make_x(("cfg1",), 1, 256)
    y = run_linear(th, xb, path)
    W0, s, U, V = th.f64()
    xf = x_f64(xb, 256)
    y_ref = oracle.linear(W0, s, U, V, xf)
    assert_close(host_f64(y), y_ref, f"{variant}/{PATH_IDS[path]}")
    if variant == "passthrough":
        # closed form: y = W0 x
        assert_close(host_f64(y), xf @ W0.T)
    if variant == "r0":
        assert_close(host_f64(y), s[None, :] * (xf @ W0.T))


# ----------------------------------------------------------------------------------
# ragged shapes and both paths, random values
# ----------------------------------------------------------------------------------
RAGGED = [(100, 72, 5, 1), (333, 200, 33, 7), (129, 1000, 64, 129), (1000, 264, 4, 63),
          (2000, 128, 130, 65), (48, 4096, 16, 300), (520, 512, 256, 1000)]


@pytest.mark.parametrize("path", PATHS, ids=lambda p: PATH_IDS[p])
@pytest.mark.parametrize("shape", RAGGED, ids=lambda s: "x".join(map(str, s)))
def test_ragged_random(shape, path):
    out, inp, r, M = shape
    th = synth.make_theta(("rag", *shape), out, inp, r)
    xb = synth.make_x(("rag", *shape), M, inp)
    if decode_refused(th, xb, path):
        return
    y = run_linear(th, xb, path)
    assert_close(host_f64(y), oracle.linear(*th.f64(), x_f64(xb, inp)), str(shape))


def test_padded_leading_dims_and_canaries():
    """x, y with padded leading dimensions inside larger buffers: everything outside
    the output window keeps its sentinel."""
    out, inp, r, M = 200, 136, 12, 9
    th = synth.make_theta(("pad",), out, inp, r)
    xb = synth.make_x(("pad",), M, inp)
    xbuf = torch.zeros(M, 160, dtype=torch.bfloat16, device="cuda")
    xbuf[:, :inp] = dev(xb)[:, :inp]
    for path in PATHS:
        aq.aq_set_path(path)
        ybuf = torch.full((M + 2, 224), -7.0, dtype=torch.bfloat16, device="cuda")
        y = ybuf[1:M + 1, 8:8 + out]
        aq.aq_linear(dev_theta(th), xbuf[:, :inp], y=y)
        torch.cuda.synchronize()
        assert_close(host_f64(y), oracle.linear(*th.f64(), x_f64(xb, inp)))
        yb = host_f64(ybuf)
        mask = np.ones_like(yb, dtype=bool)
        mask[1:M + 1, 8:8 + out] = False
        assert np.all(yb[mask] == -7.0)


def test_workspace_shared_across_paths_stays_clean():
    """One zero-filled workspace serves decode and prefill calls of different shapes in
    any order; every call leaves the sync region zero."""
    shapes = [((700, 264, 24), 7), ((300, 520, 40), 100), ((1000, 264, 8), 32), ((700, 264, 24), 1)]
    need = max(aq.aq_linear_workspace_bytes(dev_theta(synth.make_theta(("ws", *sh), *sh)), M)
               for sh, M in shapes)
    ws = aq.binding.new_workspace(need, "cuda")
    for sh, M in shapes * 2:
        th = synth.make_theta(("ws", *sh), *sh)
        xb = synth.make_x(("ws", M), M, sh[1])
        y = aq.aq_linear(dev_theta(th), dev(xb)[:, : sh[1]], workspace=ws)
        torch.cuda.synchronize()
        assert_close(host_f64(y), oracle.linear(*th.f64(), x_f64(xb, sh[1])), str((sh, M)))
        assert int(ws[: aq.binding.AQ_WORKSPACE_SYNC_BYTES].count_nonzero()) == 0
    assert aq.aq_device_status() == aq.AQ_OK


def test_m_zero_noop():
    th = synth.make_theta(("m0",), 64, 64, 4)
    x = torch.empty(0, 64, dtype=torch.bfloat16, device="cuda")
    y = aq.aq_linear(dev_theta(th), x)
    assert y.shape == (0, 64)


def test_batch_rows_match_single_token_calls():
    out, inp, r = 640, 384, 16
    th = synth.make_theta(("rows",), out, inp, r)
    xb = synth.make_x(("rows",), 12, inp)
    y_all = host_f64(run_linear(th, xb))
    for m in (0, 5, 11):
        y1 = host_f64(run_linear(th, xb[m:m + 1]))
        assert_close(y1[0], y_all[m])


# ----------------------------------------------------------------------------------
# Gemma-3-1B-shaped decode layer (r = 16, M in {1, 4, 16}), Q/K/V batched
# ----------------------------------------------------------------------------------
def _gemma_layer(layer, r, M, row_scale=None):
    fam = synth.GEMMA3_1B_FAMILIES
    thetas = {}
    for name, (out, inp) in fam.items():
        W0 = synth.make_w0(("gemma", name), out, inp)          # G = 1: shared by all layers
        thetas[name] = synth.make_theta(("gemma", name, layer), out, inp, r, W0=W0)
    xs = {inp: synth.make_x(("gemma-x", layer, inp, M), M, inp, row_scale) for inp in (1152, 1024, 6912)}
    return thetas, xs


@pytest.mark.parametrize("M", [1, 4, 16])
@pytest.mark.parametrize("layer", [0, 25])
def test_gemma_decode_layer(layer, M):
    thetas, xs = _gemma_layer(layer, 16, M)
    qkv = [thetas[n] for n in ("q_proj", "k_proj", "v_proj")]
    ys = aq.aq_linear_qkv([dev_theta(t) for t in qkv], dev(xs[1152])[:, :1152])
    torch.cuda.synchronize()
    for t, y in zip(qkv, ys):
        assert_close(host_f64(y), oracle.linear(*t.f64(), x_f64(xs[1152], 1152)), "qkv")
    for name in ("o_proj", "gate_proj", "up_proj", "down_proj"):
        t = thetas[name]
        y = run_linear(t, xs[t.inp])
        assert_close(host_f64(y), oracle.linear(*t.f64(), x_f64(xs[t.inp], t.inp)), name)


@pytest.mark.parametrize("M", [1, 16, 100, 512])
def test_qkv_stacked_layout(M):
    """y_q, y_k, y_v as column slices of one [M, 1536] buffer (the concatenated layout)."""
    thetas, xs = _gemma_layer(3, 16, M)
    qkv = [thetas[n] for n in ("q_proj", "k_proj", "v_proj")]
    Y = torch.zeros(M, 1536, dtype=torch.bfloat16, device="cuda")
    views = [Y[:, :1024], Y[:, 1024:1280], Y[:, 1280:]]
    aq.aq_linear_qkv([dev_theta(t) for t in qkv], dev(xs[1152])[:, :1152], ys=views)
    torch.cuda.synchronize()
    Yh = host_f64(Y)
    xf = x_f64(xs[1152], 1152)
    ref = np.concatenate([oracle.linear(*t.f64(), xf) for t in qkv], axis=1)
    assert_close(Yh, ref)


def test_qkv_mixed_ranks():
    out_in = [(512, 256), (128, 256), (136, 256)]
    ths = [synth.make_theta(("mix", j), o, i, r) for j, ((o, i), r) in enumerate(zip(out_in, (0, 8, 40)))]
    for M in (3, 70):
        xb = synth.make_x(("mix", M), M, 256)
        ys = aq.aq_linear_qkv([dev_theta(t) for t in ths], dev(xb)[:, :256])
        torch.cuda.synchronize()
        for t, y in zip(ths, ys):
            assert_close(host_f64(y), oracle.linear(*t.f64(), x_f64(xb, 256)))


@pytest.mark.parametrize("M", [3000, 4096])
def test_prefill_mixed_ranks_many_tiles(M):
    """Prefill with families of rank 0, 16 and 40 in one launch, at token counts where every
    CTA (pair) takes several tiles: tiles without a rank-r part (and the t = x V tiles) run
    between tiles with one on the same accumulator buffer. 3000 tokens leave an odd number
    of 128-token tiles."""
    out_in = [(2048, 1152), (640, 1152), (1024, 1152)]
    ths = [synth.make_theta(("mix-many", j), o, i, r) for j, ((o, i), r) in enumerate(zip(out_in, (16, 0, 40)))]
    xb = synth.make_x(("mix-many", M), M, 1152)
    ys = aq.aq_linear_qkv([dev_theta(t) for t in ths], dev(xb)[:, :1152])
    torch.cuda.synchronize()
    assert aq.aq_last_path() == aq.AQ_PATH_PREFILL
    xf = x_f64(xb, 1152)
    for t, y in zip(ths, ys):
        assert_close(host_f64(y), oracle.linear(*t.f64(), xf), f"out={t.out} r={t.r}")


@pytest.mark.parametrize("M", [1, 4, 16, 512])
def test_gate_up_batched(M):
    """gate and up of one layer over the same x in one aq_linear_multi call (n = 2), and
    n = 1 bit-identical to aq_linear."""
    thetas, xs = _gemma_layer(4, 16, M)
    pair = [thetas["gate_proj"], thetas["up_proj"]]
    x = dev(xs[1152])[:, :1152]
    ys = aq.aq_linear_multi([dev_theta(t) for t in pair], x)
    torch.cuda.synchronize()
    xf = x_f64(xs[1152], 1152)
    for t, y in zip(pair, ys):
        assert_close(host_f64(y), oracle.linear(*t.f64(), xf))
    one = aq.aq_linear_multi([dev_theta(pair[0])], x)[0]
    ref = aq.aq_linear(dev_theta(pair[0]), x)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(bits(one), bits(ref))


# ----------------------------------------------------------------------------------
# Gemma-3-1B shapes at prefill (r = 64, rows of x scaled by U(0.5, 2))
# ----------------------------------------------------------------------------------
@pytest.mark.parametrize("M", [512, 2048, 8192])
def test_gemma_prefill(M):
    thetas, xs = _gemma_layer(7, 64, M, row_scale=(0.5, 2.0))
    names = list(thetas) if M < 8192 else ["gate_proj", "down_proj", "o_proj"]
    for name in names:
        t = thetas[name]
        y = run_linear(t, xs[t.inp])
        assert_close(host_f64(y), oracle.linear(*t.f64(), x_f64(xs[t.inp], t.inp)), f"{name} M={M}")
    qkv = [thetas[n] for n in ("q_proj", "k_proj", "v_proj")]
    ys = aq.aq_linear_qkv([dev_theta(t) for t in qkv], dev(xs[1152])[:, :1152])
    torch.cuda.synchronize()
    for t, y in zip(qkv, ys):
        assert_close(host_f64(y), oracle.linear(*t.f64(), x_f64(xs[1152], 1152)), f"qkv M={M}")


# ----------------------------------------------------------------------------------
# rank / shape sweep on gate-like and down-like projections
# ----------------------------------------------------------------------------------
@pytest.mark.parametrize("M", [1, 8, 64, 512, 4096])
@pytest.mark.parametrize("r", [0, 4, 16, 64, 256])
@pytest.mark.parametrize("shape", [(6912, 1152), (1152, 6912)], ids=["gate", "down"])
def test_rank_sweep(shape, r, M):
    out, inp = shape
    th = synth.make_theta(("sweep", out, inp, r), out, inp, r)
    xb = synth.make_x(("sweep", out, inp, M), M, inp)
    y = host_f64(run_linear(th, xb))
    st, ok = close_over_rows(y, *th.f64(), x_f64(xb, inp))
    assert ok, st


# ----------------------------------------------------------------------------------
# 31B-class projection: out 21504, in 5376, r 128, M in {1, 32, 8192}
# ----------------------------------------------------------------------------------
@pytest.mark.parametrize("path", [aq.AQ_PATH_MIDM, aq.AQ_PATH_PREFILL], ids=lambda p: PATH_IDS[p])
@pytest.mark.parametrize("r", [0, 5, 64])
def test_split_k_dispatch(r, path):
    """A down-like projection at 64 tokens has few output tiles over a K of 6912 (9 tiles of
    128 rows on the mid-M GEMM, 18 tiles of 64 rows on the prefill GEMM): up to rank 16 its
    K is split across CTAs and a finalize kernel sums the slices (one more launch); at rank 64
    it stays one GEMM. All within tolerance of the oracle."""
    out, inp, M = 1152, 6912, 64
    th = synth.make_theta(("split", r), out, inp, r)
    xb = synth.make_x(("split", r), M, inp)
    y = run_linear(th, xb, path)
    assert aq.aq_last_path() == path
    gemm_launches = 1 if r == 0 else 2             # (V^T transpose,) GEMM
    split = r <= 16
    assert aq.aq_last_launch_count() == gemm_launches + (1 if split else 0)
    assert_close(host_f64(y), oracle.linear(*th.f64(), x_f64(xb, inp)), f"r={r}")
    assert aq.aq_device_status() == aq.AQ_OK


@pytest.mark.parametrize("M", [1, 32, 8192])
def test_31b_projection(M):
    out, inp = synth.CLASS31B_SHAPES["wide"]
    th = synth.make_theta(("31b", "wide", 0), out, inp, 128)
    xb = synth.make_x(("31b-x", M), M, inp)
    y = host_f64(run_linear(th, xb))
    # a W0 of 231 MB takes the tcgen05 GEMM from 16 tokens on
    assert aq.aq_last_path() == (aq.AQ_PATH_DECODE if M < 16 else aq.AQ_PATH_PREFILL)
    # the whole output, every token tile of the persistent multi-wave schedule included
    st, ok = close_over_rows(y, *th.f64(), x_f64(xb, inp), chunk=512)
    assert ok, st


@pytest.mark.parametrize("M", [16, 32])
def test_31b_projection_decode_forced(M):
    """The decode kernel on the 31B-class projection where the automatic choice is the GEMM."""
    out, inp = synth.CLASS31B_SHAPES["wide"]
    th = synth.make_theta(("31b", "wide", 0), out, inp, 128)
    xb = synth.make_x(("31b-x", M), M, inp)
    y = host_f64(run_linear(th, xb, path=aq.AQ_PATH_DECODE))
    assert aq.aq_last_path() == aq.AQ_PATH_DECODE
    assert_close(y, oracle.linear(*th.f64(), x_f64(xb, inp)))


def test_path_choice_by_size():
    """Up to 32 tokens the decode kernel, except from 16 tokens on for a W0 of 128 MB or more;
    the prefill GEMM above; the swapped-operand GEMM for 1024 to 4096 tokens on a deep K with
    at most 16 tiles of 128 rows."""
    sq = synth.CLASS31B_SHAPES["square"]
    th = synth.make_theta(("31b", "square", 0), sq[0], sq[1], 128)
    for M, path in ((1, aq.AQ_PATH_DECODE), (16, aq.AQ_PATH_DECODE), (32, aq.AQ_PATH_DECODE),
                    (33, aq.AQ_PATH_PREFILL), (1024, aq.AQ_PATH_PREFILL)):
        y = host_f64(run_linear(th, synth.make_x(("path", M), M, sq[1])))
        assert aq.aq_last_path() == path, M
        if M == 33:
            xb = synth.make_x(("path", M), M, sq[1])
            st, ok = close_over_rows(y, *th.f64(), x_f64(xb, sq[1]))
            assert ok, (M, st)
    # down-like: 9 tiles of 128 rows over K = 6912
    dn = synth.make_theta(("path", "down"), 1152, 6912, 16)
    for M, path in ((512, aq.AQ_PATH_PREFILL), (1024, aq.AQ_PATH_MIDM), (4096, aq.AQ_PATH_MIDM),
                    (4097, aq.AQ_PATH_PREFILL)):
        xb = synth.make_x(("path", "down", M), M, 6912)
        y = host_f64(run_linear(dn, xb))
        assert aq.aq_last_path() == path, M
        st, ok = close_over_rows(y, *dn.f64(), x_f64(xb, 6912))
        assert ok, (M, st)


# ----------------------------------------------------------------------------------
# precompute W_eff
# ----------------------------------------------------------------------------------
def _ulp_diff(got_bits, ref_value):
    ref_bits = oracle.bf16_bits_of_value(ref_value)
    return np.abs(oracle.bf16_ordinal(got_bits) - oracle.bf16_ordinal(ref_bits))


def assert_weight_ok(W, th, what=""):
    acc = oracle.weight_acceptance(bits(W), *th.f64())
    # what the acceptance actually used: elements beyond 1 ulp and the largest distance
    print(f"W_eff {what or (th.out, th.inp, th.r)}: {acc['elements'] - acc['within_1ulp']} of "
          f"{acc['elements']} elements beyond 1 ulp, max {acc['max_ulp']} ulp")
    assert acc["all_ok"], acc
    # the 1-ulp bar holds everywhere except on near-cancelling elements: measured on GB300,
    # at most 72 of 115.6 M elements of a 21504 x 5376 layer (0.6 per million), 3 of 8 M at
    # 6912 x 1152, r = 130, and 1 of 0.2 M at 520 x 384, r = 256
    assert acc["within_1ulp"] >= acc["elements"] - max(4, acc["elements"] // 1000000), acc
    return acc


@pytest.mark.parametrize("shape", [(256, 256, 8), (300, 200, 17), (129, 1000, 64), (1000, 136, 0),
                                   (520, 384, 256), (64, 72, 4), (1152, 6912, 16), (6912, 1152, 130)],
                         ids=lambda s: "x".join(map(str, s)))
def test_precompute_within_one_ulp(shape):
    out, inp, r = shape
    th = synth.make_theta(("pre", *shape), out, inp, r)
    W = aq.aq_precompute(dev_theta(th))
    torch.cuda.synchronize()
    assert_weight_ok(W, th)


def test_precompute_passthrough_and_pow2_scale_exact():
    th = synth.passthrough_theta(("pre-pt",), 300, 264, 16)
    W = aq.aq_precompute(dev_theta(th))
    torch.cuda.synchronize()
    np.testing.assert_array_equal(bits(W), th.W0[:, :264])
    th0 = synth.make_theta(("pre-r0",), 200, 136, 0)
    th0.s = synth.bf16_bits_from_f64(np.ldexp(1.0, np.arange(200) % 5 - 2))
    W = aq.aq_precompute(dev_theta(th0))
    torch.cuda.synchronize()
    np.testing.assert_array_equal(bits(W), oracle.bf16_bits_of_value(oracle.effective_weight_bf16(*th0.f64())))


def test_precompute_integer_exact():
    th = synth.sparse_int_theta(("pre-int",), 260, 200, 40)
    W = aq.aq_precompute(dev_theta(th))
    torch.cuda.synchronize()
    ref = oracle.effective_weight(*th.f64())
    assert np.all(np.abs(ref) <= 128)
    np.testing.assert_array_equal(host_f64(W), ref)


def test_precompute_into_padded_buffer_with_canaries():
    th = synth.make_theta(("pre-pad",), 130, 72, 8)
    buf = torch.full((132, 96), 3.0, dtype=torch.bfloat16, device="cuda")
    W = buf[1:131, 8:80]
    aq.aq_precompute(dev_theta(th), W_eff=W)
    torch.cuda.synchronize()
    assert_weight_ok(W, th)
    b = host_f64(buf)
    mask = np.ones_like(b, dtype=bool)
    mask[1:131, 8:80] = False
    assert np.all(b[mask] == 3.0)


def test_weight_then_dense_matches_identity():
    """y computed as W_eff x (torch matmul consuming the GPU-built W_eff) agrees with the
    oracle's factorised y: the load-time and in-graph forms are the same projection."""
    th = synth.make_theta(("weffx",), 1152, 1024, 16)
    W = aq.aq_precompute(dev_theta(th))
    xb = synth.make_x(("weffx",), 8, 1024)
    y = (dev(xb)[:, :1024].float() @ W.float().t())
    assert_close(y.double().cpu().numpy(), oracle.linear(*th.f64(), x_f64(xb, 1024)))


@pytest.mark.parametrize("M", [1, 200])
def test_precompute_then_linear_on_same_stream(M):
    """W_eff built by aq_precompute serves as W0 of the very next call on the same stream
    (no synchronisation, no kernel in between). The linear kernels fetch W0 before their
    dependency wait, so this only holds because precompute does not release its
    dependents early: a stale read would see the NaN fill."""
    out, inp, r = 2304, 1536, 32
    th = synth.make_theta(("pre-chain", M), out, inp, r)
    xb = synth.make_x(("pre-chain", M), M, inp)
    x = dev(xb)[:, :inp]
    W = torch.full((out, inp), float("nan"), dtype=torch.bfloat16, device="cuda")
    ones = torch.ones(out, dtype=torch.bfloat16, device="cuda")
    dense = aq.Theta(W0=W, s=ones)
    ws = aq.new_workspace(aq.aq_linear_workspace_bytes(dense, M), "cuda")
    y1 = torch.empty((M, out), dtype=torch.bfloat16, device="cuda")
    torch.cuda.synchronize()
    aq.aq_precompute(dev_theta(th), W_eff=W)
    aq.aq_linear(dense, x, y=y1, workspace=ws)
    torch.cuda.synchronize()
    y2 = aq.aq_linear(dense, x, workspace=ws)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(bits(y1), bits(y2))
    assert_weight_ok(W, th)
    # the second call is a plain dense product over the W that was built
    Wf = host_f64(W)
    ref = oracle.linear(Wf, np.ones(out), np.zeros((out, 0)), np.zeros((inp, 0)), x_f64(xb, inp))
    assert_close(host_f64(y1), ref)


@pytest.mark.parametrize("shape", ["square", "wide"])
def test_31b_band_precompute(shape):
    """60-layer stack with G = 4 bands: the first and last layer (bands 0 and 3) checked
    in full, element by element."""
    out, inp = synth.CLASS31B_SHAPES[shape]
    W0b = {b: synth.make_w0(("31b-band", shape, b), out, inp) for b in (0, 3)}
    for layer in (0, 59):
        band = oracle.band_of_layer(layer, 60, 4)
        th = synth.make_theta(("31b-layer", shape, layer), out, inp, 128, W0=W0b[band])
        W = aq.aq_precompute(dev_theta(th))
        torch.cuda.synchronize()
        assert_weight_ok(W, th, f"31B {shape} layer {layer}")
        del W
    assert aq.aq_device_status() == aq.AQ_OK
