"""Pins of the NVFP4 quantization oracle against what the formats and the pages fix
("Internals and extension", "Nvfp4Spec"; "Execution paths", "Precompute-outside: the
production path"): the E2M1 and E4M3 tables, a library FP8 cast, brute-force nearest
rounding, exact round trips, error bounds, a hand-worked row and the layouts' shapes."""
import os

import numpy as np
import pytest
import torch

from oracle import nvfp4

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_e2m1_table_is_the_format():
    # E2M1: 1 sign, 2 exponent bits (bias 1), 1 mantissa bit; exponent 0 is subnormal
    want = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    np.testing.assert_array_equal(nvfp4.e2m1_value(np.arange(8)), want)
    np.testing.assert_array_equal(nvfp4.e2m1_value(np.arange(8, 16)), [-v for v in want])
    assert np.signbit(nvfp4.e2m1_value(8))
    # every code survives value -> code
    for c in range(16):
        assert nvfp4.e2m1_round(np.float32(nvfp4.e2m1_value(c))) == c


def _e2m1_brute(q):
    """Nearest of the 15 distinct E2M1 values by exhaustive comparison, ties to the code
    with a zero mantissa bit, magnitudes above 6 clamped, the sign taken from q."""
    out = []
    for v in np.asarray(q, dtype=np.float64):
        a = min(abs(v), 6.0)
        best = None
        for c in range(8):
            m = float(nvfp4.e2m1_value(c))
            dist = abs(a - m)
            if best is None or dist < best[0] or (dist == best[0] and c % 2 == 0):
                best = (dist, c)
        out.append(best[1] | (8 if np.signbit(v) else 0))
    return np.array(out, dtype=np.uint8)


def test_e2m1_rounding_brute_force():
    rng = np.random.default_rng(7)
    q = np.concatenate([rng.uniform(-8, 8, 4000), rng.uniform(-0.3, 0.3, 500),
                        [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -0.25, -5.0, 6.0, 6.5, 1e9, -1e9,
                         0.0, -0.0, np.nextafter(0.25, 1), np.nextafter(0.25, 0)]]).astype(np.float32)
    np.testing.assert_array_equal(nvfp4.e2m1_round(q), _e2m1_brute(q))


def test_e4m3_matches_a_library_cast():
    """Inside the finite range, round-to-nearest-even to E4M3 is what torch's FP8 cast
    does; its decode of all 256 patterns matches the table too."""
    rng = np.random.default_rng(3)
    vals = nvfp4.e4m3_value(np.arange(0x7F))
    mids = (vals[1:] + vals[:-1]) / 2
    t = np.concatenate([rng.uniform(0, 447.9, 20000), rng.uniform(0, 0.02, 20000), vals, mids,
                        np.nextafter(mids, 0), np.nextafter(mids, 1e9)]).astype(np.float32)
    t = t[t < 448]
    ref = torch.from_numpy(t).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(nvfp4.e4m3_round(t), ref)
    tv = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy()
    mine = nvfp4.e4m3_value(np.arange(256))
    assert np.all((mine == tv) | (np.isnan(mine) & np.isnan(tv)))


def test_e4m3_saturates_at_448():
    t = np.array([448.0, 455.0, 464.0, 470.0, 480.0, 1e6, 3e38], dtype=np.float32)
    assert np.all(nvfp4.e4m3_round(t) == 0x7E)
    assert nvfp4.e4m3_value(0x7E) == 448.0
    assert nvfp4.e4m3_round(np.float32(432.0)) == 0x7E   # tie 416|448 -> even mantissa 6
    assert nvfp4.e4m3_round(np.float32(431.9)) == 0x7D


def _golden_row():
    g, blocks, packed, scales = None, [], None, None
    for line in open(os.path.join(GOLDEN, "nvfp4_row.txt")):
        f = line.split()
        if not f or f[0].startswith("#"):
            continue
        if f[0] == "g":
            g = np.float32(float.fromhex(f[1]))
        elif f[0] == "block":
            blocks.append([float(v) for v in f[1:]])
        elif f[0] == "packed":
            packed = np.array([int(v, 16) for v in f[1:]], dtype=np.uint8)
        elif f[0] == "scales":
            scales = np.array([int(v, 16) for v in f[1:]], dtype=np.uint8)
    x = (np.array(blocks, dtype=np.float64).reshape(1, -1) * np.float64(g)).astype(np.float32)
    return x, g, packed, scales


def test_hand_worked_row():
    x, g, packed, scales = _golden_row()
    codes, sf = nvfp4.quantize(x, g)
    np.testing.assert_array_equal(nvfp4.pack(codes)[0], packed)
    np.testing.assert_array_equal(sf[0], scales)
    np.testing.assert_array_equal(nvfp4.unpack(nvfp4.pack(codes)), codes)


def test_exact_values_round_trip():
    """A block whose values are E2M1 values times a representable d, with a 6 in it,
    quantizes to exactly those codes and scale and decodes to itself."""
    rng = np.random.default_rng(11)
    N, K = 64, 256
    g = np.float32(2.0 ** -7)
    sf_true = rng.integers(0x08, 0x7E, size=(N, K // 16))          # normal E4M3 scales
    codes_true = rng.integers(0, 16, size=(N, K)).astype(np.uint8)
    codes_true[:, ::16] = 7                                          # block max is +6
    x = nvfp4.dequantize(codes_true, sf_true.astype(np.uint8), g).astype(np.float32)
    codes, sf = nvfp4.quantize(x, g)
    np.testing.assert_array_equal(sf, sf_true)
    np.testing.assert_array_equal(nvfp4.e2m1_value(codes), nvfp4.e2m1_value(codes_true))
    np.testing.assert_array_equal(nvfp4.dequantize(codes, sf, g), x.astype(np.float64))


def test_quantization_error_bound():
    """Each decoded value is within half an E2M1 step of x·(1/d), in units of d; values
    beyond 6d (the scale rounded down) saturate to ±6, by at most the E4M3 rounding of the
    scale (2^-4)."""
    rng = np.random.default_rng(5)
    x = (rng.standard_normal((96, 512)) * np.exp(rng.uniform(-3, 3, (96, 1)))).astype(np.float32)
    g = nvfp4.global_scale(np.max(np.abs(x)))
    codes, sf = nvfp4.quantize(x, g)
    deq = nvfp4.dequantize(codes, sf, g)
    d = np.repeat(nvfp4.e4m3_value(sf) * np.float64(g), 16, axis=1)
    q = np.abs(x) / d
    half_step = np.where(q <= 2, 0.25, np.where(q <= 4, 0.5, 1.0))
    err = np.abs(deq - x) / d
    sat = q > 6
    assert np.all(err[~sat] <= half_step[~sat] * (1 + 1e-6))
    assert np.all(np.abs(x)[sat] <= 6 * d[sat] * (1 + 2.0 ** -4) + 1e-30)
    assert np.all((codes[sat] & 7) == 7)
    assert np.all(np.sign(deq[deq != 0]) == np.sign(x[deq != 0]))


def test_global_scale_puts_the_largest_block_on_448():
    rng = np.random.default_rng(9)
    x = rng.standard_normal((40, 160)).astype(np.float32)
    amax = np.max(np.abs(x))
    g = nvfp4.global_scale(amax)
    _, sf = nvfp4.quantize(x, g)
    r, c = np.unravel_index(np.argmax(np.abs(x)), x.shape)
    assert sf[r, c // 16] == 0x7E
    assert np.all(nvfp4.e4m3_value(sf) <= 448)
    assert nvfp4.global_scale(np.float32(2688 * 2.0 ** -8)) == np.float32(2.0 ** -8)


def test_zero_and_tiny_blocks():
    x = np.zeros((2, 32), dtype=np.float32)
    x[1, 16] = -1e-30          # the scale underflows to 0: the block stores +0 codes
    codes, sf = nvfp4.quantize(x, np.float32(1.0))
    assert np.all(codes == 0) and np.all(sf == 0)
    # a zero global scale (all-zero weight) gives zero scales and codes, no NaN
    codes, sf = nvfp4.quantize(np.ones((1, 16), np.float32), np.float32(0.0))
    assert np.all(codes == 0) and np.all(sf == 0)


def test_128x4_layout_shape_padding_and_bijection():
    """The padded shape is the pages'; the order inside a tile is a reading (parity
    unpinned): here only that it places every entry once and pads with zeros."""
    for N, KB in [(1, 1), (130, 5), (256, 8), (300, 72)]:
        sf = (np.arange(N * KB) % 251 + 1).astype(np.uint8).reshape(N, KB)
        out = nvfp4.scales_128x4(sf)
        NP, KBP = -(-N // 128) * 128, -(-KB // 4) * 4
        assert out.size == NP * KBP
        assert np.count_nonzero(out) == N * KB
        assert sorted(out[out != 0].tolist()) == sorted(sf.reshape(-1).tolist())
    # one 128x4 tile: each row's 4 scales are contiguous; rows 32 apart interleave
    sf = np.arange(1, 129 * 4 + 1).reshape(129, 4) % 256
    out = nvfp4.scales_128x4(sf.astype(np.uint8))
    np.testing.assert_array_equal(out[0:4], sf[0])
    np.testing.assert_array_equal(out[4:8], sf[32])
    np.testing.assert_array_equal(out[16:20], sf[1])
    np.testing.assert_array_equal(out[512:516], sf[128])


def test_weff_f32_and_bound():
    """W_eff in fp32 is the exact sum rounded once; with the passthrough bundle (s = 1,
    r = 0) it is W0 itself and the bound is zero."""
    rng = np.random.default_rng(2)
    W0 = np.round(rng.standard_normal((8, 32)) * 64) / 64
    s = np.ones(8)
    U, V = np.zeros((8, 0)), np.zeros((32, 0))
    np.testing.assert_array_equal(nvfp4.weff_f32(W0, s, U, V), W0.astype(np.float32))
    b = nvfp4.weff_error_bound(W0, s, U, V)
    assert np.all(b <= 3 * 2.0 ** -23 * np.abs(W0) * 1.0001)


def test_ambiguity_flags_only_near_boundaries():
    """With no evaluation error the flags sit exactly on decision boundaries; widening
    the error widens them; nothing else is flagged."""
    x, g, _, _ = _golden_row()
    ele, blk = nvfp4.ambiguous(x.astype(np.float64), np.zeros(x.shape), g)
    # block 3's scale input is an exact E4M3 tie; blocks 1 and 2 are not on a boundary
    assert blk[0].tolist() == [False, False, True]
    q = np.abs(x[0, :16].astype(np.float64)) / np.float64(g)
    at_tie = np.isin(q, [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]) | (q == 0)
    np.testing.assert_array_equal(ele[0, :16], at_tie)
    rng = np.random.default_rng(1)
    y = rng.standard_normal((16, 64))
    gy = nvfp4.global_scale(np.max(np.abs(y)))
    e0, b0 = nvfp4.ambiguous(y, np.zeros(y.shape), gy)
    e1, b1 = nvfp4.ambiguous(y, np.full(y.shape, 1e-3), gy)
    assert not e0.any() and not b0.any()
    assert e1.sum() > 0 and np.all(e1 | ~e0)
