"""Oracle for quantizing the effective weight W_eff = s·W0 + U·Vᵀ to NVFP4.

TEST INFRASTRUCTURE ONLY: imported by the tests, the smoke check and the benchmark's
CPU-baseline leg, never by the library, and sharing no code with it.

Sources (page title, then section):
* "Execution paths", "Precompute-outside: the production path": with NVFP4 selected,
  every W_eff is quantized to 4 bits when the model loads.
* "Internals and extension", "Nvfp4Spec": two E2M1 values share a byte,
  so a logical (N, K) weight is held as (N, K // 2) bytes; each run of 16 values along K
  has one FP8-E4M3 block scale, and the whole tensor one fp32 global scale. The block
  scales come in a "linear" (N, K // 16) layout or a "128x4" layout padded to
  (ceil(N, 128), ceil(K // 16, 4)) for Blackwell GEMMs, chosen for sm >= 100.

The formats themselves are the published ones: E2M1 is 1 sign, 2 exponent (bias 1) and 1
mantissa bit, magnitudes {0, 0.5, 1, 1.5, 2, 3, 4, 6}; E4M3 (the OCP 8-bit float
"E4M3") is 1 sign, 4 exponent (bias 7) and 3 mantissa bits, subnormal step 2^-9, largest
finite 448, the all-ones exponent-and-mantissa pattern being NaN.

Readings where the pages are silent (each also listed in the design notes):
* The value quantized is W_eff in fp32 (the exact sum rounded once to fp32), not a bf16
  copy of it: the fused precompute never forms the bf16 weight.
* The stored global scale g is the decode multiplier: a weight decodes as
  e2m1 · e4m3 · g. Unless the caller gives g, it is amax / 2688 in fp32, amax = max|W_eff|
  and 2688 = 6 · 448, so that the largest block scale lands on the largest E4M3 value.
* One block: a = max|x|; t = a · (1/(6·g)), the factor 1/(6·g) formed once per tensor; the
  stored scale is E4M3(t), rounded to nearest even and clamped to 448 ("satfinite");
  d = E4M3(t) · g; each x becomes E2M1(x · (1/d)), rounded to nearest even (ties to the even
  code), clamped to ±6, keeping the sign of x (a small negative x gives −0). A block whose d
  is 0 stores +0 codes. Every one of these operations is a single fp32 operation rounded to
  nearest even (6·g, 1/(6·g), a·that, value·g, 1/d, x·that); they are the decision steps both
  sides take in the same precision.
* Two codes per byte, the even column in the low nibble.
* The "128x4" layout's order inside a tile is not on the pages. Taken here: 128-row by
  4-column tiles of 512 bytes, tiles ordered with the K direction fastest, and inside a
  tile the byte of (row r, column c) at 16·(r mod 32) + 4·(r div 32) + c. Padding is 0.
  Parity unpinned: the pages fix the padded shape, not this order.

Parity status: the E2M1 and E4M3 rounding, the block rule, packing and the linear layout
are pinned by ``tests/test_nvfp4_pins.py`` (format tables, a library FP8 cast, brute
force, exact round trips, error bounds, a hand-worked block under ``tests/golden/``).
The 128x4 tile order is "parity unpinned" (only its shape, padding and bijectivity are
checked).
"""
from __future__ import annotations

import numpy as np

E2M1_MAX = 6.0
E4M3_MAX = 448.0
GLOBAL_DIV = np.float32(6.0 * 448.0)
BLOCK = 16

# magnitude of each 3-bit E2M1 code: exponent bits e, mantissa bit m; e = 0 is subnormal
E2M1_MAGNITUDES = np.array(
    [(m * 0.5) if e == 0 else (1.0 + 0.5 * m) * 2.0 ** (e - 1) for e in range(4) for m in range(2)])


def e2m1_value(codes) -> np.ndarray:
    """Value of each 4-bit E2M1 code (bit 3 the sign)."""
    c = np.asarray(codes, dtype=np.int64)
    mag = E2M1_MAGNITUDES[c & 7]
    return np.where(c & 8, -mag, mag)


def e2m1_round(q) -> np.ndarray:
    """Nearest E2M1 code of each fp32 value, ties to the even code, clamped to ±6,
    the sign of q kept (−0 for negative values that round to zero)."""
    q = np.asarray(q, dtype=np.float32).astype(np.float64)
    a = np.minimum(np.abs(q), E2M1_MAX)
    hi = np.searchsorted(E2M1_MAGNITUDES, a, side="left")   # first magnitude >= a
    hi = np.minimum(hi, 7)
    lo = np.maximum(hi - 1, 0)
    dlo = a - E2M1_MAGNITUDES[lo]
    dhi = E2M1_MAGNITUDES[hi] - a
    pick_hi = (dhi < dlo) | ((dhi == dlo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo)
    return (code | np.where(np.signbit(q), 8, 0)).astype(np.uint8)


def e4m3_value(bits) -> np.ndarray:
    """Value of each E4M3 byte (finite patterns; 0x7F / 0xFF are NaN)."""
    b = np.asarray(bits, dtype=np.int64)
    e = (b >> 3) & 15
    m = b & 7
    mag = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.ldexp(1.0, e - 7))
    mag = np.where((b & 0x7F) == 0x7F, np.nan, mag)
    return np.where(b & 0x80, -mag, mag)


def e4m3_round(t) -> np.ndarray:
    """Nearest E4M3 byte of each fp32 value, ties to even, magnitudes clamped to 448
    ("satfinite"), the sign kept."""
    t = np.asarray(t, dtype=np.float32).astype(np.float64)
    a = np.abs(t)
    out = np.zeros(a.shape, dtype=np.int64)
    sub = a < 2.0 ** -6
    # subnormal range: multiples of 2^-9 (a result of 8 is the smallest normal, bits 0x08)
    out[sub] = np.rint(a[sub] * 2.0 ** 9).astype(np.int64)
    nrm = ~sub
    mant, ex = np.frexp(a[nrm])                  # a = mant · 2^ex, mant in [0.5, 1)
    e = ex - 1                                   # a = (2·mant) · 2^e, 2·mant in [1, 2)
    k = np.rint((2.0 * mant - 1.0) * 8.0).astype(np.int64)   # ties to even (exact)
    carry = k == 8
    e = np.where(carry, e + 1, e)
    k = np.where(carry, 0, k)
    bits = ((e + 7) << 3) | k
    bits = np.where((e + 7 > 15) | (bits > 0x7E), 0x7E, bits)   # satfinite: 448 = 0x7E
    out[nrm] = bits
    return (out | np.where(np.signbit(t), 0x80, 0)).astype(np.uint8)


def weff_f32(W0, s, U, V) -> np.ndarray:
    """W_eff = s·W0 + U·Vᵀ, exact in float64 then rounded once to fp32 (the value the
    quantizer sees). "Execution paths", "Precompute-outside: the production path"."""
    W0, s, U, V = (np.asarray(a, dtype=np.float64) for a in (W0, s, U, V))
    return (s[:, None] * W0 + U @ V.T).astype(np.float32)


def global_scale(amax) -> np.float32:
    """g = amax / (6·448) in fp32 ("Nvfp4Spec": one fp32 global scale)."""
    return np.float32(np.float32(amax) / GLOBAL_DIV)


def quantize(x32, g):
    """Codes (N, K) uint8 (one 4-bit code per value) and linear block scales (N, K/16)
    uint8 of fp32 values x32 under the global scale g, by the block rule stated in the
    module header ("Nvfp4Spec": 16 values per E4M3 scale, one fp32 global scale)."""
    x = np.asarray(x32, dtype=np.float32)
    N, K = x.shape
    if K % BLOCK:
        raise ValueError("K must be a multiple of 16")
    g = np.float32(g)
    blocks = x.reshape(N, K // BLOCK, BLOCK)
    a = np.max(np.abs(blocks), axis=2)                        # exact in fp32
    six_g = np.float32(np.float32(6.0) * g)
    inv6 = np.float32(np.float32(1.0) / six_g) if six_g > 0 else np.float32(0.0)
    t = (a * inv6).astype(np.float32)
    sf = e4m3_round(t)
    d = (e4m3_value(sf).astype(np.float32) * g).astype(np.float32)
    with np.errstate(divide="ignore"):
        inv = np.where(d > 0, np.float32(1.0) / d, np.float32(0)).astype(np.float32)
    q = (blocks * inv[:, :, None]).astype(np.float32)
    codes = e2m1_round(q)
    codes = np.where((d > 0)[:, :, None], codes, 0).astype(np.uint8)
    return codes.reshape(N, K), sf


def pack(codes) -> np.ndarray:
    """(N, K) 4-bit codes -> (N, K/2) bytes, column 2j in the low nibble of byte j."""
    c = np.asarray(codes, dtype=np.uint8)
    return (c[:, 0::2] | (c[:, 1::2] << 4)).astype(np.uint8)


def unpack(packed) -> np.ndarray:
    """Inverse of ``pack``."""
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty((p.shape[0], 2 * p.shape[1]), dtype=np.uint8)
    out[:, 0::2] = p & 15
    out[:, 1::2] = p >> 4
    return out


def dequantize(codes, sf, g) -> np.ndarray:
    """e2m1 · e4m3 · g per value, in float64."""
    c = np.asarray(codes)
    N, K = c.shape
    scale = np.repeat(e4m3_value(sf), BLOCK, axis=1)[:, :K] * np.float64(np.float32(g))
    return e2m1_value(c) * scale


def scales_128x4(sf) -> np.ndarray:
    """The linear (N, K/16) scales placed in the padded 128x4 layout, as a flat byte
    array of ceil(N, 128) · ceil(K/16, 4) entries (tile order: module header; parity
    unpinned)."""
    sf = np.asarray(sf, dtype=np.uint8)
    N, KB = sf.shape
    NP, KBP = -(-N // 128) * 128, -(-KB // 4) * 4
    out = np.zeros(NP * KBP, dtype=np.uint8)
    n_kt = KBP // 4
    for r in range(N):
        for c in range(KB):
            tile = (r // 128) * n_kt + c // 4
            rr, cc = r % 128, c % 4
            out[tile * 512 + 16 * (rr % 32) + 4 * (rr // 32) + cc] = sf[r, c]
    return out


def weff_error_bound(W0, s, U, V, unit_roundoff: float = 2.0 ** -23) -> np.ndarray:
    """Bound on |fp32 evaluation of W_eff − exact W_eff| per element: the dot-product
    bound of Higham, "Accuracy and Stability of Numerical Algorithms", sec. 3.1, over the
    r + 2 roundings of an fp32 evaluation (r products summed, then s·W0 added), with
    u = 2^-23 so that truncating accumulation is covered too."""
    W0, s, U, V = (np.asarray(a, dtype=np.float64) for a in (W0, s, U, V))
    n = U.shape[1] + 2
    gamma = n * unit_roundoff / (1.0 - n * unit_roundoff)
    return gamma * (np.abs(s[:, None] * W0) + np.abs(U) @ np.abs(V).T)


_E2M1_CUTS = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])


def _e4m3_cuts() -> np.ndarray:
    vals = np.unique(e4m3_value(np.arange(0x7F)))
    return (vals[1:] + vals[:-1]) / 2.0


def ambiguous(x, bound, g, g_rel: float = 0.0):
    """Where an fp32 evaluation within ``bound`` of the exact W_eff ``x`` may take a
    different decision than the exact one: (element flags (N, K), block flags (N, K/16)).

    A block is flagged when its scale's input t = a / (6g) can fall on either side of an
    E4M3 rounding boundary (a moved by the largest bound in the block, g by the relative
    ``g_rel``, plus the fp32 roundings of the rule); an element when x · (1/d) can fall on
    either side of an E2M1 boundary or of zero. Outside the flags the decisions are
    unique, so codes and scales must match bit for bit there."""
    x = np.asarray(x, dtype=np.float64)
    bound = np.asarray(bound, dtype=np.float64) + np.abs(x) * 2.0 ** -24
    N, K = x.shape
    g64 = np.float64(np.float32(g))
    rel = g_rel + 4 * 2.0 ** -24
    xb = np.abs(x).reshape(N, K // BLOCK, BLOCK)
    bb = bound.reshape(N, K // BLOCK, BLOCK)
    a = xb.max(axis=2)
    b = bb.max(axis=2)
    with np.errstate(divide="ignore", invalid="ignore"):
        t_lo = (a - b) / (6.0 * g64) * (1 - rel)
        t_hi = (a + b) / (6.0 * g64) * (1 + rel)
    cuts = _e4m3_cuts()
    blk = (np.searchsorted(cuts, t_lo, side="left") != np.searchsorted(cuts, t_hi, side="right"))
    blk |= ~np.isfinite(t_lo) | ~np.isfinite(t_hi)
    _, sf = quantize(x.astype(np.float32), g)
    d = e4m3_value(sf) * g64
    with np.errstate(divide="ignore", invalid="ignore"):
        q = np.abs(x).reshape(N, K // BLOCK, BLOCK) / d[:, :, None]
        dq = bb / d[:, :, None] + q * (rel + 2.0 ** -23)
    q_lo, q_hi = q - dq, q + dq
    ele = (np.searchsorted(_E2M1_CUTS, q_lo, side="left") != np.searchsorted(_E2M1_CUTS, q_hi, side="right"))
    ele |= np.abs(x).reshape(N, K // BLOCK, BLOCK) <= bb          # sign of a zero code
    ele &= (d > 0)[:, :, None]
    return ele.reshape(N, K), blk
