"""Seeded synthetic inputs for the theta-bundle reconstruction linear.

This module only draws numbers: it holds none of the reconstruction's arithmetic.
Both the CUDA path (through the tests and the benchmark) and the fp64 oracle are fed
from it, so that they see the very same bf16 values.

Generator
---------
* ``splitmix64`` (Steele, Lea and Flood, "Fast splittable pseudorandom number
  generators", OOPSLA 2014; the 64-bit finaliser popularised by Vigna): the n-th
  output of a stream with state ``S`` is ``mix(S + (n + 1) * 0x9E3779B97F4A7C15)``,
  so any element can be drawn from its index alone (counter-based).
* uniform doubles from the top 53 bits of an output;
* normal doubles by Box-Muller (cosine branch), element ``j`` using the two
  outputs ``2j`` and ``2j + 1`` of its stream;
* every stored value is rounded from double to bfloat16 with round-to-nearest-even,
  written from the format's definition (1 sign bit, 8 exponent bits, 7 fraction
  bits, subnormals down to 2**-133).

Value distributions follow the workloads the pages' models imply (Gemma-shaped
projections): W0 ~ N(0, 0.02^2), s ~ U(0.9, 1.1), U, V ~ N(0, 0.01^2), x ~ N(0, 1),
optionally with each token row of x scaled by a ~ U(0.5, 2).

Everything is returned as ``uint16`` arrays of bf16 bit patterns (row-major, with
an optional padded leading dimension) plus helpers to widen them to float64 or to
view them as torch bf16 tensors.
"""
from __future__ import annotations

import hashlib
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def splitmix64(state: int, counters: np.ndarray) -> np.ndarray:
    """Outputs number ``counters`` (0-based) of a splitmix64 stream started at ``state``."""
    with np.errstate(over="ignore"):
        c = np.asarray(counters, dtype=np.uint64)
        z = np.uint64(state & 0xFFFFFFFFFFFFFFFF) + (c + np.uint64(1)) * _GOLDEN
        return _mix(z)


def stream_seed(*keys) -> int:
    """A 64-bit stream state derived from any tuple of ints/strings (e.g. config,
    layer, family, tensor name). Uses SHA-256 so that nearby keys give unrelated streams."""
    h = hashlib.sha256(repr(tuple(keys)).encode()).digest()
    return int.from_bytes(h[:8], "little")


def _uniform01(state: int, start: int, n: int) -> np.ndarray:
    z = splitmix64(state, np.arange(start, start + n, dtype=np.uint64))
    return (z >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def _chunked(n: int, fn) -> None:
    """Run fn(a, b) over [0, n) in chunks; numpy releases the GIL inside its
    ufuncs, so a thread pool spreads large draws over the host cores."""
    spans = [(a, min(n, a + _CHUNK)) for a in range(0, n, _CHUNK)]
    if len(spans) <= 1:
        for a, b in spans:
            fn(a, b)
        return
    with ThreadPoolExecutor(max_workers=min(len(spans), os.cpu_count() or 1)) as ex:
        list(ex.map(lambda ab: fn(*ab), spans))


def normal_f64(state: int, n: int, sigma: float = 1.0, mean: float = 0.0) -> np.ndarray:
    out = np.empty(n, dtype=np.float64)

    def fill(a, b):
        u = _uniform01(state, 2 * a, 2 * (b - a)).reshape(-1, 2)
        u1 = 1.0 - u[:, 0]                      # (0, 1]: log is finite
        out[a:b] = np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u[:, 1]) * sigma + mean

    _chunked(n, fill)
    return out


def uniform_f64(state: int, n: int, lo: float, hi: float) -> np.ndarray:
    out = np.empty(n, dtype=np.float64)

    def fill(a, b):
        out[a:b] = lo + (hi - lo) * _uniform01(state, a, b - a)

    _chunked(n, fill)
    return out


def bf16_bits_from_f64(v: np.ndarray) -> np.ndarray:
    """Round doubles to bfloat16 (nearest, ties to even) and return the bit patterns.

    Uses exact power-of-two scaling: for |v| in [2**(e-1), 2**e) the bf16 spacing is
    2**(e-8) (never below the subnormal spacing 2**-133), so ``round(v / q) * q`` is
    the correctly rounded value (numpy's ``round`` is half-to-even and exact here).
    """
    v = np.asarray(v, dtype=np.float64)
    out = np.empty(v.shape, dtype=np.uint16)
    flat_v = v.reshape(-1)
    flat_o = out.reshape(-1)

    def fill(a, b):
        x = flat_v[a:b]
        _, e = np.frexp(x)
        q = np.maximum(e.astype(np.int64) - 8, -133)
        r = np.ldexp(np.round(np.ldexp(x, -q)), q)
        with np.errstate(over="ignore"):
            f = r.astype(np.float32)            # exact (or +-inf past the bf16 range)
        flat_o[a:b] = (f.view(np.uint32) >> np.uint32(16)).astype(np.uint16)

    _chunked(flat_v.size, fill)
    return out


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float64 (exact)."""
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


def round_up(a: int, b: int) -> int:
    return (a + b - 1) // b * b


def _matrix(vals: np.ndarray, rows: int, cols: int, ld: int | None) -> np.ndarray:
    """bf16 bits of a rows x cols matrix stored row-major with leading dimension ld
    (padding columns are zero). Returns the full [rows, ld] array."""
    ld = cols if ld is None else ld
    assert ld >= cols
    bits = bf16_bits_from_f64(vals).reshape(rows, cols)
    if ld == cols:
        return bits
    out = np.zeros((rows, ld), dtype=np.uint16)
    out[:, :cols] = bits
    return out


@dataclass
class Theta:
    """One projection's theta bundle as bf16 bit arrays (row-major, padded ld).

    W0: [out, ld_w0]   s: [out]   U: [out, ld_u]   V: [in, ld_v]
    Shapes follow the GEMM formulation on the "Execution paths" page
    (``x @ W0.T``, ``x @ V``, ``@ U.T``)."""
    W0: np.ndarray
    s: np.ndarray
    U: np.ndarray | None
    V: np.ndarray | None
    out: int
    inp: int
    r: int

    def f64(self):
        """(W0, s, U, V) widened to float64 with the padding columns dropped."""
        W0 = bf16_bits_to_f64(self.W0[:, : self.inp])
        s = bf16_bits_to_f64(self.s)
        if self.r == 0:
            U = np.zeros((self.out, 0))
            V = np.zeros((self.inp, 0))
        else:
            U = bf16_bits_to_f64(self.U[:, : self.r])
            V = bf16_bits_to_f64(self.V[:, : self.r])
        return W0, s, U, V


def ld_for(cols: int) -> int:
    """Smallest leading dimension (elements) keeping bf16 rows 16-byte aligned."""
    return round_up(max(cols, 1), 8)


def make_w0(seed_keys, out: int, inp: int, sigma: float = 0.02) -> np.ndarray:
    st = stream_seed(*seed_keys, "W0")
    return _matrix(normal_f64(st, out * inp, sigma), out, inp, ld_for(inp))


def make_theta(seed_keys, out: int, inp: int, r: int, W0: np.ndarray | None = None,
               w0_sigma: float = 0.02, s_range=(0.9, 1.1), uv_sigma: float = 0.01) -> Theta:
    """Theta bundle with the stated distributions. ``W0`` may be passed in to share
    one block across the layers of a band."""
    if W0 is None:
        W0 = make_w0(seed_keys, out, inp, w0_sigma)
    s = bf16_bits_from_f64(uniform_f64(stream_seed(*seed_keys, "s"), out, *s_range))
    if r == 0:
        U = V = None
    else:
        U = _matrix(normal_f64(stream_seed(*seed_keys, "U"), out * r, uv_sigma), out, r, ld_for(r))
        V = _matrix(normal_f64(stream_seed(*seed_keys, "V"), inp * r, uv_sigma), inp, r, ld_for(r))
    return Theta(W0=W0, s=s, U=U, V=V, out=out, inp=inp, r=r)


def passthrough_theta(seed_keys, out: int, inp: int, r: int) -> Theta:
    """s = 1, U = V = 0: the passthrough operating point ("How attnquant works",
    "The passthrough operating point")."""
    W0 = make_w0(seed_keys, out, inp)
    s = bf16_bits_from_f64(np.ones(out))
    if r == 0:
        return Theta(W0, s, None, None, out, inp, 0)
    U = np.zeros((out, ld_for(r)), dtype=np.uint16)
    V = np.zeros((inp, ld_for(r)), dtype=np.uint16)
    return Theta(W0, s, U, V, out, inp, r)


def make_x(seed_keys, M: int, inp: int, row_scale=None) -> np.ndarray:
    """Activations x [M, inp] ~ N(0,1); with ``row_scale=(lo, hi)`` each token row is
    multiplied by a ~ U(lo, hi) before rounding (token-norm spread)."""
    v = normal_f64(stream_seed(*seed_keys, "x"), M * inp).reshape(M, inp)
    if row_scale is not None:
        a = uniform_f64(stream_seed(*seed_keys, "xscale"), M, *row_scale)
        v = v * a[:, None]
    return _matrix(v.reshape(-1), M, inp, ld_for(inp))


def small_int_theta(seed_keys, out: int, inp: int, r: int, lim: int = 3) -> Theta:
    """Integer-valued theta: W0, U, V in [-lim, lim], s in {0.5, 1, 2}. With small
    sizes every partial sum is an integer (or half-integer) well inside 2**8, so
    any fp32 summation order gives the exact value and bf16 holds it exactly."""
    def ints(tag, n):
        z = splitmix64(stream_seed(*seed_keys, tag), np.arange(n, dtype=np.uint64))
        return (z % np.uint64(2 * lim + 1)).astype(np.int64) - lim
    W0 = _matrix(ints("W0", out * inp).astype(np.float64), out, inp, ld_for(inp))
    choice = np.array([0.5, 1.0, 2.0])
    z = splitmix64(stream_seed(*seed_keys, "s"), np.arange(out, dtype=np.uint64))
    s = bf16_bits_from_f64(choice[(z % np.uint64(3)).astype(np.int64)])
    if r == 0:
        return Theta(W0, s, None, None, out, inp, 0)
    U = _matrix(ints("U", out * r).astype(np.float64), out, r, ld_for(r))
    V = _matrix(ints("V", inp * r).astype(np.float64), inp, r, ld_for(r))
    return Theta(W0, s, U, V, out, inp, r)


def small_int_x(seed_keys, M: int, inp: int, lim: int = 3) -> np.ndarray:
    z = splitmix64(stream_seed(*seed_keys, "x"), np.arange(M * inp, dtype=np.uint64))
    v = ((z % np.uint64(2 * lim + 1)).astype(np.int64) - lim).astype(np.float64)
    return _matrix(v, M, inp, ld_for(inp))


def _sparse_ints(state: int, n: int, lim: int, density: float) -> np.ndarray:
    """Integers in [-lim, lim] \\ {0} with probability ``density``, else 0."""
    z = splitmix64(state, np.arange(2 * n, dtype=np.uint64)).reshape(n, 2)
    keep = (z[:, 0] >> np.uint64(11)).astype(np.float64) * (2.0 ** -53) < density
    mag = (z[:, 1] % np.uint64(lim)).astype(np.int64) + 1
    sign = np.where((z[:, 1] >> np.uint64(32)) & np.uint64(1), -1, 1)
    return np.where(keep, sign * mag, 0).astype(np.float64)


def sparse_int_theta(seed_keys, out: int, inp: int, r: int, w_lim: int = 2, uv_lim: int = 1,
                     w_density: float = 0.5, v_density: float = 0.1, u_density: float = 0.5) -> Theta:
    """Integer-valued bundle for bit-exact checks: sparse small integers keep every
    partial sum (W0 x, Vᵀx and the final y) small enough to be exact in fp32 and,
    for t and y, in bf16 as well; s is drawn from {0.5, 1, 2}."""
    W0 = _matrix(_sparse_ints(stream_seed(*seed_keys, "W0"), out * inp, w_lim, w_density), out, inp,
                 ld_for(inp))
    choice = np.array([0.5, 1.0, 2.0])
    z = splitmix64(stream_seed(*seed_keys, "s"), np.arange(out, dtype=np.uint64))
    s = bf16_bits_from_f64(choice[(z % np.uint64(3)).astype(np.int64)])
    if r == 0:
        return Theta(W0, s, None, None, out, inp, 0)
    U = _matrix(_sparse_ints(stream_seed(*seed_keys, "U"), out * r, w_lim, u_density), out, r, ld_for(r))
    V = _matrix(_sparse_ints(stream_seed(*seed_keys, "V"), inp * r, uv_lim, v_density), inp, r, ld_for(r))
    return Theta(W0, s, U, V, out, inp, r)


def sparse_int_x(seed_keys, M: int, inp: int, density: float = 0.3) -> np.ndarray:
    return _matrix(_sparse_ints(stream_seed(*seed_keys, "x"), M * inp, 1, density), M, inp, ld_for(inp))


# ----------------------------------------------------------------------------------
# Workload shapes (sizes only; no trained weights are involved anywhere)
# ----------------------------------------------------------------------------------
GEMMA3_1B_FAMILIES = {
    # family: (out, in)
    "q_proj": (1024, 1152),
    "k_proj": (256, 1152),
    "v_proj": (256, 1152),
    "o_proj": (1152, 1024),
    "gate_proj": (6912, 1152),
    "up_proj": (6912, 1152),
    "down_proj": (1152, 6912),
}
GEMMA3_1B_LAYERS = 26
CLASS31B_SHAPES = {"wide": (21504, 5376), "square": (5376, 5376)}
CLASS31B_LAYERS = 60
