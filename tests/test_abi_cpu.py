"""The C-ABI library builds, loads and exports every declared symbol; host-side argument
validation works without a GPU (no compute calls are made here)."""
import ctypes
import os
import re

import pytest

import rank_weight_reconstruction_gb300 as aq
from rank_weight_reconstruction_gb300 import binding, build_lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build_lib.build()
    return binding.load()


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "aq.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(aq_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_boundary():
    syms = declared_symbols()
    for name in ("aq_linear", "aq_linear_qkv", "aq_precompute", "aq_linear_workspace_bytes"):
        assert name in syms
    assert sorted(binding.EXPORTED_SYMBOLS) == syms


def test_library_exports_every_declared_symbol(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_status_strings_and_version(lib):
    assert binding.aq_abi_version() == 1
    assert binding.aq_status_string(0) == "AQ_OK"
    assert binding.aq_status_string(8) == "AQ_ERR_TIMEOUT"
    assert binding.aq_status_string(99) == "AQ_ERR_UNKNOWN"
    assert aq.aq_decode_max_m() == 32


def _theta(out=64, inp=32, r=4, W0=0x1000, s=0x2000, U=0x3000, V=0x4000, ld_w0=None, ld_u=8, ld_v=8):
    return binding.c_theta(W0=W0, ld_w0=ld_w0 or inp, s=s, U=U if r else 0, ld_u=ld_u if r else 0,
                           V=V if r else 0, ld_v=ld_v if r else 0, out=out, in_=inp, r=r)


def _linear(lib, th, x=0x100000, M=4, ldx=32, y=0x200000, ldy=64, ws=0x300000, ws_bytes=1 << 20):
    return lib.aq_linear(ctypes.byref(th), x, M, ldx, y, ldy, ws, ws_bytes, None)


def test_workspace_bytes(lib):
    """Layout: a zero-initialised sync region of AQ_WORKSPACE_SYNC_BYTES (all the decode
    kernel needs), then prefill scratch: t as bf16 [M, sum round_up(r, 8)] (rounded to
    256 B) and V^T of all families stacked as [sum round_up(r, 8), round_up(in, 8)] (rounded
    to 256 B). For M <= 32 the workspace covers both paths."""
    sync = binding.AQ_WORKSPACE_SYNC_BYTES
    th = _theta(out=64, inp=32, r=4)
    # M = 4: t 4 x 8 x 2 = 64 -> 256, V^T 8 x 32 x 2 = 512
    assert lib.aq_linear_workspace_bytes(ctypes.byref(th), 1, 4) == sync + 256 + 512
    assert lib.aq_linear_workspace_bytes(ctypes.byref(th), 1, 0) == 0
    # M = 100: prefill only: t 100 x 8 x 2 = 1600 -> 1792, V^T 512
    assert lib.aq_linear_workspace_bytes(ctypes.byref(th), 1, 100) == sync + 1792 + 512
    th0 = _theta(r=0)
    assert lib.aq_linear_workspace_bytes(ctypes.byref(th0), 1, 1000) == 0
    assert lib.aq_linear_workspace_bytes(ctypes.byref(th0), 1, 8) == sync
    arr = (binding.c_theta * 3)(_theta(r=4), _theta(r=0), _theta(r=12))
    # M = 8: t 8 x (8 + 16) x 2 = 384 -> 512, V^T (8 + 16) x 32 x 2 = 1536
    assert lib.aq_linear_workspace_bytes(arr, 3, 8) == sync + 512 + 1536
    # M = 40: t 40 x 24 x 2 = 1920 -> 2048
    assert lib.aq_linear_workspace_bytes(arr, 3, 40) == sync + 2048 + 1536
    assert lib.aq_linear_workspace_bytes(ctypes.byref(th), 2, 8) == ctypes.c_size_t(-1).value


def test_workspace_error_names_the_minimum(lib):
    """The preferred size includes split-K partials. A call is refused only below its
    minimum, and the message names that minimum. The call is refused before any device
    access, so the placeholder pointers are never dereferenced."""
    th = _theta(out=1152, inp=6912, r=16, ld_u=16, ld_v=16)
    minimum = binding.AQ_WORKSPACE_SYNC_BYTES + 64 * 16 * 2 + 16 * 6912 * 2
    assert lib.aq_linear_workspace_bytes(ctypes.byref(th), 1, 64) > minimum
    st = lib.aq_linear(ctypes.byref(th), 0x10000000, 64, 6912, 0x20000000, 1152, 0x30000000, minimum - 256, None)
    assert st == binding.AQ_ERR_WORKSPACE
    assert str(minimum) in binding.aq_last_error()


def test_workspace_bytes_split_k(lib):
    """A down-like projection (1152 x 6912) at 64 tokens may split its K (at most 16
    slices: 108 k blocks, 5 output tiles of 256 rows at the fewest). The workspace then
    also holds, after the rest, fp32 partial sums per slice: [M][round_up(out, 4)] of W0 x
    and [M][sum round_up(r, 8)] of x V. Ranks above 16 never split."""
    sync = binding.AQ_WORKSPACE_SYNC_BYTES
    M, slices = 64, 16
    th = _theta(out=1152, inp=6912, r=16, ld_u=16, ld_v=16)
    base = sync + 64 * 16 * 2 + 16 * 6912 * 2            # t bf16, V^T (both whole 256-B units)
    assert lib.aq_linear_workspace_bytes(ctypes.byref(th), 1, M) == base + slices * M * (1152 + 16) * 4
    th0 = _theta(out=1152, inp=6912, r=0)
    assert lib.aq_linear_workspace_bytes(ctypes.byref(th0), 1, M) == slices * M * 1152 * 4
    th64 = _theta(out=1152, inp=6912, r=64, ld_u=64, ld_v=64)
    assert lib.aq_linear_workspace_bytes(ctypes.byref(th64), 1, M) == sync + 64 * 64 * 2 + 64 * 6912 * 2
    # many output tiles (8192 tokens): nothing to split
    assert lib.aq_linear_workspace_bytes(ctypes.byref(th0), 1, 8192) == 0


@pytest.mark.parametrize("kw,status", [
    (dict(r=257), binding.AQ_ERR_UNSUPPORTED),
    (dict(r=-1), binding.AQ_ERR_SHAPE),
    (dict(out=0), binding.AQ_ERR_SHAPE),
    (dict(ld_w0=16), binding.AQ_ERR_SHAPE),
    (dict(ld_w0=36), binding.AQ_ERR_ALIGNMENT),
    (dict(W0=0x1008), binding.AQ_ERR_ALIGNMENT),
    (dict(U=0), binding.AQ_ERR_INVALID_ARG),
    (dict(ld_u=2), binding.AQ_ERR_SHAPE),
    (dict(ld_v=12), binding.AQ_ERR_ALIGNMENT),
    (dict(s=0), binding.AQ_ERR_INVALID_ARG),
])
def test_theta_validation(lib, kw, status):
    assert _linear(lib, _theta(**kw)) == status
    assert binding.aq_last_error()


@pytest.mark.parametrize("kw,status", [
    (dict(M=-1), binding.AQ_ERR_SHAPE),
    (dict(x=0), binding.AQ_ERR_INVALID_ARG),
    (dict(ldx=16), binding.AQ_ERR_SHAPE),
    (dict(ldx=36), binding.AQ_ERR_ALIGNMENT),
    (dict(y=0), binding.AQ_ERR_INVALID_ARG),
    (dict(ldy=40), binding.AQ_ERR_SHAPE),
    (dict(y=0x200004), binding.AQ_ERR_ALIGNMENT),
    (dict(ws=0), binding.AQ_ERR_WORKSPACE),
    (dict(ws_bytes=16), binding.AQ_ERR_WORKSPACE),
    (dict(ws=0x300010), binding.AQ_ERR_WORKSPACE),
    (dict(y=0x100000 + 64), binding.AQ_ERR_OVERLAP),      # y inside x
    (dict(y=0x1000), binding.AQ_ERR_OVERLAP),             # y on W0
    (dict(ws=0x200000 + 256), binding.AQ_ERR_OVERLAP),    # workspace inside y
])
def test_call_validation(lib, kw, status):
    assert _linear(lib, _theta(), **kw) == status, binding.aq_last_error()


def test_m_zero_is_noop(lib):
    assert _linear(lib, _theta(), M=0, x=0, y=0, ws=0, ws_bytes=0) == binding.AQ_OK


def test_qkv_validation(lib):
    th = (binding.c_theta * 3)(_theta(out=16, r=4, W0=0x10000), _theta(out=8, r=4, W0=0x20000),
                               _theta(out=8, r=4, W0=0x30000))
    ys = (ctypes.c_void_p * 3)(0x200000, 0x200000 + 32, 0x200000 + 48)
    ld = (ctypes.c_int64 * 3)(32, 32, 32)
    # column slices of one [M, 32] buffer at 0/16/24 overlap: 16-wide q slice covers columns 0..15
    ys_bad = (ctypes.c_void_p * 3)(0x200000, 0x200000 + 16, 0x200000 + 48)
    assert lib.aq_linear_qkv(th, 0x100000, 4, 32, ys_bad, ld, 0x300000, 1 << 20, None) == binding.AQ_ERR_OVERLAP
    th_in = (binding.c_theta * 3)(_theta(inp=32), _theta(inp=40, ld_w0=40), _theta(inp=32))
    assert lib.aq_linear_qkv(th_in, 0x100000, 4, 40, ys, ld, 0x300000, 1 << 20, None) == binding.AQ_ERR_SHAPE


def test_multi_validation(lib):
    th = (binding.c_theta * 3)(_theta(out=16, r=4, W0=0x10000), _theta(out=8, r=4, W0=0x20000),
                               _theta(out=8, r=4, W0=0x30000))
    ys = (ctypes.c_void_p * 3)(0x200000, 0x200000 + 32, 0x200000 + 48)
    ld = (ctypes.c_int64 * 3)(32, 32, 32)
    for n in (0, 4, -1):
        assert lib.aq_linear_multi(th, n, 0x100000, 4, 32, ys, ld, 0x300000, 1 << 20, None) == binding.AQ_ERR_INVALID_ARG
    assert "n=" in binding.aq_last_error()
    assert lib.aq_linear_multi(None, 2, 0x100000, 4, 32, ys, ld, 0x300000, 1 << 20, None) == binding.AQ_ERR_INVALID_ARG
    # two families whose outputs overlap are refused like aq_linear_qkv's
    ys_bad = (ctypes.c_void_p * 3)(0x200000, 0x200000 + 16, 0)
    assert lib.aq_linear_multi(th, 2, 0x100000, 4, 32, ys_bad, ld, 0x300000, 1 << 20, None) == binding.AQ_ERR_OVERLAP
    # n == 2 needs the workspace of the two bundles together; n outside [1, 3] is invalid
    invalid = ctypes.c_size_t(-1).value
    two, one = lib.aq_linear_workspace_bytes(th, 2, 100), lib.aq_linear_workspace_bytes(th, 1, 100)
    assert invalid not in (two, one) and two > one
    assert lib.aq_linear_workspace_bytes(th, 4, 100) == invalid
    assert lib.aq_linear_workspace_bytes(th, 0, 100) == invalid


def test_precompute_validation(lib):
    th = _theta()
    assert lib.aq_precompute(ctypes.byref(th), 0, 32, None) == binding.AQ_ERR_INVALID_ARG
    assert lib.aq_precompute(ctypes.byref(th), 0x500000, 16, None) == binding.AQ_ERR_SHAPE
    assert lib.aq_precompute(ctypes.byref(th), 0x1000 + 64, 32, None) == binding.AQ_ERR_OVERLAP


def test_path_setting(lib):
    assert lib.aq_set_path(7) == binding.AQ_ERR_INVALID_ARG
    assert lib.aq_set_path(binding.AQ_PATH_AUTO) == binding.AQ_OK


def test_selftest_argument_check(lib):
    assert lib.aq_selftest_bounded_wait(0, None) == binding.AQ_ERR_INVALID_ARG
    assert lib.aq_selftest_bounded_wait(2_000_000, None) == binding.AQ_ERR_INVALID_ARG
    th = binding.c_theta(W0=0x1000, s=0x2000, U=None, V=None, ld_w0=64, ld_u=0, ld_v=0, out=64, in_=64, r=0)
    for us in (0, 2_000_000):
        assert lib.aq_selftest_prefill_timeout(ctypes.byref(th), 0x3000, 4, 64, 0x4000, 64, 0x5000, 1 << 20, us,
                                               None) == binding.AQ_ERR_INVALID_ARG
    # r = 0: no t tiles to wait for
    assert lib.aq_selftest_prefill_timeout(ctypes.byref(th), 0x3000, 4, 64, 0x4000, 64, 0x5000, 1 << 20, 1000,
                                           None) == binding.AQ_ERR_INVALID_ARG


def _mlp_thetas(inter=256, inp=128, out=128, r=4, down_in=None):
    def th(o, i, W0):
        return binding.c_theta(W0=W0, s=W0 + 0x100000, U=W0 + 0x200000, V=W0 + 0x300000, ld_w0=i, ld_u=8, ld_v=8,
                               out=o, in_=i, r=r)
    return th(inter, inp, 0x1000000), th(inter, inp, 0x2000000), th(out, down_in or inter, 0x3000000)


def _mlp(lib, g, u, d, act=binding.AQ_ACT_GELU_TANH, x=0x4000000, M=2, ldx=128, y=0x5000000, ldy=128,
         ws=0x6000000, ws_bytes=1 << 20):
    return lib.aq_mlp(ctypes.byref(g), ctypes.byref(u), ctypes.byref(d), act, x, M, ldx, y, ldy, ws, ws_bytes, None)


def test_mlp_validation(lib):
    """aq_mlp refuses bad calls before any device work: the families' shapes must chain
    (gate and up [inter, in], down [out, inter]), the activation must be known, and the
    workspace must hold g and u besides the projections' own scratch."""
    g, u, d = _mlp_thetas()
    assert _mlp(lib, *_mlp_thetas(down_in=200)) == binding.AQ_ERR_SHAPE
    assert "down.in" in binding.aq_last_error()
    g2, _, _ = _mlp_thetas(inp=64)
    assert _mlp(lib, g2, u, d) == binding.AQ_ERR_SHAPE
    assert _mlp(lib, g, u, d, act=9) == binding.AQ_ERR_INVALID_ARG
    assert "activation" in binding.aq_last_error()
    need = lib.aq_mlp_workspace_bytes(ctypes.byref(g), ctypes.byref(u), ctypes.byref(d), 2)
    # g and u in bf16 at least, plus what the projections need
    assert need >= 2 * 2 * 256 * 2
    assert need > lib.aq_mlp_workspace_bytes(ctypes.byref(g), ctypes.byref(u), ctypes.byref(d), 1)
    assert _mlp(lib, g, u, d, ws_bytes=need - 256) == binding.AQ_ERR_WORKSPACE
    assert _mlp(lib, g, u, d, x=0) == binding.AQ_ERR_INVALID_ARG
