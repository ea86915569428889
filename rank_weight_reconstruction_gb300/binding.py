"""ctypes binding of the C ABI in ``include/aq.h`` (argument marshalling only).

Every function here has the C entry point's name and does nothing but turn torch
tensors into device pointers, leading dimensions and the current CUDA stream, call the
library, and turn a non-zero ``aq_status`` into an exception. All arithmetic happens in
the CUDA kernels of ``libaq_gb300.so``; if that library is missing the first call raises.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

from . import build_lib

AQ_OK = 0
AQ_ERR_INVALID_ARG = 1
AQ_ERR_SHAPE = 2
AQ_ERR_ALIGNMENT = 3
AQ_ERR_UNSUPPORTED = 4
AQ_ERR_WORKSPACE = 5
AQ_ERR_OVERLAP = 6
AQ_ERR_CUDA = 7
AQ_ERR_TIMEOUT = 8
AQ_ERR_NUMERIC = 9
AQ_ERR_BOUNDS = 10
AQ_MAX_RANK = 256

AQ_PATH_AUTO = 0
AQ_PATH_DECODE = 1
AQ_PATH_PREFILL = 2
AQ_PATH_MIDM = 3
AQ_ACT_GELU_TANH = 0
AQ_ACT_SILU = 1
AQ_SF_LINEAR = 0
AQ_SF_128X4 = 1
AQ_NVFP4_SCALE_FROM_AMAX = 0
AQ_NVFP4_SCALE_GIVEN = 1

EXPORTED_SYMBOLS = [
    "aq_linear_workspace_bytes", "aq_linear", "aq_linear_qkv", "aq_precompute",
    "aq_device_status", "aq_selftest_bounded_wait", "aq_set_path", "aq_decode_max_m",
    "aq_last_path", "aq_last_launch_count", "aq_status_string", "aq_last_error",
    "aq_abi_version", "aq_linear_noalloc", "aq_linear_multi", "aq_noalloc_scratch_read",
    "aq_band_mean", "aq_ls_residual", "aq_randomized_svd_workspace_bytes", "aq_randomized_svd",
    "aq_mlp_workspace_bytes", "aq_mlp", "aq_precompute_nvfp4_workspace_bytes", "aq_precompute_nvfp4",
    "aq_selftest_prefill_timeout", "aq_checked_build", "aq_selftest_bounds_check",
]
AQ_MAX_FAMILIES = 3
AQ_NOALLOC_WORKSPACE_BYTES = 8 * 1024 * 1024
AQ_WORKSPACE_SYNC_BYTES = 128 * 1024


class AqError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{_status_name(status)}: {message}")
        self.status = status


class c_theta(ctypes.Structure):
    _fields_ = [
        ("W0", ctypes.c_void_p), ("ld_w0", ctypes.c_int64),
        ("s", ctypes.c_void_p),
        ("U", ctypes.c_void_p), ("ld_u", ctypes.c_int64),
        ("V", ctypes.c_void_p), ("ld_v", ctypes.c_int64),
        ("out", ctypes.c_int32), ("in_", ctypes.c_int32), ("r", ctypes.c_int32),
    ]


_lib = None


def library_path() -> str:
    return build_lib.LIB_PATH


def load(path: str | None = None) -> ctypes.CDLL:
    """Load libaq_gb300.so (built in-tree by ``build_lib.build()``)."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or library_path()
    if not os.path.exists(path):
        raise RuntimeError(
            f"{path} is missing: build it with rank_weight_reconstruction_gb300.build_lib.build() "
            "(there is no CPU fallback)")
    lib = ctypes.CDLL(path)
    vp, i64, i32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_size_t
    th_p = ctypes.POINTER(c_theta)
    lib.aq_linear_workspace_bytes.argtypes = [th_p, i32, i64]
    lib.aq_linear_workspace_bytes.restype = sz
    lib.aq_linear.argtypes = [th_p, vp, i64, i64, vp, i64, vp, sz, vp]
    lib.aq_linear.restype = ctypes.c_int
    lib.aq_linear_qkv.argtypes = [th_p, vp, i64, i64, ctypes.POINTER(vp), ctypes.POINTER(i64), vp, sz, vp]
    lib.aq_linear_qkv.restype = ctypes.c_int
    lib.aq_linear_multi.argtypes = [th_p, i32, vp, i64, i64, ctypes.POINTER(vp), ctypes.POINTER(i64), vp, sz, vp]
    lib.aq_linear_multi.restype = ctypes.c_int
    lib.aq_linear_noalloc.argtypes = [th_p, vp, i64, i64, vp, i64, vp]
    lib.aq_linear_noalloc.restype = ctypes.c_int
    lib.aq_noalloc_scratch_read.argtypes = [vp, sz, sz, vp]
    lib.aq_noalloc_scratch_read.restype = ctypes.c_int
    lib.aq_mlp_workspace_bytes.argtypes = [th_p, th_p, th_p, i64]
    lib.aq_mlp_workspace_bytes.restype = sz
    lib.aq_mlp.argtypes = [th_p, th_p, th_p, ctypes.c_int, vp, i64, i64, vp, i64, vp, sz, vp]
    lib.aq_mlp.restype = ctypes.c_int
    lib.aq_band_mean.argtypes = [ctypes.POINTER(vp), i32, i32, i32, i64, vp, i64, vp]
    lib.aq_band_mean.restype = ctypes.c_int
    lib.aq_ls_residual.argtypes = [vp, i64, vp, i64, i32, i32, vp, vp, i64, vp]
    lib.aq_ls_residual.restype = ctypes.c_int
    lib.aq_randomized_svd_workspace_bytes.argtypes = [i32, i32, i32, i32]
    lib.aq_randomized_svd_workspace_bytes.restype = sz
    lib.aq_randomized_svd.argtypes = [vp, i64, i32, i32, i32, vp, i64, i32, i32, vp, i64, vp, i64, vp, sz, vp]
    lib.aq_randomized_svd.restype = ctypes.c_int
    lib.aq_precompute.argtypes = [th_p, vp, i64, vp]
    lib.aq_precompute.restype = ctypes.c_int
    lib.aq_precompute_nvfp4_workspace_bytes.argtypes = []
    lib.aq_precompute_nvfp4_workspace_bytes.restype = sz
    lib.aq_precompute_nvfp4.argtypes = [th_p, vp, i64, vp, ctypes.c_int, vp, ctypes.c_int, vp, sz, vp]
    lib.aq_precompute_nvfp4.restype = ctypes.c_int
    lib.aq_device_status.argtypes = [vp]
    lib.aq_device_status.restype = ctypes.c_int
    lib.aq_selftest_bounded_wait.argtypes = [ctypes.c_uint32, vp]
    lib.aq_selftest_bounded_wait.restype = ctypes.c_int
    lib.aq_selftest_prefill_timeout.argtypes = [th_p, vp, i64, i64, vp, i64, vp, sz, ctypes.c_uint32, vp]
    lib.aq_selftest_prefill_timeout.restype = ctypes.c_int
    lib.aq_checked_build.argtypes = []
    lib.aq_checked_build.restype = ctypes.c_int32
    lib.aq_selftest_bounds_check.argtypes = [vp]
    lib.aq_selftest_bounds_check.restype = ctypes.c_int
    lib.aq_set_path.argtypes = [ctypes.c_int]
    lib.aq_set_path.restype = ctypes.c_int
    for name in ("aq_decode_max_m", "aq_last_path", "aq_last_launch_count", "aq_abi_version"):
        getattr(lib, name).argtypes = []
        getattr(lib, name).restype = i32
    lib.aq_status_string.argtypes = [ctypes.c_int]
    lib.aq_status_string.restype = ctypes.c_char_p
    lib.aq_last_error.argtypes = []
    lib.aq_last_error.restype = ctypes.c_char_p
    _lib = lib
    return lib


def _status_name(st: int) -> str:
    names = {0: "AQ_OK", 1: "AQ_ERR_INVALID_ARG", 2: "AQ_ERR_SHAPE", 3: "AQ_ERR_ALIGNMENT",
             4: "AQ_ERR_UNSUPPORTED", 5: "AQ_ERR_WORKSPACE", 6: "AQ_ERR_OVERLAP", 7: "AQ_ERR_CUDA",
             8: "AQ_ERR_TIMEOUT"}
    return names.get(st, f"status {st}")


def _check(st: int) -> None:
    if st != AQ_OK:
        msg = load().aq_last_error().decode(errors="replace")
        raise AqError(st, msg)


# ----------------------------------------------------------------------------------
# tensor marshalling
# ----------------------------------------------------------------------------------
def _ptr(t) -> int:
    return 0 if t is None else int(t.data_ptr())


def _ld(t) -> int:
    """Leading dimension (elements) of a row-major 2-D bf16 tensor or view."""
    import torch
    if t.dtype != torch.bfloat16:
        raise TypeError(f"expected a bfloat16 tensor, got {t.dtype}")
    if t.dim() != 2 or (t.size(1) > 1 and t.stride(1) != 1):
        raise ValueError("expected a 2-D row-major tensor (unit column stride)")
    return int(t.stride(0)) if t.size(0) > 1 else int(max(t.stride(0), t.size(1)))


def _ld_any(t) -> int:
    """Leading dimension (elements) of a row-major 2-D tensor of any dtype."""
    if t.dim() != 2 or (t.size(1) > 1 and t.stride(1) != 1):
        raise ValueError("expected a 2-D row-major tensor (unit column stride)")
    return int(t.stride(0)) if t.size(0) > 1 else int(max(t.stride(0), t.size(1)))


def _stream(stream) -> int:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


@dataclass
class Theta:
    """A theta bundle on the device: W0 [out, in], s [out], U [out, r], V [in, r], each a
    bf16 tensor (views with padded leading dimensions are fine); U, V None when r == 0."""
    W0: object
    s: object
    U: object = None
    V: object = None

    @property
    def out(self) -> int:
        return int(self.W0.size(0))

    @property
    def inp(self) -> int:
        return int(self.W0.size(1))

    @property
    def r(self) -> int:
        return 0 if self.U is None else int(self.U.size(1))

    def c(self) -> c_theta:
        r = self.r
        return c_theta(
            W0=_ptr(self.W0), ld_w0=_ld(self.W0), s=_ptr(self.s),
            U=_ptr(self.U) if r else 0, ld_u=_ld(self.U) if r else 0,
            V=_ptr(self.V) if r else 0, ld_v=_ld(self.V) if r else 0,
            out=self.out, in_=self.inp, r=r)


def aq_linear_workspace_bytes(thetas, M: int) -> int:
    ths = [thetas] if isinstance(thetas, Theta) else list(thetas)
    arr = (c_theta * len(ths))(*[t.c() for t in ths])
    n = load().aq_linear_workspace_bytes(arr, len(ths), int(M))
    if n == ctypes.c_size_t(-1).value:
        raise AqError(AQ_ERR_INVALID_ARG, "aq_linear_workspace_bytes: invalid arguments")
    return int(n)


def _padded_empty(rows: int, cols: int, device):
    """[rows, cols] bf16 view of a buffer whose leading dimension is a multiple of 8
    (the ABI wants 16-byte aligned rows)."""
    import torch
    ld = (cols + 7) // 8 * 8
    return torch.empty(rows, ld, dtype=torch.bfloat16, device=device)[:, :cols]


def new_workspace(nbytes: int, device):
    """A workspace for aq_linear / aq_linear_qkv: zero-filled (its sync part must start
    at zero; the library keeps it zero), 256-byte aligned (torch's caching allocator
    returns 512-byte aligned blocks). Reuse it across calls on one stream."""
    import torch
    if nbytes == 0:
        return None
    return torch.zeros(nbytes, dtype=torch.uint8, device=device)


_workspace = new_workspace


def aq_linear(theta: Theta, x, y=None, workspace=None, stream=None):
    """y = s * (W0 x) + U (V^T x) for x [M, in] -> y [M, out] (bf16)."""
    import torch
    M = int(x.size(0))
    if y is None:
        y = _padded_empty(M, theta.out, x.device)
    nbytes = aq_linear_workspace_bytes(theta, M)
    if workspace is None:
        workspace = _workspace(nbytes, x.device)
    th = theta.c()
    _check(load().aq_linear(ctypes.byref(th), _ptr(x), M, _ld(x), _ptr(y), _ld(y), _ptr(workspace),
                            0 if workspace is None else workspace.numel() * workspace.element_size(),
                            _stream(stream)))
    return y


def aq_linear_noalloc(theta: Theta, x, y=None, stream=None):
    """aq_linear without a workspace argument: the library's built-in scratch array is
    used, so the library itself allocates nothing (y is allocated here only if not
    given)."""
    M = int(x.size(0))
    if y is None:
        y = _padded_empty(M, theta.out, x.device)
    th = theta.c()
    _check(load().aq_linear_noalloc(ctypes.byref(th), _ptr(x), M, _ld(x), _ptr(y), _ld(y), _stream(stream)))
    return y


def aq_linear_qkv(thetas, x, ys=None, workspace=None, stream=None):
    """The q, k, v projections over one x in one pass; returns the three outputs."""
    import torch
    thetas = list(thetas)
    assert len(thetas) == 3
    M = int(x.size(0))
    if ys is None:
        ys = [_padded_empty(M, t.out, x.device) for t in thetas]
    nbytes = aq_linear_workspace_bytes(thetas, M)
    if workspace is None:
        workspace = _workspace(nbytes, x.device)
    arr = (c_theta * 3)(*[t.c() for t in thetas])
    yp = (ctypes.c_void_p * 3)(*[_ptr(y) for y in ys])
    ldy = (ctypes.c_int64 * 3)(*[_ld(y) for y in ys])
    _check(load().aq_linear_qkv(arr, _ptr(x), M, _ld(x), yp, ldy, _ptr(workspace),
                                0 if workspace is None else workspace.numel() * workspace.element_size(),
                                _stream(stream)))
    return ys


def aq_linear_multi(thetas, x, ys=None, workspace=None, stream=None):
    """1..3 projections sharing one x (e.g. gate and up) in one pass; returns the outputs."""
    thetas = list(thetas)
    n = len(thetas)
    M = int(x.size(0))
    if ys is None:
        ys = [_padded_empty(M, t.out, x.device) for t in thetas]
    nbytes = aq_linear_workspace_bytes(thetas, M)
    if workspace is None:
        workspace = _workspace(nbytes, x.device)
    arr = (c_theta * max(1, n))(*[t.c() for t in thetas])
    yp = (ctypes.c_void_p * max(1, n))(*[_ptr(y) for y in ys])
    ldy = (ctypes.c_int64 * max(1, n))(*[_ld(y) for y in ys])
    _check(load().aq_linear_multi(arr, n, _ptr(x), M, _ld(x), yp, ldy, _ptr(workspace),
                                  0 if workspace is None else workspace.numel() * workspace.element_size(),
                                  _stream(stream)))
    return ys


def aq_precompute(theta: Theta, W_eff=None, stream=None):
    """W_eff = diag(s) W0 + U V^T as a bf16 [out, in] tensor."""
    import torch
    if W_eff is None:
        W_eff = _padded_empty(theta.out, theta.inp, theta.W0.device)
    th = theta.c()
    _check(load().aq_precompute(ctypes.byref(th), _ptr(W_eff), _ld(W_eff), _stream(stream)))
    return W_eff


def nvfp4_scale_bytes(out: int, inp: int, layout: int) -> int:
    """Bytes of the block-scale array of an [out, inp] weight in the given layout."""
    if layout == AQ_SF_LINEAR:
        return out * (inp // 16)
    return -(-out // 128) * 128 * (-(-(inp // 16) // 4) * 4)


def aq_precompute_nvfp4(theta: Theta, sf_layout: int = AQ_SF_LINEAR, global_scale=None, scale_given=None,
                        q=None, sf=None, workspace=None, stream=None):
    """W_eff quantized to NVFP4 without forming it in bf16: returns (q, sf, global_scale) with
    q a uint8 [out, in/2] tensor of E2M1 code pairs, sf the uint8 E4M3 block scales (a 2-D
    [out, in/16] tensor for AQ_SF_LINEAR, a flat tensor for AQ_SF_128X4) and global_scale a
    one-element float32 device tensor. With ``scale_given`` (default: whether
    ``global_scale`` is passed) the scale in ``global_scale`` is used; otherwise it is
    computed from max|W_eff| and written to ``global_scale`` (allocated if None)."""
    import torch
    dev = theta.W0.device
    if q is None:
        q = torch.empty(theta.out, theta.inp // 2, dtype=torch.uint8, device=dev)
    if sf is None:
        n = nvfp4_scale_bytes(theta.out, theta.inp, sf_layout)
        sf = torch.empty(n, dtype=torch.uint8, device=dev)
        if sf_layout == AQ_SF_LINEAR:
            sf = sf.view(theta.out, theta.inp // 16)
    given = (global_scale is not None) if scale_given is None else bool(scale_given)
    if global_scale is None:
        if given:
            raise ValueError("scale_given needs a global_scale tensor")
        global_scale = torch.empty(1, dtype=torch.float32, device=dev)
    if workspace is None and not given:
        workspace = torch.empty(int(load().aq_precompute_nvfp4_workspace_bytes()), dtype=torch.uint8, device=dev)
    th = theta.c()
    _check(load().aq_precompute_nvfp4(
        ctypes.byref(th), _ptr(q), _ld_any(q), _ptr(sf), int(sf_layout), _ptr(global_scale),
        AQ_NVFP4_SCALE_GIVEN if given else AQ_NVFP4_SCALE_FROM_AMAX, _ptr(workspace),
        0 if workspace is None else workspace.numel() * workspace.element_size(), _stream(stream)))
    return q, sf, global_scale


def aq_device_status(stream=None) -> int:
    """Synchronises the stream and returns (and clears) the device status word."""
    return int(load().aq_device_status(_stream(stream)))


def aq_selftest_bounded_wait(timeout_us: int, stream=None) -> None:
    _check(load().aq_selftest_bounded_wait(int(timeout_us), _stream(stream)))


def aq_selftest_prefill_timeout(theta: Theta, x, timeout_us: int, y=None, workspace=None, stream=None):
    """aq_linear on the prefill GEMM with its t-flag wait made unreachable (test hook)."""
    M = int(x.shape[0])
    if y is None:
        y = _padded_empty(M, theta.out, x.device)
    if workspace is None:
        workspace = new_workspace(aq_linear_workspace_bytes(theta, M), x.device)
    th = theta.c()
    _check(load().aq_selftest_prefill_timeout(ctypes.byref(th), _ptr(x), M, _ld(x), _ptr(y), _ld(y), _ptr(workspace),
                                              workspace.numel() * workspace.element_size(), int(timeout_us),
                                              _stream(stream)))
    return y


def aq_set_path(path: int) -> None:
    _check(load().aq_set_path(int(path)))


def aq_decode_max_m() -> int:
    return int(load().aq_decode_max_m())


def aq_last_path() -> int:
    return int(load().aq_last_path())


def aq_last_launch_count() -> int:
    return int(load().aq_last_launch_count())


def aq_abi_version() -> int:
    return int(load().aq_abi_version())


def aq_last_error() -> str:
    return load().aq_last_error().decode(errors="replace")


def aq_status_string(st: int) -> str:
    return load().aq_status_string(int(st)).decode()


# ----------------------------------------------------------------------------------
# the decomposition (load time): band mean, least-squares scale and residual, randomized SVD
# ----------------------------------------------------------------------------------
def aq_band_mean(weights, W0=None, stream=None):
    """W0 = RN_bf16(mean of the band's bf16 [out, in] weights), on the GPU."""
    import torch
    weights = list(weights)
    out, inp = int(weights[0].size(0)), int(weights[0].size(1))
    ld = _ld(weights[0])
    for w in weights:
        assert w.shape == weights[0].shape and _ld(w) == ld, "band weights must share shape and row stride"
    if W0 is None:
        W0 = _padded_empty(out, inp, weights[0].device)
    ptrs = (ctypes.c_void_p * len(weights))(*[_ptr(w) for w in weights])
    _check(load().aq_band_mean(ptrs, len(weights), out, inp, ld, _ptr(W0), _ld(W0), _stream(stream)))
    return W0


def aq_ls_residual(weight, W0, s=None, resid=None, stream=None):
    """s = RN_bf16(per-row least-squares scale of W0 toward weight) and resid = weight − s·W0
    (float64), on the GPU. Returns (s, resid)."""
    import torch
    out, inp = int(weight.size(0)), int(weight.size(1))
    if s is None:
        s = torch.empty(out, dtype=torch.bfloat16, device=weight.device)
    if resid is None:
        resid = torch.empty(out, inp, dtype=torch.float64, device=weight.device)
    _check(load().aq_ls_residual(_ptr(weight), _ld(weight), _ptr(W0), _ld(W0), out, inp, _ptr(s), _ptr(resid),
                                 _ld_any(resid), _stream(stream)))
    return s, resid


def aq_randomized_svd(A, r, omega, power_iters=0, U=None, V=None, stream=None):
    """Rank-r factors (U [m, r], V [n, r], bf16) of the float64 matrix A by the randomized SVD
    with the caller's test matrix omega [n, k] (float64), on the GPU."""
    import torch
    m, n = int(A.size(0)), int(A.size(1))
    k = int(omega.size(1))
    if U is None:
        U = _padded_empty(m, r, A.device) if r > 0 else torch.empty(m, 0, dtype=torch.bfloat16, device=A.device)
    if V is None:
        V = _padded_empty(n, r, A.device) if r > 0 else torch.empty(n, 0, dtype=torch.bfloat16, device=A.device)
    need = load().aq_randomized_svd_workspace_bytes(m, n, k, r)
    if need == ctypes.c_size_t(-1).value:
        raise AqError(AQ_ERR_SHAPE, f"aq_randomized_svd: bad sizes m={m} n={n} k={k} r={r}")
    ws = torch.empty(max(int(need), 16), dtype=torch.uint8, device=A.device)
    _check(load().aq_randomized_svd(_ptr(A), _ld_any(A), m, n, r, _ptr(omega), _ld_any(omega), k, power_iters,
                                    _ptr(U) if r > 0 else None, _ld(U) if r > 0 else max(r, 1),
                                    _ptr(V) if r > 0 else None, _ld(V) if r > 0 else max(r, 1),
                                    _ptr(ws), ws.numel(), _stream(stream)))
    return U, V


def aq_mlp_workspace_bytes(gate: Theta, up: Theta, down: Theta, M: int) -> int:
    g, u, d = gate.c(), up.c(), down.c()
    return int(load().aq_mlp_workspace_bytes(ctypes.byref(g), ctypes.byref(u), ctypes.byref(d), M))


def aq_mlp(gate: Theta, up: Theta, down: Theta, x, act=AQ_ACT_GELU_TANH, y=None, workspace=None, stream=None):
    """y = down(act(gate(x)) * up(x)) with every projection a reconstruction linear."""
    M = int(x.size(0))
    if y is None:
        y = _padded_empty(M, down.out, x.device)
    if workspace is None:
        workspace = new_workspace(max(aq_mlp_workspace_bytes(gate, up, down, M), 256), x.device)
    g, u, d = gate.c(), up.c(), down.c()
    _check(load().aq_mlp(ctypes.byref(g), ctypes.byref(u), ctypes.byref(d), int(act), _ptr(x), M, _ld(x), _ptr(y),
                         _ld(y), _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))
    return y
