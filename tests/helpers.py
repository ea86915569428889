"""Shared test helpers: moving seeded bf16 bit arrays to and from the GPU."""
import inspect

import numpy as np

from rank_weight_reconstruction_gb300 import synth


def dev(bits):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def bits(t):
    import torch
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def host_f64(t):
    return synth.bf16_bits_to_f64(bits(t))


def dev_theta(th):
    """synth.Theta (host bit arrays) -> binding.Theta of device views."""
    from rank_weight_reconstruction_gb300 import Theta
    W0 = dev(th.W0)[:, : th.inp]
    s = dev(th.s)
    if th.r == 0:
        return Theta(W0=W0, s=s)
    return Theta(W0=W0, s=s, U=dev(th.U)[:, : th.r], V=dev(th.V)[:, : th.r])


def x_f64(xbits, inp):
    return synth.bf16_bits_to_f64(xbits)[:, :inp]


def close_over_rows(y, W0, s, U, V, xf, chunk=1024):
    """Acceptance of the whole output y [M, out] against the fp64 oracle, evaluated in row
    chunks so that large outputs need no [M, out] float64 reference at once. Returns the
    statistics oracle.error_stats gives for the full tensor (max |Δ|, max |y_ref|, relative
    L2), and whether they meet oracle.within_tolerance's bars."""
    import oracle
    max_err = max_ref = 0.0
    d2 = r2 = 0.0
    for m0 in range(0, xf.shape[0], chunk):
        ref = oracle.linear(W0, s, U, V, xf[m0:m0 + chunk])
        d = np.asarray(y[m0:m0 + chunk], dtype=np.float64) - ref
        max_err = max(max_err, float(np.max(np.abs(d))))
        max_ref = max(max_ref, float(np.max(np.abs(ref))))
        d2 += float(np.sum(d * d))
        r2 += float(np.sum(ref * ref))
    rel = (d2 ** 0.5) / (r2 ** 0.5) if r2 > 0 else d2 ** 0.5
    st = {"max_abs_err": max_err, "max_abs_ref": max_ref, "rel_l2": rel}
    bars = inspect.signature(oracle.within_tolerance).parameters
    ok = max_err <= bars["elem_tol"].default * max_ref and rel <= bars["l2_tol"].default
    return st, ok
