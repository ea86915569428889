"""Shared test helpers: moving seeded bf16 bit arrays to and from the GPU."""
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
