"""Banded-sharing bookkeeping (rank_weight_reconstruction_gb300/stack.py) on the CPU: which
band's W0 each layer uses, and the error that lists the layers whose pieces do not fit it.
"""
import pytest
import torch

import oracle
from rank_weight_reconstruction_gb300.stack import StackMismatchError, ThetaStack, band_of


def _stack(L, G, out=6, inp=4, r=2, broken=None):
    """G blocks [out, inp] and L layers (s, U, V); `broken` maps a layer to the piece to
    give the wrong shape ("s", "U", "V", "rank", "half")."""
    broken = broken or {}
    blocks = [torch.full((out, inp), float(b)) for b in range(G)]
    layers = []
    for l in range(L):
        s, U, V = torch.ones(out), torch.zeros(out, r), torch.zeros(inp, r)
        kind = broken.get(l)
        if kind == "s":
            s = torch.ones(out + 1)
        elif kind == "U":
            U = torch.zeros(out - 1, r)
        elif kind == "V":
            V = torch.zeros(inp + 2, r)
        elif kind == "rank":
            V = torch.zeros(inp, r + 1)
        elif kind == "half":
            V = None
        layers.append((s, U, V))
    return blocks, layers


@pytest.mark.parametrize("L,G", [(26, 1), (26, 26), (60, 4), (7, 3), (5, 2)])
def test_bands_match_the_oracle(L, G):
    assert [band_of(l, L, G) for l in range(L)] == [oracle.band_of_layer(l, L, G) for l in range(L)]


def test_sixty_layers_in_four_bands_of_fifteen():
    stack = ThetaStack(*_stack(60, 4))
    assert [sum(stack.band(l) == b for l in range(60)) for b in range(4)] == [15] * 4
    for l in (0, 14, 15, 59):
        th = stack.theta(l)
        assert th.W0 is stack.blocks[l // 15]        # shared by pointer, not copied
        assert th.s is stack.layers[l][0] and th.r == 2


def test_passthrough_gives_every_layer_its_own_block():
    stack = ThetaStack(*_stack(5, 5))
    assert [stack.theta(l).W0 is stack.blocks[l] for l in range(5)] == [True] * 5


def test_rank_zero_layers():
    blocks, layers = _stack(3, 1)
    layers = [(s, None, None) for s, _, _ in layers]
    stack = ThetaStack(blocks, layers)
    assert stack.theta(2).r == 0


def test_mismatch_lists_every_offending_layer():
    broken = {1: "s", 4: "U", 5: "V", 8: "rank", 9: "half"}
    with pytest.raises(StackMismatchError) as e:
        ThetaStack(*_stack(10, 2, broken=broken))
    assert e.value.layers == sorted(broken)
    msg = str(e.value)
    for l in broken:
        assert f"layer {l} (band {l * 2 // 10})" in msg


def test_band_counts_out_of_range():
    with pytest.raises(ValueError):
        ThetaStack(*_stack(3, 4))
    with pytest.raises(ValueError):
        band_of(3, 3, 1)
    with pytest.raises(ValueError):
        band_of(0, 3, 0)
