"""Banded sharing bookkeeping for a stack of layers of one projection family.

"How attnquant works" ("The theta bundle", "How the decomposition produces s, U, and V",
"The passthrough operating point"): each projection family stores one W0 per band of
layers (G bands over L layers; G = 1 shares one block across the stack, G = L gives
one block per layer), and every layer keeps its own s, U, V. Layer l uses band
floor(l * G / L) (contiguous bands). "Execution paths", "Precompute-outside": a layer
whose pieces do not match a shape-compatible W0 is an error that lists the offending
layers.
"""
from __future__ import annotations

from .binding import Theta


def band_of(layer: int, num_layers: int, num_blocks: int) -> int:
    if not (1 <= num_blocks <= num_layers) or not (0 <= layer < num_layers):
        raise ValueError(f"layer {layer} / {num_layers} layers / {num_blocks} blocks out of range")
    return (layer * num_blocks) // num_layers


class StackMismatchError(ValueError):
    """Raised when layers cannot be matched to a shape-compatible band block."""

    def __init__(self, layers, details):
        self.layers = list(layers)
        super().__init__(f"theta pieces of layers {self.layers} do not match their band's W0: "
                         + "; ".join(details))


class ThetaStack:
    """One projection family over L layers: ``blocks`` holds the G shared W0 tensors,
    ``layers`` the per-layer (s, U, V) tensors (U, V None for r = 0)."""

    def __init__(self, blocks, layers):
        self.blocks = list(blocks)
        self.layers = list(layers)
        L, G = len(self.layers), len(self.blocks)
        if L == 0 or not (1 <= G <= L):
            raise ValueError(f"need 1 <= G <= L, got G={G}, L={L}")
        bad, details = [], []
        for l, (s, U, V) in enumerate(self.layers):
            W0 = self.blocks[band_of(l, L, G)]
            out, inp = int(W0.size(0)), int(W0.size(1))
            msg = []
            if s is None or s.dim() != 1 or int(s.size(0)) != out:
                msg.append(f"s has shape {None if s is None else tuple(s.shape)}, want ({out},)")
            if (U is None) != (V is None):
                msg.append("U and V must both be given or both be None")
            elif U is not None:
                if U.dim() != 2 or int(U.size(0)) != out:
                    msg.append(f"U has shape {tuple(U.shape)}, want ({out}, r)")
                if V.dim() != 2 or int(V.size(0)) != inp:
                    msg.append(f"V has shape {tuple(V.shape)}, want ({inp}, r)")
                if U.dim() == 2 and V.dim() == 2 and int(U.size(1)) != int(V.size(1)):
                    msg.append(f"U rank {int(U.size(1))} != V rank {int(V.size(1))}")
            if msg:
                bad.append(l)
                details.append(f"layer {l} (band {band_of(l, L, G)}): " + ", ".join(msg))
        if bad:
            raise StackMismatchError(bad, details)

    @property
    def num_layers(self) -> int:
        return len(self.layers)

    @property
    def num_blocks(self) -> int:
        return len(self.blocks)

    def band(self, layer: int) -> int:
        return band_of(layer, self.num_layers, self.num_blocks)

    def theta(self, layer: int) -> Theta:
        s, U, V = self.layers[layer]
        return Theta(W0=self.blocks[self.band(layer)], s=s, U=U, V=V)
