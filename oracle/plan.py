"""Oracle patch plan: band boundaries of a spatial split.

TEST INFRASTRUCTURE ONLY (see the package header).

Band rule (DistVAE PR #14 "Add tiled VAE parallelism & extended model support", Patchify
commit): bands are cut in whole multiples of the factor by which the VAE widens the axis, no
rows are invented, and when the count does not divide, the first bands get one extra row.  At a
layer of scale s the band edges are s times the latent edges.  A patch narrower than the
kernel's reach is refused (narrow-patch commit of the same page).

Parity: pinned by the CPU tests (sizes sum to the extent, differ by at most one, the larger ones
come first; the refusal case).
"""
from __future__ import annotations

from typing import List


class PatchTooNarrow(ValueError):
    """A patch narrower than the convolution's reach; carries rows and reach as fields."""

    def __init__(self, rows: int, reach: int):
        super().__init__(f"patch of {rows} rows is narrower than the kernel reach {reach}")
        self.rows = rows
        self.reach = reach


def band_sizes(length: int, n: int) -> List[int]:
    """Sizes of n bands over ``length`` latent rows: the first length % n get ceil, the rest floor."""
    if n < 1:
        raise ValueError("need at least one patch")
    q, r = divmod(length, n)
    return [q + 1 if i < r else q for i in range(n)]


def band_edges(length: int, n: int, scale: int = 1, reach: int = 1) -> List[int]:
    """Edges [0, e1, ..., length*scale] of n bands at a layer of the given scale."""
    sizes = band_sizes(length, n)
    for s in sizes:
        if s * scale < reach:
            raise PatchTooNarrow(s * scale, reach)
    edges = [0]
    for s in sizes:
        edges.append(edges[-1] + s * scale)
    return edges
