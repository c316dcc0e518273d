"""Oracle tile plan, blend ramps, overlap blend and sequential tiled decode.

TEST INFRASTRUCTURE ONLY (see the package header).

What it follows:
  * TensorRT-LLM PR #15753 "LTX-2 tile-parallel VAE decode", Approach: tiled decode runs over
    overlapping spatial/temporal tiles; each tile is decoded on its own, weighted by a blend
    mask assembled from 1-D parts, summed into a full-size buffer next to a weight buffer, and
    the buffer is divided by the weights.
  * vllm-omni PR #4831 "VAE tiling parallel encode for LTX-2": an LTX-2.5 grid of a 576 px
    frame with tile 512 and stride 448 is 2 x 2.

Readings (the pages give neither the start rule nor the ramp):
  * per axis, starts 0, stride, 2 stride, ... (stride = tile - overlap) up to the first tile
    that reaches the end; the last tile is clipped;
  * spatial pixels of a tile: [s*a0, s*(a0+n)); temporal pixel frames of a causal tile starting
    at latent frame t0 with n frames: [st*t0, st*(t0+n-1)] (its first latent frame decodes to one
    frame), so consecutive temporal tiles overlap by st*(overlap-1)+1 frames;
  * on an edge shared with a neighbour, over the P-pixel overlap the weight rises as
    (y+1)/(P+1) (or falls as its mirror); elsewhere it is 1; image borders get no ramp; the tile
    weight is the outer product of the three 1-D ramps;
  * out = sum_i w_i x_i / sum_i w_i, tiles in raster order (t, h, w).

Parity: pinned by the CPU tests (2-tile ramps sum to one, a single tile reproduces the untiled
decode, constant tiles blend to the constant, the 576 px LTX-2.5 grid, brute-force blend).
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional, Sequence, Tuple

import numpy as np

from . import decoder


def axis_tiles(length: int, tile: int, overlap: int) -> List[Tuple[int, int]]:
    """(start, extent) of each tile along one axis, latent units."""
    stride = tile - overlap
    assert stride > 0 and length > 0
    starts = [0]
    while starts[-1] + tile < length:
        starts.append(starts[-1] + stride)
    return [(s, min(tile, length - s)) for s in starts]


@dataclasses.dataclass
class Tile:
    lat: Tuple[int, int, int, int, int, int]   # t0, nt, h0, nh, w0, nw (latent)
    pix: Tuple[int, int, int, int, int, int]   # t0, nt, h0, nh, w0, nw (pixels)
    ovl: Tuple[int, int, int, int, int, int]   # P before / after, per axis t, h, w (pixels)


def _pix(axis: str, a0: int, n: int, scale: int, causal: bool) -> Tuple[int, int]:
    if axis == "t" and causal:
        return scale * a0, scale * (n - 1) + 1
    return scale * a0, scale * n


def tile_plan(lat_thw: Sequence[int], tile_thw: Sequence[int], ovl_thw: Sequence[int],
              scale_t: int, scale_s: int, causal_t: bool = True) -> List[Tile]:
    axes = []
    for k, (name, sc) in enumerate((("t", scale_t), ("h", scale_s), ("w", scale_s))):
        at = axis_tiles(lat_thw[k], tile_thw[k], ovl_thw[k])
        px = [_pix(name, a0, n, sc, causal_t) for a0, n in at]
        ov = []
        for i, (p0, pn) in enumerate(px):
            lo = (px[i - 1][0] + px[i - 1][1] - p0) if i > 0 else 0
            hi = (p0 + pn - px[i + 1][0]) if i + 1 < len(px) else 0
            ov.append((lo, hi))
        axes.append(list(zip(at, px, ov)))
    tiles = []
    for (lt, pt, ot) in axes[0]:
        for (lh, ph, oh) in axes[1]:
            for (lw, pw, ow) in axes[2]:
                tiles.append(Tile(lat=lt + lh + lw, pix=pt + ph + pw, ovl=ot + oh + ow))
    return tiles


def ramp(n: int, p_lo: int, p_hi: int) -> np.ndarray:
    """1-D weight of a tile of n pixels with overlaps p_lo before and p_hi after."""
    w = np.ones(n, dtype=np.float64)
    for y in range(n):
        if y < p_lo:
            w[y] *= (y + 1) / (p_lo + 1)
        if y >= n - p_hi:
            w[y] *= (n - y) / (p_hi + 1)
    return w


def tile_weight(t: Tile) -> np.ndarray:
    _, nt, _, nh, _, nw = t.pix
    a, b, c, d, e, f = t.ovl
    return np.einsum("t,h,w->thw", ramp(nt, a, b), ramp(nh, c, d), ramp(nw, e, f))


def blend(tiles: Sequence[Tile], data: Sequence[np.ndarray], out_shape: Sequence[int],
          frames: Optional[Tuple[int, int]] = None) -> np.ndarray:
    """sum_i w_i x_i / sum_i w_i in float64, raster order.  data[i] is [B, C, nt, nh, nw].

    frames = (f0, f1): form only output frames f0 .. f1-1 (every tile keeps its whole weight; a
    tile not covering those frames contributes nothing and its data may be None)."""
    f0, f1 = frames if frames is not None else (0, out_shape[2])
    shape = (out_shape[0], out_shape[1], f1 - f0) + tuple(out_shape[3:])
    acc = np.zeros(shape, dtype=np.float64)
    wsum = np.zeros(shape[2:], dtype=np.float64)
    for t, x in zip(tiles, data):
        t0, nt, h0, nh, w0, nw = t.pix
        a, b = max(t0, f0), min(t0 + nt, f1)
        if a >= b:
            continue
        wt = tile_weight(t)[a - t0:b - t0]
        acc[:, :, a - f0:b - f0, h0:h0 + nh, w0:w0 + nw] += wt * x[:, :, a - t0:b - t0].astype(np.float64)
        wsum[a - f0:b - f0, h0:h0 + nh, w0:w0 + nw] += wt
    return acc / wsum


def tiled_decode(cfg, params: dict, latent: np.ndarray, tile_thw, ovl_thw, tier: str = "A"):
    """Sequential tiled decode: each tile decoded causally on its own, then blended."""
    st, sh, sw = cfg.scale()
    assert sh == sw
    b, _, t, h, w = latent.shape
    plan = tile_plan((t, h, w), tile_thw, ovl_thw, st, sh)
    outs = []
    for tl in plan:
        t0, nt, h0, nh, w0, nw = tl.lat
        outs.append(decoder.decode(cfg, params, latent[:, :, t0:t0 + nt, h0:h0 + nh, w0:w0 + nw], tier=tier))
    return blend(plan, outs, cfg.output_shape(latent.shape)), plan, outs
