"""Oracle encoder: the unpatched causal video-VAE encode, whole or overlap-tiled.

TEST INFRASTRUCTURE ONLY (see the package header).

Structure (DistVAE PR #14 "Add tiled VAE parallelism & extended model support"):
  * encoder commits: the encoders are their decoders read backwards -- a causal convolution in, a
    run of down blocks (residual blocks, then a down-sampler), a mid block, a normalisation and a
    causal convolution out;
  * HunyuanVideo / 1.5 and LTX-2 encoder commits: a down-sampler either folds space into channels
    after a stride-1 convolution ("fold"), or is a bare strided convolution;
  * Qwen-Image / Wan 2.1 and AutoencoderKL encoder commits: the strided down-sampler pads one row
    below and one column to the right, (0, 1, 0, 1), and strides 2 over the result ("stride");
  * Patchify commit: bands are cut in whole multiples of what the encoder narrows the axis by.
The tiled encode follows vllm-omni PR #4831 "VAE tiling parallel encode for LTX-2" (split into
tiles, encode each, merge), with the tile plan and blend of the tiled decode applied in latent units.

Readings where the pages are silent (each is listed in the design notes):
  * the pixels may first be folded into channels (patchify, space-to-depth of the pixel grid), the
    mirror of the decoders' final depth-to-space;
  * space-to-depth order: position (c, st t + dt, sh y + dy, sw x + dx) -> channel
    c*(st sh sw) + dt sh sw + dy sw + dx (PixelUnshuffle in 3-D, the inverse of the decoders'
    depth-to-space); a causal temporal fold puts st - 1 copies of frame 0 in front first, so the
    first frame folds into one latent frame (the inverse of the decoders' first-frame drop);
  * the fold down-sampler's conv maps C_i -> C_{i+1} / (st sh sw) channels, so the fold lands on
    C_{i+1}; the strided one is a 3 x 3 conv of each frame (no temporal taps) C_i -> C_{i+1};
  * the down-sampler takes the residual stream directly (no norm in front), as the decoders' up-
    samplers do; the head is norm + SiLU + causal conv to 2 * latent_c moment channels;
  * tiled encode: spatial tiles only (the whole clip in time), planned on the latent grid by the
    tile plan's start rule; each tile's pixels are the tile's latent box times the compression;
    the latent tiles are blended with the same ramps and normalised weighted sum as decoded tiles.

Parity: pinned by the CPU tests through its parts (space-to-depth as the inverse of depth-to-space
and against torch's pixel_unshuffle; the strided conv against torch's conv2d and brute force), a
library-op formulation of the whole encoder, causality, Tier A == Tier B, and a single tile ==
the untiled encode.
"""
from __future__ import annotations

from typing import List, Sequence, Tuple

import numpy as np

from . import ops, tiles


def _down(cfg, p: dict, i: int, x: np.ndarray, conv, tier: str) -> np.ndarray:
    kind, s = cfg.down[i]
    name = f"stage{i}.down"
    if kind == "fold":
        return ops.space_to_depth(conv(name, x), s, pad_first=True)
    assert kind == "stride" and tuple(s) == (1, 2, 2), cfg.down[i]
    return ops.conv2d_stride2_pad_end(x, p[name + ".weight"], p[name + ".bias"], tier=tier).astype(x.dtype)


def encode(cfg, params: dict, video: np.ndarray, tier: str = "A") -> np.ndarray:
    """Encode pixels [B, C_pix, T, H, W] -> latent moments [B, 2*latent_c, T', h, w].

    tier "A": float64 throughout; "B": float32 activations (statistics in float64)."""
    dtype = np.float64 if tier == "A" else np.float32
    p = params
    g, eps, kind = cfg.gn_groups, cfg.gn_eps, cfg.norm

    def conv(name, x):
        return ops.conv3d_causal(x, p[name + ".weight"], p[name + ".bias"], tier=tier).astype(dtype)

    x = video.astype(dtype)
    if tuple(cfg.patchify) != (1, 1):
        x = ops.space_to_depth(x, (1,) + tuple(cfg.patchify), pad_first=False)
    x = conv("conv_in", x)
    for i in range(cfg.n_stages):
        for r in range(cfg.n_res[i]):
            x = ops.resblock(x, p, f"stage{i}.res{r}", g, eps, conv, kind).astype(dtype)
        if i + 1 < cfg.n_stages:
            x = _down(cfg, p, i, x, conv, tier)
    for r in range(cfg.mid_res):
        x = ops.resblock(x, p, f"mid.res{r}", g, eps, conv, kind).astype(dtype)
    x = ops.silu(ops.norm(x, p["head.norm.gamma"], p["head.norm.beta"], g, eps, kind)).astype(dtype)
    return conv("head.conv", x)


def tile_plan(cfg, video_shape: Sequence[int], tile_hw: Sequence[int], ovl_hw: Sequence[int]) -> List[tiles.Tile]:
    """Spatial tiles on the latent grid (the whole clip in time), boxes in latent units."""
    t_lat = cfg.latent_shape(video_shape)[2:]
    return tiles.tile_plan(t_lat, (t_lat[0],) + tuple(tile_hw), (0,) + tuple(ovl_hw), 1, 1, causal_t=False)


def tiled_encode(cfg, params: dict, video: np.ndarray, tile_hw, ovl_hw, tier: str = "A"):
    """Encode each tile's pixels on its own, then blend the latent tiles; returns (moments, plan, tiles)."""
    _, sh, sw = cfg.scale()
    plan_ = tile_plan(cfg, video.shape, tile_hw, ovl_hw)
    outs = []
    for tl in plan_:
        _, _, h0, nh, w0, nw = tl.lat
        outs.append(encode(cfg, params, video[:, :, :, h0 * sh:(h0 + nh) * sh, w0 * sw:(w0 + nw) * sw], tier=tier))
    return tiles.blend(plan_, outs, cfg.latent_shape(video.shape)), plan_, outs
