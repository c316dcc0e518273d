"""Oracle patched decode: split -> per-patch decode with explicit halo reads -> merge.

TEST INFRASTRUCTURE ONLY (see the package header).

What it follows (DistVAE PR #14 "Add tiled VAE parallelism & extended model support"):
  * PatchConv3d padding commit: each patch convolves its halo-extended input; the halo rows and
    columns are read from the neighbouring patches, and zero padding applies only where the
    patch edge is an image edge.  Time is never split.
  * PatchGroupNorm and two-collective commits: each patch contributes its count and sum; the
    merged totals give the global mean; each patch then contributes its squares about that
    mean; the merged total over the merged count is the population variance.
  * LTX-2 adapter commit: depth-to-space reads one input position per output position, so each
    patch up-samples its own rows.
  * HunyuanVideo commit: an attention that needs the whole frame runs on the gathered frame.
  * Patchify commit: band edges on the latent grid, first bands one row larger.

The central invariant of the pages, split -> decode -> merge == unsplit decode, is pinned by
the CPU tests against ``decoder.decode``.
"""
from __future__ import annotations

from typing import List

import numpy as np

from . import ops
from .plan import band_edges

Grid = List[List[np.ndarray]]  # [patch row][patch col] -> [B, C, T, Hp, Wp]


def split(x: np.ndarray, eh: List[int], ew: List[int]) -> Grid:
    return [[x[:, :, :, eh[i]:eh[i + 1], ew[j]:ew[j + 1]].copy() for j in range(len(ew) - 1)]
            for i in range(len(eh) - 1)]


def merge(g: Grid) -> np.ndarray:
    return np.concatenate([np.concatenate(row, axis=4) for row in g], axis=3)


def _halo_extend(g: Grid, i: int, j: int) -> np.ndarray:
    """Patch (i, j) with a 1-pixel ring read from its eight neighbours; zeros at image edges."""
    p = g[i][j]
    n, c, t, hp, wp = p.shape
    ext = np.zeros((n, c, t, hp + 2, wp + 2), dtype=p.dtype)
    ext[:, :, :, 1:-1, 1:-1] = p
    nh, nw = len(g), len(g[0])
    for di in (-1, 0, 1):
        for dj in (-1, 0, 1):
            if (di, dj) == (0, 0):
                continue
            a, b = i + di, j + dj
            if not (0 <= a < nh and 0 <= b < nw):
                continue  # image edge: stays zero
            q = g[a][b]
            rs = slice(-1, None) if di == -1 else (slice(0, 1) if di == 1 else slice(None))
            cs = slice(-1, None) if dj == -1 else (slice(0, 1) if dj == 1 else slice(None))
            rd = slice(0, 1) if di == -1 else (slice(hp + 1, hp + 2) if di == 1 else slice(1, hp + 1))
            cd = slice(0, 1) if dj == -1 else (slice(wp + 1, wp + 2) if dj == 1 else slice(1, wp + 1))
            ext[:, :, :, rd, cd] = q[:, :, :, rs, cs]
    return ext


class _PatchedConv:
    def __init__(self, params: dict):
        self.p = params

    def __call__(self, name: str, g: Grid) -> Grid:
        w, b = self.p[name + ".weight"], self.p[name + ".bias"]
        out: Grid = []
        for i in range(len(g)):
            row = []
            for j in range(len(g[0])):
                ext = _halo_extend(g, i, j)
                xp = ops.causal_pad(ext, None, k_t=w.shape[2], pad_s=0)  # space: halo ring already there
                row.append(ops.conv3d_valid_tierA(xp, w, b))
            out.append(row)
        return out


def _patch_group_norm(g: Grid, gamma, beta, groups: int, eps: float) -> Grid:
    """Two-pass merge of per-patch partial sums: (count, sum) -> mean; (sum of squares about
    the mean) -> population variance."""
    def grouped(p):
        n, c, t, h, w = p.shape
        return p.astype(np.float64).transpose(0, 2, 1, 3, 4).reshape(n, t, groups, (c // groups) * h * w)

    flat = [grouped(p) for row in g for p in row]
    count = sum(f.shape[-1] for f in flat)
    total = sum(f.sum(axis=-1) for f in flat)
    mean = total / count
    sq = sum(((f - mean[..., None]) ** 2).sum(axis=-1) for f in flat)
    var = sq / count
    out: Grid = []
    for row in g:
        orow = []
        for p in row:
            n, c, t, h, w = p.shape
            cg = c // groups
            m = np.repeat(mean, cg, axis=2).transpose(0, 2, 1)[..., None, None]
            v = np.repeat(var, cg, axis=2).transpose(0, 2, 1)[..., None, None]
            y = (p.astype(np.float64) - m) / np.sqrt(v + eps)
            orow.append(y * gamma.astype(np.float64)[None, :, None, None, None]
                        + beta.astype(np.float64)[None, :, None, None, None])
        out.append(orow)
    return out


def _map(g: Grid, f) -> Grid:
    return [[f(p) for p in row] for row in g]


def _patch_norm(g: Grid, gamma, beta, groups: int, eps: float, kind: str) -> Grid:
    """Group norm merges per-patch sums; a channel RMS norm needs nothing from other patches."""
    if kind == "rms":
        return _map(g, lambda a: ops.channel_rms_norm(a, gamma, beta, eps))
    return _patch_group_norm(g, gamma, beta, groups, eps)


def _resblock(g: Grid, p: dict, prefix: str, groups: int, eps: float, conv: _PatchedConv,
              kind: str = "group") -> Grid:
    h = _map(_patch_norm(g, p[prefix + ".norm1.gamma"], p[prefix + ".norm1.beta"], groups, eps, kind), ops.silu)
    h = conv(prefix + ".conv1", h)
    h = _map(_patch_norm(h, p[prefix + ".norm2.gamma"], p[prefix + ".norm2.beta"], groups, eps, kind), ops.silu)
    h = conv(prefix + ".conv2", h)
    return [[a + b for a, b in zip(ra, rb)] for ra, rb in zip(g, h)]


def decode_patched(cfg, params: dict, latent: np.ndarray, n_patch_h: int, n_patch_w: int) -> np.ndarray:
    """Float64 patched decode; the result is merged back into one [B, out_c, T', H, W] array."""
    gr, eps, kind = cfg.gn_groups, cfg.gn_eps, cfg.norm
    lh, lw = latent.shape[3], latent.shape[4]
    eh, ew = band_edges(lh, n_patch_h), band_edges(lw, n_patch_w)
    conv = _PatchedConv(params)
    g = split(latent.astype(np.float64), eh, ew)
    g = conv("conv_in", g)
    for r in range(cfg.mid_res):
        g = _resblock(g, params, f"mid.res{r}", gr, eps, conv, kind)
    if cfg.mid_attn:
        # the attention sees the whole frame: gather, attend, split on the same edges
        whole = ops.spatial_attention(merge(g), params, "mid.attn", gr, eps, kind=kind)
        g = split(whole, eh, ew)
    sh_tot = sw_tot = 1
    for i in range(cfg.n_stages):
        for r in range(cfg.n_res[i]):
            g = _resblock(g, params, f"stage{i}.res{r}", gr, eps, conv, kind)
        if i + 1 < cfg.n_stages:
            g = conv(f"stage{i}.up", g)
            g = _map(g, lambda a, s=cfg.up[i]: ops.depth_to_space(a, s, drop_first=True))
            sh_tot *= cfg.up[i][1]
            sw_tot *= cfg.up[i][2]
    g = _map(_patch_norm(g, params["head.norm.gamma"], params["head.norm.beta"], gr, eps, kind), ops.silu)
    g = conv("head.conv", g)
    g = _map(g, lambda a: ops.depth_to_space(a, cfg.out_d2s, drop_first=True))
    return merge(g)
