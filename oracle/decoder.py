"""Oracle decoder: the unpatched causal video-VAE decode, whole or in temporal chunks.

TEST INFRASTRUCTURE ONLY (see the package header).

Structure (DistVAE PR #14 "Add tiled VAE parallelism & extended model support", Wan and LTX-2
adapter commits; TensorRT-LLM PR #16066 "ParallelVAE_TrtllmWan for native Wan VAE"):
  conv_in -> [mid residual blocks] -> [mid attention] -> for each stage: residual blocks, then
  (except after the last stage) the up-sampling conv + depth-to-space -> norm + SiLU -> conv_out
  -> final depth-to-space.  The norms are group norms, or channel RMS norms (``cfg.norm == "rms"``).

Chunked temporal decode (Wan-family decoders thread a per-convolution temporal cache through
a chunked decode; DistVAE PR #14, Wan adapter and HunyuanVideo commits): the latent is cut into
frame chunks; every causal conv keeps the last 2 frames of its (padded) input and puts them in
front of the next chunk instead of the copies of frame 0; the temporal depth-to-space drops its
first frame only in the first chunk.  With per-frame group statistics the chunked decode equals
the whole decode.

Parity: the pages print no output value for any input, so the whole decoder is pinned against a
second formulation of the same architecture written only with library routines (torch conv3d,
group_norm / rms_norm, silu, pixel-shuffle-style reshapes, softmax attention; tests/test_oracle_pins.py,
1e-10), on small configs of every family, together with: every parameter reaching the output, the
causality invariant, chunked == whole, patched == unpatched, Tier A / Tier B agreement, and planted
mistakes in the layer order and the residual block that those pins must catch
(tests/test_oracle_mutations.py).
"""
from __future__ import annotations

from typing import Dict, Iterable, List, Optional, Sequence

import numpy as np

from . import ops


class _ConvRunner:
    """Runs named causal convs, keeping a 2-frame cache per conv across chunks."""

    def __init__(self, params: dict, tier: str):
        self.p = params
        self.tier = tier
        self.cache: Dict[str, np.ndarray] = {}
        self.first = True

    def __call__(self, name: str, x: np.ndarray) -> np.ndarray:
        w = self.p[name + ".weight"]
        b = self.p[name + ".bias"]
        kt = w.shape[2]
        cache = None if self.first else self.cache[name]
        y = ops.conv3d_causal(x, w, b, cache=cache, tier=self.tier)
        front = cache if cache is not None else np.repeat(x[:, :, :1], kt - 1, axis=2)
        self.cache[name] = np.concatenate([front.astype(x.dtype), x], axis=2)[:, :, -(kt - 1):].copy()
        return y.astype(x.dtype)


def _decode_chunk(cfg, p: dict, z: np.ndarray, conv: _ConvRunner, dtype) -> np.ndarray:
    g, eps, kind = cfg.gn_groups, cfg.gn_eps, cfg.norm
    x = conv("conv_in", z.astype(dtype))
    for r in range(cfg.mid_res):
        x = ops.resblock(x, p, f"mid.res{r}", g, eps, conv, kind).astype(dtype)
    if cfg.mid_attn:
        x = ops.spatial_attention(x, p, "mid.attn", g, eps, dtype=dtype, kind=kind).astype(dtype)
    for i in range(cfg.n_stages):
        for r in range(cfg.n_res[i]):
            x = ops.resblock(x, p, f"stage{i}.res{r}", g, eps, conv, kind).astype(dtype)
        if i + 1 < cfg.n_stages:
            x = conv(f"stage{i}.up", x)
            x = ops.depth_to_space(x, cfg.up[i], drop_first=conv.first)
    x = ops.silu(ops.norm(x, p["head.norm.gamma"], p["head.norm.beta"], g, eps, kind)).astype(dtype)
    x = conv("head.conv", x)
    return ops.depth_to_space(x, cfg.out_d2s, drop_first=conv.first)


def decode(cfg, params: dict, latent: np.ndarray, tier: str = "A",
           chunks: Optional[Sequence[int]] = None) -> np.ndarray:
    """Decode latent [B, C, T, h, w] -> pixels [B, out_c, T', H, W].

    tier "A": float64 throughout; "B": float32 activations (statistics in float64).
    chunks: latent frame counts per chunk (summing to T); None decodes in one piece.
    """
    dtype = np.float64 if tier == "A" else np.float32
    t = latent.shape[2]
    sizes: List[int] = list(chunks) if chunks is not None else [t]
    assert sum(sizes) == t and all(s > 0 for s in sizes), sizes
    conv = _ConvRunner(params, tier)
    outs = []
    t0 = 0
    for s in sizes:
        outs.append(_decode_chunk(cfg, params, latent[:, :, t0:t0 + s], conv, dtype))
        conv.first = False
        t0 += s
    return np.concatenate(outs, axis=2)


def chunk_sizes(t: int, per_chunk: int) -> List[int]:
    """Chunk 0 is latent frame 0 alone, then chunks of ``per_chunk`` latent frames."""
    out = [1]
    rest = t - 1
    while rest > 0:
        out.append(min(per_chunk, rest))
        rest -= out[-1]
    return out if t > 0 else []
