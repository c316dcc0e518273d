"""Seeded synthetic workloads: decoder configurations, parameter lists and random draws.

This module holds no arithmetic of the decode itself (no convolution, norm, blend or
up-sampling).  It names the workloads, lists every parameter of a decoder in declaration
order with its shape, and draws the latent and the parameters from seeded generators.
Both the CUDA path (through the Python binding) and the CPU oracle take their inputs from
here, as plain host arrays.

Draw rules:
  * generator ``numpy.random.Generator(PCG64(seed))``, float32;
  * the latent comes from ``seed``; the parameters from ``seed + 1``, drawn in declaration
    order;
  * convolution / projection weights ~ N(0, 1/fan_in), fan_in = C_in * k_t * k_h * k_w;
  * biases 0, norm scale 1, norm shift 0, unless ``rand_affine`` is set, in which case each
    of them is drawn too (bias, shift ~ N(0, 0.1^2); scale ~ 1 + N(0, 0.1^2)).

The architectures follow the video-VAE decoders the pages describe (DistVAE PR #14 "Add tiled
VAE parallelism & extended model support", LTX-2 and Wan adapter commits; TensorRT-LLM PR #16066
"ParallelVAE_TrtllmWan for native Wan VAE"): a causal 3x3x3 convolution in, an optional mid block
(residual block, then single-head spatial attention), stages of residual blocks each followed by a
depth-to-space up-sampler, and a norm + SiLU + causal convolution out with a final depth-to-space.
"""
from __future__ import annotations

import dataclasses
from collections import OrderedDict
from typing import Dict, List, Optional, Sequence, Tuple

import numpy as np


@dataclasses.dataclass(frozen=True)
class DecoderConfig:
    """Architecture hyper-parameters of a causal video-VAE decoder.

    stage_c[i]  channels of stage i; n_res[i] residual blocks in stage i.
    up[i]       (s_t, s_h, s_w) of the up-sampler after stage i (i < n_stages - 1); it maps
                stage_c[i] -> s_t*s_h*s_w*stage_c[i+1] channels, then depth-to-space.
    mid_res     residual blocks at the start (after conv_in), at stage_c[0] channels.
    mid_attn    1 = single-head per-frame spatial self-attention after the mid residual blocks.
    out_c       pixel channels; out_d2s the final depth-to-space factors of conv_out.
    norm        "group": every norm is a per-frame group norm; "rms": a channel RMS norm per pixel
                (the Wan / Qwen-Image, HunyuanVideo 1.5 and LTX-2 decoders' norms).
    """

    name: str
    latent_shape: Tuple[int, int, int, int, int]  # [B, C, T, h, w]
    stage_c: Tuple[int, ...]
    n_res: Tuple[int, ...]
    up: Tuple[Tuple[int, int, int], ...]
    mid_res: int = 0
    mid_attn: int = 0
    gn_groups: int = 32
    gn_eps: float = 1e-6
    out_c: int = 3
    out_d2s: Tuple[int, int, int] = (1, 1, 1)
    norm: str = "group"  # "group" (per-frame group norm) or "rms" (channel RMS norm per pixel)

    @property
    def latent_c(self) -> int:
        return self.latent_shape[1]

    @property
    def n_stages(self) -> int:
        return len(self.stage_c)

    def scale(self) -> Tuple[int, int, int]:
        """Total (t, h, w) up-sampling factor from latent to pixels."""
        st, sh, sw = self.out_d2s
        for u in self.up:
            st *= u[0]
            sh *= u[1]
            sw *= u[2]
        return st, sh, sw

    def output_shape(self, latent_shape: Optional[Sequence[int]] = None) -> Tuple[int, ...]:
        """[B, out_c, T', H', W'] for a latent of the given shape (causal: first latent frame -> 1 frame)."""
        b, _, t, h, w = latent_shape if latent_shape is not None else self.latent_shape
        st, sh, sw = self.scale()
        return (b, self.out_c, st * (t - 1) + 1, sh * h, sw * w)


@dataclasses.dataclass(frozen=True)
class EncoderConfig:
    """Architecture hyper-parameters of a causal video-VAE encoder (a decoder read backwards).

    video_shape  [B, C_pix, T, H, W] pixels.
    patchify     (s_h, s_w): space-to-depth of the pixels before conv_in ((1, 1) = none).
    stage_c[i]   channels of stage i; n_res[i] residual blocks in stage i.
    down[i]      (kind, (s_t, s_h, s_w)) of the down-sampler after stage i (i < n_stages - 1):
                 "fold"   a stride-1 causal conv to stage_c[i+1] / (s_t*s_h*s_w) channels, then
                          space-to-depth by (s_t, s_h, s_w);
                 "stride" zero padding of one row below and one column right, then a 3x3 stride-2
                          conv of each frame to stage_c[i+1] channels ((s_t, s_h, s_w) = (1, 2, 2)).
    mid_res      residual blocks after the last stage.
    latent_c     latent channels; conv_out writes 2 * latent_c (the moments: mean, log-variance).
    norm         "group" (per-frame group norm) or "rms" (channel RMS norm per pixel).
    """

    name: str
    video_shape: Tuple[int, int, int, int, int]
    stage_c: Tuple[int, ...]
    n_res: Tuple[int, ...]
    down: Tuple[Tuple[str, Tuple[int, int, int]], ...]
    patchify: Tuple[int, int] = (1, 1)
    mid_res: int = 0
    gn_groups: int = 32
    gn_eps: float = 1e-6
    latent_c: int = 16
    norm: str = "group"

    @property
    def pix_c(self) -> int:
        return self.video_shape[1]

    @property
    def n_stages(self) -> int:
        return len(self.stage_c)

    def scale(self) -> Tuple[int, int, int]:
        """Total (t, h, w) down-sampling factor from pixels to latent."""
        st, sh, sw = 1, self.patchify[0], self.patchify[1]
        for _, f in self.down:
            st *= f[0]
            sh *= f[1]
            sw *= f[2]
        return st, sh, sw

    def latent_shape(self, video_shape: Optional[Sequence[int]] = None) -> Tuple[int, ...]:
        """[B, 2*latent_c, T', h, w]: causal time, the first pixel frame -> one latent frame."""
        b, _, t, h, w = video_shape if video_shape is not None else self.video_shape
        st, sh, sw = self.scale()
        return (b, 2 * self.latent_c, (t - 1) // st + 1, h // sh, w // sw)


@dataclasses.dataclass(frozen=True)
class TilingConfig:
    """Overlap-tiled decode: tile length and overlap per axis, in latent units (t, h, w)."""

    tile: Tuple[int, int, int]
    overlap: Tuple[int, int, int]


# ---------------------------------------------------------------------------------------------
# Named workloads.  Sizes follow the five workloads of the hot path; the small "mini" ones are
# test cases that still span several 128-pixel tiles, ragged tails and every channel path.
# ---------------------------------------------------------------------------------------------

TINY = DecoderConfig(
    name="tiny", latent_shape=(1, 16, 3, 16, 16), stage_c=(32, 32), n_res=(2, 0),
    up=((1, 2, 2),), gn_groups=8, out_d2s=(1, 1, 1))

WAN = DecoderConfig(
    name="wan", latent_shape=(1, 48, 21, 44, 80), stage_c=(1024, 1024, 512, 256),
    n_res=(2, 2, 2, 2), up=((2, 2, 2), (2, 2, 2), (1, 2, 2)), mid_res=1, mid_attn=1,
    gn_groups=32, out_d2s=(1, 2, 2))

LTX = DecoderConfig(
    name="ltx", latent_shape=(1, 128, 11, 22, 40), stage_c=(1024, 512, 256, 128),
    n_res=(3, 3, 3, 3), up=((2, 2, 2), (2, 2, 2), (2, 2, 2)), gn_groups=32, out_d2s=(1, 4, 4))

LTX_TILED = dataclasses.replace(LTX, name="ltx_tiled", latent_shape=(2, 128, 17, 34, 60))
LTX_TILING = TilingConfig(tile=(8, 16, 16), overlap=(1, 4, 4))

# Reduced-width stand-ins with the same structure (every conv path, GN groups of 1..4
# channels, temporal and spatial depth-to-space, attention) and sizes the oracle runs in
# seconds.  Channel counts are multiples of 64 so the tensor-core convolution takes them.
MINI_LTX = DecoderConfig(
    name="mini_ltx", latent_shape=(1, 64, 3, 10, 13), stage_c=(128, 64), n_res=(1, 1),
    up=((2, 2, 2),), gn_groups=32, out_d2s=(1, 4, 4))

MINI_WAN = DecoderConfig(
    name="mini_wan", latent_shape=(1, 48, 3, 9, 11), stage_c=(128, 128, 64), n_res=(1, 1, 1),
    up=((2, 2, 2), (1, 2, 2)), mid_res=1, mid_attn=1, gn_groups=32, out_d2s=(1, 2, 2))

# The Wan-family block structure with channel RMS norms instead of group norms (the norm the
# Wan / Qwen-Image decoders use); same architecture otherwise.
WAN_RMS = dataclasses.replace(WAN, name="wan_rms", norm="rms")
MINI_WAN_RMS = dataclasses.replace(MINI_WAN, name="mini_wan_rms", norm="rms")

MINI_TILED = dataclasses.replace(MINI_LTX, name="mini_tiled", latent_shape=(2, 64, 5, 7, 9))
MINI_TILING = TilingConfig(tile=(3, 4, 4), overlap=(1, 1, 2))

CONFIGS: Dict[str, DecoderConfig] = {c.name: c for c in (
    TINY, WAN, LTX, LTX_TILED, MINI_LTX, MINI_WAN, MINI_TILED, WAN_RMS, MINI_WAN_RMS)}

# Encoders: the LTX-shaped decoder read backwards (720p x 81f pixels -> latent [1, 256, 11, 22, 40]
# moments: patchify 4 x 4, three space-to-depth down-samplers (2, 2, 2)), and small ones that the
# oracle runs in seconds, one per down-sampler kind.
LTX_ENC = EncoderConfig(
    name="ltx_enc", video_shape=(1, 3, 81, 704, 1280), stage_c=(128, 256, 512, 1024), n_res=(3, 3, 3, 3),
    down=(("fold", (2, 2, 2)),) * 3, patchify=(4, 4), gn_groups=32, latent_c=128)
TINY_ENC = EncoderConfig(
    name="tiny_enc", video_shape=(1, 3, 5, 16, 16), stage_c=(32, 32), n_res=(1, 1),
    down=(("fold", (2, 2, 2)),), gn_groups=8, latent_c=4)
TINY_ENC_STRIDE = EncoderConfig(
    name="tiny_enc_stride", video_shape=(1, 3, 3, 16, 16), stage_c=(32, 32), n_res=(1, 1),
    down=(("stride", (1, 2, 2)),), gn_groups=8, latent_c=4)
MINI_ENC = EncoderConfig(
    name="mini_enc", video_shape=(1, 3, 9, 40, 56), stage_c=(128, 128), n_res=(1, 1),
    down=(("fold", (2, 2, 2)),), patchify=(4, 4), mid_res=1, gn_groups=32, latent_c=16)
MINI_ENC_STRIDE = EncoderConfig(
    name="mini_enc_stride", video_shape=(1, 3, 5, 24, 40), stage_c=(64, 128), n_res=(1, 1),
    down=(("stride", (1, 2, 2)),), patchify=(2, 2), gn_groups=32, latent_c=16)
MINI_ENC_RMS = dataclasses.replace(MINI_ENC, name="mini_enc_rms", norm="rms")

ENCODERS: Dict[str, EncoderConfig] = {c.name: c for c in (
    LTX_ENC, TINY_ENC, TINY_ENC_STRIDE, MINI_ENC, MINI_ENC_STRIDE, MINI_ENC_RMS)}


# ---------------------------------------------------------------------------------------------
# Parameter list (declaration order) and draws.
# ---------------------------------------------------------------------------------------------

def _resblock_params(prefix: str, c: int) -> List[Tuple[str, Tuple[int, ...]]]:
    return [
        (f"{prefix}.norm1.gamma", (c,)), (f"{prefix}.norm1.beta", (c,)),
        (f"{prefix}.conv1.weight", (c, c, 3, 3, 3)), (f"{prefix}.conv1.bias", (c,)),
        (f"{prefix}.norm2.gamma", (c,)), (f"{prefix}.norm2.beta", (c,)),
        (f"{prefix}.conv2.weight", (c, c, 3, 3, 3)), (f"{prefix}.conv2.bias", (c,)),
    ]


def encoder_param_specs(cfg: EncoderConfig) -> "OrderedDict[str, Tuple[int, ...]]":
    """Every parameter of the encoder, in declaration order, with its shape.

    Causal conv weights are [C_out, C_in, 3, 3, 3]; the stride-2 down-sampler's [C_out, C_in, 3, 3].
    """
    specs: List[Tuple[str, Tuple[int, ...]]] = []
    c0 = cfg.stage_c[0]
    cin = cfg.pix_c * cfg.patchify[0] * cfg.patchify[1]
    specs += [("conv_in.weight", (c0, cin, 3, 3, 3)), ("conv_in.bias", (c0,))]
    for i, c in enumerate(cfg.stage_c):
        for r in range(cfg.n_res[i]):
            specs += _resblock_params(f"stage{i}.res{r}", c)
        if i + 1 < cfg.n_stages:
            kind, (st, sh, sw) = cfg.down[i]
            if kind == "fold":
                co = cfg.stage_c[i + 1] // (st * sh * sw)
                specs += [(f"stage{i}.down.weight", (co, c, 3, 3, 3)), (f"stage{i}.down.bias", (co,))]
            else:
                co = cfg.stage_c[i + 1]
                specs += [(f"stage{i}.down.weight", (co, c, 3, 3)), (f"stage{i}.down.bias", (co,))]
    cl = cfg.stage_c[-1]
    for r in range(cfg.mid_res):
        specs += _resblock_params(f"mid.res{r}", cl)
    specs += [("head.norm.gamma", (cl,)), ("head.norm.beta", (cl,)),
              ("head.conv.weight", (2 * cfg.latent_c, cl, 3, 3, 3)), ("head.conv.bias", (2 * cfg.latent_c,))]
    return OrderedDict(specs)


def param_specs(cfg) -> "OrderedDict[str, Tuple[int, ...]]":
    """Every parameter of the decoder (or encoder), in declaration order, with its shape.

    Convolution weights are [C_out, C_in, k_t, k_h, k_w]; attention projections [C_out, C_in].
    """
    if isinstance(cfg, EncoderConfig):
        return encoder_param_specs(cfg)
    specs: List[Tuple[str, Tuple[int, ...]]] = []
    c0 = cfg.stage_c[0]
    specs += [("conv_in.weight", (c0, cfg.latent_c, 3, 3, 3)), ("conv_in.bias", (c0,))]
    for r in range(cfg.mid_res):
        specs += _resblock_params(f"mid.res{r}", c0)
    if cfg.mid_attn:
        specs += [("mid.attn.norm.gamma", (c0,)), ("mid.attn.norm.beta", (c0,))]
        for p in ("q", "k", "v", "o"):
            specs += [(f"mid.attn.{p}.weight", (c0, c0)), (f"mid.attn.{p}.bias", (c0,))]
    for i, c in enumerate(cfg.stage_c):
        for r in range(cfg.n_res[i]):
            specs += _resblock_params(f"stage{i}.res{r}", c)
        if i + 1 < cfg.n_stages:
            st, sh, sw = cfg.up[i]
            co = st * sh * sw * cfg.stage_c[i + 1]
            specs += [(f"stage{i}.up.weight", (co, c, 3, 3, 3)), (f"stage{i}.up.bias", (co,))]
    cl = cfg.stage_c[-1]
    st, sh, sw = cfg.out_d2s
    specs += [("head.norm.gamma", (cl,)), ("head.norm.beta", (cl,)),
              ("head.conv.weight", (cfg.out_c * st * sh * sw, cl, 3, 3, 3)),
              ("head.conv.bias", (cfg.out_c * st * sh * sw,))]
    return OrderedDict(specs)


def draw_video(cfg: EncoderConfig, seed: int = 0, shape: Optional[Sequence[int]] = None) -> np.ndarray:
    """Pixels [B, C_pix, T, H, W] ~ N(0, 1), float32, from PCG64(seed)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    return rng.standard_normal(tuple(shape or cfg.video_shape), dtype=np.float32)


def draw_latent(cfg: DecoderConfig, seed: int = 0,
                shape: Optional[Sequence[int]] = None) -> np.ndarray:
    """Latent [B, C, T, h, w] ~ N(0, 1), float32, from PCG64(seed)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    return rng.standard_normal(tuple(shape or cfg.latent_shape), dtype=np.float32)


def draw_params(cfg: DecoderConfig, seed: int = 0,
                rand_affine: bool = False) -> "OrderedDict[str, np.ndarray]":
    """All parameters, float32, drawn from PCG64(seed + 1) in declaration order."""
    rng = np.random.Generator(np.random.PCG64(seed + 1))
    out: "OrderedDict[str, np.ndarray]" = OrderedDict()
    for name, shape in param_specs(cfg).items():
        kind = name.rsplit(".", 1)[1]
        if kind == "weight":
            fan_in = int(np.prod(shape[1:]))
            a = rng.standard_normal(shape, dtype=np.float32)
            a *= np.float32(1.0 / np.sqrt(fan_in))
        elif not rand_affine:
            a = (np.ones if kind == "gamma" else np.zeros)(shape, dtype=np.float32)
        else:
            a = rng.standard_normal(shape, dtype=np.float32) * np.float32(0.1)
            if kind == "gamma":
                a += np.float32(1.0)
        out[name] = a
    return out


def draw_normal(shape: Sequence[int], seed: int, offset: float = 0.0,
                std: float = 1.0) -> np.ndarray:
    """A tensor ~ N(offset, std^2), float32, from PCG64(seed) (op-level test inputs)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    a = rng.standard_normal(tuple(shape), dtype=np.float32)
    if std != 1.0:
        a *= np.float32(std)
    if offset:
        a += np.float32(offset)
    return a


def conv_weight(c_out: int, c_in: int, seed: int, k: Tuple[int, int, int] = (3, 3, 3)) -> np.ndarray:
    """A convolution weight [C_out, C_in, k_t, k_h, k_w] ~ N(0, 1/fan_in), float32."""
    fan_in = c_in * k[0] * k[1] * k[2]
    return draw_normal((c_out, c_in) + tuple(k), seed, std=1.0 / np.sqrt(fan_in))
