"""Oracle operations of the causal video-VAE decoder, NCTHW layout.

TEST INFRASTRUCTURE ONLY (see the package header).  Plain NumPy, written for reading, not speed.

Sources (page titles; the section is the commit or heading of the page named):
  * DistVAE PR #14 "Add tiled VAE parallelism & extended model support":
      - PatchConv3d padding commit: zero padding pads both sides of the halo-extended input and
        crops the halo off the output; spatial padding of a causal conv lives in the conv.
      - HunyuanVideo / LTX-2 commits: the temporal half of a causal padding is one-sided and
        repeats frames along an axis nobody splits; the LTX-2 up-sampler moves channels into
        space, one input position per output position.
      - PatchGroupNorm commit: group statistics are the exact global mean and the population
        variance (divide by the count, no Bessel correction), as nn.GroupNorm computes them.
      - Two-collective PatchGroupNorm commit: sums and counts first (the mean), then squares
        about that mean; the two passes are not folded.
  * TensorRT-LLM PR #16066 "ParallelVAE_TrtllmWan for native Wan VAE": the Wan decoder family
    (causal convs, residual blocks, mid-block attention, temporal cache).

Readings where the pages are silent (each is listed in the design notes):
  * group statistics are per frame: one (mean, variance) per (batch, frame, group), taken over
    the group's channels and the frame's pixels (nn.GroupNorm on the [B*T, C, H, W] view);
  * causal temporal padding = 2 copies of frame 0 in front of a 3-tap kernel (or, in chunked
    decode, the previous chunk's last 2 input frames); spatial padding = 1 zero on each side;
  * residual block = x + conv2(SiLU(GN2(conv1(SiLU(GN1(x))))));
  * depth-to-space channel order c*(s_t*s_h*s_w) + dt*s_h*s_w + dy*s_w + dx -> (c, s_t*t+dt,
    s_h*y+dy, s_w*x+dx) (PixelShuffle order in 3-D); with s_t > 1 the first s_t - 1 output
    frames of the first chunk are dropped (first latent frame -> one frame);
  * attention: one head over the H*W tokens of each frame, 1x1 q/k/v/o projections with bias,
    scale 1/sqrt(C), softmax over keys, residual add; its input is group-normed (no SiLU).

Parity: conv, group norm, channel RMS norm, SiLU, depth-to-space and attention are pinned by the
CPU tests (brute force, library routines, closed forms, invariants); the residual block against a
library-routine formulation, with planted mistakes (swapped norms, a dropped SiLU) that must fail.
"""
from __future__ import annotations

from typing import Optional, Sequence, Tuple

import numpy as np


# ---------------------------------------------------------------------------------------------
# Causal Conv3d
# ---------------------------------------------------------------------------------------------

def causal_pad(x: np.ndarray, cache: Optional[np.ndarray] = None, k_t: int = 3,
               pad_s: int = 1) -> np.ndarray:
    """Pad [B,C,T,H,W] for a causal k_t x (2 pad_s+1)^2 conv.

    Time: k_t - 1 frames in front, copies of frame 0, or the given cache ([B,C,k_t-1,H,W]: the
    last k_t - 1 input frames of the previous chunk).  Space: pad_s zeros on every side.
    """
    front = cache if cache is not None else np.repeat(x[:, :, :1], k_t - 1, axis=2)
    xt = np.concatenate([front.astype(x.dtype), x], axis=2)
    if pad_s:
        xt = np.pad(xt, ((0, 0), (0, 0), (0, 0), (pad_s, pad_s), (pad_s, pad_s)))
    return xt


def conv3d_valid_tierA(xp: np.ndarray, w: np.ndarray, b: np.ndarray) -> np.ndarray:
    """Valid 3-D convolution (cross-correlation) in float64: a direct sum over the taps.

    y[n,o,t,h,x] = b[o] + sum_{kt,kh,kw} sum_c w[o,c,kt,kh,kw] * xp[n,c,t+kt,h+kh,x+kw]
    """
    xp = xp.astype(np.float64)
    w = w.astype(np.float64)
    co, ci, kt_, kh_, kw_ = w.shape
    n, c, tp, hp, wp = xp.shape
    assert c == ci, (c, ci)
    t, h, wd = tp - kt_ + 1, hp - kh_ + 1, wp - kw_ + 1
    y = np.zeros((n, co, t, h, wd), dtype=np.float64)
    for kt in range(kt_):
        for kh in range(kh_):
            for kw in range(kw_):
                sl = xp[:, :, kt:kt + t, kh:kh + h, kw:kw + wd]
                # contract channels: [O, C] x [N, C, T, H, W] -> [N, O, T, H, W]
                y += np.tensordot(w[:, :, kt, kh, kw], sl, axes=([1], [1])).transpose(1, 0, 2, 3, 4)
    y += b.astype(np.float64)[None, :, None, None, None]
    return y


def conv3d_valid_tierB(xp: np.ndarray, w: np.ndarray, b: np.ndarray,
                       max_chunk_bytes: int = 1 << 29) -> np.ndarray:
    """Valid 3-D convolution in float32: per tap one BLAS product over channels-last frame chunks."""
    co, ci, kt_, kh_, kw_ = w.shape
    n, c, tp, hp, wp = xp.shape
    t, h, wd = tp - kt_ + 1, hp - kh_ + 1, wp - kw_ + 1
    xcl = np.ascontiguousarray(xp.astype(np.float32).transpose(0, 2, 3, 4, 1))  # [N,Tp,Hp,Wp,C]
    wt = w.astype(np.float32).transpose(2, 3, 4, 1, 0)  # [kt,kh,kw,C,O]
    y = np.empty((n, t, h, wd, co), dtype=np.float32)
    per_frame = h * wd * max(c, co) * 4
    tc = max(1, min(t, max_chunk_bytes // max(per_frame, 1)))
    for bi in range(n):
        for t0 in range(0, t, tc):
            t1 = min(t, t0 + tc)
            acc = np.zeros((t1 - t0, h, wd, co), dtype=np.float32)
            for kt in range(kt_):
                for kh in range(kh_):
                    for kw in range(kw_):
                        sl = xcl[bi, t0 + kt:t1 + kt, kh:kh + h, kw:kw + wd, :]
                        acc += np.matmul(sl, wt[kt, kh, kw])
            acc += b.astype(np.float32)
            y[bi, t0:t1] = acc
    return np.ascontiguousarray(y.transpose(0, 4, 1, 2, 3))


def conv3d_causal(x: np.ndarray, w: np.ndarray, b: np.ndarray, cache: Optional[np.ndarray] = None,
                  tier: str = "A") -> np.ndarray:
    """Causal 3x3x3 conv, stride 1: temporal front padding (frame 0 repeated, or the cache) and
    spatial zero padding of 1; output has the input's T, H, W."""
    xp = causal_pad(x, cache, k_t=w.shape[2], pad_s=w.shape[3] // 2)
    return conv3d_valid_tierA(xp, w, b) if tier == "A" else conv3d_valid_tierB(xp, w, b)


# ---------------------------------------------------------------------------------------------
# Group norm (per frame), SiLU
# ---------------------------------------------------------------------------------------------

def group_norm_stats(x: np.ndarray, groups: int) -> Tuple[np.ndarray, np.ndarray]:
    """Two-pass float64 statistics per (b, t, g): mean = sum/N, var = sum((x-mean)^2)/N."""
    n, c, t, h, w = x.shape
    xg = x.astype(np.float64).transpose(0, 2, 1, 3, 4).reshape(n, t, groups, (c // groups) * h * w)
    cnt = xg.shape[-1]
    mean = xg.sum(axis=-1) / cnt
    d = xg - mean[..., None]
    var = (d * d).sum(axis=-1) / cnt
    return mean, var


def group_norm(x: np.ndarray, gamma: np.ndarray, beta: np.ndarray, groups: int,
               eps: float) -> np.ndarray:
    """y = (x - mean) / sqrt(var + eps) * gamma[c] + beta[c], statistics per (b, t, g), float64."""
    n, c, t, h, w = x.shape
    mean, var = group_norm_stats(x, groups)  # [N, T, G]
    cg = c // groups
    mean_c = np.repeat(mean, cg, axis=2).transpose(0, 2, 1)[..., None, None]  # [N, C, T, 1, 1]
    var_c = np.repeat(var, cg, axis=2).transpose(0, 2, 1)[..., None, None]
    y = (x.astype(np.float64) - mean_c) / np.sqrt(var_c + eps)
    return y * gamma.astype(np.float64)[None, :, None, None, None] + \
        beta.astype(np.float64)[None, :, None, None, None]


def channel_rms_norm(x: np.ndarray, gamma: np.ndarray, beta: np.ndarray, eps: float) -> np.ndarray:
    """y = x / sqrt(mean_c(x^2) + eps) * gamma[c] + beta[c]: one statistic per (b, t, h, w) over
    the channels, float64.  The channel RMS norms of the Wan / Qwen-Image, HunyuanVideo 1.5 and
    LTX-2 decoders reduce over channels only, so a patch needs nothing from its neighbours (DistVAE
    PR #14 "Add tiled VAE parallelism & extended model support": Qwen-Image, HunyuanVideo/1.5 and
    LTX-2 adapter commits)."""
    xd = x.astype(np.float64)
    ms = (xd * xd).mean(axis=1, keepdims=True)
    y = xd / np.sqrt(ms + eps)
    return y * gamma.astype(np.float64)[None, :, None, None, None] + beta.astype(np.float64)[None, :, None, None, None]


def norm(x: np.ndarray, gamma: np.ndarray, beta: np.ndarray, groups: int, eps: float,
         kind: str = "group") -> np.ndarray:
    """The decoder's norm: group norm (kind "group") or channel RMS norm (kind "rms")."""
    if kind == "rms":
        return channel_rms_norm(x, gamma, beta, eps)
    return group_norm(x, gamma, beta, groups, eps)


def silu(x: np.ndarray) -> np.ndarray:
    """SiLU(x) = x * sigmoid(x) = x / (1 + exp(-x))."""
    with np.errstate(over="ignore"):
        return x / (1.0 + np.exp(-x))


# ---------------------------------------------------------------------------------------------
# Depth-to-space
# ---------------------------------------------------------------------------------------------

def depth_to_space(x: np.ndarray, s: Sequence[int], drop_first: bool) -> np.ndarray:
    """[B, C*st*sh*sw, T, H, W] -> [B, C, st*T, sh*H, sw*W]; channel c*(st sh sw) +
    dt*sh*sw + dy*sw + dx goes to (c, st*t+dt, sh*y+dy, sw*x+dx).  With drop_first and st > 1
    the first st-1 output frames are dropped."""
    st, sh, sw = s
    n, cs, t, h, w = x.shape
    c = cs // (st * sh * sw)
    y = x.reshape(n, c, st, sh, sw, t, h, w).transpose(0, 1, 5, 2, 6, 3, 7, 4)
    y = y.reshape(n, c, t * st, h * sh, w * sw)
    if drop_first and st > 1:
        y = y[:, :, st - 1:]
    return np.ascontiguousarray(y)


def space_to_depth(x: np.ndarray, s: Sequence[int], pad_first: bool) -> np.ndarray:
    """[B, C, T, H, W] -> [B, C*st*sh*sw, T/st, H/sh, W/sw]: position (c, st*t+dt, sh*y+dy, sw*x+dx)
    goes to channel c*(st sh sw) + dt*sh*sw + dy*sw + dx (PixelUnshuffle order in 3-D, the inverse of
    depth_to_space).  With pad_first and st > 1, st-1 copies of frame 0 are put in front first (a
    causal sequence of T frames folds into (T + st - 1) / st, its first frame into one)."""
    st, sh, sw = s
    if pad_first and st > 1:
        x = np.concatenate([np.repeat(x[:, :, :1], st - 1, axis=2), x], axis=2)
    n, c, t, h, w = x.shape
    assert t % st == 0 and h % sh == 0 and w % sw == 0, (x.shape, s)
    y = x.reshape(n, c, t // st, st, h // sh, sh, w // sw, sw).transpose(0, 1, 3, 5, 7, 2, 4, 6)
    return np.ascontiguousarray(y.reshape(n, c * st * sh * sw, t // st, h // sh, w // sw))


def conv2d_stride2_pad_end(x: np.ndarray, w: np.ndarray, b: np.ndarray, tier: str = "A") -> np.ndarray:
    """The stride-2 down-sampler of each frame: one zero row below and one zero column to the right,
    then y[n,o,t,i,j] = b[o] + sum_{kh,kw,c} w[o,c,kh,kw] * xp[n,c,t,2i+kh,2j+kw] (H, W even)."""
    dt = np.float64 if tier == "A" else np.float32
    n, c, t, h, wd = x.shape
    assert h % 2 == 0 and wd % 2 == 0, x.shape
    xp = np.pad(x.astype(dt), ((0, 0), (0, 0), (0, 0), (0, 1), (0, 1)))
    wt = w.astype(dt)
    y = np.zeros((n, w.shape[0], t, h // 2, wd // 2), dtype=dt)
    for kh in range(3):
        for kw in range(3):
            sl = xp[:, :, :, kh:kh + h:2, kw:kw + wd:2]
            y += np.tensordot(wt[:, :, kh, kw], sl, axes=([1], [1])).transpose(1, 0, 2, 3, 4)
    return y + b.astype(dt)[None, :, None, None, None]


# ---------------------------------------------------------------------------------------------
# Mid-block spatial attention
# ---------------------------------------------------------------------------------------------

def softmax(s: np.ndarray, axis: int = -1) -> np.ndarray:
    m = s.max(axis=axis, keepdims=True)
    e = np.exp(s - m)
    return e / e.sum(axis=axis, keepdims=True)


def spatial_attention(x: np.ndarray, p: dict, prefix: str, groups: int, eps: float,
                      dtype=np.float64, kind: str = "group") -> np.ndarray:
    """x + o_proj(softmax(q k^T / sqrt(C)) v) over the H*W tokens of each frame, one head;
    q, k, v are 1x1 projections of the normed x (group or channel RMS norm, no SiLU)."""
    n, c, t, h, w = x.shape
    hn = norm(x, p[prefix + ".norm.gamma"], p[prefix + ".norm.beta"], groups, eps, kind).astype(dtype)
    tok = hn.transpose(0, 2, 3, 4, 1).reshape(n * t, h * w, c)  # [frames, N, C]

    def proj(a, name):
        return a @ p[f"{prefix}.{name}.weight"].astype(dtype).T + p[f"{prefix}.{name}.bias"].astype(dtype)

    q, k, v = proj(tok, "q"), proj(tok, "k"), proj(tok, "v")
    s = (q @ k.transpose(0, 2, 1)).astype(np.float64) / np.sqrt(c)
    a = softmax(s, axis=-1).astype(dtype)
    o = proj(a @ v, "o")
    o = o.reshape(n, t, h, w, c).transpose(0, 4, 1, 2, 3)
    return x.astype(dtype) + o


# ---------------------------------------------------------------------------------------------
# Residual block
# ---------------------------------------------------------------------------------------------

def resblock(x: np.ndarray, p: dict, prefix: str, groups: int, eps: float, conv,
             kind: str = "group") -> np.ndarray:
    """x + conv2(SiLU(N2(conv1(SiLU(N1(x)))))), N = group or channel RMS norm; ``conv(name, input)``
    runs a causal conv."""
    dt = x.dtype
    hmid = silu(norm(x, p[prefix + ".norm1.gamma"], p[prefix + ".norm1.beta"], groups, eps, kind)).astype(dt)
    hmid = conv(prefix + ".conv1", hmid)
    hmid = silu(norm(hmid, p[prefix + ".norm2.gamma"], p[prefix + ".norm2.beta"], groups, eps, kind)).astype(dt)
    hmid = conv(prefix + ".conv2", hmid)
    return x + hmid
