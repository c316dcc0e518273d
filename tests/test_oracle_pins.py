"""Pins of the CPU oracle against things other than itself.

Each test checks one oracle function against a brute-force loop, a library routine used only
here, a closed form, an invariant the pages state, or a value the pages print (tests/golden).
"""
import json
import os

import numpy as np
import pytest
import torch

from oracle import decoder, metrics, ops, patched, plan, tiles
from patch_tiled_causal_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ----------------------------------------------------------------------------- convolution

def _brute_conv(x, w, b):
    """Causal 3-D conv by explicit loops: frame index clamped at 0 (frame 0 replicated in front),
    spatial taps outside the image read zero."""
    n, ci, t, h, wd = x.shape
    co, _, kt_, kh_, kw_ = w.shape
    y = np.zeros((n, co, t, h, wd))
    for bn in range(n):
        for o in range(co):
            for tt in range(t):
                for hh in range(h):
                    for ww in range(wd):
                        s = float(b[o])
                        for kt in range(kt_):
                            ti = max(tt + kt - (kt_ - 1), 0)
                            for kh in range(kh_):
                                hi = hh + kh - kh_ // 2
                                if hi < 0 or hi >= h:
                                    continue
                                for kw in range(kw_):
                                    wi = ww + kw - kw_ // 2
                                    if wi < 0 or wi >= wd:
                                        continue
                                    for c in range(ci):
                                        s += w[o, c, kt, kh, kw] * x[bn, c, ti, hi, wi]
                        y[bn, o, tt, hh, ww] = s
    return y


def _im2col_conv(x, w, b):
    """Second formulation: gather the 27-tap patch of every output voxel, one matrix product."""
    n, ci, t, h, wd = x.shape
    co = w.shape[0]
    ti = np.clip(np.arange(t)[:, None] + np.arange(3)[None, :] - 2, 0, None)       # [t, 3]
    xp = np.pad(x, ((0, 0), (0, 0), (0, 0), (1, 1), (1, 1)))
    cols = np.empty((n, t, h, wd, ci, 3, 3, 3))
    for kt in range(3):
        for kh in range(3):
            for kw in range(3):
                cols[..., kt, kh, kw] = xp[:, :, ti[:, kt], kh:kh + h, kw:kw + wd].transpose(0, 2, 3, 4, 1)
    y = cols.reshape(n, t, h, wd, -1) @ w.reshape(co, -1).T + b
    return y.transpose(0, 4, 1, 2, 3)


@pytest.mark.parametrize("shape", [(1, 3, 4, 4, 4), (2, 2, 3, 2, 4), (1, 4, 1, 3, 2)])
def test_conv_brute_force(shape):
    x = synth.draw_normal(shape, 3).astype(np.float64)
    w = synth.draw_normal((3, shape[1], 3, 3, 3), 4).astype(np.float64)
    b = synth.draw_normal((3,), 5).astype(np.float64)
    ref = _brute_conv(x, w, b)
    np.testing.assert_allclose(ops.conv3d_causal(x, w, b, tier="A"), ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(_im2col_conv(x, w, b), ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(ops.conv3d_causal(x, w, b, tier="B"), ref, rtol=2e-5, atol=2e-5)


def test_conv_vs_torch_library():
    x = synth.draw_normal((1, 5, 4, 6, 7), 6).astype(np.float64)
    w = synth.draw_normal((4, 5, 3, 3, 3), 7).astype(np.float64)
    b = synth.draw_normal((4,), 8).astype(np.float64)
    xt = torch.from_numpy(x)
    xt = torch.cat([xt[:, :, :1], xt[:, :, :1], xt], dim=2)              # causal: frame 0 twice
    ref = torch.nn.functional.conv3d(xt, torch.from_numpy(w), torch.from_numpy(b), padding=(0, 1, 1))
    np.testing.assert_allclose(ops.conv3d_causal(x, w, b), ref.numpy(), rtol=1e-12, atol=1e-12)


def test_conv_special_cases():
    x = synth.draw_normal((1, 3, 3, 5, 6), 9).astype(np.float64)
    # delta kernel at (kt=2, kh=1, kw=1) of channel 1 -> copy of channel 1
    w = np.zeros((2, 3, 3, 3, 3))
    w[0, 1, 2, 1, 1] = 1.0
    # delta at (kt=1, kh=0, kw=2): previous frame (clamped), one row up, one column right
    w[1, 2, 1, 0, 2] = 1.0
    y = ops.conv3d_causal(x, w, np.zeros(2))
    np.testing.assert_array_equal(y[0, 0], x[0, 1])
    prev = x[0, 2, np.maximum(np.arange(3) - 1, 0)]
    exp = np.zeros_like(prev)
    exp[:, 1:, :-1] = prev[:, :-1, 1:]
    np.testing.assert_array_equal(y[0, 1], exp)
    # 1x1x1 kernel = channel matmul
    w1 = synth.draw_normal((4, 3, 1, 1, 1), 10).astype(np.float64)
    y1 = ops.conv3d_causal(x, w1, np.zeros(4))
    np.testing.assert_allclose(y1, np.einsum("oc,ncthw->nothw", w1[:, :, 0, 0, 0], x), rtol=1e-13)
    # constant input: interior output = sum of the weights (+ bias)
    wc = synth.draw_normal((2, 3, 3, 3, 3), 11).astype(np.float64)
    yc = ops.conv3d_causal(np.full((1, 3, 3, 5, 6), 2.0), wc, np.array([0.5, -1.0]))
    np.testing.assert_allclose(yc[0, :, :, 1:-1, 1:-1],
                               (2.0 * wc.sum(axis=(1, 2, 3, 4)) + [0.5, -1.0])[:, None, None, None]
                               * np.ones((2, 3, 3, 4)), rtol=1e-12)


def test_conv_cache_is_front_padding():
    x = synth.draw_normal((1, 2, 5, 4, 4), 12).astype(np.float64)
    w = synth.draw_normal((3, 2, 3, 3, 3), 13).astype(np.float64)
    b = np.zeros(3)
    whole = ops.conv3d_causal(x, w, b)
    tail = ops.conv3d_causal(x[:, :, 3:], w, b, cache=x[:, :, 1:3])
    np.testing.assert_allclose(tail, whole[:, :, 3:], rtol=1e-13, atol=1e-13)


# ----------------------------------------------------------------------------- group norm

@pytest.mark.parametrize("offset", [0.0, 100.0])
def test_group_norm_vs_torch(offset):
    x = synth.draw_normal((2, 8, 3, 5, 6), 14, offset=offset).astype(np.float64)
    g = synth.draw_normal((8,), 15) * 0.1 + 1.0
    bt = synth.draw_normal((8,), 16) * 0.1
    y = ops.group_norm(x, g, bt, 4, 1e-6)
    # library routine on the [B*T, C, H, W] view (per-frame statistics)
    xv = torch.from_numpy(x).permute(0, 2, 1, 3, 4).reshape(6, 8, 5, 6)
    gn = torch.nn.GroupNorm(4, 8, eps=1e-6).double()
    with torch.no_grad():
        gn.weight.copy_(torch.from_numpy(g.astype(np.float64)))
        gn.bias.copy_(torch.from_numpy(bt.astype(np.float64)))
        ref = gn(xv).reshape(2, 3, 8, 5, 6).permute(0, 2, 1, 3, 4).numpy()
    np.testing.assert_allclose(y, ref, rtol=1e-9, atol=1e-9)


def test_group_norm_population_variance():
    # one group of values {0, 2}: mean 1, population variance 1 (Bessel would give 2)
    x = np.array([0.0, 2.0, 0.0, 2.0]).reshape(1, 1, 1, 2, 2)
    mean, var = ops.group_norm_stats(x, 1)
    assert mean[0, 0, 0] == 1.0 and var[0, 0, 0] == 1.0
    y = ops.group_norm(x, np.ones(1), np.zeros(1), 1, 0.0)
    np.testing.assert_allclose(y.ravel(), [-1, 1, -1, 1])


def test_group_norm_per_frame():
    # a frame-wise offset must not leak into other frames (statistics per (b, t, g))
    x = synth.draw_normal((1, 4, 3, 4, 4), 17).astype(np.float64)
    x2 = x.copy()
    x2[:, :, 2] += 50.0
    y, y2 = (ops.group_norm(a, np.ones(4), np.zeros(4), 2, 1e-6) for a in (x, x2))
    np.testing.assert_allclose(y2[:, :, :2], y[:, :, :2], rtol=0, atol=0)
    np.testing.assert_allclose(y2[:, :, 2], y[:, :, 2], rtol=1e-9, atol=1e-9)


def test_channel_rms_norm_vs_torch():
    # library routine: rms_norm over the channel axis of the channels-last view
    x = synth.draw_normal((2, 12, 3, 5, 6), 26, offset=0.5).astype(np.float64)
    g = synth.draw_normal((12,), 27) * 0.1 + 1.0
    bt = synth.draw_normal((12,), 28) * 0.1
    y = ops.channel_rms_norm(x, g, bt, 1e-6)
    xv = torch.from_numpy(x).permute(0, 2, 3, 4, 1)
    ref = torch.nn.functional.rms_norm(xv, (12,), torch.from_numpy(g.astype(np.float64)), eps=1e-6)
    ref = (ref + torch.from_numpy(bt.astype(np.float64))).permute(0, 4, 1, 2, 3).numpy()
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)


def test_channel_rms_norm_brute_force_and_closed_forms():
    x = synth.draw_normal((1, 5, 2, 2, 3), 29).astype(np.float64)
    g = synth.draw_normal((5,), 30) * 0.1 + 1.0
    bt = synth.draw_normal((5,), 31) * 0.1
    y = ops.channel_rms_norm(x, g, bt, 1e-3)
    for t in range(2):
        for i in range(2):
            for j in range(3):
                v = x[0, :, t, i, j]
                r = (sum(float(a) * float(a) for a in v) / 5 + 1e-3) ** 0.5
                for ch in range(5):
                    assert abs(y[0, ch, t, i, j] - (v[ch] / r * g[ch] + bt[ch])) < 1e-12
    # a constant vector a*1 normalises to sign(a) (eps 0), whatever |a|
    for a in (-3.0, 0.25, 1e4):
        c = np.full((1, 4, 1, 1, 1), a)
        np.testing.assert_allclose(ops.channel_rms_norm(c, np.ones(4), np.zeros(4), 0.0).ravel(), np.sign(a))
    # scale invariance (eps 0) and per-pixel independence: a pixel's change leaves the others alone
    np.testing.assert_allclose(ops.channel_rms_norm(7.5 * x, g, bt, 0.0), ops.channel_rms_norm(x, g, bt, 0.0),
                               rtol=1e-12, atol=1e-12)
    x2 = x.copy()
    x2[0, :, 1, 1, 2] *= -40.0
    y0, y2 = (ops.channel_rms_norm(a, g, bt, 1e-6) for a in (x, x2))
    mask = np.ones(y0.shape, bool)
    mask[0, :, 1, 1, 2] = False
    np.testing.assert_array_equal(y2[mask], y0[mask])


def test_silu_closed_form():
    x = np.array([-1000.0, -2.0, 0.0, 1.0, 3.0, 1000.0])
    ref = torch.nn.functional.silu(torch.from_numpy(x)).numpy()
    np.testing.assert_allclose(ops.silu(x), ref, rtol=1e-14, atol=1e-300)
    assert ops.silu(np.array([0.0]))[0] == 0.0


# ----------------------------------------------------------------------------- depth-to-space

def test_d2s_vs_pixel_shuffle_and_inverse():
    x = synth.draw_normal((1, 3 * 8, 2, 3, 4), 18).astype(np.float64)
    y = ops.depth_to_space(x, (2, 2, 2), drop_first=False)
    assert y.shape == (1, 3, 4, 6, 8)
    # inverse by explicit index loops
    inv = np.empty_like(x)
    for c in range(3):
        for dt in range(2):
            for dy in range(2):
                for dx in range(2):
                    ch = c * 8 + dt * 4 + dy * 2 + dx
                    inv[0, ch] = y[0, c, dt::2, dy::2, dx::2]
    np.testing.assert_array_equal(inv, x)
    # 2-D case equals the library pixel shuffle, frame by frame
    x2 = synth.draw_normal((1, 2 * 4, 3, 3, 5), 19)
    y2 = ops.depth_to_space(x2, (1, 2, 2), drop_first=True)
    for t in range(3):
        ref = torch.nn.functional.pixel_shuffle(torch.from_numpy(x2[:, :, t]), 2).numpy()
        np.testing.assert_array_equal(y2[:, :, t], ref)


def test_d2s_first_frame_drop_counts():
    for base, counts in ((synth.WAN, [21, 41, 81, 81]), (synth.LTX, [11, 21, 41, 81])):
        t = base.latent_shape[2]
        seen = [t]
        for u in base.up:
            t = u[0] * t - (u[0] - 1)
            seen.append(t)
        assert seen == counts
        assert base.output_shape()[2] == 81


# ----------------------------------------------------------------------------- attention

def _attn_params(c, seed, zero_qk=False):
    p = {"a.norm.gamma": np.ones(c), "a.norm.beta": np.zeros(c)}
    for i, n in enumerate("qkvo"):
        w = synth.draw_normal((c, c), seed + i) / np.sqrt(c)
        if zero_qk and n in "qk":
            w = np.zeros((c, c))
        p[f"a.{n}.weight"] = w
        p[f"a.{n}.bias"] = synth.draw_normal((c,), seed + 10 + i) * 0.1
    return p


def test_attention_vs_library():
    c = 8
    x = synth.draw_normal((1, c, 2, 3, 4), 20).astype(np.float64)
    p = _attn_params(c, 21)
    y = ops.spatial_attention(x, p, "a", 4, 1e-6)
    hn = ops.group_norm(x, p["a.norm.gamma"], p["a.norm.beta"], 4, 1e-6)
    tok = torch.from_numpy(hn.transpose(0, 2, 3, 4, 1).reshape(2, 12, c))
    lin = lambda a, n: a @ torch.from_numpy(p[f"a.{n}.weight"]).T + torch.from_numpy(p[f"a.{n}.bias"])
    o = torch.nn.functional.scaled_dot_product_attention(lin(tok, "q"), lin(tok, "k"), lin(tok, "v"))
    ref = x + lin(o, "o").numpy().reshape(1, 2, 3, 4, c).transpose(0, 4, 1, 2, 3)
    np.testing.assert_allclose(y, ref, rtol=1e-10, atol=1e-10)


def test_attention_special_cases():
    c = 4
    x = synth.draw_normal((1, c, 1, 2, 3), 22).astype(np.float64)
    p = _attn_params(c, 23, zero_qk=True)
    y = ops.spatial_attention(x, p, "a", 2, 1e-6)
    hn = ops.group_norm(x, p["a.norm.gamma"], p["a.norm.beta"], 2, 1e-6)[0, :, 0].reshape(c, -1)
    v = p["a.v.weight"] @ hn + p["a.v.bias"][:, None]           # [C, N]
    o = p["a.o.weight"] @ v.mean(axis=1) + p["a.o.bias"]        # uniform scores -> mean of v
    np.testing.assert_allclose((y - x)[0, :, 0].reshape(c, -1), np.repeat(o[:, None], 6, 1), rtol=1e-12)


# ----------------------------------------------------------------------------- decoder invariants

def test_resblock_zero_conv2_is_identity():
    cfg = synth.TINY
    p = synth.draw_params(cfg, 0, rand_affine=True)
    p["stage0.res0.conv2.weight"][:] = 0
    p["stage0.res0.conv2.bias"][:] = 0
    x = synth.draw_normal((1, 32, 2, 4, 4), 24).astype(np.float64)
    run = decoder._ConvRunner(p, "A")
    np.testing.assert_array_equal(ops.resblock(x, p, "stage0.res0", 8, 1e-6, run), x)


# A second formulation of the residual block and of the whole decoder, written from the stated
# architecture with library routines only (torch.nn.functional conv3d, group_norm, rms_norm, silu,
# linear, scaled_dot_product_attention; depth-to-space as strided assignments).  It shares no code
# with the oracle, so a wiring mistake in the oracle (parameters of one norm used for the other, a
# missing activation, a skipped block, a stage's layers in the wrong order) shows up as a mismatch.

def _lt(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float64))


def _lib_conv(x, p, name):
    """Causal 3x3x3 conv: frame 0 twice in front, one zero pixel on each spatial side."""
    w = _lt(p[name + ".weight"])
    front = x[:, :, :1].expand(-1, -1, w.shape[2] - 1, -1, -1)
    return torch.nn.functional.conv3d(torch.cat([front, x], dim=2), w, _lt(p[name + ".bias"]), padding=(0, 1, 1))


def _lib_norm(x, p, name, groups, eps, kind):
    """Group norm of each frame ([B*T, C, H, W] view), or RMS norm over the channels of each pixel."""
    b, c, t, h, w = x.shape
    g, bt = _lt(p[name + ".gamma"]), _lt(p[name + ".beta"])
    if kind == "rms":
        y = torch.nn.functional.rms_norm(x.permute(0, 2, 3, 4, 1), (c,), eps=eps) * g + bt
        return y.permute(0, 4, 1, 2, 3)
    v = x.permute(0, 2, 1, 3, 4).reshape(b * t, c, h, w)
    y = torch.nn.functional.group_norm(v, groups, g, bt, eps)
    return y.reshape(b, t, c, h, w).permute(0, 2, 1, 3, 4)


def _lib_d2s(x, s, drop_first):
    """Channel c*S + dt*sh*sw + dy*sw + dx -> (c, st*t + dt, sh*y + dy, sw*x + dx), by strided writes."""
    st, sh, sw = s
    S = st * sh * sw
    b, cs, t, h, w = x.shape
    y = torch.empty((b, cs // S, st * t, sh * h, sw * w), dtype=x.dtype)
    for dt in range(st):
        for dy in range(sh):
            for dx in range(sw):
                y[:, :, dt::st, dy::sh, dx::sw] = x[:, dt * sh * sw + dy * sw + dx::S]
    return y[:, :, st - 1:] if drop_first and st > 1 else y


def _lib_resblock(x, p, prefix, groups, eps, kind):
    silu = torch.nn.functional.silu
    hmid = _lib_conv(silu(_lib_norm(x, p, prefix + ".norm1", groups, eps, kind)), p, prefix + ".conv1")
    hmid = _lib_conv(silu(_lib_norm(hmid, p, prefix + ".norm2", groups, eps, kind)), p, prefix + ".conv2")
    return x + hmid


def _lib_attention(x, p, prefix, groups, eps, kind):
    b, c, t, h, w = x.shape
    tok = _lib_norm(x, p, prefix + ".norm", groups, eps, kind).permute(0, 2, 3, 4, 1).reshape(b * t, 1, h * w, c)
    lin = lambda a, n: torch.nn.functional.linear(a, _lt(p[f"{prefix}.{n}.weight"]), _lt(p[f"{prefix}.{n}.bias"]))
    o = torch.nn.functional.scaled_dot_product_attention(lin(tok, "q"), lin(tok, "k"), lin(tok, "v"))
    return x + lin(o, "o").reshape(b, t, h, w, c).permute(0, 4, 1, 2, 3)


def _lib_decode(cfg, p, z):
    g, eps, kind = cfg.gn_groups, cfg.gn_eps, cfg.norm
    x = _lib_conv(_lt(z), p, "conv_in")
    for r in range(cfg.mid_res):
        x = _lib_resblock(x, p, f"mid.res{r}", g, eps, kind)
    if cfg.mid_attn:
        x = _lib_attention(x, p, "mid.attn", g, eps, kind)
    for i in range(cfg.n_stages):
        for r in range(cfg.n_res[i]):
            x = _lib_resblock(x, p, f"stage{i}.res{r}", g, eps, kind)
        if i + 1 < cfg.n_stages:
            x = _lib_d2s(_lib_conv(x, p, f"stage{i}.up"), cfg.up[i], True)
    x = torch.nn.functional.silu(_lib_norm(x, p, "head.norm", g, eps, kind))
    return _lib_d2s(_lib_conv(x, p, "head.conv"), cfg.out_d2s, True).numpy()


@pytest.mark.parametrize("kind", ["group", "rms"])
def test_resblock_vs_library(kind):
    # random norm affines and conv biases, so that norm1 / norm2 and conv1 / conv2 are told apart
    cfg = synth.TINY
    p = synth.draw_params(cfg, 0, rand_affine=True)
    x = synth.draw_normal((1, 32, 3, 5, 6), 26).astype(np.float64)
    y = ops.resblock(x, p, "stage0.res1", 8, 1e-6, decoder._ConvRunner(p, "A"), kind)
    ref = _lib_resblock(_lt(x), p, "stage0.res1", 8, 1e-6, kind).numpy()
    np.testing.assert_allclose(y, ref, rtol=1e-10, atol=1e-10)


@pytest.mark.parametrize("name", ["tiny", "mini_wan", "mini_ltx", "mini_wan_rms"])
def test_decoder_vs_library(name):
    cfg = synth.CONFIGS[name]
    p = synth.draw_params(cfg, 0, rand_affine=True)
    z = synth.draw_latent(cfg, 0)
    y = decoder.decode(cfg, p, z)
    ref = _lib_decode(cfg, p, z)
    assert y.shape == ref.shape
    assert metrics.max_rel(y, ref) < 1e-10


@pytest.mark.parametrize("name", ["tiny", "mini_wan"])
def test_every_parameter_reaches_the_output(name):
    # a skipped layer, norm or projection would leave its parameters without effect on the pixels.
    # The one exception is exact: a key bias adds q.b_k to every score of a query, and the softmax
    # over keys ignores a per-query constant, so that bias must have no effect.
    cfg = synth.CONFIGS[name]
    p = synth.draw_params(cfg, 0, rand_affine=True)
    z = synth.draw_latent(cfg, 0)
    y = decoder.decode(cfg, p, z, tier="B")
    for k in p:
        q = dict(p)
        q[k] = p[k] + synth.draw_normal(p[k].shape, 27, std=0.5)
        change = np.abs(decoder.decode(cfg, q, z, tier="B") - y).max() / np.abs(y).max()
        if k.endswith("attn.k.bias"):
            assert change < 1e-5, k
        else:
            assert change > 1e-4, k


@pytest.mark.parametrize("name", ["tiny", "mini_wan", "mini_wan_rms"])
def test_causality(name):
    cfg = synth.CONFIGS[name]
    p = synth.draw_params(cfg, 0)
    z = synth.draw_latent(cfg, 0)
    y = decoder.decode(cfg, p, z)
    st = cfg.scale()[0]
    k = 1
    z2 = z.copy()
    z2[:, :, k + 1:] += synth.draw_normal(z2[:, :, k + 1:].shape, 25)
    y2 = decoder.decode(cfg, p, z2)
    keep = st * k + 1  # output frames 0 .. st*k depend on latent frames 0..k only
    np.testing.assert_array_equal(y2[:, :, :keep], y[:, :, :keep])
    assert np.abs(y2[:, :, keep:] - y[:, :, keep:]).max() > 1e-3


@pytest.mark.parametrize("name", ["tiny", "mini_wan", "mini_wan_rms", "mini_ltx"])
def test_chunked_equals_whole(name):
    cfg = synth.CONFIGS[name]
    p = synth.draw_params(cfg, 0, rand_affine=True)
    z = synth.draw_latent(cfg, 0)
    y = decoder.decode(cfg, p, z)
    for per in (1, 2, z.shape[2]):
        yc = decoder.decode(cfg, p, z, chunks=decoder.chunk_sizes(z.shape[2], per))
        np.testing.assert_allclose(yc, y, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("name,ph,pw", [("tiny", 2, 2), ("tiny", 1, 3), ("mini_wan", 2, 4), ("mini_ltx", 3, 2),
                                        ("mini_wan_rms", 2, 3)])
def test_patched_equals_unpatched(name, ph, pw):
    cfg = synth.CONFIGS[name]
    p = synth.draw_params(cfg, 0, rand_affine=True)
    z = synth.draw_latent(cfg, 0)
    np.testing.assert_allclose(patched.decode_patched(cfg, p, z, ph, pw), decoder.decode(cfg, p, z),
                               rtol=1e-11, atol=1e-11)


def test_patched_halo_matters():
    # a patched decode that ignored the neighbours (zero halo) would differ: guards the invariant
    cfg = synth.TINY
    p = synth.draw_params(cfg, 0)
    z = synth.draw_latent(cfg, 0)
    orig = patched._halo_extend
    try:
        def no_halo(g, i, j):
            e = orig(g, i, j)
            e[:, :, :, 0, :] = e[:, :, :, -1, :] = 0
            e[:, :, :, :, 0] = e[:, :, :, :, -1] = 0
            return e
        patched._halo_extend = no_halo
        bad = patched.decode_patched(cfg, p, z, 2, 2)
    finally:
        patched._halo_extend = orig
    assert metrics.max_rel(bad, decoder.decode(cfg, p, z)) > 1e-3


def test_tier_b_matches_tier_a():
    cfg = synth.MINI_WAN
    p = synth.draw_params(cfg, 0, rand_affine=True)
    z = synth.draw_latent(cfg, 0)
    assert metrics.max_rel(decoder.decode(cfg, p, z, tier="B"), decoder.decode(cfg, p, z)) < 1e-5


# ----------------------------------------------------------------------------- plans

def test_band_rule_golden():
    with open(os.path.join(GOLDEN, "band_rule.json")) as f:
        g = json.load(f)
    for case in g["cases"]:
        assert plan.band_sizes(case["rows"], case["n"]) == case["sizes"]
    for length in range(1, 40):
        for n in range(1, min(length, 9) + 1):
            s = plan.band_sizes(length, n)
            assert sum(s) == length and max(s) - min(s) <= 1 and s == sorted(s, reverse=True)
    with pytest.raises(plan.PatchTooNarrow) as e:
        plan.band_edges(3, 4)
    assert e.value.rows == 0 and e.value.reach == 1
    assert plan.band_edges(10, 4, scale=8) == [0, 24, 48, 64, 80]


def test_tile_plan_golden():
    with open(os.path.join(GOLDEN, "tile_grids.json")) as f:
        g = json.load(f)
    for case in g["axis_cases"]:
        got = tiles.axis_tiles(case["length"], case["tile"], case["overlap"])
        assert [s for s, _ in got] == case["starts"], case
        assert [n for _, n in got] == case["extents"], case
    t = tiles.tile_plan((17, 34, 60), (8, 16, 16), (1, 4, 4), 8, 32)
    assert len(t) == 45
    assert t[0].pix == (0, 57, 0, 512, 0, 512)
    assert t[-1].lat == (14, 3, 24, 10, 48, 12) and t[-1].pix == (112, 17, 768, 320, 1536, 384)
    assert all(tl.ovl[2:] in [(0, 128, 0, 128), (128, 128, 0, 128), (128, 0, 0, 128), (0, 128, 128, 128),
                              (128, 128, 128, 128), (128, 0, 128, 128), (0, 128, 128, 0),
                              (128, 128, 128, 0), (128, 0, 128, 0)] for tl in t)
    assert {tl.ovl[:2] for tl in t} == {(0, 1), (1, 1), (1, 0)}


def test_ramps_sum_to_one_in_overlaps():
    for p in (1, 3, 64, 128):
        n = 2 * p + 5
        a = tiles.ramp(n, 0, p)
        b = tiles.ramp(n, p, 0)
        np.testing.assert_allclose(a[n - p:] + b[:p], 1.0, rtol=0, atol=1e-15)
        assert (a[:n - p] == 1).all() and (b[p:] == 1).all()


def test_blend_brute_force_and_constant():
    t = tiles.tile_plan((1, 24, 20), (1, 10, 8), (0, 3, 3), 1, 1, causal_t=False)
    shape = (1, 2, 1, 24, 20)
    data = [synth.draw_normal((1, 2) + (tl.pix[1], tl.pix[3], tl.pix[5]), 30 + i).astype(np.float64)
            for i, tl in enumerate(t)]
    out = tiles.blend(t, data, shape)
    # brute force per pixel: weights from the per-axis ramps, normalised
    for y in range(24):
        for x in range(20):
            num = np.zeros(2)
            den = 0.0
            for tl, d in zip(t, data):
                _, _, h0, nh, w0, nw = tl.pix
                if h0 <= y < h0 + nh and w0 <= x < w0 + nw:
                    wy = tiles.ramp(nh, tl.ovl[2], tl.ovl[3])[y - h0]
                    wx = tiles.ramp(nw, tl.ovl[4], tl.ovl[5])[x - w0]
                    num += wy * wx * d[0, :, 0, y - h0, x - w0]
                    den += wy * wx
            np.testing.assert_allclose(out[0, :, 0, y, x], num / den, rtol=1e-13)
    const = tiles.blend(t, [np.full_like(d, 3.25) for d in data], shape)
    np.testing.assert_allclose(const, 3.25, rtol=1e-15)


def test_blend_frame_window_equals_full_blend():
    # forming only a window of output frames gives exactly those frames of the full blend
    t = tiles.tile_plan((4, 10, 9), (2, 6, 5), (1, 2, 2), 4, 1)  # causal time: 13 frames, 1-frame overlaps
    shape = (1, 2, 13, 10, 9)
    data = [synth.draw_normal((1, 2) + (tl.pix[1], tl.pix[3], tl.pix[5]), 40 + i).astype(np.float64)
            for i, tl in enumerate(t)]
    full = tiles.blend(t, data, shape)
    for f0, f1 in [(0, 13), (3, 6), (4, 5), (12, 13)]:
        np.testing.assert_array_equal(tiles.blend(t, data, shape, frames=(f0, f1)), full[:, :, f0:f1])


def test_single_tile_equals_untiled_decode():
    cfg = synth.TINY
    p = synth.draw_params(cfg, 0)
    z = synth.draw_latent(cfg, 0)
    out, plan_, _ = tiles.tiled_decode(cfg, p, z, (3, 16, 16), (1, 4, 4))
    assert len(plan_) == 1
    np.testing.assert_array_equal(out, decoder.decode(cfg, p, z))


def test_metrics_closed_forms():
    r = np.array([0.0, 1.0, -1.0, 2.0])
    g = r + np.array([0.0, 0.1, 0.0, -0.2])
    assert abs(metrics.max_rel(g, r) - 0.1) < 1e-15
    assert abs(metrics.rel_l2(g, r) - np.sqrt(0.05) / np.sqrt(6)) < 1e-15
    assert abs(metrics.psnr(g, r) - 20 * np.log10(3 / np.sqrt(0.05 / 4))) < 1e-12
