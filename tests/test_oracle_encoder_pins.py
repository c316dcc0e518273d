"""Pins of the CPU oracle's encoder against things other than itself.

Space-to-depth against torch's pixel_unshuffle and as the exact inverse of depth-to-space; the
stride-2 down-sampler against torch's conv2d after F.pad and against brute-force loops; the whole
encoder against a second formulation built from library routines; causality, Tier A == Tier B,
every parameter reaching the output, and the tiled encode's single-tile and constant cases.
"""
import numpy as np
import pytest
import torch

from oracle import encoder, metrics, ops, tiles
from patch_tiled_causal_gb300 import synth


def _lt(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float64))


# ----------------------------------------------------------------------------- space-to-depth

def test_space_to_depth_is_pixel_unshuffle_per_frame():
    x = synth.draw_normal((2, 3, 4, 8, 12), 50).astype(np.float64)
    y = ops.space_to_depth(x, (1, 2, 2), pad_first=False)
    for t in range(4):
        ref = torch.nn.functional.pixel_unshuffle(_lt(x[:, :, t]), 2).numpy()
        np.testing.assert_array_equal(y[:, :, t], ref)


@pytest.mark.parametrize("s", [(2, 2, 2), (1, 4, 4), (2, 1, 3)])
def test_space_to_depth_inverts_depth_to_space(s):
    st = s[0]
    x = synth.draw_normal((1, 5, 1 + st * 3, 3 * s[1], 2 * s[2]), 51).astype(np.float64)
    y = ops.space_to_depth(x, s, pad_first=True)
    assert y.shape[2] == (x.shape[2] - 1) // st + 1        # causal: first frame -> one frame
    np.testing.assert_array_equal(ops.depth_to_space(y, s, drop_first=True), x)
    z = synth.draw_normal((1, 5 * s[0] * s[1] * s[2], 3, 2, 2), 52).astype(np.float64)
    np.testing.assert_array_equal(ops.space_to_depth(ops.depth_to_space(z, s, drop_first=False), s, pad_first=False), z)


def test_space_to_depth_brute_force():
    st, sh, sw = 2, 2, 3
    x = synth.draw_normal((1, 2, 3, 4, 6), 53).astype(np.float64)
    y = ops.space_to_depth(x, (st, sh, sw), pad_first=True)
    for c in range(2):
        for t in range(y.shape[2]):
            for i in range(y.shape[3]):
                for j in range(y.shape[4]):
                    for dt in range(st):
                        for dy in range(sh):
                            for dx in range(sw):
                                src_t = max(st * t + dt - (st - 1), 0)   # frame 0 repeated in front
                                ch = c * st * sh * sw + dt * sh * sw + dy * sw + dx
                                assert y[0, ch, t, i, j] == x[0, c, src_t, sh * i + dy, sw * j + dx]


# ----------------------------------------------------------------------------- stride-2 down-sampler

def test_stride2_conv_vs_torch_and_brute_force():
    x = synth.draw_normal((1, 3, 2, 6, 8), 54).astype(np.float64)
    w = synth.draw_normal((4, 3, 3, 3), 55).astype(np.float64)
    b = synth.draw_normal((4,), 56).astype(np.float64)
    y = ops.conv2d_stride2_pad_end(x, w, b)
    for t in range(2):
        ref = torch.nn.functional.conv2d(torch.nn.functional.pad(_lt(x[:, :, t]), (0, 1, 0, 1)), _lt(w), _lt(b), stride=2)
        np.testing.assert_allclose(y[:, :, t], ref.numpy(), rtol=1e-12, atol=1e-12)
    for o in range(4):
        for i in range(3):
            for j in range(4):
                s = b[o]
                for kh in range(3):
                    for kw in range(3):
                        r, c = 2 * i + kh, 2 * j + kw
                        if r < 6 and c < 8:                     # one zero row below, one column right
                            s += (w[o, :, kh, kw] * x[0, :, 1, r, c]).sum()
                np.testing.assert_allclose(y[0, o, 1, i, j], s, rtol=1e-12)
    np.testing.assert_allclose(ops.conv2d_stride2_pad_end(x, w, b, tier="B"), y, rtol=1e-5, atol=1e-5)


# ----------------------------------------------------------------------------- whole encoder

def _lib_conv(x, p, name):
    w = _lt(p[name + ".weight"])
    front = x[:, :, :1].expand(-1, -1, w.shape[2] - 1, -1, -1)
    return torch.nn.functional.conv3d(torch.cat([front, x], dim=2), w, _lt(p[name + ".bias"]), padding=(0, 1, 1))


def _lib_norm(x, p, name, groups, eps, kind):
    b, c, t, h, w = x.shape
    g, bt = _lt(p[name + ".gamma"]), _lt(p[name + ".beta"])
    if kind == "rms":
        return (torch.nn.functional.rms_norm(x.permute(0, 2, 3, 4, 1), (c,), eps=eps) * g + bt).permute(0, 4, 1, 2, 3)
    y = torch.nn.functional.group_norm(x.permute(0, 2, 1, 3, 4).reshape(b * t, c, h, w), groups, g, bt, eps)
    return y.reshape(b, t, c, h, w).permute(0, 2, 1, 3, 4)


def _lib_s2d(x, s, pad_first):
    """Fold by strided reads: channel c*S + dt*sh*sw + dy*sw + dx <- (c, st*t+dt, sh*y+dy, sw*x+dx)."""
    st, sh, sw = s
    if pad_first and st > 1:
        x = torch.cat([x[:, :, :1].expand(-1, -1, st - 1, -1, -1), x], dim=2)
    b, c, t, h, w = x.shape
    S = st * sh * sw
    y = torch.empty((b, c * S, t // st, h // sh, w // sw), dtype=x.dtype)
    for dt in range(st):
        for dy in range(sh):
            for dx in range(sw):
                y[:, dt * sh * sw + dy * sw + dx::S] = x[:, :, dt::st, dy::sh, dx::sw]
    return y


def _lib_resblock(x, p, prefix, g, eps, kind):
    silu = torch.nn.functional.silu
    h = _lib_conv(silu(_lib_norm(x, p, prefix + ".norm1", g, eps, kind)), p, prefix + ".conv1")
    return x + _lib_conv(silu(_lib_norm(h, p, prefix + ".norm2", g, eps, kind)), p, prefix + ".conv2")


def _lib_encode(cfg, p, video):
    g, eps, kind = cfg.gn_groups, cfg.gn_eps, cfg.norm
    x = _lt(video)
    if tuple(cfg.patchify) != (1, 1):
        x = _lib_s2d(x, (1,) + tuple(cfg.patchify), False)
    x = _lib_conv(x, p, "conv_in")
    for i in range(cfg.n_stages):
        for r in range(cfg.n_res[i]):
            x = _lib_resblock(x, p, f"stage{i}.res{r}", g, eps, kind)
        if i + 1 < cfg.n_stages:
            dkind, s = cfg.down[i]
            if dkind == "fold":
                x = _lib_s2d(_lib_conv(x, p, f"stage{i}.down"), s, True)
            else:
                b, c, t, h, w = x.shape
                f = x.permute(0, 2, 1, 3, 4).reshape(b * t, c, h, w)
                f = torch.nn.functional.conv2d(torch.nn.functional.pad(f, (0, 1, 0, 1)), _lt(p[f"stage{i}.down.weight"]),
                                               _lt(p[f"stage{i}.down.bias"]), stride=2)
                x = f.reshape(b, t, f.shape[1], h // 2, w // 2).permute(0, 2, 1, 3, 4)
    for r in range(cfg.mid_res):
        x = _lib_resblock(x, p, f"mid.res{r}", g, eps, kind)
    x = torch.nn.functional.silu(_lib_norm(x, p, "head.norm", g, eps, kind))
    return _lib_conv(x, p, "head.conv").numpy()


@pytest.mark.parametrize("name", ["tiny_enc", "tiny_enc_stride", "mini_enc", "mini_enc_stride", "mini_enc_rms"])
def test_encoder_vs_library(name):
    cfg = synth.ENCODERS[name]
    p = synth.draw_params(cfg, 0, rand_affine=True)
    v = synth.draw_video(cfg, 0)
    y = encoder.encode(cfg, p, v)
    ref = _lib_encode(cfg, p, v)
    assert y.shape == ref.shape == cfg.latent_shape()
    assert metrics.max_rel(y, ref) < 1e-10


@pytest.mark.parametrize("name", ["tiny_enc", "mini_enc_stride"])
def test_encoder_causality(name):
    cfg = synth.ENCODERS[name]
    p = synth.draw_params(cfg, 0)
    v = synth.draw_video(cfg, 0)
    y = encoder.encode(cfg, p, v)
    st = cfg.scale()[0]
    k = 1                                   # latent frames 0..k depend on pixel frames 0..st*k only
    v2 = v.copy()
    v2[:, :, st * k + 1:] += synth.draw_normal(v2[:, :, st * k + 1:].shape, 57)
    y2 = encoder.encode(cfg, p, v2)
    np.testing.assert_array_equal(y2[:, :, :k + 1], y[:, :, :k + 1])
    assert np.abs(y2[:, :, k + 1:] - y[:, :, k + 1:]).max() > 1e-3


def test_encoder_tier_b_matches_tier_a():
    cfg = synth.MINI_ENC
    p = synth.draw_params(cfg, 0, rand_affine=True)
    v = synth.draw_video(cfg, 0)
    assert metrics.max_rel(encoder.encode(cfg, p, v, tier="B"), encoder.encode(cfg, p, v)) < 1e-5


@pytest.mark.parametrize("name", ["tiny_enc", "tiny_enc_stride"])
def test_every_encoder_parameter_reaches_the_output(name):
    # One exception is exact: after a fold, a conv channel's bias is one constant on its S folded
    # channels; when every group of the group norms that follow lies inside one such block, each
    # norm (down to the head's, at the end of the residual stream) removes that per-group constant.
    cfg = synth.ENCODERS[name]
    p = synth.draw_params(cfg, 0, rand_affine=True)
    v = synth.draw_video(cfg, 0)
    y = encoder.encode(cfg, p, v, tier="B")
    invariant = set()
    for i, (kind, s) in enumerate(cfg.down):
        cpg = cfg.stage_c[i + 1] // cfg.gn_groups
        if kind == "fold" and cfg.norm == "group" and (s[0] * s[1] * s[2]) % cpg == 0:
            invariant.add(f"stage{i}.down.bias")
    for k in p:
        q = dict(p)
        q[k] = p[k] + synth.draw_normal(p[k].shape, 58, std=0.5)
        change = np.abs(encoder.encode(cfg, q, v, tier="B") - y).max() / np.abs(y).max()
        assert (change < 1e-5) if k in invariant else (change > 1e-4), (k, change)


# ----------------------------------------------------------------------------- tiled encode

def test_single_tile_equals_untiled_encode():
    cfg = synth.TINY_ENC
    p = synth.draw_params(cfg, 0, rand_affine=True)
    v = synth.draw_video(cfg, 0)
    lat = cfg.latent_shape()
    out, plan_, _ = encoder.tiled_encode(cfg, p, v, lat[3:], (0, 0))
    assert len(plan_) == 1
    np.testing.assert_allclose(out, encoder.encode(cfg, p, v), rtol=1e-13, atol=1e-13)


def test_tiled_encode_plan_and_constant_blend():
    cfg = synth.MINI_ENC_STRIDE                              # latent 6 x 10
    plan_ = encoder.tile_plan(cfg, cfg.video_shape, (4, 4), (2, 1))
    assert [t.lat[2:4] for t in plan_[::3]] == [(0, 4), (2, 4)]
    assert sorted({t.lat[4:6] for t in plan_}) == [(0, 4), (3, 4), (6, 4)]
    consts = [np.full((1, 32, 5, t.pix[3], t.pix[5]), -1.5) for t in plan_]
    np.testing.assert_allclose(tiles.blend(plan_, consts, cfg.latent_shape()), -1.5, rtol=1e-15)
