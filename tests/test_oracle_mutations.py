"""The oracle's pins catch plausible mistakes.

Each case plants one mistake in an oracle function (a dropped term, a wrong sign, index or operand
order, the wrong padding or estimator), on the CPU, for the duration of the case only, and checks
that the pin written for that function now fails.  The pins themselves live in
test_oracle_pins.py and are imported, not restated.
"""
import numpy as np
import pytest

from oracle import decoder, ops, tiles
from tests import test_oracle_pins as pins


def _fails(pin, *args):
    with pytest.raises(AssertionError):
        pin(*args)


def test_pins_pass_unmutated():
    # the same pins, run here on the untouched oracle, so a failure below can only be the mutation
    pins.test_conv_vs_torch_library()
    pins.test_conv_special_cases()
    pins.test_group_norm_population_variance()
    pins.test_group_norm_vs_torch(0.0)
    pins.test_d2s_vs_pixel_shuffle_and_inverse()
    pins.test_channel_rms_norm_vs_torch()
    pins.test_ramps_sum_to_one_in_overlaps()
    pins.test_silu_closed_form()
    pins.test_resblock_vs_library("group")
    pins.test_decoder_vs_library("mini_wan")


def test_flipped_kernel_is_caught(monkeypatch):
    # convolution instead of cross-correlation: taps reversed
    orig = ops.conv3d_valid_tierA
    monkeypatch.setattr(ops, "conv3d_valid_tierA", lambda xp, w, b: orig(xp, w[:, :, ::-1, ::-1, ::-1], b))
    _fails(pins.test_conv_vs_torch_library)


def test_zero_temporal_padding_is_caught(monkeypatch):
    # zeros in front instead of copies of frame 0
    orig = ops.causal_pad

    def zero_front(x, cache=None, k_t=3, pad_s=1):
        if cache is None:
            cache = np.zeros_like(x[:, :, :1]).repeat(k_t - 1, axis=2)
        return orig(x, cache, k_t, pad_s)
    monkeypatch.setattr(ops, "causal_pad", zero_front)
    _fails(pins.test_conv_vs_torch_library)


def test_bessel_corrected_variance_is_caught(monkeypatch):
    def bessel(x, groups):
        n, c, t, h, w = x.shape
        xg = x.astype(np.float64).transpose(0, 2, 1, 3, 4).reshape(n, t, groups, (c // groups) * h * w)
        return xg.mean(axis=-1), xg.var(axis=-1, ddof=1)
    monkeypatch.setattr(ops, "group_norm_stats", bessel)
    _fails(pins.test_group_norm_population_variance)
    _fails(pins.test_group_norm_vs_torch, 0.0)


def test_dropped_shift_is_caught(monkeypatch):
    orig = ops.group_norm
    monkeypatch.setattr(ops, "group_norm", lambda x, g, b, groups, eps: orig(x, g, 0.0 * b, groups, eps))
    _fails(pins.test_group_norm_vs_torch, 0.0)


def test_swapped_depth_to_space_order_is_caught(monkeypatch):
    # (dx, dy) read in the wrong order from the channel index
    orig = ops.depth_to_space

    def swapped(x, s, drop_first):
        st, sh, sw = s
        n, cs, t, h, w = x.shape
        c = cs // (st * sh * sw)
        xr = x.reshape(n, c, st, sh, sw, t, h, w).transpose(0, 1, 2, 4, 3, 5, 6, 7).reshape(n, cs, t, h, w)
        return orig(xr, s, drop_first)
    monkeypatch.setattr(ops, "depth_to_space", swapped)
    _fails(pins.test_d2s_vs_pixel_shuffle_and_inverse)


def test_rms_over_the_wrong_axis_is_caught(monkeypatch):
    # mean of squares over the width instead of the channels
    def wrong_axis(x, gamma, beta, eps):
        xd = x.astype(np.float64)
        y = xd / np.sqrt((xd * xd).mean(axis=4, keepdims=True) + eps)
        return y * gamma[None, :, None, None, None] + beta[None, :, None, None, None]
    monkeypatch.setattr(ops, "channel_rms_norm", wrong_axis)
    _fails(pins.test_channel_rms_norm_vs_torch)


def test_unshifted_ramp_is_caught(monkeypatch):
    # y / P instead of (y + 1) / (P + 1): the overlap weights no longer sum to one
    def shifted(n, p_lo, p_hi):
        w = np.ones(n)
        for y in range(n):
            if y < p_lo:
                w[y] *= y / p_lo
            if y >= n - p_hi:
                w[y] *= (n - 1 - y) / p_hi
        return w
    monkeypatch.setattr(tiles, "ramp", shifted)
    _fails(pins.test_ramps_sum_to_one_in_overlaps)


def test_sign_error_in_silu_is_caught(monkeypatch):
    def wrong_sign(x):
        with np.errstate(over="ignore"):
            return x / (1.0 + np.exp(x))
    monkeypatch.setattr(ops, "silu", wrong_sign)
    _fails(pins.test_silu_closed_form)


def test_swapped_norm_parameters_in_resblock_are_caught(monkeypatch):
    # norm2's scale and shift used for the first norm and norm1's for the second
    orig = ops.resblock

    def swapped(x, p, prefix, groups, eps, conv, kind="group"):
        q = dict(p)
        for k in ("gamma", "beta"):
            q[f"{prefix}.norm1.{k}"], q[f"{prefix}.norm2.{k}"] = p[f"{prefix}.norm2.{k}"], p[f"{prefix}.norm1.{k}"]
        return orig(x, q, prefix, groups, eps, conv, kind)
    monkeypatch.setattr(ops, "resblock", swapped)
    _fails(pins.test_resblock_vs_library, "group")
    _fails(pins.test_decoder_vs_library, "mini_wan")


def test_dropped_silu_before_conv2_is_caught(monkeypatch):
    def no_second_silu(x, p, prefix, groups, eps, conv, kind="group"):
        dt = x.dtype
        h = ops.silu(ops.norm(x, p[prefix + ".norm1.gamma"], p[prefix + ".norm1.beta"], groups, eps, kind)).astype(dt)
        h = conv(prefix + ".conv1", h)
        h = ops.norm(h, p[prefix + ".norm2.gamma"], p[prefix + ".norm2.beta"], groups, eps, kind).astype(dt)
        return x + conv(prefix + ".conv2", h)
    monkeypatch.setattr(ops, "resblock", no_second_silu)
    _fails(pins.test_resblock_vs_library, "group")
    _fails(pins.test_decoder_vs_library, "mini_wan")


def _mutated_chunk(skip=None, up_first=False):
    """The decoder's layer sequence with one residual block skipped, or with a stage's up-sampling
    conv run before that stage's residual blocks (where the channel counts allow it)."""
    def run(cfg, p, z, conv, dtype):
        g, eps, kind = cfg.gn_groups, cfg.gn_eps, cfg.norm
        x = conv("conv_in", z.astype(dtype))
        for r in range(cfg.mid_res):
            x = ops.resblock(x, p, f"mid.res{r}", g, eps, conv, kind).astype(dtype)
        if cfg.mid_attn:
            x = ops.spatial_attention(x, p, "mid.attn", g, eps, dtype=dtype, kind=kind).astype(dtype)
        for i in range(cfg.n_stages):
            early = up_first and i + 1 < cfg.n_stages and cfg.stage_c[i] == cfg.stage_c[i + 1]
            if early:
                x = ops.depth_to_space(conv(f"stage{i}.up", x), cfg.up[i], drop_first=conv.first)
            for r in range(cfg.n_res[i]):
                if (i, r) != skip:
                    x = ops.resblock(x, p, f"stage{i}.res{r}", g, eps, conv, kind).astype(dtype)
            if i + 1 < cfg.n_stages and not early:
                x = ops.depth_to_space(conv(f"stage{i}.up", x), cfg.up[i], drop_first=conv.first)
        x = ops.silu(ops.norm(x, p["head.norm.gamma"], p["head.norm.beta"], g, eps, kind)).astype(dtype)
        return ops.depth_to_space(conv("head.conv", x), cfg.out_d2s, drop_first=conv.first)
    return run


def test_skipped_resblock_is_caught(monkeypatch):
    monkeypatch.setattr(decoder, "_decode_chunk", _mutated_chunk(skip=(1, 0)))
    _fails(pins.test_decoder_vs_library, "mini_wan")


def test_up_conv_before_the_stage_resblocks_is_caught(monkeypatch):
    # mini_wan's first two stages have the same width, so the reordered decoder still runs
    monkeypatch.setattr(decoder, "_decode_chunk", _mutated_chunk(up_first=True))
    _fails(pins.test_decoder_vs_library, "mini_wan")


def test_unmutated_copy_of_the_layer_sequence_passes(monkeypatch):
    # the copy above, with no mutation switched on, is the oracle's sequence: the pin passes on it
    monkeypatch.setattr(decoder, "_decode_chunk", _mutated_chunk())
    pins.test_decoder_vs_library("mini_wan")
