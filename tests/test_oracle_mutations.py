"""The oracle's pins catch plausible mistakes.

Each case plants one mistake in an oracle function (a dropped term, a wrong sign, index or operand
order, the wrong padding or estimator), on the CPU, for the duration of the case only, and checks
that the pin written for that function now fails.  The pins themselves live in
test_oracle_pins.py and are imported, not restated.
"""
import numpy as np
import pytest

from oracle import ops, tiles
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
