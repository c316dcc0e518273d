"""Whole-decoder parity on the GPU through the C ABI, against the CPU oracle.

Bars: fp32 storage mode max relative error <= 1e-4 (max|g - r| / max|r|); bf16 mode relative
L2 <= 1e-2 and PSNR >= 50 dB (peak = max - min of the fp32 reference) against the fp32 oracle;
bit-identical output across patch counts, and chunked == whole, on the GPU.
"""
import dataclasses

import numpy as np
import pytest
import torch

from oracle import decoder as odec
from oracle import metrics, tiles
from patch_tiled_causal_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def vd():
    from patch_tiled_causal_gb300 import build, vaedec
    build.build()
    vaedec.load()
    return vaedec


_cache = {}


def oracle_out(cfg, rand_affine, tier="A"):
    key = (cfg.name, cfg.latent_shape, rand_affine, tier)
    if key not in _cache:
        p = synth.draw_params(cfg, 0, rand_affine=rand_affine)
        z = synth.draw_latent(cfg, 0)
        _cache[key] = odec.decode(cfg, p, z, tier=tier)
    return _cache[key]


def gpu_decode(vd, cfg, dtype, nph=1, npw=1, rand_affine=True):
    p = synth.draw_params(cfg, 0, rand_affine=rand_affine)
    z = torch.from_numpy(synth.draw_latent(cfg, 0)).cuda()
    dec = vd.Decoder(cfg, p, dtype)
    y = dec.decode(z, n_patch_h=nph, n_patch_w=npw)
    torch.cuda.synchronize()
    code, msg = vd.last_error(dec.h)
    assert code == vd.VAE_OK, msg
    dec.close()
    return y.float().cpu().numpy()


@pytest.mark.parametrize("name", ["tiny", "mini_ltx", "mini_wan", "mini_wan_rms"])
@pytest.mark.parametrize("dt", ["fp32", "fp32tc"])
def test_fp32_mode_matches_oracle(vd, name, dt):
    # fp32tc: the convs as three TF32 products on the tensor cores (the small decoders' sums of at most
    # 27 x 128 terms stay within the fp32 bar)
    cfg = synth.CONFIGS[name]
    g = gpu_decode(vd, cfg, vd.VAE_FP32 if dt == "fp32" else vd.VAE_FP32_TC, 2, 2)
    r = oracle_out(cfg, True)
    assert g.shape == r.shape
    assert metrics.max_rel(g, r) <= 1e-4


@pytest.mark.parametrize("name", ["tiny", "mini_ltx", "mini_wan", "mini_wan_rms", "mini_wan_rms_g0"])
def test_bf16_mode_matches_oracle(vd, name):
    # mini_wan_rms_g0: the channel-RMS decoder handed gn_groups = 0 (it keeps no group statistics)
    cfg = synth.CONFIGS[name.replace("_g0", "")]
    gcfg = dataclasses.replace(cfg, gn_groups=0) if name.endswith("_g0") else cfg
    g = gpu_decode(vd, gcfg, vd.VAE_BF16, 2, 3)
    r = oracle_out(cfg, True)
    assert metrics.rel_l2(g, r) <= 1e-2
    assert metrics.psnr(g, r) >= 50.0


@pytest.mark.parametrize("name,grids", [("mini_ltx", [(1, 1), (2, 2), (2, 4), (3, 5), (10, 13)]),
                                        ("mini_wan", [(1, 1), (1, 4), (3, 2), (9, 11)]),
                                        ("mini_wan_rms", [(1, 1), (2, 3), (9, 11)]),
                                        ("tiny", [(1, 1), (2, 2), (4, 4), (16, 16)])])
@pytest.mark.parametrize("dt", ["bf16", "fp32", "fp32tc"])
def test_bit_identical_across_patch_counts(vd, name, grids, dt):
    cfg = synth.CONFIGS[name]
    dtc = {"bf16": vd.VAE_BF16, "fp32": vd.VAE_FP32, "fp32tc": vd.VAE_FP32_TC}[dt]
    outs = [gpu_decode(vd, cfg, dtc, ph, pw) for ph, pw in grids]
    for o in outs[1:]:
        np.testing.assert_array_equal(o, outs[0])


@pytest.mark.parametrize("dt", ["bf16", "fp32", "fp32tc"])
@pytest.mark.parametrize("per", [1, 2])
@pytest.mark.parametrize("base", ["mini_wan", "mini_wan_rms", "mini_ltx"])
def test_chunked_equals_whole(vd, dt, per, base):
    c0 = synth.CONFIGS[base]
    cfg = dataclasses.replace(c0, latent_shape=(1, c0.latent_c, 4, 9, 11))
    dtc = {"bf16": vd.VAE_BF16, "fp32": vd.VAE_FP32, "fp32tc": vd.VAE_FP32_TC}[dt]
    p = synth.draw_params(cfg, 0, rand_affine=True)
    z = torch.from_numpy(synth.draw_latent(cfg, 0)).cuda()
    dec = vd.Decoder(cfg, p, dtc)
    whole = dec.decode(z, n_patch_h=1, n_patch_w=2).float().cpu().numpy()
    outs, t0 = [], 0
    for i, s in enumerate(odec.chunk_sizes(z.shape[2], per)):
        outs.append(dec.decode_chunk(z[:, :, t0:t0 + s].contiguous(), i == 0, n_patch_h=1, n_patch_w=2))
        t0 += s
    torch.cuda.synchronize()
    chunked = torch.cat(outs, dim=2).float().cpu().numpy()
    dec.close()
    np.testing.assert_array_equal(chunked, whole)


@pytest.mark.parametrize("dt", ["bf16", "fp32"])
@pytest.mark.parametrize("per", [0, 1, 3])
@pytest.mark.parametrize("base", ["mini_wan", "mini_ltx"])
def test_host_decode_equals_device_decode(vd, dt, per, base):
    # host latent in, host pixels out, copies overlapped with the chunked decode: the same bits as decode()
    c0 = synth.CONFIGS[base]
    cfg = dataclasses.replace(c0, latent_shape=(2, c0.latent_c, 6, 9, 11))
    dtc = vd.VAE_BF16 if dt == "bf16" else vd.VAE_FP32
    p = synth.draw_params(cfg, 0, rand_affine=True)
    zn = synth.draw_latent(cfg, 0)
    dec = vd.Decoder(cfg, p, dtc)
    ref = dec.decode(torch.from_numpy(zn).cuda(), n_patch_h=2, n_patch_w=1).cpu()
    got = dec.decode_host(torch.from_numpy(zn).pin_memory(), n_patch_h=2, n_patch_w=1, frames_per_chunk=per)
    torch.cuda.synchronize()
    assert vd.last_error(dec.h)[0] == vd.VAE_OK
    dec.close()
    assert torch.equal(got, ref)


@pytest.mark.parametrize("dt", ["bf16", "fp32"])
def test_tiled_decode_matches_oracle(vd, dt):
    cfg = synth.MINI_TILED
    dtc = vd.VAE_BF16 if dt == "bf16" else vd.VAE_FP32
    p = synth.draw_params(cfg, 0, rand_affine=True)
    zn = synth.draw_latent(cfg, 0)
    ref, plan_, _ = tiles.tiled_decode(cfg, p, zn, synth.MINI_TILING.tile, synth.MINI_TILING.overlap)
    dec = vd.Decoder(cfg, p, dtc)
    g = dec.decode_tiled(torch.from_numpy(zn).cuda(), synth.MINI_TILING.tile, synth.MINI_TILING.overlap)
    torch.cuda.synchronize()
    g = g.float().cpu().numpy()
    dec.close()
    assert g.shape == ref.shape
    if dt == "fp32":
        assert metrics.max_rel(g, ref) <= 1e-4
    else:
        assert metrics.rel_l2(g, ref) <= 1e-2 and metrics.psnr(g, ref) >= 50.0


def test_refusals(vd):
    cfg = synth.TINY
    p = synth.draw_params(cfg, 0)
    dec = vd.Decoder(cfg, p, vd.VAE_BF16)
    z = torch.from_numpy(synth.draw_latent(cfg, 0)).cuda()
    with pytest.raises(vd.VaeError) as e:
        dec.decode(z, n_patch_h=17, n_patch_w=1)  # 16 latent rows cannot make 17 bands
    assert e.value.code == vd.VAE_ERR_PATCH_TOO_NARROW
    with pytest.raises(vd.VaeError) as e:
        dec.decode_chunk(z[:, :, 1:].contiguous(), False)  # a later chunk before the first
    assert e.value.code == vd.VAE_ERR_INVALID_ARG
    dec.close()
