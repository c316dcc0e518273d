"""Encoder parity on the GPU through the C ABI, against the CPU oracle's encoder.

The encoder is the decoder read backwards (DistVAE PR #14 "Add tiled VAE parallelism & extended model
support", encoder commits), with fold (stride-1 conv + space-to-depth) and strided down-samplers;
the tiled encode follows vllm-omni PR #4831 "VAE tiling parallel encode for LTX-2".

Bars as for the decoder: fp32 storage (CUDA-core or three-TF32 tensor-core convs) max relative error
<= 1e-4; bf16 relative L2 <= 1e-2 and
PSNR >= 50 dB against the fp32 oracle; fp8 (e4m3 operands) relative L2 <= 0.15 and PSNR >= 35 dB;
bit-identical moments across patch grids (the strided down-sampler's halo follows the patch's
place in the global stride grid).
"""
import dataclasses

import numpy as np
import pytest
import torch

from oracle import encoder as oenc
from oracle import metrics
from patch_tiled_causal_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def vd():
    from patch_tiled_causal_gb300 import build, vaedec
    build.build()
    vaedec.load()
    return vaedec


_cache = {}


def oracle_out(cfg, tier="A"):
    key = (cfg.name, cfg.video_shape, tier)
    if key not in _cache:
        p = synth.draw_params(cfg, 0, rand_affine=True)
        _cache[key] = oenc.encode(cfg, p, synth.draw_video(cfg, 0), tier=tier)
    return _cache[key]


def gpu_encode(vd, cfg, dtype, nph=1, npw=1):
    p = synth.draw_params(cfg, 0, rand_affine=True)
    enc = vd.Encoder(cfg, p, dtype)
    y = enc.encode(torch.from_numpy(synth.draw_video(cfg, 0)).cuda(), n_patch_h=nph, n_patch_w=npw)
    torch.cuda.synchronize()
    code, msg = enc.last_error()
    assert code == vd.VAE_OK, msg
    enc.close()
    return y.cpu().numpy()


NAMES = ["tiny_enc", "tiny_enc_stride", "mini_enc", "mini_enc_stride", "mini_enc_rms"]


@pytest.mark.parametrize("name", NAMES)
@pytest.mark.parametrize("dt", ["fp32", "fp32tc"])
def test_fp32_encoder_matches_oracle(vd, name, dt):
    # fp32tc: the convs as three TF32 products on the tensor cores
    cfg = synth.ENCODERS[name]
    g, r = gpu_encode(vd, cfg, vd.VAE_FP32 if dt == "fp32" else vd.VAE_FP32_TC, 2, 2), oracle_out(cfg)
    assert g.shape == r.shape == cfg.latent_shape()
    assert metrics.max_rel(g, r) <= 1e-4


@pytest.mark.parametrize("name", NAMES)
def test_bf16_encoder_matches_oracle(vd, name):
    cfg = synth.ENCODERS[name]
    g, r = gpu_encode(vd, cfg, vd.VAE_BF16, 2, 3 if cfg.latent_shape()[4] >= 3 else 1), oracle_out(cfg)
    rl2, ps = metrics.rel_l2(g, r), metrics.psnr(g, r)
    print(f"{name} bf16: rel L2 {rl2:.3e}, PSNR {ps:.1f} dB")
    assert rl2 <= 1e-2 and ps >= 50.0


@pytest.mark.parametrize("name", ["mini_enc", "mini_enc_stride"])
def test_fp8_encoder_matches_oracle(vd, name):
    cfg = synth.ENCODERS[name]
    g, r = gpu_encode(vd, cfg, vd.VAE_FP8, 1, 2), oracle_out(cfg)
    rl2, ps = metrics.rel_l2(g, r), metrics.psnr(g, r)
    print(f"{name} fp8: rel L2 {rl2:.3e}, PSNR {ps:.1f} dB")
    assert rl2 <= 0.15 and ps >= 35.0


@pytest.mark.parametrize("name,grids", [("mini_enc", [(1, 1), (2, 2), (5, 7), (3, 2)]),
                                        ("mini_enc_stride", [(1, 1), (2, 5), (6, 10), (3, 3)]),
                                        ("tiny_enc_stride", [(1, 1), (8, 8), (3, 5)])])
@pytest.mark.parametrize("dt", ["bf16", "fp32"])
def test_encoder_bit_identical_across_patch_counts(vd, name, grids, dt):
    cfg = synth.ENCODERS[name]
    dtc = vd.VAE_BF16 if dt == "bf16" else vd.VAE_FP32
    outs = [gpu_encode(vd, cfg, dtc, ph, pw) for ph, pw in grids]
    for o in outs[1:]:
        np.testing.assert_array_equal(o, outs[0])


@pytest.mark.parametrize("dt", ["bf16", "fp32"])
def test_tiled_encode_matches_oracle(vd, dt):
    cfg = dataclasses.replace(synth.MINI_ENC_STRIDE, video_shape=(2, 3, 5, 40, 56))   # latent 10 x 14
    tile, ovl = (4, 6), (1, 2)
    p = synth.draw_params(cfg, 0, rand_affine=True)
    v = synth.draw_video(cfg, 0)
    ref, plan_, _ = oenc.tiled_encode(cfg, p, v, tile, ovl)
    assert len(plan_) > 4
    dtc = vd.VAE_BF16 if dt == "bf16" else vd.VAE_FP32
    enc = vd.Encoder(cfg, p, dtc)
    g = enc.encode_tiled(torch.from_numpy(v).cuda(), tile, ovl)
    torch.cuda.synchronize()
    assert enc.last_error()[0] == vd.VAE_OK
    g = g.cpu().numpy()
    enc.close()
    if dt == "fp32":
        assert metrics.max_rel(g, ref) <= 1e-4
    else:
        assert metrics.rel_l2(g, ref) <= 1e-2 and metrics.psnr(g, ref) >= 50.0


@pytest.mark.parametrize("dt", ["bf16", "fp32"])
def test_tiled_encode_equals_blend_of_separate_tile_encodes(vd, dt):
    # the tiled driver batches the 9 equal-shape tiles into one encode of 18 items; each tile's moments
    # must be those of encoding its pixels on their own, and the blend the library blend of those
    cfg = dataclasses.replace(synth.MINI_ENC_STRIDE, video_shape=(2, 3, 5, 40, 56))   # latent 10 x 14
    tile, ovl = (4, 6), (1, 2)
    p = synth.draw_params(cfg, 0, rand_affine=True)
    dtc = vd.VAE_BF16 if dt == "bf16" else vd.VAE_FP32
    enc = vd.Encoder(cfg, p, dtc)
    vt = torch.from_numpy(synth.draw_video(cfg, 0)).cuda()
    out = enc.encode_tiled(vt, tile, ovl)
    lat = cfg.latent_shape()
    s = cfg.video_shape[3] // lat[3]
    meta = vd.tile_plan(lat[2:], (lat[2],) + tile, (0,) + ovl, 1, 1, False)
    assert len(meta) == 9
    parts = []
    for m in meta:
        _, _, h0, nh, w0, nw = m["lat"]
        parts.append(enc.encode(vt[:, :, :, h0 * s:(h0 + nh) * s, w0 * s:(w0 + nw) * s].contiguous()))
    out2 = vd.tile_blend(parts, meta, torch.full_like(out, float("nan")))
    torch.cuda.synchronize()
    assert enc.last_error()[0] == vd.VAE_OK
    enc.close()
    assert torch.equal(out2, out)


def test_encoder_refusals(vd):
    cfg = synth.MINI_ENC
    enc = vd.Encoder(cfg, synth.draw_params(cfg, 0), vd.VAE_BF16)
    v = torch.zeros((1, 3, 8, 40, 56), device="cuda")          # 8 frames: (T - 1) is not a multiple of 2
    with pytest.raises(vd.VaeError) as e:
        enc.encode(v, out=torch.empty(16, device="cuda"))
    assert e.value.code == vd.VAE_ERR_INVALID_ARG
    v = torch.zeros((1, 3, 9, 44, 56), device="cuda")          # 44 rows: not a multiple of 8
    with pytest.raises(vd.VaeError) as e:
        enc.encode(v, out=torch.empty(16, device="cuda"))
    assert e.value.code == vd.VAE_ERR_INVALID_ARG
    v = torch.zeros((1, 3, 9, 40, 56), device="cuda")          # 5 latent rows cannot make 6 bands
    with pytest.raises(vd.VaeError) as e:
        enc.encode(v, n_patch_h=6)
    assert e.value.code == vd.VAE_ERR_PATCH_TOO_NARROW
    enc.close()


def test_full_size_ltx_encoder(vd):
    # LTX-shaped encoder on 720p x 81 frames -> latent [1, 256, 11, 22, 40]: bit-identical across patch
    # grids; causal, so latent frame 0 depends on pixel frame 0 only and matches the oracle's encode of it
    cfg = synth.LTX_ENC
    p = synth.draw_params(cfg, 0)
    v = synth.draw_video(cfg, 0)
    enc = vd.Encoder(cfg, p, vd.VAE_BF16)
    vt = torch.from_numpy(v).cuda()
    ref = enc.encode(vt, n_patch_h=1, n_patch_w=1)
    out = torch.empty_like(ref)
    for ph, pw in ((2, 4), (1, 4)):
        enc.encode(vt, out, n_patch_h=ph, n_patch_w=pw)
        torch.cuda.synchronize()
        assert torch.equal(out, ref), (ph, pw)
    assert enc.last_error()[0] == vd.VAE_OK
    got = ref[:, :, :1].cpu().numpy()
    enc.close()
    sub = dataclasses.replace(cfg, video_shape=(1, 3, 1) + cfg.video_shape[3:])
    r = oenc.encode(sub, p, v[:, :, :1].copy(), tier="B")
    rl2, ps = metrics.rel_l2(got, r), metrics.psnr(got, r)
    print(f"ltx_enc: latent frame 0, rel L2 {rl2:.3e}, PSNR {ps:.1f} dB")
    assert rl2 <= 1e-2 and ps >= 50.0
