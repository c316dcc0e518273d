"""Full-size parity (720p x 81 frames) in the launch configuration the benchmark times.

The CPU oracle cannot decode a whole 720p x 81f video in test time, so full-size checks use
properties that hold at any size plus a prefix the oracle can afford:
  * bit-identical output across patch grids (1x1, 2x2, 2x4 / 1x4), and chunked == whole (chunks of
    1, 4 and 21 latent frames for the Wan-shaped decoder, 1 and 4 for the LTX-shaped one);
  * causality: output frames 0 .. s_t*(k-1) depend only on latent frames 0 .. k-1, so the first
    frames of the full decode must match the oracle's decode of the first latent frame(s) at full
    spatial size (bf16 bar: relative L2 <= 1e-2, PSNR >= 50 dB against the fp32 oracle; the fp32
    parity mode: max relative error <= 1e-4; the fp32 mode with three-TF32 tensor-core convs:
    relative L2 <= 1e-3).
"""
import dataclasses

import numpy as np
import pytest
import torch

from oracle import decoder as odec
from oracle import metrics
from patch_tiled_causal_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def vd():
    from patch_tiled_causal_gb300 import build, vaedec
    build.build()
    vaedec.load()
    return vaedec


def _decoder(vd, cfg):
    p = synth.draw_params(cfg, 0)
    return vd.Decoder(cfg, p, vd.VAE_BF16), p


@pytest.mark.parametrize("name,grids", [("ltx", [(1, 1), (2, 2), (2, 4)]), ("wan", [(1, 1), (1, 4), (2, 2)])])
def test_full_size_bit_identical_across_patch_grids(vd, name, grids):
    cfg = synth.CONFIGS[name]
    dec, _ = _decoder(vd, cfg)
    z = torch.from_numpy(synth.draw_latent(cfg, 0)).cuda()
    ref = dec.decode(z, n_patch_h=grids[0][0], n_patch_w=grids[0][1])
    out = torch.empty_like(ref)
    for ph, pw in grids[1:]:
        dec.decode(z, out, n_patch_h=ph, n_patch_w=pw)
        torch.cuda.synchronize()
        assert torch.equal(out, ref), (name, ph, pw)
    assert vd.last_error(dec.h)[0] == vd.VAE_OK
    dec.close()


@pytest.mark.parametrize("name,pers", [("wan", (1, 4, 21)), ("ltx", (1, 4))])
def test_full_size_chunked_equals_whole(vd, name, pers):
    # chunk 0 = latent frame 0, then chunks of `per` latent frames (per = 21: the rest in one piece)
    cfg = synth.CONFIGS[name]
    st = cfg.scale()[0]
    dec, _ = _decoder(vd, cfg)
    z = torch.from_numpy(synth.draw_latent(cfg, 0)).cuda()
    whole = dec.decode(z, n_patch_h=1, n_patch_w=4)
    for per in pers:
        t0 = 0
        for i, s in enumerate(odec.chunk_sizes(z.shape[2], per)):
            part = dec.decode_chunk(z[:, :, t0:t0 + s].contiguous(), i == 0, n_patch_h=1, n_patch_w=4)
            f0 = 0 if i == 0 else 1 + st * (t0 - 1)
            assert torch.equal(part, whole[:, :, f0:f0 + part.shape[2]]), (per, i)
            t0 += s
    assert vd.last_error(dec.h)[0] == vd.VAE_OK
    dec.close()


_prefix_refs = {}


def _prefix_ref(cfg, p, zn, k):
    # the oracle's decode of the first k latent frames at full spatial size (shared by the dtype cases)
    if (cfg.name, k) not in _prefix_refs:
        sub = dataclasses.replace(cfg, latent_shape=(1, cfg.latent_c, k) + cfg.latent_shape[3:])
        _prefix_refs[(cfg.name, k)] = odec.decode(sub, p, zn[:, :, :k].copy(), tier="B")
    return _prefix_refs[(cfg.name, k)]


@pytest.mark.parametrize("name,k,dt", [("ltx", 2, "bf16"), ("ltx", 2, "fp32"), ("ltx", 2, "fp32tc"),
                                       ("wan", 1, "bf16")])
def test_full_size_prefix_matches_oracle(vd, name, k, dt):
    # bf16 bar: relative L2 <= 1e-2 and PSNR >= 50 dB; fp32 (the CUDA-core parity mode): max relative
    # error <= 1e-4 against the oracle's float32 tier (itself within 1e-6 of its float64 tier here);
    # fp32tc (convs as three TF32 products on the tensor cores, whose fp32 accumulation over up to
    # 27 x 1024 terms measured 2.8e-4): relative L2 <= 1e-3
    cfg = synth.CONFIGS[name]
    p = synth.draw_params(cfg, 0)
    dec = vd.Decoder(cfg, p, {"bf16": vd.VAE_BF16, "fp32": vd.VAE_FP32, "fp32tc": vd.VAE_FP32_TC}[dt])
    zn = synth.draw_latent(cfg, 0)
    y = dec.decode(torch.from_numpy(zn).cuda(), n_patch_h=1, n_patch_w=4)
    st = cfg.scale()[0]
    nf = st * (k - 1) + 1
    got = y[:, :, :nf].float().cpu().numpy()
    assert vd.last_error(dec.h)[0] == vd.VAE_OK
    dec.close()
    ref = _prefix_ref(cfg, p, zn, k)
    assert ref.shape == got.shape
    rl2, ps = metrics.rel_l2(got, ref), metrics.psnr(got, ref)
    print(f"{name} {dt}: first {nf} frames, rel L2 {rl2:.3e}, PSNR {ps:.1f} dB")
    if dt == "bf16":
        assert rl2 <= 1e-2 and ps >= 50.0
    elif dt == "fp32":
        assert metrics.max_rel(got, ref) <= 1e-4
    else:
        assert rl2 <= 1e-3
