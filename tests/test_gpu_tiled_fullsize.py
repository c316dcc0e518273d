"""Full-size overlap-tiled decode: the LTX-shaped decoder on latent [2, 128, 17, 34, 60] (batch 2,
output [2, 3, 129, 1088, 1920]) in 3 x 3 x 5 = 45 tiles of 8 x 16 x 16 latents with a 1 x 4 x 4
overlap, blended linearly (TensorRT-LLM PR #15753 "LTX-2 tile-parallel VAE decode", Approach).

The oracle cannot decode 45 full tiles in test time, so the checks split the work:
  * the tile plan equals the oracle's, bit for bit;
  * vae_decode_tiled equals, bit for bit, vae_tile_blend over the 45 tiles decoded one by one with
    vae_decode (the tiled driver adds nothing of its own to the arithmetic);
  * those GPU tile outputs blended by the oracle's blend, over a window of output frames that spans
    the temporal overlap (and every spatial seam of those frames), match the GPU blend element by
    element within the bf16 bar of the op tests;
  * the first output frame of the corner tile matches the oracle's decode of that tile's first
    latent frame (relative L2 <= 1e-2, PSNR >= 50 dB against the fp32 oracle).
"""
import dataclasses

import numpy as np
import pytest
import torch

from oracle import decoder as odec
from oracle import metrics, tiles
from patch_tiled_causal_gb300 import synth

pytestmark = pytest.mark.gpu

BF16_TOL = 2.0 ** -8


@pytest.fixture(scope="module")
def vd():
    from patch_tiled_causal_gb300 import build, vaedec
    build.build()
    vaedec.load()
    return vaedec


@pytest.fixture(scope="module")
def tiled(vd):
    cfg, tl = synth.LTX_TILED, synth.LTX_TILING
    p = synth.draw_params(cfg, 0)
    zn = synth.draw_latent(cfg, 0)
    dec = vd.Decoder(cfg, p, vd.VAE_BF16)
    z = torch.from_numpy(zn).cuda()
    out = dec.decode_tiled(z, tl.tile, tl.overlap)
    torch.cuda.synchronize()
    assert vd.last_error(dec.h)[0] == vd.VAE_OK
    st, sh, _ = cfg.scale()
    meta = vd.tile_plan(zn.shape[2:], tl.tile, tl.overlap, st, sh)
    parts = []
    for m in meta:
        t0, nt, h0, nh, w0, nw = m["lat"]
        parts.append(dec.decode(z[:, :, t0:t0 + nt, h0:h0 + nh, w0:w0 + nw].contiguous()))
    torch.cuda.synchronize()
    assert vd.last_error(dec.h)[0] == vd.VAE_OK
    yield {"cfg": cfg, "params": p, "latent": zn, "out": out, "meta": meta, "parts": parts}
    dec.close()


def test_plan_is_the_oracle_plan(tiled):
    cfg, tl = tiled["cfg"], synth.LTX_TILING
    st, sh, _ = cfg.scale()
    ref = tiles.tile_plan(tiled["latent"].shape[2:], tl.tile, tl.overlap, st, sh)
    assert len(tiled["meta"]) == len(ref) == 45
    for m, r in zip(tiled["meta"], ref):
        assert (m["lat"], m["pix"], m["ovl"]) == (tuple(r.lat), tuple(r.pix), tuple(r.ovl))
    assert tuple(tiled["out"].shape) == (2, 3, 129, 1088, 1920)


def test_tiled_equals_blend_of_separate_tile_decodes(vd, tiled):
    out2 = torch.full_like(tiled["out"], float("nan"))
    vd.tile_blend(tiled["parts"], tiled["meta"], out2)
    torch.cuda.synchronize()
    assert torch.equal(out2, tiled["out"])


class _Frames:
    """A tile's data of which only tile frames [first, first + n) were copied to the host."""

    def __init__(self, arr, first):
        self.arr, self.first = arr, first

    def __getitem__(self, idx):
        ts = idx[2]
        assert ts.start >= self.first and ts.stop <= self.first + self.arr.shape[2]
        return self.arr[:, :, ts.start - self.first:ts.stop - self.first]


def test_blend_window_matches_oracle_blend(tiled):
    # output frames 54..58 hold the 1-frame temporal overlap (frame 56) of the first two tile rows
    f0, f1 = 54, 59
    plan_ = [tiles.Tile(lat=m["lat"], pix=m["pix"], ovl=m["ovl"]) for m in tiled["meta"]]
    data = []
    for t, x in zip(plan_, tiled["parts"]):
        a, b = max(t.pix[0], f0), min(t.pix[0] + t.pix[1], f1)
        data.append(_Frames(x[:, :, a - t.pix[0]:b - t.pix[0]].float().cpu().numpy(), a - t.pix[0]) if a < b else None)
    ref = tiles.blend(plan_, data, tuple(tiled["out"].shape), frames=(f0, f1))
    got = tiled["out"][:, :, f0:f1].float().cpu().numpy()
    err = np.abs(got - ref).max() / np.abs(ref).max()
    assert err < BF16_TOL, err


def test_corner_tile_first_frame_matches_oracle(tiled):
    cfg, p, zn = tiled["cfg"], tiled["params"], tiled["latent"]
    t0, nt, h0, nh, w0, nw = tiled["meta"][0]["lat"]
    sub = dataclasses.replace(cfg, latent_shape=(zn.shape[0], cfg.latent_c, 1, nh, nw))
    ref = odec.decode(sub, p, zn[:, :, t0:t0 + 1, h0:h0 + nh, w0:w0 + nw].copy(), tier="B")
    got = tiled["parts"][0][:, :, :1].float().cpu().numpy()
    assert got.shape == ref.shape
    rl2, ps = metrics.rel_l2(got, ref), metrics.psnr(got, ref)
    print(f"corner tile, first frame: rel L2 {rl2:.3e}, PSNR {ps:.1f} dB")
    assert rl2 <= 1e-2 and ps >= 50.0
