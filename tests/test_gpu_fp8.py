"""e4m3 (FP8) convolution operands on the tcgen05 tensor cores (kind::f8f6f4), through the C ABI.

The low-precision conv with the norm + SiLU -> quantisation fusion follows TensorRT-LLM PR #16066
"ParallelVAE_TrtllmWan for native Wan VAE" (reviewer comment: FP4 conv quantisation and
RMSNorm/SiLU -> quantisation fusion); here at 8 bits.

What is checked, and against what:
  * weight packing: the library's e4m3 bytes and per-output-channel scales equal a host
    quantisation written here from the definition (scale = max|w| / 448 in fp32, bytes = w / scale
    rounded to nearest even, saturated at 448), bit for bit;
  * the conv itself: on the same e4m3 inputs and dequantised weights the oracle (float64) and the
    GPU differ only by fp32 accumulation and the final store: bf16 outputs within 2^-8 of max|ref|,
    fp32 outputs within 2e-5; bit-identical across patch grids;
  * the norms' e4m3 outputs: every element within one e4m3 step of the oracle's value (the oracle
    is float64, the kernel fp32, so a value next to a rounding boundary may round the other way),
    and almost all equal to its rounding;
  * whole decoders in fp8 mode against the fp32 oracle: relative L2 <= 0.15 and PSNR >= 35 dB.  Each
    e4m3 rounding has unit roundoff 2^-4 (3 mantissa bits), an RMS relative error of about 2^-4/sqrt(3)
    per operand; a conv with both operands rounded carries about sqrt(2) times that (~5%) on its
    output, and the residual stream and the bf16 layers dilute it.  An emulation of the same rounding
    points in the oracle gave relative L2 0.05-0.07 on the mini decoders and 0.094 (40.8 dB) on the
    first frame of the Wan-shaped decode; the bar is 1.5 times the largest.
"""
import dataclasses

import numpy as np
import pytest
import torch

from oracle import decoder as odec
from oracle import metrics, ops, plan
from patch_tiled_causal_gb300 import synth

pytestmark = pytest.mark.gpu

BF16_TOL = 2.0 ** -8
F32_TOL = 2e-5
FP8_REL_L2 = 0.15
FP8_PSNR = 35.0


@pytest.fixture(scope="module")
def vd():
    from patch_tiled_causal_gb300 import build, vaedec
    build.build()
    vaedec.load()
    return vaedec


def e4m3(a) -> torch.Tensor:
    """Round to e4m3 (nearest even), saturating at +-448: a torch float8_e4m3fn CPU tensor."""
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).clamp(-448.0, 448.0).to(torch.float8_e4m3fn)


def e4m3_step(v):
    """Spacing of e4m3 values at |v| (2^-9 in the subnormal range below 2^-6)."""
    a = np.maximum(np.abs(np.asarray(v, dtype=np.float64)), 2.0 ** -6)
    return 2.0 ** (np.floor(np.log2(a)) - 3)


def quantise_weight(w):
    """Per output channel: scale = max|w| / 448 (fp32), e4m3 bytes of w / scale; returns (bytes, scales)."""
    wf = np.ascontiguousarray(w, dtype=np.float32).reshape(w.shape[0], -1)
    s = np.abs(wf).max(axis=1).astype(np.float32) / np.float32(448.0)
    s = np.where(s > 0, s, np.float32(1.0)).astype(np.float32)
    return e4m3(wf / s[:, None]), s


def bf16_round(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16).float().numpy()


def rel_err(g, r):
    g, r = np.asarray(g, np.float64), np.asarray(r, np.float64)
    return float(np.abs(g - r).max() / max(np.abs(r).max(), 1e-30))


# ----------------------------------------------------------------------------- weight packing

@pytest.mark.parametrize("Co,Ci,d2s", [(256, 128, (1, 1, 1)), (48, 128, (1, 4, 4)), (1024, 256, (2, 2, 2))])
def test_fp8_weight_packing_is_the_host_quantisation(vd, Co, Ci, d2s):
    w = synth.conv_weight(Co, Ci, 5)
    d = vd.conv_desc(1, 1, 4, 4, Ci, Co, [0, 4], [0, 4], d2s=d2s, in_dtype=vd.VAE_FP8)
    wp = vd.conv3d_pack_weights(torch.from_numpy(w).cuda(), d).cpu()
    q, s = quantise_weight(w)
    S = d2s[0] * d2s[1] * d2s[2]
    n_pad = (Co + 15) // 16 * 16
    # packed row n = sub * (Co / S) + c holds output channel c * S + sub; K order (tap, channel)
    co = np.array([(n % (Co // S)) * S + n // (Co // S) for n in range(Co)])
    want = q.view(torch.uint8).numpy().reshape(Co, Ci, 27).transpose(0, 2, 1).reshape(Co, -1)[co]
    nbytes = n_pad * 27 * Ci
    got = wp[:nbytes].numpy().reshape(n_pad, -1)
    np.testing.assert_array_equal(got[:Co], want)
    assert not got[Co:].any()
    off = (nbytes + 255) // 256 * 256
    scales = wp[off:off + 4 * n_pad].view(torch.float32).numpy()
    np.testing.assert_array_equal(scales[:Co], s[co])


# ----------------------------------------------------------------------------- causal conv

def _conv_fp8_case(vd, B, T, H, W, Ci, Co, ph, pw, cache, d2s, drop, ncthw, resid, out_dt, seed):
    S = d2s[0] * d2s[1] * d2s[2]
    x = synth.draw_normal((B, T + cache, H, W, Ci), seed)
    xq = e4m3(x)
    w = synth.conv_weight(Co, Ci, seed + 1)
    q, s = quantise_weight(w)
    w_deq = q.float().numpy().astype(np.float64) * s[:, None].astype(np.float64)
    b = synth.draw_normal((Co,), seed + 2) * 0.1
    tdt = torch.float32 if out_dt == vd.VAE_FP32 else torch.bfloat16
    r = synth.draw_normal((B, T, H, W, Co), seed + 3) if resid else None
    if r is not None and out_dt == vd.VAE_BF16:
        r = bf16_round(r)
    d = vd.conv_desc(B, T, H, W, Ci, Co, plan.band_edges(H, ph), plan.band_edges(W, pw), cache_frames=cache, d2s=d2s,
                     drop_first=drop, out_ncthw=ncthw, in_dtype=vd.VAE_FP8, out_dtype=out_dt, res_dtype=out_dt)
    wp = vd.conv3d_pack_weights(torch.from_numpy(w).cuda(), d)
    To = d2s[0] * T - (d2s[0] - 1 if drop else 0)
    Cd = Co // S
    shape = (B, Cd, To, H * d2s[1], W * d2s[2]) if ncthw else (B, To, H * d2s[1], W * d2s[2], Cd)
    y = torch.full(shape, float("nan"), dtype=tdt, device="cuda")
    rd = None if r is None else torch.from_numpy(r).cuda().to(tdt)
    vd.conv3d_causal(xq.cuda(), wp, torch.from_numpy(b).cuda(), rd, y, d)
    torch.cuda.synchronize()
    assert vd.last_error()[0] == vd.VAE_OK
    xn = xq.float().numpy().astype(np.float64).transpose(0, 4, 1, 2, 3)
    ref = ops.conv3d_causal(xn[:, :, cache:], w_deq.reshape(w.shape), b.astype(np.float64),
                            cache=xn[:, :, :cache] if cache else None)
    if r is not None:
        ref = ref + r.transpose(0, 4, 1, 2, 3)
    ref = ops.depth_to_space(ref, d2s, drop_first=drop)
    if not ncthw:
        ref = ref.transpose(0, 2, 3, 4, 1)
    return y.float().cpu().numpy(), ref


FP8_CASES = [
    # B, T, H, W, Ci, Co, ph, pw, cache, d2s, drop, ncthw, resid
    (1, 3, 10, 13, 128, 128, 2, 3, 0, (1, 1, 1), False, False, True),      # MMA pairs, 128-wide tile
    (2, 2, 9, 20, 256, 256, 3, 2, 2, (1, 1, 1), False, False, True),       # two k blocks per stage, cache
    (1, 3, 6, 7, 128, 256, 2, 2, 0, (2, 2, 2), True, False, False),        # depth-to-space + frame drop
    (1, 2, 5, 9, 128, 48, 1, 3, 0, (1, 4, 4), False, True, False),         # 48-wide tile, NCTHW pixels
    (1, 2, 33, 40, 128, 320, 1, 1, 0, (1, 1, 1), False, False, False),     # N past 256 (two weight tiles)
    (1, 2, 8, 12, 512, 512, 2, 2, 0, (1, 1, 1), False, False, False),      # 4 channel chunks per tap
]


@pytest.mark.parametrize("case", FP8_CASES)
@pytest.mark.parametrize("out", ["bf16", "fp32"])
def test_conv_fp8_matches_oracle_on_the_same_operands(vd, case, out):
    B, T, H, W, Ci, Co, ph, pw, cache, d2s, drop, ncthw, resid = case
    out_dt = vd.VAE_BF16 if out == "bf16" else vd.VAE_FP32
    g, r = _conv_fp8_case(vd, B, T, H, W, Ci, Co, ph, pw, cache, d2s, drop, ncthw, resid, out_dt, 90)
    assert not np.isnan(g).any()
    assert rel_err(g, r) < (BF16_TOL if out == "bf16" else F32_TOL)


def test_conv_fp8_bit_identical_across_patch_counts(vd):
    outs = [_conv_fp8_case(vd, 1, 2, 24, 40, 128, 128, ph, pw, 0, (1, 1, 1), False, False, True, vd.VAE_BF16, 91)[0]
            for ph, pw in ((1, 1), (2, 2), (4, 8), (3, 5))]
    for o in outs[1:]:
        np.testing.assert_array_equal(o, outs[0])


def test_conv_fp8_refuses_unsupported(vd):
    d = vd.conv_desc(1, 1, 4, 4, 64, 64, [0, 4], [0, 4], in_dtype=vd.VAE_FP8)  # needs C_in % 128 == 0
    x = torch.zeros(16, dtype=torch.uint8, device="cuda")  # never read: refused on the host
    with pytest.raises(vd.VaeError) as e:
        vd.conv3d_causal(x, x, None, None, torch.zeros(16, device="cuda"), d)
    assert e.value.code == vd.VAE_ERR_UNSUPPORTED


# ----------------------------------------------------------------------------- norm -> e4m3

def _check_e4m3(got, ref):
    rq = e4m3(ref).float().numpy()
    diff = np.abs(got - ref)
    assert (diff <= e4m3_step(ref) * (1 + 1e-6)).all(), float((diff / e4m3_step(ref)).max())
    assert np.mean(got == rq) > 0.995


@pytest.mark.parametrize("din", ["bf16", "fp32"])
def test_groupnorm_silu_e4m3_output(vd, din):
    shape, groups = (1, 3, 9, 13, 256), 32
    x = synth.draw_normal(shape, 92, offset=0.5)
    g = synth.draw_normal((256,), 93) * 0.1 + 1.0
    bt = synth.draw_normal((256,), 94) * 0.1
    tin = torch.bfloat16 if din == "bf16" else torch.float32
    if din == "bf16":
        x = bf16_round(x)
    d = vd.gn_desc(*shape, groups, plan.band_edges(9, 2), plan.band_edges(13, 3),
                   in_dtype=vd.VAE_BF16 if din == "bf16" else vd.VAE_FP32, out_dtype=vd.VAE_FP8)
    y = torch.empty(shape, dtype=torch.float8_e4m3fn, device="cuda")
    vd.patch_groupnorm_silu(torch.from_numpy(x).cuda().to(tin), torch.from_numpy(g).cuda(), torch.from_numpy(bt).cuda(),
                            y, vd.gn_workspace(d, "cuda"), d)
    torch.cuda.synchronize()
    assert vd.last_error()[0] == vd.VAE_OK
    ref = ops.silu(ops.group_norm(x.transpose(0, 4, 1, 2, 3).astype(np.float64), g, bt, groups, 1e-6))
    _check_e4m3(y.float().cpu().numpy(), ref.transpose(0, 2, 3, 4, 1))


def test_rmsnorm_silu_e4m3_output(vd):
    shape = (2, 2, 7, 13, 512)
    x = synth.draw_normal(shape, 95, offset=0.3)
    g = synth.draw_normal((512,), 96) * 0.1 + 1.0
    bt = synth.draw_normal((512,), 97) * 0.1
    y = torch.empty(shape, dtype=torch.float8_e4m3fn, device="cuda")
    vd.channel_rmsnorm_silu(torch.from_numpy(x).cuda(), torch.from_numpy(g).cuda(), torch.from_numpy(bt).cuda(), y,
                            *shape)
    torch.cuda.synchronize()
    assert vd.last_error()[0] == vd.VAE_OK
    ref = ops.silu(ops.channel_rms_norm(x.transpose(0, 4, 1, 2, 3).astype(np.float64), g, bt, 1e-6))
    _check_e4m3(y.float().cpu().numpy(), ref.transpose(0, 2, 3, 4, 1))


def test_e4m3_overflow_is_flagged(vd):
    # a scale of 1000 on a unit-variance norm output cannot fit e4m3's +-448
    shape = (1, 1, 4, 4, 64)
    x = torch.from_numpy(synth.draw_normal(shape, 98)).cuda()
    d = vd.gn_desc(*shape, 32, [0, 4], [0, 4], silu=False, in_dtype=vd.VAE_FP32, out_dtype=vd.VAE_FP8)
    y = torch.empty(shape, dtype=torch.float8_e4m3fn, device="cuda")
    vd.patch_groupnorm_silu(x, torch.full((64,), 1000.0, device="cuda"), torch.zeros(64, device="cuda"), y,
                            vd.gn_workspace(d, "cuda"), d)
    assert vd.last_error()[0] == vd.VAE_ERR_RANGE
    assert vd.last_error()[0] == vd.VAE_OK  # cleared


# ----------------------------------------------------------------------------- decoders

_cache = {}


def _oracle(cfg):
    if cfg.name not in _cache:
        p = synth.draw_params(cfg, 0, rand_affine=True)
        _cache[cfg.name] = odec.decode(cfg, p, synth.draw_latent(cfg, 0), tier="A")
    return _cache[cfg.name]


def _fp8_decode(vd, cfg, nph, npw):
    p = synth.draw_params(cfg, 0, rand_affine=True)
    dec = vd.Decoder(cfg, p, vd.VAE_FP8)
    y = dec.decode(torch.from_numpy(synth.draw_latent(cfg, 0)).cuda(), n_patch_h=nph, n_patch_w=npw)
    torch.cuda.synchronize()
    code, msg = vd.last_error(dec.h)
    assert code == vd.VAE_OK, msg
    dec.close()
    assert y.dtype == torch.bfloat16
    return y.float().cpu().numpy()


@pytest.mark.parametrize("name", ["mini_wan", "mini_ltx", "mini_wan_rms"])
def test_fp8_decoder_matches_oracle(vd, name):
    cfg = synth.CONFIGS[name]
    g, r = _fp8_decode(vd, cfg, 2, 3), _oracle(cfg)
    rl2, ps = metrics.rel_l2(g, r), metrics.psnr(g, r)
    print(f"{name} fp8: rel L2 {rl2:.3e}, PSNR {ps:.1f} dB")
    assert rl2 <= FP8_REL_L2 and ps >= FP8_PSNR


@pytest.mark.parametrize("name,grids", [("mini_wan", [(1, 1), (1, 4), (3, 2)]), ("mini_ltx", [(1, 1), (2, 2), (3, 5)])])
def test_fp8_decoder_bit_identical_across_patch_counts(vd, name, grids):
    cfg = synth.CONFIGS[name]
    outs = [_fp8_decode(vd, cfg, ph, pw) for ph, pw in grids]
    for o in outs[1:]:
        np.testing.assert_array_equal(o, outs[0])


def test_fp8_decoder_chunked_equals_whole(vd):
    cfg = dataclasses.replace(synth.MINI_WAN, latent_shape=(1, 48, 4, 9, 11))
    p = synth.draw_params(cfg, 0, rand_affine=True)
    z = torch.from_numpy(synth.draw_latent(cfg, 0)).cuda()
    dec = vd.Decoder(cfg, p, vd.VAE_FP8)
    whole = dec.decode(z, n_patch_h=1, n_patch_w=2).float().cpu().numpy()
    outs, t0 = [], 0
    for i, s in enumerate(odec.chunk_sizes(z.shape[2], 1)):
        outs.append(dec.decode_chunk(z[:, :, t0:t0 + s].contiguous(), i == 0, n_patch_h=1, n_patch_w=2))
        t0 += s
    torch.cuda.synchronize()
    chunked = torch.cat(outs, dim=2).float().cpu().numpy()
    dec.close()
    np.testing.assert_array_equal(chunked, whole)


@pytest.mark.parametrize("name,k", [("ltx", 2), ("wan", 1)])
def test_fp8_full_size_prefix_matches_oracle(vd, name, k):
    # causal: the first s_t*(k-1)+1 output frames depend only on latent frames 0..k-1
    cfg = synth.CONFIGS[name]
    p = synth.draw_params(cfg, 0)
    zn = synth.draw_latent(cfg, 0)
    dec = vd.Decoder(cfg, p, vd.VAE_FP8)
    y = dec.decode(torch.from_numpy(zn).cuda(), n_patch_h=1, n_patch_w=4)
    torch.cuda.synchronize()
    assert vd.last_error(dec.h)[0] == vd.VAE_OK
    nf = cfg.scale()[0] * (k - 1) + 1
    got = y[:, :, :nf].float().cpu().numpy()
    dec.close()
    sub = dataclasses.replace(cfg, latent_shape=(1, cfg.latent_c, k) + cfg.latent_shape[3:])
    ref = odec.decode(sub, p, zn[:, :, :k].copy(), tier="B")
    rl2, ps = metrics.rel_l2(got, ref), metrics.psnr(got, ref)
    print(f"{name} fp8: first {nf} frames, rel L2 {rl2:.3e}, PSNR {ps:.1f} dB")
    assert rl2 <= FP8_REL_L2 and ps >= FP8_PSNR
