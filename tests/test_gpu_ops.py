"""Op-level parity on the GPU, through the C ABI, against the CPU oracle on the same seeded inputs.

Tolerances: the oracle runs in float64 on the values the kernel actually reads (bf16 inputs and
weights rounded to nearest even on the host), so the only differences are fp32 accumulation order
and the final store: fp32 outputs within 2e-5 of max|ref|, bf16 outputs within 2^-8 of max|ref|.
"""
import numpy as np
import pytest
import torch

from oracle import ops, plan, tiles
from patch_tiled_causal_gb300 import synth

pytestmark = pytest.mark.gpu

BF16_TOL = 2.0 ** -8
F32_TOL = 2e-5


@pytest.fixture(scope="module")
def vd():
    from patch_tiled_causal_gb300 import build, vaedec
    build.build()
    vaedec.load()
    return vaedec


def bf16_round(a: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16).float().numpy()


def to_dev(a, dtype):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to("cuda").to(dtype).contiguous()


def rel_err(g, r):
    g = np.asarray(g, dtype=np.float64)
    r = np.asarray(r, dtype=np.float64)
    return float(np.abs(g - r).max() / max(np.abs(r).max(), 1e-30))


# ----------------------------------------------------------------------------- GEMM core

# unbatched GEMMs with 128- or 256-wide weight tiles run as cta_group::2 pairs (odd M-tile counts leave
# the last pair's second CTA with no tile of its own; an odd k-block count takes one k block per stage)
@pytest.mark.parametrize("M,N,K,batch", [(200, 96, 128, 2), (128, 256, 64, 1), (77, 48, 192, 3), (300, 512, 256, 1),
                                         (700, 128, 256, 1), (520, 128, 192, 1), (260, 384, 128, 1), (90, 256, 320, 1)])
def test_gemm_bf16(vd, M, N, K, batch):
    A = bf16_round(synth.draw_normal((batch, M, K), 1))
    B = bf16_round(synth.draw_normal((batch, N, K), 2))
    bias = synth.draw_normal((N,), 3)
    ref = np.einsum("bmk,bnk->bmn", A.astype(np.float64), B.astype(np.float64)) * 0.5 + bias
    D = torch.empty((batch, M, N), dtype=torch.float32, device="cuda")
    vd.gemm_bf16(to_dev(A, torch.bfloat16), to_dev(B, torch.bfloat16), D, to_dev(bias, torch.float32), alpha=0.5)
    torch.cuda.synchronize()
    assert rel_err(D.cpu().numpy(), ref) < F32_TOL


# ----------------------------------------------------------------------------- causal conv

def _conv_case(vd, B, T, H, W, Ci, Co, ph, pw, cache, d2s, drop, ncthw, dt, resid, seed):
    S = d2s[0] * d2s[1] * d2s[2]
    x = synth.draw_normal((B, T + cache, H, W, Ci), seed)            # channels-last
    w = synth.conv_weight(Co, Ci, seed + 1)
    b = synth.draw_normal((Co,), seed + 2) * 0.1
    r = synth.draw_normal((B, T, H, W, Co), seed + 3) if resid else None
    tdt = torch.bfloat16 if dt == vd.VAE_BF16 else torch.float32
    if dt == vd.VAE_BF16:
        x, w_ref = bf16_round(x), bf16_round(w)
        r = bf16_round(r) if r is not None else None
    else:
        w_ref = w
    eh, ew = plan.band_edges(H, ph), plan.band_edges(W, pw)
    d = vd.conv_desc(B, T, H, W, Ci, Co, eh, ew, cache_frames=cache, d2s=d2s, drop_first=drop, out_ncthw=ncthw,
                     in_dtype=dt, out_dtype=dt, res_dtype=dt)
    wp = vd.conv3d_pack_weights(to_dev(w, torch.float32), d)
    To = d2s[0] * T - (d2s[0] - 1 if drop else 0)
    Cd = Co // S
    shape = (B, Cd, To, H * d2s[1], W * d2s[2]) if ncthw else (B, To, H * d2s[1], W * d2s[2], Cd)
    y = torch.full(shape, float("nan"), dtype=tdt, device="cuda")
    vd.conv3d_causal(to_dev(x, tdt), wp, to_dev(b, torch.float32), None if r is None else to_dev(r, tdt), y, d)
    torch.cuda.synchronize()
    # oracle: NCTHW float64
    xn = x.transpose(0, 4, 1, 2, 3).astype(np.float64)
    cache_arr = xn[:, :, :cache] if cache else None
    ref = ops.conv3d_causal(xn[:, :, cache:], w_ref.astype(np.float64), b.astype(np.float64), cache=cache_arr)
    if r is not None:
        ref = ref + r.transpose(0, 4, 1, 2, 3)
    ref = ops.depth_to_space(ref, d2s, drop_first=drop)
    if not ncthw:
        ref = ref.transpose(0, 2, 3, 4, 1)
    return y.float().cpu().numpy(), ref


CONV_CASES = [
    # B, T, H, W, Ci, Co, ph, pw, cache, d2s, drop, ncthw, resid
    (1, 3, 10, 13, 64, 64, 1, 1, 0, (1, 1, 1), False, False, False),
    (1, 3, 10, 13, 64, 64, 2, 3, 0, (1, 1, 1), False, False, True),
    (2, 2, 9, 20, 128, 128, 3, 2, 2, (1, 1, 1), False, False, True),
    (1, 3, 6, 7, 64, 256, 2, 2, 0, (2, 2, 2), True, False, False),
    (1, 2, 6, 7, 64, 256, 1, 2, 2, (2, 2, 2), False, False, False),
    (1, 2, 5, 9, 128, 512, 1, 3, 0, (1, 2, 2), False, False, False),
    (1, 3, 8, 11, 64, 48, 2, 2, 0, (1, 4, 4), False, True, False),
    (1, 2, 7, 6, 64, 12, 1, 2, 0, (1, 2, 2), False, True, False),
    (1, 2, 33, 40, 64, 320, 1, 1, 0, (1, 1, 1), False, False, False),
    # narrow convs (at most 32 channels): one shared halo box per (kt, channel chunk)
    (1, 3, 21, 19, 128, 32, 2, 3, 2, (1, 1, 1), False, False, True),
    (2, 2, 35, 17, 64, 16, 3, 1, 0, (1, 2, 2), False, True, False),
    # at most 12 channels: tap-stacked weights (all 9 spatial taps in one MMA of N = 112)
    (2, 3, 30, 33, 128, 12, 3, 2, 2, (1, 2, 2), False, True, False),
    (1, 3, 29, 31, 64, 8, 2, 3, 0, (1, 1, 1), False, False, True),
    (1, 2, 17, 45, 192, 3, 1, 4, 2, (1, 1, 1), False, True, False),
    (1, 4, 15, 14, 64, 12, 1, 1, 0, (2, 1, 2), True, False, False),
]


@pytest.mark.parametrize("case", CONV_CASES)
def test_conv_tensor_core_bf16(vd, case):
    B, T, H, W, Ci, Co, ph, pw, cache, d2s, drop, ncthw, resid = case
    g, r = _conv_case(vd, B, T, H, W, Ci, Co, ph, pw, cache, d2s, drop, ncthw, vd.VAE_BF16, resid, 10)
    assert not np.isnan(g).any()
    assert rel_err(g, r) < BF16_TOL


@pytest.mark.parametrize("case", [CONV_CASES[1], CONV_CASES[3], CONV_CASES[6],
                                  (1, 3, 6, 9, 16, 32, 2, 2, 2, (1, 1, 1), False, False, True),
                                  (1, 2, 5, 6, 48, 24, 1, 2, 0, (1, 2, 2), False, True, False)])
def test_conv_cuda_core_fp32(vd, case):
    B, T, H, W, Ci, Co, ph, pw, cache, d2s, drop, ncthw, resid = case
    g, r = _conv_case(vd, B, T, H, W, Ci, Co, ph, pw, cache, d2s, drop, ncthw, vd.VAE_FP32, resid, 20)
    assert rel_err(g, r) < F32_TOL


def test_conv_cuda_core_bf16_small_channels(vd):
    g, r = _conv_case(vd, 1, 3, 6, 9, 32, 32, 2, 1, 0, (1, 1, 1), False, False, vd.VAE_BF16, True, 30)
    assert rel_err(g, r) < BF16_TOL


@pytest.mark.parametrize("dt", ["bf16", "fp32"])
def test_conv_bit_identical_across_patch_counts(vd, dt):
    dtc = vd.VAE_BF16 if dt == "bf16" else vd.VAE_FP32
    outs = [_conv_case(vd, 1, 2, 24, 40, 64, 128, ph, pw, 0, (1, 1, 1), False, False, dtc, True, 40)[0]
            for ph, pw in ((1, 1), (2, 2), (2, 4), (4, 8), (3, 5))]
    for o in outs[1:]:
        np.testing.assert_array_equal(o, outs[0])


@pytest.mark.parametrize("Co,d2s,ncthw", [(16, (1, 1, 1), False), (12, (1, 2, 2), True), (8, (1, 1, 1), False)])
def test_conv_halo_path_bit_identical_across_patch_counts(vd, Co, d2s, ncthw):
    outs = [_conv_case(vd, 1, 2, 40, 36, 64, Co, ph, pw, 2, d2s, False, ncthw, vd.VAE_BF16, d2s == (1, 1, 1), 45)[0]
            for ph, pw in ((1, 1), (2, 2), (3, 4), (5, 2))]
    for o in outs[1:]:
        np.testing.assert_array_equal(o, outs[0])


@pytest.mark.parametrize("Co,Ci,d2s,ncthw", [(12, 64, (1, 2, 2), True), (8, 128, (1, 1, 1), False),
                                             (12, 64, (1, 2, 2), False)])
def test_tap_stacked_weight_packing(vd, Co, Ci, d2s, ncthw):
    # [3 kt][112 rows][Ci]: row (kh*3 + kw)*12 + n holds packed column n of tap (kh, kw), the columns in
    # PyTorch order for NCTHW outputs, else (depth-to-space sub-position, channel); zeros elsewhere
    w = synth.conv_weight(Co, Ci, 6)
    d = vd.conv_desc(1, 1, 4, 4, Ci, Co, [0, 4], [0, 4], d2s=d2s, out_ncthw=ncthw)
    wp = vd.conv3d_pack_weights(torch.from_numpy(w).cuda(), d).cpu()
    assert wp.numel() * wp.element_size() == 3 * 112 * Ci * 2
    got = wp.view(torch.bfloat16).float().numpy().reshape(3, 112, Ci)
    S = d2s[0] * d2s[1] * d2s[2]
    Cd = Co // S
    co = np.arange(Co) if ncthw else np.array([(n % Cd) * S + n // Cd for n in range(Co)])
    wr = torch.from_numpy(w).to(torch.bfloat16).float().numpy().reshape(Co, Ci, 3, 9)
    want = np.zeros((3, 112, Ci), np.float32)
    for t9 in range(9):
        want[:, t9 * 12:t9 * 12 + Co] = wr[co][:, :, :, t9].transpose(2, 0, 1)
    np.testing.assert_array_equal(got, want)


# ----------------------------------------------------------------------------- channel RMS norm

@pytest.mark.parametrize("Cc,din,dout,silu", [(64, "fp32", "fp32", True), (256, "bf16", "bf16", True),
                                             (1024, "fp32", "bf16", True), (128, "bf16", "fp32", False),
                                             (512, "fp32", "fp32", False), (8, "fp32", "fp32", True)])
def test_channel_rmsnorm(vd, Cc, din, dout, silu):
    shape = (2, 3, 7, 13, Cc)  # ragged pixel count: the last warp's teams run partly masked
    x = synth.draw_normal(shape, 80, offset=0.3)
    g = synth.draw_normal((Cc,), 81) * 0.1 + 1.0
    b = synth.draw_normal((Cc,), 82) * 0.1
    tin = torch.bfloat16 if din == "bf16" else torch.float32
    tout = torch.bfloat16 if dout == "bf16" else torch.float32
    if din == "bf16":
        x = bf16_round(x)
    y = torch.full(shape, float("nan"), dtype=tout, device="cuda")
    vd.channel_rmsnorm_silu(to_dev(x, tin), to_dev(g, torch.float32), to_dev(b, torch.float32), y, *shape, eps=1e-6,
                            silu=silu)
    torch.cuda.synchronize()
    ref = ops.channel_rms_norm(x.transpose(0, 4, 1, 2, 3).astype(np.float64), g, b, 1e-6)
    if silu:
        ref = ops.silu(ref)
    ref = ref.transpose(0, 2, 3, 4, 1)
    out = y.float().cpu().numpy()
    assert np.isfinite(out).all()
    assert rel_err(out, ref) < (BF16_TOL if dout == "bf16" else F32_TOL)


def test_channel_rmsnorm_refuses_unsupported_channels(vd):
    x = torch.zeros(16, dtype=torch.float32, device="cuda")  # never read: refused on the host
    one = torch.ones(2048, device="cuda")
    for Cc in (2048, 1032, 12):
        with pytest.raises(vd.VaeError) as e:
            vd.channel_rmsnorm_silu(x, one, one, x, 1, 1, 1, 1, Cc)
        assert e.value.code in (vd.VAE_ERR_UNSUPPORTED,)


# ----------------------------------------------------------------------------- PatchGroupNorm

def _gn_case(vd, shape, groups, ph, pw, dt_in, dt_out, offset=0.0, silu=True, seed=50):
    B, T, H, W, Cc = shape
    x = synth.draw_normal(shape, seed, offset=offset)
    g = synth.draw_normal((Cc,), seed + 1) * 0.1 + 1.0
    bt = synth.draw_normal((Cc,), seed + 2) * 0.1
    tin = torch.bfloat16 if dt_in == vd.VAE_BF16 else torch.float32
    tout = torch.bfloat16 if dt_out == vd.VAE_BF16 else torch.float32
    if dt_in == vd.VAE_BF16:
        x = bf16_round(x)
    d = vd.gn_desc(B, T, H, W, Cc, groups, plan.band_edges(H, ph), plan.band_edges(W, pw), eps=1e-6, silu=silu,
                   in_dtype=dt_in, out_dtype=dt_out)
    ws = vd.gn_workspace(d, "cuda")
    y = torch.empty(shape, dtype=tout, device="cuda")
    vd.patch_groupnorm_silu(to_dev(x, tin), to_dev(g, torch.float32), to_dev(bt, torch.float32), y, ws, d)
    torch.cuda.synchronize()
    ref = ops.group_norm(x.transpose(0, 4, 1, 2, 3).astype(np.float64), g, bt, groups, 1e-6)
    if silu:
        ref = ops.silu(ref)
    return y.float().cpu().numpy(), ref.transpose(0, 2, 3, 4, 1)


@pytest.mark.parametrize("Cc,groups", [(64, 32), (128, 32), (256, 32), (512, 32), (32, 8), (1024, 32)])
def test_groupnorm_silu_fp32(vd, Cc, groups):
    g, r = _gn_case(vd, (1, 3, 7, 13, Cc), groups, 2, 3, vd.VAE_FP32, vd.VAE_FP32)
    assert rel_err(g, r) < 1e-5


def test_groupnorm_bf16_and_large_mean(vd):
    g, r = _gn_case(vd, (2, 2, 9, 11, 128), 32, 3, 2, vd.VAE_BF16, vd.VAE_BF16)
    assert rel_err(g, r) < BF16_TOL
    # mean 100, spread 1: E[x^2] - E[x]^2 in float would lose the variance; exact sums do not
    g, r = _gn_case(vd, (1, 2, 16, 16, 64), 32, 2, 2, vd.VAE_FP32, vd.VAE_FP32, offset=100.0, silu=False)
    assert rel_err(g, r) < 1e-4


def test_groupnorm_bit_identical_across_patch_counts(vd):
    outs = [_gn_case(vd, (1, 2, 24, 40, 256), 32, ph, pw, vd.VAE_BF16, vd.VAE_BF16)[0]
            for ph, pw in ((1, 1), (2, 2), (4, 8), (3, 7))]
    for o in outs[1:]:
        np.testing.assert_array_equal(o, outs[0])


def test_groupnorm_range_is_flagged(vd):
    B, T, H, W, Cc = 1, 1, 4, 4, 64
    x = torch.zeros((B, T, H, W, Cc), dtype=torch.float32, device="cuda")
    x[0, 0, 1, 1, 3] = 9000.0
    d = vd.gn_desc(B, T, H, W, Cc, 32, [0, 4], [0, 4], in_dtype=vd.VAE_FP32, out_dtype=vd.VAE_FP32)
    ws = vd.gn_workspace(d, "cuda")
    y = torch.empty_like(x)
    one = torch.ones(Cc, device="cuda")
    vd.patch_groupnorm_silu(x, one, torch.zeros(Cc, device="cuda"), y, ws, d)
    code, _ = vd.last_error()
    assert code == vd.VAE_ERR_RANGE
    assert vd.last_error()[0] == vd.VAE_OK  # cleared


# ----------------------------------------------------------------------------- depth-to-space, blend

@pytest.mark.parametrize("s,drop", [((2, 2, 2), True), ((1, 2, 2), False), ((2, 1, 3), False)])
def test_d2s(vd, s, drop):
    B, T, H, W, Cc = 1, 3, 4, 5, 16
    S = s[0] * s[1] * s[2]
    x = synth.draw_normal((B, T, H, W, Cc * S), 60)
    To = s[0] * T - (s[0] - 1 if drop else 0)
    y = torch.empty((B, To, H * s[1], W * s[2], Cc), dtype=torch.float32, device="cuda")
    vd.upsample_d2s(to_dev(x, torch.float32), y, B, T, H, W, Cc, s, drop)
    torch.cuda.synchronize()
    ref = ops.depth_to_space(x.transpose(0, 4, 1, 2, 3), s, drop_first=drop).transpose(0, 2, 3, 4, 1)
    np.testing.assert_array_equal(y.cpu().numpy(), ref)


@pytest.mark.parametrize("dt,order,W", [("bf16", "raster", 56), ("fp32", "raster", 56), ("fp32", "reversed", 56),
                                         ("bf16", "raster", 136)])
def test_tile_blend(vd, dt, order, W):
    # raster order is a grid (factorised kernel); any other order takes the general gather kernel.
    # W = 136: 13 column intervals, so rows covered by 4 (t, y) pairs have 52 source rows per warp
    tdt = torch.bfloat16 if dt == "bf16" else torch.float32
    plan_ = tiles.tile_plan((3, 40, W), (2, 16, 16), (1, 4, 6), 4, 1)   # causal time, ragged last tiles
    if order == "reversed":
        plan_ = plan_[::-1]
    B, Cc = 2, 3
    out_shape = (B, Cc, 4 * 2 + 1, 40, W)
    data = []
    for i, t in enumerate(plan_):
        a = synth.draw_normal((B, Cc, t.pix[1], t.pix[3], t.pix[5]), 70 + i)
        data.append(bf16_round(a) if dt == "bf16" else a)
    ref = tiles.blend(plan_, data, out_shape)
    out = torch.empty(out_shape, dtype=tdt, device="cuda")
    meta = [{"lat": t.lat, "pix": t.pix, "ovl": t.ovl} for t in plan_]
    from patch_tiled_causal_gb300 import vaedec
    vaedec.tile_blend([to_dev(a, tdt) for a in data], meta, out)
    torch.cuda.synchronize()
    assert rel_err(out.float().cpu().numpy(), ref) < (BF16_TOL if dt == "bf16" else F32_TOL)


@pytest.mark.parametrize("dt", ["bf16", "fp32"])
def test_tile_blend_aligned_grid(vd, dt):
    # tile edges on 8-pixel boundaries: every vector takes the vector path, including rows whose frames
    # and rows both lie in overlaps (4 (t, y) pairs, 2 column intervals: 8 source vectors)
    tdt = torch.bfloat16 if dt == "bf16" else torch.float32
    plan_ = tiles.tile_plan((3, 56, 112), (2, 32, 32), (1, 8, 8), 4, 1)
    B, Cc = 2, 3
    out_shape = (B, Cc, 4 * 2 + 1, 56, 112)
    data = []
    for i, t in enumerate(plan_):
        a = synth.draw_normal((B, Cc, t.pix[1], t.pix[3], t.pix[5]), 90 + i)
        data.append(bf16_round(a) if dt == "bf16" else a)
    ref = tiles.blend(plan_, data, out_shape)
    out = torch.full(out_shape, float("nan"), dtype=tdt, device="cuda")
    meta = [{"lat": t.lat, "pix": t.pix, "ovl": t.ovl} for t in plan_]
    vd.tile_blend([to_dev(a, tdt) for a in data], meta, out)
    torch.cuda.synchronize()
    g = out.float().cpu().numpy()
    assert not np.isnan(g).any()
    assert rel_err(g, ref) < (BF16_TOL if dt == "bf16" else F32_TOL)


# ----------------------------------------------------------------------------- watchdog

def test_watchdog_times_out_and_context_survives(vd):
    assert vd.watchdog_selftest(20000) == vd.VAE_ERR_TIMEOUT
    assert vd.last_error()[0] == vd.VAE_OK
    test_gemm_bf16(vd, 128, 64, 64, 1)  # the context still works
