"""ctypes binding of libvaedec (include/vaedec.h): argument marshalling only.

Every function below forwards to the C ABI of the same name; all arithmetic runs in the library's
CUDA kernels.  Tensors are PyTorch CUDA tensors (PyTorch provides device memory and streams); the
binding checks dtype/contiguity/device, passes raw pointers and raises ``VaeError`` on a non-zero
status.  There is no fallback: without the built library on a CUDA device, importing or calling
fails loudly.
"""
from __future__ import annotations

import ctypes as C
import os
from typing import Dict, List, Optional, Sequence, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libvaedec.so")

VAE_OK, VAE_ERR_INVALID_ARG, VAE_ERR_UNSUPPORTED, VAE_ERR_PATCH_TOO_NARROW = 0, 1, 2, 3
VAE_ERR_ALIGNMENT, VAE_ERR_OOM, VAE_ERR_CUDA, VAE_ERR_TIMEOUT, VAE_ERR_RANGE = 4, 5, 6, 7, 8
VAE_BF16, VAE_FP32, VAE_FP8, VAE_FP32_TC = 0, 1, 2, 3
VAE_NORM_GROUP, VAE_NORM_CHANNEL_RMS = 0, 1
MAX_STAGES, MAX_PATCHES, MAX_TILES = 8, 64, 512

STATUS_NAMES = {0: "VAE_OK", 1: "VAE_ERR_INVALID_ARG", 2: "VAE_ERR_UNSUPPORTED", 3: "VAE_ERR_PATCH_TOO_NARROW",
                4: "VAE_ERR_ALIGNMENT", 5: "VAE_ERR_OOM", 6: "VAE_ERR_CUDA", 7: "VAE_ERR_TIMEOUT", 8: "VAE_ERR_RANGE"}


class VaeConfig(C.Structure):
    _fields_ = [("latent_c", C.c_int), ("n_stages", C.c_int), ("stage_c", C.c_int * MAX_STAGES),
                ("n_res", C.c_int * MAX_STAGES), ("up_t", C.c_int * MAX_STAGES), ("up_h", C.c_int * MAX_STAGES),
                ("up_w", C.c_int * MAX_STAGES), ("mid_res", C.c_int), ("mid_attn", C.c_int),
                ("gn_groups", C.c_int), ("gn_eps", C.c_float), ("out_c", C.c_int), ("out_d2s_t", C.c_int),
                ("out_d2s_h", C.c_int), ("out_d2s_w", C.c_int), ("dtype", C.c_int), ("norm_type", C.c_int)]


VAE_DOWN_FOLD, VAE_DOWN_STRIDE = 0, 1


class VaeEncoderConfig(C.Structure):
    _fields_ = [("pix_c", C.c_int), ("patch_h", C.c_int), ("patch_w", C.c_int), ("n_stages", C.c_int),
                ("stage_c", C.c_int * MAX_STAGES), ("n_res", C.c_int * MAX_STAGES),
                ("down_kind", C.c_int * MAX_STAGES), ("down_t", C.c_int * MAX_STAGES),
                ("down_h", C.c_int * MAX_STAGES), ("down_w", C.c_int * MAX_STAGES), ("mid_res", C.c_int),
                ("gn_groups", C.c_int), ("gn_eps", C.c_float), ("latent_c", C.c_int), ("dtype", C.c_int),
                ("norm_type", C.c_int)]


class VaeErrorInfo(C.Structure):
    _fields_ = [("code", C.c_int), ("rows", C.c_int), ("factor", C.c_int), ("message", C.c_char * 256)]


class VaeTile(C.Structure):
    _fields_ = [("lat", C.c_int * 6), ("pix", C.c_int * 6), ("ovl", C.c_int * 6)]


_EDGES = C.c_int * (MAX_PATCHES + 1)


class VaeConvDesc(C.Structure):
    _fields_ = [("B", C.c_int), ("T", C.c_int), ("H", C.c_int), ("W", C.c_int), ("C_in", C.c_int),
                ("C_out", C.c_int), ("cache_frames", C.c_int), ("n_patch_h", C.c_int), ("n_patch_w", C.c_int),
                ("patch_h_edges", _EDGES), ("patch_w_edges", _EDGES), ("d2s_t", C.c_int), ("d2s_h", C.c_int),
                ("d2s_w", C.c_int), ("drop_first", C.c_int), ("out_ncthw", C.c_int), ("in_dtype", C.c_int),
                ("out_dtype", C.c_int), ("res_dtype", C.c_int)]


class VaeGnDesc(C.Structure):
    _fields_ = [("B", C.c_int), ("T", C.c_int), ("H", C.c_int), ("W", C.c_int), ("C", C.c_int),
                ("groups", C.c_int), ("eps", C.c_float), ("silu", C.c_int), ("n_patch_h", C.c_int),
                ("n_patch_w", C.c_int), ("patch_h_edges", _EDGES), ("patch_w_edges", _EDGES),
                ("in_dtype", C.c_int), ("out_dtype", C.c_int)]


class VaeRmsDesc(C.Structure):
    _fields_ = [("B", C.c_int), ("T", C.c_int), ("H", C.c_int), ("W", C.c_int), ("C", C.c_int),
                ("eps", C.c_float), ("silu", C.c_int), ("in_dtype", C.c_int), ("out_dtype", C.c_int)]


class VaeD2sDesc(C.Structure):
    _fields_ = [("B", C.c_int), ("T", C.c_int), ("H", C.c_int), ("W", C.c_int), ("C", C.c_int),
                ("s_t", C.c_int), ("s_h", C.c_int), ("s_w", C.c_int), ("drop_first", C.c_int), ("dtype", C.c_int)]


class VaeBlendDesc(C.Structure):
    _fields_ = [("B", C.c_int), ("C", C.c_int), ("T", C.c_int), ("H", C.c_int), ("W", C.c_int),
                ("tile_dtype", C.c_int), ("out_dtype", C.c_int)]


class VaeProf(C.Structure):
    _fields_ = [("name", C.c_char * 32), ("launches", C.c_int), ("ms", C.c_double), ("flops", C.c_double),
                ("bytes", C.c_double)]


_P = C.c_void_p
_SIGS = {
    "vae_decoder_profile": (C.c_int, [_P, C.c_int]),
    "vae_decoder_profile_read": (C.c_int, [_P, C.POINTER(VaeProf), C.POINTER(C.c_int)]),
    "vae_decoder_n_weights": (C.c_int, [C.POINTER(VaeConfig), C.POINTER(C.c_int)]),
    "vae_decoder_create": (C.c_int, [C.POINTER(VaeConfig), C.POINTER(_P), C.c_int, C.POINTER(_P)]),
    "vae_decoder_destroy": (None, [_P]),
    "vae_decoder_reserve": (C.c_int, [_P, C.POINTER(C.c_int64), C.c_int, C.c_int]),
    "vae_decode": (C.c_int, [_P, _P, C.POINTER(C.c_int64), _P, C.c_int, C.c_int, _P]),
    "vae_decode_chunk": (C.c_int, [_P, _P, C.POINTER(C.c_int64), C.c_int, _P, C.c_int, C.c_int, _P]),
    "vae_decode_host": (C.c_int, [_P, _P, C.POINTER(C.c_int64), _P, C.c_int, C.c_int, C.c_int, _P]),
    "vae_decode_tiled": (C.c_int, [_P, _P, C.POINTER(C.c_int64), _P, C.POINTER(C.c_int), C.POINTER(C.c_int), _P]),
    "vae_last_error": (C.c_int, [_P, C.POINTER(VaeErrorInfo)]),
    "vae_patch_edges": (C.c_int, [C.c_int, C.c_int, C.c_int, C.c_int, C.POINTER(C.c_int)]),
    "vae_tile_plan": (C.c_int, [C.POINTER(C.c_int), C.POINTER(C.c_int), C.POINTER(C.c_int), C.c_int, C.c_int,
                                C.c_int, C.POINTER(VaeTile), C.POINTER(C.c_int)]),
    "vae_conv3d_packed_bytes": (C.c_size_t, [C.POINTER(VaeConvDesc)]),
    "vae_conv3d_pack_weights": (C.c_int, [_P, C.POINTER(VaeConvDesc), _P, _P]),
    "vae_conv3d_causal": (C.c_int, [_P, _P, _P, _P, _P, C.POINTER(VaeConvDesc), _P]),
    "vae_patch_groupnorm_workspace_bytes": (C.c_size_t, [C.POINTER(VaeGnDesc)]),
    "vae_patch_groupnorm_silu": (C.c_int, [_P, _P, _P, _P, _P, C.POINTER(VaeGnDesc), _P]),
    "vae_patch_groupnorm_silu_noalloc": (C.c_int, [_P, _P, _P, _P, C.POINTER(VaeGnDesc), _P]),
    "vae_channel_rmsnorm_silu": (C.c_int, [_P, _P, _P, _P, C.POINTER(VaeRmsDesc), _P]),
    "vae_upsample_d2s": (C.c_int, [_P, _P, C.POINTER(VaeD2sDesc), _P]),
    "vae_tile_blend": (C.c_int, [C.POINTER(_P), C.POINTER(VaeTile), C.c_int, _P, C.POINTER(VaeBlendDesc), _P]),
    "vae_gemm_bf16": (C.c_int, [_P, _P, _P, _P, C.c_int, C.c_int, C.c_int, C.c_int, C.c_int64, C.c_int64,
                                C.c_int64, C.c_float, C.c_int, _P]),
    "vae_watchdog_selftest": (C.c_int, [C.c_int, _P]),
    "vae_encoder_n_weights": (C.c_int, [C.POINTER(VaeEncoderConfig), C.POINTER(C.c_int)]),
    "vae_encoder_create": (C.c_int, [C.POINTER(VaeEncoderConfig), C.POINTER(_P), C.c_int, C.POINTER(_P)]),
    "vae_encoder_destroy": (None, [_P]),
    "vae_encode": (C.c_int, [_P, _P, C.POINTER(C.c_int64), _P, C.c_int, C.c_int, _P]),
    "vae_encode_tiled": (C.c_int, [_P, _P, C.POINTER(C.c_int64), _P, C.POINTER(C.c_int), C.POINTER(C.c_int), _P]),
    "vae_encoder_profile": (C.c_int, [_P, C.c_int]),
    "vae_encoder_profile_read": (C.c_int, [_P, C.POINTER(VaeProf), C.POINTER(C.c_int)]),
    "vae_encoder_last_error": (C.c_int, [_P, C.POINTER(VaeErrorInfo)]),
}

_lib: Optional[C.CDLL] = None


def load() -> C.CDLL:
    """Load libvaedec.so (built by ``patch_tiled_causal_gb300.build``); raises if it is missing."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with patch_tiled_causal_gb300.build.build()")
        lib = C.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            f = getattr(lib, name)
            f.restype = res
            f.argtypes = args
        _lib = lib
    return _lib


def declared_symbols() -> List[str]:
    return sorted(_SIGS)


class VaeError(RuntimeError):
    def __init__(self, code: int, info: Optional[VaeErrorInfo] = None, where: str = ""):
        self.code = code
        self.rows = info.rows if info is not None else 0
        self.factor = info.factor if info is not None else 0
        msg = info.message.decode(errors="replace") if info is not None else ""
        super().__init__(f"{where}: {STATUS_NAMES.get(code, code)} {msg}".strip())


def _check(code: int, where: str, dec=None, enc=None):
    if code != VAE_OK:
        info = VaeErrorInfo()
        if enc is not None:
            load().vae_encoder_last_error(enc, C.byref(info))
        else:
            load().vae_last_error(dec, C.byref(info))
        raise VaeError(code, info, where)


def last_error(dec=None) -> Tuple[int, str]:
    info = VaeErrorInfo()
    code = load().vae_last_error(dec, C.byref(info))
    return code, info.message.decode(errors="replace")


# --------------------------------------------------------------------------- torch marshalling
def _torch():
    import torch
    return torch


def _stream(stream=None) -> int:
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _hptr(t, dtype) -> int:
    """Pointer to a contiguous host (CPU) tensor of the given dtype."""
    if t.is_cuda:
        raise ValueError("expected a host (CPU) tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    if t.dtype != dtype:
        raise ValueError(f"expected {dtype}, got {t.dtype}")
    return t.data_ptr()


def _ptr(t, dtype=None) -> Optional[int]:
    if t is None:
        return None
    torch = _torch()
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"expected {dtype}, got {t.dtype}")
    return t.data_ptr()


def _dt(t) -> int:
    torch = _torch()
    if t.dtype == torch.float32:
        return VAE_FP32
    return VAE_FP8 if t.dtype == torch.float8_e4m3fn else VAE_BF16


def _edges_array(edges: Sequence[int]):
    a = _EDGES()
    for i, e in enumerate(edges):
        a[i] = int(e)
    return a


# --------------------------------------------------------------------------- host plans
def patch_edges(length: int, n: int, scale: int = 1, reach: int = 1) -> List[int]:
    out = (C.c_int * (n + 1))()
    _check(load().vae_patch_edges(length, n, scale, reach, out), "vae_patch_edges")
    return list(out)


def tile_plan(lat_thw, tile_thw, ovl_thw, scale_t: int, scale_s: int, causal_t: bool = True) -> List[dict]:
    lib = load()
    a, b, c = ((C.c_int * 3)(*x) for x in (lat_thw, tile_thw, ovl_thw))
    n = C.c_int(0)
    _check(lib.vae_tile_plan(a, b, c, scale_t, scale_s, int(causal_t), None, C.byref(n)), "vae_tile_plan")
    arr = (VaeTile * n.value)()
    _check(lib.vae_tile_plan(a, b, c, scale_t, scale_s, int(causal_t), arr, C.byref(n)), "vae_tile_plan")
    return [{"lat": tuple(t.lat), "pix": tuple(t.pix), "ovl": tuple(t.ovl)} for t in arr]


# --------------------------------------------------------------------------- op level
def conv_desc(B, T, H, W, C_in, C_out, ph_edges, pw_edges, cache_frames=0, d2s=(1, 1, 1), drop_first=False,
              out_ncthw=False, in_dtype=VAE_BF16, out_dtype=VAE_BF16, res_dtype=VAE_BF16) -> VaeConvDesc:
    d = VaeConvDesc()
    d.B, d.T, d.H, d.W, d.C_in, d.C_out = B, T, H, W, C_in, C_out
    d.cache_frames = cache_frames
    d.n_patch_h, d.n_patch_w = len(ph_edges) - 1, len(pw_edges) - 1
    d.patch_h_edges, d.patch_w_edges = _edges_array(ph_edges), _edges_array(pw_edges)
    d.d2s_t, d.d2s_h, d.d2s_w = d2s
    d.drop_first, d.out_ncthw = int(drop_first), int(out_ncthw)
    d.in_dtype, d.out_dtype, d.res_dtype = in_dtype, out_dtype, res_dtype
    return d


def conv3d_pack_weights(w, d: VaeConvDesc, stream=None):
    torch = _torch()
    nbytes = load().vae_conv3d_packed_bytes(C.byref(d))
    out = torch.empty(nbytes, dtype=torch.uint8, device=w.device)
    _check(load().vae_conv3d_pack_weights(_ptr(w, torch.float32), C.byref(d), _ptr(out), _stream(stream)),
           "vae_conv3d_pack_weights")
    return out


def conv3d_causal(x, w_packed, bias, residual, y, d: VaeConvDesc, stream=None):
    torch = _torch()
    _check(load().vae_conv3d_causal(_ptr(x), _ptr(w_packed), _ptr(bias, torch.float32), _ptr(residual), _ptr(y),
                                    C.byref(d), _stream(stream)), "vae_conv3d_causal")
    return y


def gn_desc(B, T, H, W, Cc, groups, ph_edges, pw_edges, eps=1e-6, silu=True, in_dtype=VAE_BF16,
            out_dtype=VAE_BF16) -> VaeGnDesc:
    d = VaeGnDesc()
    d.B, d.T, d.H, d.W, d.C, d.groups, d.eps, d.silu = B, T, H, W, Cc, groups, eps, int(silu)
    d.n_patch_h, d.n_patch_w = len(ph_edges) - 1, len(pw_edges) - 1
    d.patch_h_edges, d.patch_w_edges = _edges_array(ph_edges), _edges_array(pw_edges)
    d.in_dtype, d.out_dtype = in_dtype, out_dtype
    return d


def gn_workspace(d: VaeGnDesc, device):
    torch = _torch()
    return torch.empty(load().vae_patch_groupnorm_workspace_bytes(C.byref(d)), dtype=torch.uint8, device=device)


def patch_groupnorm_silu(x, gamma, beta, y, workspace, d: VaeGnDesc, stream=None):
    torch = _torch()
    _check(load().vae_patch_groupnorm_silu(_ptr(x), _ptr(gamma, torch.float32), _ptr(beta, torch.float32), _ptr(y),
                                           _ptr(workspace), C.byref(d), _stream(stream)), "vae_patch_groupnorm_silu")
    return y


def prepare_patch_groupnorm_silu(x, gamma, beta, y, workspace, d: VaeGnDesc, stream=None):
    """Marshal the arguments of vae_patch_groupnorm_silu once; returns a function that only makes the
    C call."""
    torch = _torch()
    args = (_ptr(x), _ptr(gamma, torch.float32), _ptr(beta, torch.float32), _ptr(y), _ptr(workspace), C.byref(d),
            _stream(stream))
    lib = load()
    keep = (x, gamma, beta, y, workspace, d)

    def call():
        _check(lib.vae_patch_groupnorm_silu(*args), "vae_patch_groupnorm_silu")
    call.keep = keep
    return call


def patch_groupnorm_silu_noalloc(x, gamma, beta, y, d: VaeGnDesc, stream=None):
    """Same as patch_groupnorm_silu, with the scratch in the library's fixed device array."""
    torch = _torch()
    _check(load().vae_patch_groupnorm_silu_noalloc(_ptr(x), _ptr(gamma, torch.float32), _ptr(beta, torch.float32),
                                                   _ptr(y), C.byref(d), _stream(stream)),
           "vae_patch_groupnorm_silu_noalloc")
    return y


def channel_rmsnorm_silu(x, gamma, beta, y, B, T, H, W, Cc, eps=1e-6, silu=True, stream=None):
    """Channel RMS norm (+ SiLU) of channels-last x [B, T, H, W, C] into y (vae_channel_rmsnorm_silu)."""
    torch = _torch()
    d = VaeRmsDesc()
    d.B, d.T, d.H, d.W, d.C = B, T, H, W, Cc
    d.eps, d.silu = eps, int(silu)
    d.in_dtype, d.out_dtype = _dt(x), _dt(y)
    _check(load().vae_channel_rmsnorm_silu(_ptr(x), _ptr(gamma, torch.float32), _ptr(beta, torch.float32), _ptr(y),
                                           C.byref(d), _stream(stream)), "vae_channel_rmsnorm_silu")
    return y


def prepare_channel_rmsnorm_silu(x, gamma, beta, y, B, T, H, W, Cc, eps=1e-6, silu=True, stream=None):
    """Marshal the arguments of vae_channel_rmsnorm_silu once; returns a function that only makes the call."""
    torch = _torch()
    d = VaeRmsDesc()
    d.B, d.T, d.H, d.W, d.C = B, T, H, W, Cc
    d.eps, d.silu = eps, int(silu)
    d.in_dtype, d.out_dtype = _dt(x), _dt(y)
    lib = load()
    args = (_ptr(x), _ptr(gamma, torch.float32), _ptr(beta, torch.float32), _ptr(y), C.byref(d), _stream(stream))

    def call():
        _check(lib.vae_channel_rmsnorm_silu(*args), "vae_channel_rmsnorm_silu")
    call.keep = (d, x, gamma, beta, y)
    return call


def upsample_d2s(x, y, B, T, H, W, Cc, s, drop_first, stream=None):
    d = VaeD2sDesc()
    d.B, d.T, d.H, d.W, d.C = B, T, H, W, Cc
    d.s_t, d.s_h, d.s_w = s
    d.drop_first, d.dtype = int(drop_first), _dt(x)
    _check(load().vae_upsample_d2s(_ptr(x), _ptr(y), C.byref(d), _stream(stream)), "vae_upsample_d2s")
    return y


def prepare_tile_blend(tiles: Sequence, meta: Sequence[dict], out, stream=None):
    """Marshal the arguments of vae_tile_blend once; returns a function that only makes the C call
    (for loops that call the blend repeatedly on the same buffers)."""
    n = len(tiles)
    ptrs = (_P * n)(*[_ptr(t) for t in tiles])
    arr = (VaeTile * n)()
    for i, m in enumerate(meta):
        arr[i].lat = (C.c_int * 6)(*m.get("lat", (0,) * 6))
        arr[i].pix = (C.c_int * 6)(*m["pix"])
        arr[i].ovl = (C.c_int * 6)(*m["ovl"])
    d = VaeBlendDesc()
    d.B, d.C, d.T, d.H, d.W = out.shape
    d.tile_dtype, d.out_dtype = _dt(tiles[0]), _dt(out)
    optr, s, lib = _ptr(out), _stream(stream), load()
    keep = (ptrs, arr, d, tiles, out)

    def call():
        _check(lib.vae_tile_blend(keep[0], keep[1], n, optr, C.byref(keep[2]), s), "vae_tile_blend")
    return call


def tile_blend(tiles: Sequence, meta: Sequence[dict], out, stream=None):
    n = len(tiles)
    ptrs = (_P * n)(*[_ptr(t) for t in tiles])
    arr = (VaeTile * n)()
    for i, m in enumerate(meta):
        arr[i].lat = (C.c_int * 6)(*m.get("lat", (0,) * 6))
        arr[i].pix = (C.c_int * 6)(*m["pix"])
        arr[i].ovl = (C.c_int * 6)(*m["ovl"])
    d = VaeBlendDesc()
    d.B, d.C, d.T, d.H, d.W = out.shape
    d.tile_dtype, d.out_dtype = _dt(tiles[0]), _dt(out)
    _check(load().vae_tile_blend(ptrs, arr, n, _ptr(out), C.byref(d), _stream(stream)), "vae_tile_blend")
    return out


def gemm_bf16(A, Bm, D, bias=None, alpha=1.0, stream=None):
    """D[b] = alpha A[b] B[b]^T + bias on the tensor cores; A [batch, M, K], B [batch, N, K] bf16."""
    torch = _torch()
    if A.dim() == 2:
        A, Bm, D = A[None], Bm[None], D[None]
    batch, M, K = A.shape
    N = Bm.shape[1]
    _check(load().vae_gemm_bf16(_ptr(A, torch.bfloat16), _ptr(Bm, torch.bfloat16), _ptr(D), _ptr(bias, torch.float32),
                                M, N, K, batch, M * K, N * K, M * N, float(alpha), _dt(D), _stream(stream)),
           "vae_gemm_bf16")
    return D


def watchdog_selftest(timeout_us: int = 20000, stream=None) -> int:
    return load().vae_watchdog_selftest(int(timeout_us), _stream(stream))


# --------------------------------------------------------------------------- decoder
def make_config(cfg, dtype: int = VAE_BF16) -> VaeConfig:
    """VaeConfig from a ``synth.DecoderConfig``."""
    c = VaeConfig()
    c.latent_c = cfg.latent_c
    c.n_stages = cfg.n_stages
    for i, ch in enumerate(cfg.stage_c):
        c.stage_c[i] = ch
        c.n_res[i] = cfg.n_res[i]
    for i, u in enumerate(cfg.up):
        c.up_t[i], c.up_h[i], c.up_w[i] = u
    c.mid_res, c.mid_attn = cfg.mid_res, cfg.mid_attn
    c.gn_groups, c.gn_eps = cfg.gn_groups, cfg.gn_eps
    c.out_c = cfg.out_c
    c.out_d2s_t, c.out_d2s_h, c.out_d2s_w = cfg.out_d2s
    c.dtype = dtype
    c.norm_type = VAE_NORM_CHANNEL_RMS if getattr(cfg, "norm", "group") == "rms" else VAE_NORM_GROUP
    return c


def param_order(cfg) -> List[str]:
    """Parameter names in the order vae_decoder_create takes them (same as the declaration order)."""
    from . import synth
    return list(synth.param_specs(cfg).keys())


class Decoder:
    """A libvaedec decoder handle built from a config and fp32 parameter tensors (by name)."""

    def __init__(self, cfg, params: Dict[str, "object"], dtype: int = VAE_BF16, device="cuda"):
        torch = _torch()
        lib = load()
        self.cfg = cfg
        self.dtype = dtype
        self.c = make_config(cfg, dtype)
        names = param_order(cfg)
        dev = [params[n] if isinstance(params[n], torch.Tensor) else torch.from_numpy(np.ascontiguousarray(params[n]))
               for n in names]
        dev = [t.to(device=device, dtype=torch.float32).contiguous() for t in dev]
        n = C.c_int(0)
        _check(lib.vae_decoder_n_weights(C.byref(self.c), C.byref(n)), "vae_decoder_n_weights")
        if n.value != len(dev):
            raise ValueError(f"library expects {n.value} parameters, config lists {len(dev)}")
        arr = (_P * len(dev))(*[t.data_ptr() for t in dev])
        h = _P()
        _check(lib.vae_decoder_create(C.byref(self.c), arr, len(dev), C.byref(h)), "vae_decoder_create")
        self.h = h
        del dev

    def close(self):
        if getattr(self, "h", None):
            load().vae_decoder_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def out_dtype(self):
        torch = _torch()
        return torch.float32 if self.dtype in (VAE_FP32, VAE_FP32_TC) else torch.bfloat16

    def output_shape(self, latent_shape, first_chunk=True):
        b, _, t, h, w = latent_shape
        st, sh, sw = self.cfg.scale()
        nt = st * (t - 1) + 1 if first_chunk else st * t
        return (b, self.cfg.out_c, nt, sh * h, sw * w)

    def reserve(self, latent_shape, n_patch_h=1, n_patch_w=1):
        shp = (C.c_int64 * 5)(*latent_shape)
        _check(load().vae_decoder_reserve(self.h, shp, n_patch_h, n_patch_w), "vae_decoder_reserve", self.h)

    def profile(self, enable: bool):
        _check(load().vae_decoder_profile(self.h, int(enable)), "vae_decoder_profile", self.h)

    def profile_read(self) -> Dict[str, dict]:
        arr = (VaeProf * 32)()
        n = C.c_int(32)
        _check(load().vae_decoder_profile_read(self.h, arr, C.byref(n)), "vae_decoder_profile_read", self.h)
        return {arr[i].name.decode(): {"launches": arr[i].launches, "ms": arr[i].ms, "flops": arr[i].flops,
                                        "bytes": arr[i].bytes} for i in range(n.value)}

    def decode(self, latent, out=None, n_patch_h=1, n_patch_w=1, stream=None):
        torch = _torch()
        if out is None:
            out = torch.empty(self.output_shape(latent.shape), dtype=self.out_dtype(), device=latent.device)
        shp = (C.c_int64 * 5)(*latent.shape)
        _check(load().vae_decode(self.h, _ptr(latent, torch.float32), shp, _ptr(out, self.out_dtype()), n_patch_h,
                                 n_patch_w, _stream(stream)), "vae_decode", self.h)
        return out

    def decode_host(self, latent_cpu, out_cpu=None, n_patch_h=1, n_patch_w=1, frames_per_chunk=0, stream=None):
        """Host latent (CPU fp32, page-locked for overlap) -> host pixels (vae_decode_host)."""
        torch = _torch()
        if out_cpu is None:
            out_cpu = torch.empty(self.output_shape(latent_cpu.shape), dtype=self.out_dtype(), pin_memory=True)
        shp = (C.c_int64 * 5)(*latent_cpu.shape)
        _check(load().vae_decode_host(self.h, _hptr(latent_cpu, torch.float32), shp, _hptr(out_cpu, self.out_dtype()),
                                      n_patch_h, n_patch_w, frames_per_chunk, _stream(stream)), "vae_decode_host",
               self.h)
        return out_cpu

    def decode_chunk(self, latent_chunk, first_chunk, out=None, n_patch_h=1, n_patch_w=1, stream=None):
        torch = _torch()
        if out is None:
            out = torch.empty(self.output_shape(latent_chunk.shape, first_chunk), dtype=self.out_dtype(),
                              device=latent_chunk.device)
        shp = (C.c_int64 * 5)(*latent_chunk.shape)
        _check(load().vae_decode_chunk(self.h, _ptr(latent_chunk, torch.float32), shp, int(first_chunk),
                                       _ptr(out, self.out_dtype()), n_patch_h, n_patch_w, _stream(stream)),
               "vae_decode_chunk", self.h)
        return out

    def decode_tiled(self, latent, tile_thw, ovl_thw, out=None, stream=None):
        torch = _torch()
        if out is None:
            out = torch.empty(self.output_shape(latent.shape), dtype=self.out_dtype(), device=latent.device)
        shp = (C.c_int64 * 5)(*latent.shape)
        _check(load().vae_decode_tiled(self.h, _ptr(latent, torch.float32), shp, _ptr(out, self.out_dtype()),
                                       (C.c_int * 3)(*tile_thw), (C.c_int * 3)(*ovl_thw), _stream(stream)),
               "vae_decode_tiled", self.h)
        return out


# --------------------------------------------------------------------------- encoder
def make_encoder_config(cfg, dtype: int = VAE_BF16) -> VaeEncoderConfig:
    """VaeEncoderConfig from a ``synth.EncoderConfig``."""
    c = VaeEncoderConfig()
    c.pix_c = cfg.pix_c
    c.patch_h, c.patch_w = cfg.patchify
    c.n_stages = cfg.n_stages
    for i, ch in enumerate(cfg.stage_c):
        c.stage_c[i] = ch
        c.n_res[i] = cfg.n_res[i]
    for i, (kind, f) in enumerate(cfg.down):
        c.down_kind[i] = VAE_DOWN_FOLD if kind == "fold" else VAE_DOWN_STRIDE
        c.down_t[i], c.down_h[i], c.down_w[i] = f
    c.mid_res = cfg.mid_res
    c.gn_groups, c.gn_eps = cfg.gn_groups, cfg.gn_eps
    c.latent_c = cfg.latent_c
    c.dtype = dtype
    c.norm_type = VAE_NORM_CHANNEL_RMS if cfg.norm == "rms" else VAE_NORM_GROUP
    return c


class Encoder:
    """A libvaedec encoder handle built from a config and fp32 parameter tensors (by name)."""

    def __init__(self, cfg, params: Dict[str, "object"], dtype: int = VAE_BF16, device="cuda"):
        torch = _torch()
        lib = load()
        self.cfg = cfg
        self.dtype = dtype
        self.c = make_encoder_config(cfg, dtype)
        names = param_order(cfg)
        dev = [params[n] if isinstance(params[n], torch.Tensor) else torch.from_numpy(np.ascontiguousarray(params[n]))
               for n in names]
        dev = [t.to(device=device, dtype=torch.float32).contiguous() for t in dev]
        n = C.c_int(0)
        _check(lib.vae_encoder_n_weights(C.byref(self.c), C.byref(n)), "vae_encoder_n_weights")
        if n.value != len(dev):
            raise ValueError(f"library expects {n.value} parameters, config lists {len(dev)}")
        arr = (_P * len(dev))(*[t.data_ptr() for t in dev])
        h = _P()
        _check(lib.vae_encoder_create(C.byref(self.c), arr, len(dev), C.byref(h)), "vae_encoder_create")
        self.h = h
        del dev

    def close(self):
        if getattr(self, "h", None):
            load().vae_encoder_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def output_shape(self, video_shape):
        return self.cfg.latent_shape(video_shape)

    def last_error(self) -> Tuple[int, str]:
        info = VaeErrorInfo()
        code = load().vae_encoder_last_error(self.h, C.byref(info))
        return code, info.message.decode(errors="replace")

    def profile(self, enable: bool):
        _check(load().vae_encoder_profile(self.h, int(enable)), "vae_encoder_profile", enc=self.h)

    def profile_read(self) -> Dict[str, dict]:
        arr = (VaeProf * 32)()
        n = C.c_int(32)
        _check(load().vae_encoder_profile_read(self.h, arr, C.byref(n)), "vae_encoder_profile_read", enc=self.h)
        return {arr[i].name.decode(): {"launches": arr[i].launches, "ms": arr[i].ms, "flops": arr[i].flops,
                                        "bytes": arr[i].bytes} for i in range(n.value)}

    def encode(self, video, out=None, n_patch_h=1, n_patch_w=1, stream=None):
        """Pixels [B, C, T, H, W] fp32 -> moments [B, 2*latent_c, T', h, w] fp32 (vae_encode)."""
        torch = _torch()
        if out is None:
            out = torch.empty(self.output_shape(video.shape), dtype=torch.float32, device=video.device)
        shp = (C.c_int64 * 5)(*video.shape)
        _check(load().vae_encode(self.h, _ptr(video, torch.float32), shp, _ptr(out, torch.float32), n_patch_h,
                                 n_patch_w, _stream(stream)), "vae_encode", enc=self.h)
        return out

    def encode_tiled(self, video, tile_hw, ovl_hw, out=None, stream=None):
        torch = _torch()
        if out is None:
            out = torch.empty(self.output_shape(video.shape), dtype=torch.float32, device=video.device)
        shp = (C.c_int64 * 5)(*video.shape)
        _check(load().vae_encode_tiled(self.h, _ptr(video, torch.float32), shp, _ptr(out, torch.float32),
                                       (C.c_int * 2)(*tile_hw), (C.c_int * 2)(*ovl_hw), _stream(stream)),
               "vae_encode_tiled", enc=self.h)
        return out
