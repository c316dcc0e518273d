"""The C-ABI library loads, exports every symbol include/vaedec.h declares, and its host plans
(pure integer, no GPU) agree bit for bit with the oracle's."""
import os
import re

import pytest

from oracle import plan as oplan
from oracle import tiles as otiles
from patch_tiled_causal_gb300 import build, vaedec

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return vaedec.load()


def header_symbols():
    with open(os.path.join(ROOT, "include", "vaedec.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(vae_[a-z0-9_]+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    syms = header_symbols()
    assert len(syms) >= 19
    for s in syms:
        assert hasattr(lib, s), s
    assert set(vaedec.declared_symbols()) == set(syms)


@pytest.mark.parametrize("length,n,scale", [(15, 2, 1), (16, 3, 1), (22, 4, 8), (40, 4, 32), (13, 8, 1), (80, 1, 16)])
def test_patch_edges_match_oracle(lib, length, n, scale):
    assert vaedec.patch_edges(length, n, scale) == oplan.band_edges(length, n, scale)


def test_patch_too_narrow_is_refused(lib):
    with pytest.raises(vaedec.VaeError) as e:
        vaedec.patch_edges(3, 4, 1, 1)
    assert e.value.code == vaedec.VAE_ERR_PATCH_TOO_NARROW
    assert e.value.rows == 0 and e.value.factor == 1


@pytest.mark.parametrize("case", [
    ((17, 34, 60), (8, 16, 16), (1, 4, 4), 8, 32, True),
    ((1, 704, 1280), (1, 256, 256), (0, 64, 64), 81, 1, False),
    ((5, 7, 9), (3, 4, 4), (1, 1, 2), 2, 8, True),
    ((1, 18, 18), (1, 16, 16), (0, 2, 2), 1, 32, False),
    ((21, 44, 80), (21, 44, 80), (0, 4, 4), 4, 16, True),
])
def test_tile_plan_matches_oracle(lib, case):
    lat, tile, ovl, st, ss, causal = case
    got = vaedec.tile_plan(lat, tile, ovl, st, ss, causal)
    ref = otiles.tile_plan(lat, tile, ovl, st, ss, causal_t=causal)
    assert len(got) == len(ref)
    for g, r in zip(got, ref):
        assert g["lat"] == r.lat and g["pix"] == r.pix and g["ovl"] == r.ovl


def test_invalid_arguments_are_refused(lib):
    with pytest.raises(vaedec.VaeError) as e:
        vaedec.tile_plan((4, 4, 4), (2, 2, 2), (2, 0, 0), 1, 1)  # overlap == tile
    assert e.value.code == vaedec.VAE_ERR_INVALID_ARG
    import ctypes as C
    n = C.c_int(0)
    assert lib.vae_decoder_n_weights(None, C.byref(n)) == vaedec.VAE_ERR_INVALID_ARG


# ctypes mirrors of the header's structs, checked field by field against the C compiler's layout
STRUCTS = [("VaeConfig", "vae_config_t"), ("VaeErrorInfo", "vae_error_info_t"), ("VaeTile", "vae_tile_t"),
           ("VaeConvDesc", "vae_conv_desc_t"), ("VaeGnDesc", "vae_gn_desc_t"), ("VaeRmsDesc", "vae_rms_desc_t"),
           ("VaeD2sDesc", "vae_d2s_desc_t"), ("VaeBlendDesc", "vae_blend_desc_t"), ("VaeProf", "vae_prof_t"),
           ("VaeEncoderConfig", "vae_encoder_config_t")]


def test_binding_structs_match_header_layout(tmp_path):
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no host C compiler")
    lines = ["#include <stddef.h>", "#include <stdio.h>", '#include "vaedec.h"', "int main(void) {"]
    for py, c in STRUCTS:
        cls = getattr(vaedec, py)
        lines.append(f'  printf("{py} size %zu\\n", sizeof({c}));')
        for name, _ in cls._fields_:
            lines.append(f'  printf("{py} {name} %zu\\n", offsetof({c}, {name}));')
    lines += ["  return 0;", "}"]
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "layout"
    subprocess.run([cc, "-std=c11", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    got = {}
    for line in subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.splitlines():
        py, key, val = line.split()
        got[(py, key)] = int(val)
    import ctypes as C
    for py, _ in STRUCTS:
        cls = getattr(vaedec, py)
        assert got[(py, "size")] == C.sizeof(cls), py
        for name, _ in cls._fields_:
            assert got[(py, name)] == getattr(cls, name).offset, (py, name)


def test_config_checks_for_both_norm_families(lib):
    # host-only validation (no GPU): vae_decoder_n_weights checks the config first
    import ctypes as C
    from patch_tiled_causal_gb300 import synth
    n = C.c_int(0)
    for name in ("mini_wan", "mini_wan_rms", "wan_rms"):
        cfg = vaedec.make_config(synth.CONFIGS[name])
        assert lib.vae_decoder_n_weights(C.byref(cfg), C.byref(n)) == vaedec.VAE_OK, name
        assert n.value == len(vaedec.param_order(synth.CONFIGS[name]))
    rms = vaedec.make_config(synth.MINI_WAN_RMS)
    assert rms.norm_type == vaedec.VAE_NORM_CHANNEL_RMS
    rms.gn_groups = 0  # ignored by RMS norms
    assert lib.vae_decoder_n_weights(C.byref(rms), C.byref(n)) == vaedec.VAE_OK
    for bad_c in (1032, 2048, 12):  # not a power-of-two / multiple-of-32 vector count, too wide, not / 8
        c = vaedec.make_config(synth.MINI_WAN_RMS)
        c.stage_c[1] = bad_c
        assert lib.vae_decoder_n_weights(C.byref(c), C.byref(n)) == vaedec.VAE_ERR_UNSUPPORTED, bad_c
    c = vaedec.make_config(synth.MINI_WAN)
    c.norm_type = 7
    assert lib.vae_decoder_n_weights(C.byref(c), C.byref(n)) == vaedec.VAE_ERR_INVALID_ARG
    c = vaedec.make_config(synth.MINI_WAN)
    c.gn_groups = 0  # group norms need groups
    assert lib.vae_decoder_n_weights(C.byref(c), C.byref(n)) == vaedec.VAE_ERR_INVALID_ARG


def test_encoder_config_checks(lib):
    # host-only validation (no GPU): vae_encoder_n_weights checks the config first
    import ctypes as C
    from patch_tiled_causal_gb300 import synth
    n = C.c_int(0)
    for name, cfg in synth.ENCODERS.items():
        c = vaedec.make_encoder_config(cfg)
        assert lib.vae_encoder_n_weights(C.byref(c), C.byref(n)) == vaedec.VAE_OK, name
        assert n.value == len(vaedec.param_order(cfg)), name
    bad = vaedec.make_encoder_config(synth.MINI_ENC_STRIDE)
    bad.down_h[0] = 3  # the strided down-sampler halves rows and columns only
    assert lib.vae_encoder_n_weights(C.byref(bad), C.byref(n)) == vaedec.VAE_ERR_UNSUPPORTED
    bad = vaedec.make_encoder_config(synth.MINI_ENC)
    bad.down_kind[0] = 7
    assert lib.vae_encoder_n_weights(C.byref(bad), C.byref(n)) == vaedec.VAE_ERR_INVALID_ARG
