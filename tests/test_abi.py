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
