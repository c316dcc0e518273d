"""The allocation-free group-norm entry point, for callers that cannot allocate device memory.

vae_patch_groupnorm_silu_noalloc keeps its scratch in a fixed device array inside the library instead
of taking a workspace.  Both entry points run the same kernels on the same exact integer sums, so
through the C ABI two calls in a row must give, bit for bit, what the workspace-taking
vae_patch_groupnorm_silu gives.  The first call is the larger one (more patches, frames and
groups), so that the second, smaller call would read nonzero leftovers in the shared array if it
did not clear what it needs.  A descriptor needing more scratch than the array holds is refused.
This file is collected last and must also pass on its own in a fresh process.
"""
import pytest
import torch

from patch_tiled_causal_gb300 import synth

pytestmark = pytest.mark.gpu

@pytest.fixture(scope="module")
def vd():
    from patch_tiled_causal_gb300 import build, vaedec
    build.build()
    vaedec.load()
    return vaedec


def _edges(n, parts):
    q, r = divmod(n, parts)
    e = [0]
    for i in range(parts):
        e.append(e[-1] + q + (1 if i < r else 0))
    return e


def test_noalloc_matches_workspace_entry_point_twice(vd):
    cases = [((2, 4, 20, 36, 256), 32, (4, 6), vd.VAE_BF16, 0.0, 11),   # 24 patches x 8 frames x 32 groups
             ((1, 2, 9, 24, 128), 16, (1, 4), vd.VAE_FP32, 3.0, 12)]
    for shape, groups, (ph, pw), dt, offset, seed in cases:
        B, T, H, W, Cc = shape
        tdt = torch.bfloat16 if dt == vd.VAE_BF16 else torch.float32
        x = torch.from_numpy(synth.draw_normal(shape, seed, offset=offset)).cuda().to(tdt)
        g = torch.from_numpy(synth.draw_normal((Cc,), seed + 1) * 0.1 + 1.0).cuda()
        b = torch.from_numpy(synth.draw_normal((Cc,), seed + 2) * 0.1).cuda()
        d = vd.gn_desc(B, T, H, W, Cc, groups, _edges(H, ph), _edges(W, pw), in_dtype=dt, out_dtype=dt)
        ws = vd.gn_workspace(d, "cuda")
        y_ref = torch.empty_like(x)
        y_na = torch.full_like(x, float("nan"))
        vd.patch_groupnorm_silu(x, g, b, y_ref, ws, d)
        vd.patch_groupnorm_silu_noalloc(x, g, b, y_na, d)
        torch.cuda.synchronize()
        assert vd.last_error()[0] == vd.VAE_OK
        assert torch.isfinite(y_na.float()).all()
        assert torch.equal(y_na, y_ref)


def test_noalloc_refuses_oversized_scratch(vd):
    # 64 x 64 patches x 1024 frames x 32 groups of partial sums cannot fit the fixed array
    B, T, H, W, Cc = 1, 1024, 64, 64, 64
    d = vd.gn_desc(B, T, H, W, Cc, 32, list(range(65)), list(range(65)), in_dtype=vd.VAE_BF16, out_dtype=vd.VAE_BF16)
    x = torch.zeros(16, dtype=torch.bfloat16, device="cuda")  # never read: the call is refused first
    one = torch.ones(Cc, device="cuda")
    with pytest.raises(vd.VaeError) as e:
        vd.patch_groupnorm_silu_noalloc(x, one, one, x, d)
    assert e.value.code == vd.VAE_ERR_UNSUPPORTED
