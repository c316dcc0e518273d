"""CPU oracle for the patched / tiled causal video-VAE decode.

TEST INFRASTRUCTURE ONLY.  Nothing in the library imports, links or runs this package: only
the tests, the package's smoke check and the benchmark's CPU-baseline arm do.  It shares no
code with the CUDA path; both take their inputs from the seeded generators in
``patch_tiled_causal_gb300.synth``, which hold none of the decode's arithmetic.

Layout: PyTorch's NCTHW ([B, C, T, H, W]) throughout, the layout the pages' modules use.

Two tiers:
  * Tier A (``tier="A"``): float64, each causal convolution written as a direct sum over its
    27 taps of shifted-slice channel contractions.  Used for the tiny workload and op tests.
  * Tier B (``tier="B"``): float32, the same sum with one BLAS matrix product per tap over
    channels-last frame chunks.  Used at the full sizes; checked against Tier A on small inputs.

Modules:
  ops      convolution, group norm, SiLU, depth-to-space, attention, residual block
  decoder  the unpatched decode, whole or in temporal chunks with a per-convolution frame cache
  patched  the patched decode: explicit halo reads from neighbour patches, per-patch partial sums
  tiles    tile plan, blend ramps, overlap blend and the sequential tiled decode
  plan     patch boundaries (band rule)
  metrics  parity metrics (max relative error, relative L2, PSNR)

Parity status of each part is stated in its module header.
"""
