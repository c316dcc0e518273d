"""GB300-native patched / tiled causal video-VAE decode.

The compute path is the C-ABI library ``libvaedec.so`` (hand-written CUDA for sm_103a); the
Python module ``patch_tiled_causal_gb300.vaedec`` is a thin ctypes binding over it.
``patch_tiled_causal_gb300.synth`` holds the seeded synthetic workloads.
"""
