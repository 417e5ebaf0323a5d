"""GB300-native block-scaled FP8 linear layer.

The compute path is the C-ABI library ``libfp8bs.so`` (hand-written CUDA for
sm_103a, declared in include/fp8bs.h); ``fp8_block_scaled_05_gb300.ops`` is its
thin ctypes binding.  Nothing here falls back to a CPU implementation: a call
without the built library raises.  Importing the package loads nothing, so the
input generators (``.inputs``) work without a GPU.
"""
