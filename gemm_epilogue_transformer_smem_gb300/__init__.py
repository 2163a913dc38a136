"""GB300 (sm_103a) fused GEMM + composable-epilogue engine.

The compute path is the CUDA library under ``csrc/`` behind the C ABI in
``include/gemm_epi.h``; ``native`` binds it with ctypes and ``api`` passes
torch tensors to it.  ``synth`` draws the seeded synthetic workloads.
"""
from . import synth  # noqa: F401

__all__ = ["synth", "native", "api", "build"]
