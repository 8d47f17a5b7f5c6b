"""Context-parallel exact softmax attention on one GB300 (sm_103a).

All P sequence chunks ("virtual ranks") of Ring, Ulysses, Ulysses-Anything and Unified
sequence-parallel attention live on one GPU.  The compute runs in the CUDA library
``libusp_gb300.so`` behind the C ABI in ``include/usp.h``; ``usp`` is its thin ctypes binding.
``synth`` holds the seeded input generator and the workload shapes.
"""
__all__ = ["synth", "usp"]
