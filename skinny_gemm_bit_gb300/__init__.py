"""GB300 (sm_103a) 4/8-bit group-quantised decode projections.

The compute lives in ``libtfq.so`` (CUDA, C ABI declared in ``include/tfq.h``);
``skinny_gemm_bit_gb300.tfq`` is the thin ctypes binding over it and
``skinny_gemm_bit_gb300.synth`` holds the seeded input generators. Importing
the package itself loads nothing.
"""
__all__ = ["synth", "tfq"]
