"""dense_block_scaled_gb300 -- GB300 (sm_103a) dense and block-scaled GEMM.

The compute lives in ``libtkg.so`` (hand-written CUDA for sm_103a behind a C
ABI declared in ``include/tkg_gemm.h``).  ``dense_block_scaled_gb300.tkg`` is
the thin ctypes binding; importing this package loads nothing, so the seeded
input generators in ``synth`` stay usable on machines without the library.
"""

__all__ = ["tkg", "synth"]
