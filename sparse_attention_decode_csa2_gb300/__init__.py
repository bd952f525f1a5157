"""CSA2 compressed sparse attention hot path for GB300 (sm_103a).

The compute lives in ``libcsa2.so`` (hand-written CUDA kernels behind a C ABI,
declared in ``include/csa2.h``).  ``sparse_attention_decode_csa2_gb300.csa2``
is the thin Python binding over it; importing that module loads the library
and raises if it has not been built.  ``synthetic`` holds the seeded input
generators.  Importing this package itself loads nothing.
"""

__all__ = ["csa2", "synthetic"]
