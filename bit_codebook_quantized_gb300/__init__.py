"""3.25-bit codebook-quantised decode / speculative-verify matmul for GB300.

The compute lives in the C-ABI library ``libcbq.so`` (CUDA, sm_103a) built
from ``csrc/``; ``ops`` is a thin ctypes binding with the same names as the C
entry points.  Importing this package does not load the library; the first
call into ``ops`` does, and raises if it has not been built.
"""

__all__ = ["ops", "synth", "build"]
