"""B300-native (sm_103a) Prism content-adaptive block-sparse attention.

The compute path lives in the CUDA library built from ``csrc/`` and is reached
through the C ABI declared in ``include/prism.h``; ``prism`` is the thin ctypes
binding over it and ``synth`` the seeded workload generator.  Importing the
package loads nothing: ``prism`` loads the shared library on first use and
raises if it is missing.
"""
__all__ = ["synth", "prism"]
