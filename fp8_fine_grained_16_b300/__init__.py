"""Fine-grained FP8 (E4M3) quantise + block-scaled GEMM for B300 (sm_103a).

The compute lives in ``libfp8bs.so`` (hand-written CUDA behind a C ABI,
declared in ``include/fp8bs.h``).  ``fp8_fine_grained_16_b300.fp8bs`` is the
thin ctypes binding with the same entry-point names; attributes of this
package that name an entry point load it on first use, and loading fails
loudly if the library has not been built.
"""
from __future__ import annotations

import importlib

__all__ = ["fp8bs", "synthetic", "build"]


def __getattr__(name):
    if name.startswith("fp8_") or name == "FP8Error":
        return getattr(importlib.import_module(__name__ + ".fp8bs"), name)
    raise AttributeError(name)
