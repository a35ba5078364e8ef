"""GB300 (sm_103a) hot path of 4-bit group-quantised, block-scheduled OPT
decoding: a C-ABI CUDA library (libfg, include/fg.h) with a thin ctypes
binding (``fg``) and a model driver (``model``).

Importing the package does not touch the GPU.  The first call into ``fg``
loads ``lib/libfg.so`` and raises if it has not been built; there is no
fallback path.
"""
from . import fg  # noqa: F401

__all__ = ["fg", "build"]


def build(force: bool = False) -> str:
    from ._build import build as _b
    return _b(force=force)
