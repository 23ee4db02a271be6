"""GB300 (sm_103a) attention backward with recomputed scores and softmax.

The product is the C-ABI library ``libattnbwd.so`` (declared in
``include/attn_bwd.h``); this package holds its CUDA sources (``csrc/``), the
build script, the ctypes binding and the seeded input generators.
"""
from . import inputs  # noqa: F401

__all__ = ["inputs", "binding", "build"]


def __getattr__(name):
    if name in ("binding", "build"):
        import importlib
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
