"""Quantized mixture-of-experts FFN layer for one GB300 (sm_103a).

The compute path is the CUDA library behind include/moe.h (built in-tree by
``build.build_cuda``); ``moe`` is its thin ctypes binding and ``synth`` the
seeded input generator.  There is no CPU fallback: using ``moe`` without the
CUDA library, or without a GPU, raises.
"""
from . import synth  # noqa: F401

__all__ = ["synth", "moe", "stack"]


def __getattr__(name):
    if name in ("moe", "stack"):
        import importlib
        return importlib.import_module(__name__ + "." + name)
    raise AttributeError(name)
