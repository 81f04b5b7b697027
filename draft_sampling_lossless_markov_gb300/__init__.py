"""DSpark per-step hot path on GB300: C-ABI CUDA library + thin Python binding.

`capi` mirrors include/dspark.h (ctypes, same names); `torch_api` fills its
structs from torch tensors.  The library itself is `_lib/libdspark.so`, built
in-tree by `build.py`; nothing here computes any step of the method.
"""
import importlib

from . import capi  # noqa: F401

__all__ = ["capi", "torch_api", "build"]


def __getattr__(name):
    if name in ("torch_api", "build"):
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
