"""GB300-native causal differential-attention forward (DIFF V1, DIFF V2, V2 decode).

The compute lives in libdiffattn.so (hand-written sm_103a CUDA behind a C ABI,
include/diffattn.h); ``binding`` is a thin ctypes layer over it and
``inputs`` draws the seeded synthetic workloads.  Importing this package does
not load the library; the first call through ``binding`` does, and fails
loudly if it has not been built.
"""
import importlib

from . import inputs  # noqa: F401

__all__ = ["inputs", "binding"]


def __getattr__(name):
    if name == "binding":
        return importlib.import_module(".binding", __name__)
    if name in ("v1_fwd", "v2_fwd", "v2_decode", "decode_workspace_size", "device_error"):
        return getattr(importlib.import_module(".binding", __name__), name)
    raise AttributeError(name)
