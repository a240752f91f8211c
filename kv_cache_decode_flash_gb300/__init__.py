"""Decode attention over a q8_0 / f16 grouped-query KV cache on one GB300 GPU.

The computation lives in libkvc.so (C ABI: include/kvc.h), built from
csrc/ for sm_103a.  `kvc` is the thin ctypes binding with the ABI's names;
importing this package does not load the library (so the CPU-only tests can
use `synth`), the first call does, and fails loudly if it is missing.
"""
from . import synth  # noqa: F401

__all__ = ["synth", "kvc"]


def __getattr__(name):
    if name == "kvc":
        import importlib

        return importlib.import_module(__name__ + ".kvc")
    raise AttributeError(name)
