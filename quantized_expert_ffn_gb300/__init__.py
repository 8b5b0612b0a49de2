"""Routed mixture-of-experts FFN layer on one GB300 (sm_103a): CUDA kernels
behind the C ABI of include/moe.h, with a thin ctypes binding (_lib).

The Python side only marshals arguments; every step of the layer runs in the
CUDA library, which raises if it is missing (no CPU fallback).
"""
from . import _lib  # noqa: F401
from ._lib import MoeError, load, lib_path  # noqa: F401

__all__ = ["_lib", "MoeError", "load", "lib_path"]
