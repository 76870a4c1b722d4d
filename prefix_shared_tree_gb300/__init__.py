"""Prefix-shared (tree) decode attention for GB300 (sm_103a).

``pst`` is the ctypes binding of the C ABI in include/pst.h (libpst.so, built
in-tree by ``build.build()``); ``torch_api`` binds it to torch tensors and
streams. Every step of the computation runs in the library's CUDA kernels;
there is no CPU fallback.
"""
from . import build, pst  # noqa: F401

__all__ = ["build", "pst"]
