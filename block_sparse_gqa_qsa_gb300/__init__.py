"""GB300-native QSA (Qwen Sparse Attention) block-sparse GQA.

The compute path is the C-ABI library ``libqsa.so`` (hand-written sm_103a
kernels, declared in ``include/qsa.h``); this package is its thin Python
binding.  Importing the package does not load the library; the first call does,
and raises ``RuntimeError`` when it is missing -- there is no CPU fallback.
"""
from __future__ import annotations

__all__ = ["lib", "synthetic"]


def __getattr__(name):
    if name == "lib":
        from . import _binding
        return _binding
    raise AttributeError(name)
