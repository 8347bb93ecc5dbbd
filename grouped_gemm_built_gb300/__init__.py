"""GB300-native (sm_103a) MoE SwiGLU layer: routing, no-sort schedule table, dispatch,
tcgen05 grouped GEMMs, combine and the full backward, behind the C ABI in include/mok.h.

``mok`` is the ctypes binding (same names as the C ABI); ``layer.MoELayer`` owns the
caller-side buffers as torch tensors. ``build.build()`` compiles libmok.so in-tree.
"""
from . import build, mok  # noqa: F401

__all__ = ["build", "mok"]
