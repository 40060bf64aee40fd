"""GB300 (sm_103a) MoE FFN block: router + top-K + NVFP4/MXFP4 expert FFN + combine.

The compute path is the CUDA library libmoe_gb300.so behind the C ABI in include/moe.h;
this package holds its ctypes binding (``capi``), a small layer object that owns device
buffers (``layer.MoeLayer``), the in-tree build script (``build``) and the seeded synthetic
input generator (``synth``).  Importing the package loads nothing; the first call into
``capi`` loads the library and fails loudly if it has not been built.
"""
from . import synth  # noqa: F401

__all__ = ["synth", "capi", "layer", "build"]
