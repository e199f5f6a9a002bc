"""GB300-native MoE-layer hot path: route, dispatch layout, permute, grouped
SwiGLU FFN, combine and balancedness as hand-written sm_103a CUDA kernels
behind a C ABI (include/moe.h, libmoe.so).  Python here only marshals
arguments; build the library with grouped_ffn_gb300.build.build()."""

from . import moe  # noqa: F401
from .layer import MoELayer  # noqa: F401

__all__ = ["moe", "MoELayer"]
