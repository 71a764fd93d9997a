"""GB300-native routed-expert FFN step of an offloaded-MoE serving engine.

The compute runs in a CUDA library (``csrc/``, built for sm_103a) behind the
C ABI of ``include/moe_gb300.h``; ``MoELayer`` is its Python binding.
"""

from ._abi import load as load_library, LIB_PATH, ENTRY_POINTS, MoeError
from .build import build as build_library

__all__ = ["load_library", "LIB_PATH", "ENTRY_POINTS", "MoeError", "build_library", "MoELayer"]


def __getattr__(name):
    if name == "MoELayer":
        from .layer import MoELayer
        return MoELayer
    raise AttributeError(name)
