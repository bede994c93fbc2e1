"""GB300-native fused speculative-decode verify step (sm_103a).

The CUDA library libmk.so (C ABI in include/mk.h) runs the whole verify cycle
in one persistent cooperative kernel; `mk` is its ctypes binding.
"""
from . import build  # noqa: F401


def load():
    """Import the binding (raises ImportError if libmk.so was not built)."""
    from . import mk
    return mk
