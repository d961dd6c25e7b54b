"""GB300-native speculative-decoding verification (chain, greedy, EAGLE trees).

The compute path is libspecverify.so (hand-written CUDA for sm_103a, C ABI in
include/specverify.h).  ``api`` marshals torch tensors into that ABI; ``_lib``
is the raw ctypes binding.  Importing this package does not load the library;
the first call does, and raises if it has not been built.
"""

from . import _lib  # noqa: F401
from ._lib import SpecError, SpecParams  # noqa: F401

__all__ = ["api", "_lib", "SpecError", "SpecParams"]


def __getattr__(name):
    if name == "api":
        import importlib
        return importlib.import_module(__name__ + ".api")
    raise AttributeError(name)
