"""GB300-native Q4_0 decode-step matrix-vector product and weight streaming.

The C ABI lives in libq4.so (include/q4.h); this package is its ctypes
binding (``_lib``), the in-tree build (``build``), the seeded synthetic-input
generator (``synth``) and helpers that lay out Llama-shaped synthetic models
in device or pinned host memory (``model``).  Importing the package does not
load the library; the first call does, and fails loudly if it is not built.
"""
from ._lib import *  # noqa: F401,F403
from ._lib import LayerShape, Q4Error, lib  # noqa: F401

__version__ = "0.1.0"
