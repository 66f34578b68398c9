"""GB300-native decode step of a GGUF Q8_0 / Q4_0 Llama-style decoder.

The compute lives in liber.so (hand-written CUDA for sm_103a behind the C ABI of
include/er.h).  ``er`` is its ctypes binding (same names as the header),
``runtime`` holds small owners of model/state handles, ``build`` compiles the
library.  Importing the package itself loads nothing; importing ``er`` loads
the library and fails if it has not been built.
"""

__all__ = ["build", "er", "runtime"]
