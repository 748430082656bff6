"""GB300-native persistent GPT training step.

The product is libgpt.so (CUDA C++ for sm_103a, C ABI declared in
include/gpt.h); ``binding`` is its ctypes binding and ``inputs`` the seeded
synthetic workload generators.  Importing this package loads nothing; the
library is loaded on first use and its absence is an error.
"""

__all__ = ["binding", "inputs", "build"]
