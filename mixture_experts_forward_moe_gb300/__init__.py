"""GB300-native fused Mixture-of-Experts forward pass.

The compute lives in ``libgb300moe.so`` (hand-written CUDA for sm_103a behind the C ABI in
``include/moe.h``).  ``binding`` marshals torch tensors into that ABI; ``inputs`` holds the
seeded synthetic input generators.  Importing this package loads nothing: the library is
loaded (and built if needed) on the first call into ``binding``.
"""

__all__ = ["binding", "inputs", "build"]
