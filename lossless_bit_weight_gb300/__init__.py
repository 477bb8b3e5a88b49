"""W12 lossless 12-bit weights and the skinny verification GEMM, for one GB300 (sm_103a).

The compute path is the C-ABI library ``libw12.so`` built from ``csrc/``; ``w12`` is its thin
Python binding. Importing the package does not load the library: the first call does, and it
raises if the library is missing.
"""
__all__ = ["w12", "synth"]
