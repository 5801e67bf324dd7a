"""W12: lossless 12-bit BF16 weights, a fused decode-GEMM and greedy verify on GB300.

The compute lives in ``libw12.so`` (CUDA for sm_103a behind a C ABI declared
in ``include/w12.h``); ``lossless_bit_weight_w12_gb300.w12`` is the thin ctypes
binding.  Importing this package does not load the library; the first call
into ``w12`` does, and it raises if the library has not been built.
"""
__all__ = ["w12", "synth"]
