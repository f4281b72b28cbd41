"""GB300-native block-quantized MatMulNBits (INT4 / INT8, block 32) with a fused
rank-32 FP16 LoRA term.

The compute path is the CUDA library ``libmnb.so`` (C ABI in ``include/mnb.h``);
``block_quantized_matmul_matmulnbits_gb300.mnb`` is its thin ctypes binding.
Importing this package does not load the library; the first call does, and it
raises if the library has not been built.
"""
__all__ = ["mnb", "synth"]
