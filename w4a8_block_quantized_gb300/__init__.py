"""GB300-native W4A8 block-64 quantized prefill linear.

The compute lives in hand-written CUDA kernels for sm_103a behind a C-ABI
library (``include/w4a8.h``); :mod:`w4a8_block_quantized_gb300.binding` marshals
arguments to it.  Importing this package does not load the library; the first
call into :mod:`binding` does, and fails loudly when it is missing.
"""
__all__ = ["binding", "synth"]
