"""B300 (sm_103a) quantized decode GEMM: FP8_Dynamic, W8A8_INT8 and Block_FP8
with the Standard, Split-K and Swap-AB variants.

The compute path is the C-ABI library ``libqgemm.so`` built from ``csrc/``
(see ``include/qgemm.h``); ``qgemm`` is its thin ctypes binding.
"""
