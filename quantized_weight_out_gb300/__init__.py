"""Fused quantized-weight OUT_PROD for NVIDIA GB300 (sm_103a).

dX = beta * dX + dY . deq(W): the activation gradient of a mul_mat whose base
weight W stays resident in F16, BF16, Q8_0, Q4_0, Q4_1, Q5_0, Q5_1, Q4_K,
Q5_K or Q6_K.  The compute lives
in the C-ABI library ``librg.so`` (CUDA, built in-tree); ``binding`` wraps it
with ctypes.  The library is loaded on first use and a missing build raises.
"""
from .inputs import F16, BF16, Q8_0, Q4_0, Q4_K, Q4_1, Q5_0, Q5_1, Q5_K, Q6_K, row_bytes  # noqa: F401
