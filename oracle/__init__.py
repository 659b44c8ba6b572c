"""CPU oracle for the quantized-weight OUT_PROD (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU baseline /
reference leg may import this package.  The library under
``quantized_weight_out_gb300`` never does: it has no CPU fallback.
"""
from .quant_out_prod import (  # noqa: F401
    F16, BF16, Q8_0, Q4_0, Q4_K, Q4_1, Q5_0, Q5_1, Q5_K, Q6_K, F32, Q2_K, Q3_K, MXFP4, NVFP4,
    f16_bits_to_f32, bf16_bits_to_f32,
    decode_q8_0, decode_q4_0, decode_q4_k, decode_f16, decode_bf16,
    decode_q4_1, decode_q5_0, decode_q5_1, decode_q5_k, decode_q6_k, decode_f32,
    decode_q2_k, decode_q3_k, q3_k_scales, decode_mxfp4, e8m0_to_f32, e2m1_to_f32,
    decode_nvfp4, e4m3_to_f32,
    dequant, row_bytes, out_prod, abs_bound, out_prod_at, q4_k_scale_min, mul_mat, mul_mat_bound,
    out_prod_lora, lora_bound, lora_at, batch_weight, out_prod_batched, mul_mat_at,
)
