"""Float64 CPU oracle for MLA latent-KV decode.

TEST INFRASTRUCTURE ONLY. Nothing in the product package may import this.
Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` use it.
"""
from .mla_oracle import (  # noqa: F401
    E4M3_MAX, FP8_ROW_BYTES,
    e4m3_value_table, e4m3_encode_rne,
    quantize_kv_fp8, dequantize_kv_fp8,
    V41_DIM, FP8_528_ROW_BYTES, FP4_288_ROW_BYTES, E2M1_MAX,
    e2m1_value_table, ue8m0_value, e2m1_encode_rne,
    quantize_kv_fp8_528, dequantize_kv_fp8_528, quantize_kv_fp4_288, dequantize_kv_fp4_288,
    attend, visible_rows, mla_decode, absorb_q, up_project,
    bf16_to_f64, to_f64,
)
