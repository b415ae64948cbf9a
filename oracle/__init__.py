"""Float64 CPU oracle for MLA latent-KV decode.

TEST INFRASTRUCTURE ONLY. Nothing in the product package may import this.
Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` use it.
"""
from .mla_oracle import (  # noqa: F401
    E4M3_MAX, FP8_ROW_BYTES,
    e4m3_value_table, e4m3_encode_rne,
    quantize_kv_fp8, dequantize_kv_fp8,
    attend, visible_rows, mla_decode, absorb_q, up_project,
    bf16_to_f64, to_f64,
)
