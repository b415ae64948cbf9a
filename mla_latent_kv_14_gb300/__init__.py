"""GB300-native MLA latent-KV decode.

The compute lives in ``libmla.so`` (hand-written sm_103a CUDA behind the C ABI
of ``include/mla.h``); this package is its thin Python binding.
"""
from .binding import (  # noqa: F401
    LIB_PATH, MLAError, Metadata, load_library,
    mla_num_sm_parts, mla_get_metadata, mla_decode_with_kvcache, mla_decode_splitkv, mla_combine_splits,
    mla_decode_with_kvcache_noalloc, mla_quantize_kv_fp8, mla_read_status, workspace_for,
    mla_absorb_q, mla_up_project, mla_set_test_stall,
    mla_quantize_kv_fp8_528, mla_quantize_kv_fp4_288, KV_16BIT, KV_FP8_656, KV_FP8_528, KV_FP4_288,
)
