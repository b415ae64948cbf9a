"""Seeded synthetic inputs for MLA latent-KV decode.

This package is shared by the tests, the benchmark and the smoke check. It
only draws random numbers and lays them out (queries, latent cache rows, block
tables, sequence lengths, sparse index lists); it holds none of the attention,
softmax or quantisation arithmetic.
"""
from .workloads import (  # noqa: F401
    D_K, D_V, D_ROPE, FP8_ROW_BYTES,
    DenseCase, SparseCase, AbsorbCase,
    make_dense_case, make_sparse_case, make_latent_rows, make_absorb_case,
    uniform_seqlens, paged_rows_index,
)
