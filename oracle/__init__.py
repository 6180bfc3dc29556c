"""Plain, slow, fp64 CPU oracle for decode attention over a paged KV cache.

TEST INFRASTRUCTURE. Only the tests, the package smoke check and the
benchmark's CPU-baseline / reference leg import this package. The CUDA
product path never imports, calls or links it, and it shares no code with
the CUDA library: no kernels, headers, helpers or constant tables.

Every function works on numpy arrays. Cache contents are passed as raw
storage (bf16 as uint16 bit patterns, fp8-e4m3 as uint8 codes, MXFP4 as
rows of packed E2M1 codes and E4M3 group scales) and decoded
here, exactly, to float64 before any arithmetic.

Pinned by tests/test_oracle_pins.py (closed forms, page figures, brute force,
library special cases). Parity status per function is listed in the module
docstrings of ``attention`` and ``numerics``.
"""
from .numerics import (bf16_bits_to_f64, e4m3_value_table, e4m3_codes_to_f64,
                       e4m3_encode_f32, e2m1_value_table, e2m1_codes_to_f64,
                       e2m1_encode_f32, mxfp4_row_bytes, mxfp4_encode_rows,
                       mxfp4_rows_to_f64)
from .attention import (attend, attend_scores, decode_rows, gather_positions, gather_rows, kv_append,
                        gqa_decode, mla_decode, indexer_scores, topk_select,
                        indexer_topk, sparse_decode, lse_merge, split_decode,
                        bytes_per_token, cache_bytes, paged_waste_slots,
                        sparse_schedule, POOL_BLOCK, POOL_CAP, indexer_pool,
                        pool_positions, indexer_topk_in_pool)

from .allocator import CowPool, blocks_for_lengths

__all__ = [
    "CowPool", "blocks_for_lengths",
    "bf16_bits_to_f64", "e4m3_value_table", "e4m3_codes_to_f64",
    "e4m3_encode_f32", "e2m1_value_table", "e2m1_codes_to_f64",
    "e2m1_encode_f32", "mxfp4_row_bytes", "mxfp4_encode_rows",
    "mxfp4_rows_to_f64",
    "attend", "attend_scores", "decode_rows", "gather_positions", "gather_rows", "kv_append", "gqa_decode",
    "mla_decode", "indexer_scores", "topk_select", "indexer_topk",
    "sparse_decode", "lse_merge", "split_decode", "bytes_per_token",
    "cache_bytes", "paged_waste_slots", "sparse_schedule", "POOL_BLOCK",
    "POOL_CAP", "indexer_pool", "pool_positions", "indexer_topk_in_pool",
]
