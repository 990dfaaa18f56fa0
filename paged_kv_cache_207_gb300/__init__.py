"""Paged KV-cache single-token decode attention for GB300 (sm_103a).

The kernels live in ``libpaged_kv.so`` behind the C ABI of ``include/pa.h``;
this package is the thin Python binding (``_native``) plus the seeded workload
generators (``workloads``).
"""
from ._native import (  # noqa: F401
    BLOCK_SIZE, PARTITION_TOKENS, partition_tokens, BlockManager, PagedKVError, append_kv, copy_block,
    decode_attention, append_decode_attention, decode_attention_shared_prefix,
    append_decode_attention_shared_prefix, decode_workspace,
    decode_workspace_size, lib,
    pool_shape, fp8_pool_shape, append_kv_fp8, decode_attention_fp8, append_decode_attention_fp8,
    copy_block_fp8,
    fp4_pool_shape, append_kv_fp4, decode_attention_fp4, copy_block_fp4,
    prefill_attention,
    DEV_ERR_BAD_BLOCK, DEV_ERR_BAD_POS, DEV_ERR_HINT, DEV_ERR_BAD_CU, DEV_ERR_TIMEOUT,
    DEV_ERR_BAD_PAIR, DEV_ERR_BAD_PREFIX,
)
