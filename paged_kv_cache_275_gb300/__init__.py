"""Paged KV-cache hot path for one GB300 GPU: kv_append and paged decode attention.

The computation lives in hand-written sm_103a CUDA kernels behind the C ABI
declared in ``include/pagedkv.h`` (``libpagedkv.so``, built in-tree by
``python -m paged_kv_cache_275_gb300.build``).  This package is a thin ctypes
binding with the same names; PyTorch supplies device memory and streams only.
Importing the package does not load the library; the first call does, and
raises if it is missing.
"""
from ._capi import (BLOCK_SIZE, DEVERR_BLOCK_ID_OUT_OF_RANGE, DEVERR_COPY_OUT_OF_RANGE, DEVERR_POSITION_OUT_OF_TABLE, DEVERR_SMEM_ALIGNMENT, BlockManager, copy_blocks, decode_step, paged_prefill_attention, prefill_workspace_size, prefill_default_splits, DEVERR_CONTEXT_LEN_NEGATIVE,
                    DEVERR_CONTEXT_LEN_TOO_LONG, DEVERR_PIPELINE_TIMEOUT, DEVERR_SLOT_OUT_OF_RANGE, EXPORTS,
                    LIB_PATH, MAX_SEQS, PHASE_ALL, PHASE_MERGE, PHASE_PARTITION, PagedKVError, default_partitions,
                    get_and_clear_device_error, kernel_launch_count, kv_append, load, paged_decode_attention,
                    selftest_wait_timeout, workspace_size)

__all__ = [
    "BLOCK_SIZE", "MAX_SEQS", "EXPORTS", "LIB_PATH", "PagedKVError", "PHASE_ALL", "PHASE_MERGE", "PHASE_PARTITION",
    "DEVERR_SLOT_OUT_OF_RANGE", "DEVERR_BLOCK_ID_OUT_OF_RANGE", "DEVERR_CONTEXT_LEN_NEGATIVE",
    "DEVERR_CONTEXT_LEN_TOO_LONG", "DEVERR_PIPELINE_TIMEOUT",
    "kv_append", "paged_decode_attention", "workspace_size", "default_partitions", "get_and_clear_device_error",
    "kernel_launch_count", "load", "copy_blocks", "BlockManager", "DEVERR_COPY_OUT_OF_RANGE", "decode_step",
    "DEVERR_POSITION_OUT_OF_TABLE", "paged_prefill_attention", "prefill_workspace_size", "prefill_default_splits",
    "DEVERR_SMEM_ALIGNMENT",
    "selftest_wait_timeout",
]
