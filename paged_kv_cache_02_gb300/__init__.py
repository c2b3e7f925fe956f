"""Paged multi-token attention over a block-table KV cache, for GB300 (sm_103a).

The computation lives in ``libpa.so`` (hand-written CUDA kernels behind the C
ABI of ``include/pa.h``); this package is its thin Python binding. See
``_binding`` for the functions, which carry the C entry points' names.
"""
from ._binding import (DEVERR, LIB_PATH, STATIC_WORKSPACE_BYTES, BlockManager, OutOfBlocks,
                       PagedAttentionError, Plan, library, pa_attention, pa_attention_planned, pa_attention_static,
                       pa_attention_write,
                       pa_copy_blocks, pa_get_device_error, pa_plan_create, pa_plan_upload,
                       pa_slot_mapping, pa_swap_blocks, pa_write_kv, version)

__all__ = ["DEVERR", "LIB_PATH", "STATIC_WORKSPACE_BYTES", "BlockManager", "OutOfBlocks",
           "PagedAttentionError", "Plan",
           "library", "pa_attention", "pa_attention_planned", "pa_attention_static",
           "pa_attention_write",
           "pa_copy_blocks", "pa_get_device_error", "pa_plan_create", "pa_plan_upload",
           "pa_slot_mapping", "pa_swap_blocks", "pa_write_kv", "version"]
