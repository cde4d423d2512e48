"""GB300 (sm_103a) paged KV-cache decode path: slot-mapped KV write,
zeroing of fresh blocks, PagedAttention decode with in-kernel block-table
gather, GQA, split-KV with a log-sum-exp reduce and fp8 E4M3 KV, chunked
prefill attention and shared-prefix (cascade) decode on the tcgen05 tensor
cores, block copy / swap and GPU step-input preparation.

The kernels live in ``libpagedkv.so`` (C ABI: include/pagedkv.h); this
package binds them for PyTorch tensors.  Build with
``python -m paged_kv_cache_48_gb300.build``.
"""
from .ops import (PagedKVCache, PagedKVError, paged_attention_decode,
                  paged_attention_decode_step,
                  paged_attention_cascade_workspace_bytes,
                  paged_attention_decode_cascade, paged_attention_prefill,
                  paged_attention_partition_tokens,
                  paged_attention_workspace_bytes, paged_kv_copy_blocks,
                  paged_kv_swap_in, paged_kv_swap_out, paged_kv_write,
                  paged_kv_zero_and_write, paged_kv_zero_blocks,
                  paged_prepare_inputs, pkv_check,
                  raise_on_device_error)

__all__ = [
    "PagedKVCache", "PagedKVError", "paged_attention_decode",
    "paged_attention_decode_step",
    "paged_attention_cascade_workspace_bytes", "paged_attention_decode_cascade",
    "paged_attention_prefill",
    "paged_attention_partition_tokens", "paged_attention_workspace_bytes",
    "paged_kv_copy_blocks", "paged_kv_swap_in", "paged_kv_swap_out",
    "paged_kv_write", "paged_kv_zero_and_write", "paged_kv_zero_blocks",
    "paged_prepare_inputs",
    "pkv_check",
    "raise_on_device_error",
]
