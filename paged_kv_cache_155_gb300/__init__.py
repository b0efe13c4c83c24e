"""GB300-native paged KV-cache decode: a C-ABI CUDA library (libpagedkv) and its
thin PyTorch binding.

  reshape_and_cache       write each new token's K/V rows into its cache slot
  paged_attention_decode  one query token per sequence attends over its paged cache
  copy_blocks             copy-on-write copies of shared blocks
  paged_attention_decode_shared_prefix   the decode for a batch sharing a prefix
  reshape_and_cache_int8 / paged_attention_decode_int8   the same over an INT8
                          cache with per-channel scales
  paged_attention_prefill chunked prefill: each sequence's new tokens attend causally
                          over its paged cache

Each call has a ``prepare_*`` twin that checks and marshals its arguments once
and returns a callable (``PreparedCall``) for loops that reuse their buffers.

The library must be built first (``__graft_entry__.build()``); the calls raise
if it is missing.  There is no CPU implementation in this package.
"""
from .ops import (F16, BF16, INT8, copy_blocks, debug_wait_timeout,  # noqa: F401
                  decode_int8_workspace_bytes, decode_plan, decode_workspace_bytes,
                  get_device_error, launch_count, paged_attention_decode,
                  paged_attention_decode_int8, paged_attention_decode_shared_prefix,
                  paged_attention_prefill, prefill_workspace_bytes,
                  reshape_and_cache, reshape_and_cache_int8, shared_prefix_workspace_bytes,
                  split_pool, PreparedCall, prepare_paged_attention_decode,
                  prepare_paged_attention_decode_int8,
                  prepare_paged_attention_decode_shared_prefix, prepare_reshape_and_cache,
                  prepare_reshape_and_cache_int8)
from .block_table import slot_mapping  # noqa: F401
from ._lib import PagedKVError  # noqa: F401

__all__ = ["reshape_and_cache", "paged_attention_decode", "paged_attention_decode_shared_prefix",
           "shared_prefix_workspace_bytes", "copy_blocks", "split_pool",
           "paged_attention_prefill", "prefill_workspace_bytes", "reshape_and_cache_int8", "paged_attention_decode_int8", "decode_int8_workspace_bytes",
           "decode_workspace_bytes", "decode_plan", "get_device_error", "launch_count",
           "debug_wait_timeout", "slot_mapping", "PagedKVError", "PreparedCall",
           "prepare_paged_attention_decode", "prepare_paged_attention_decode_int8",
           "prepare_paged_attention_decode_shared_prefix", "prepare_reshape_and_cache",
           "prepare_reshape_and_cache_int8"]
