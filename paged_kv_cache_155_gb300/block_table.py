"""Slot mapping of new tokens: the input of the cache write.

"KV Cache与PagedAttention深度解析" §5.3: the block holding logical position t of
a sequence is its table entry t // block_size, the token sits at offset
t % block_size of that block, and the flat slot the cache write takes is
block * block_size + offset.  The rule runs in the library
(pkv_slot_mapping on the device, pkv_slot_mapping_host on host arrays); this
module only marshals tensors to it.
"""
from __future__ import annotations

import ctypes
from typing import Optional

import torch

from ._lib import PagedKVError, lib

# default pool size for the range check of table entries when the caller does not give one
_UNBOUNDED = 1 << 62


def slot_mapping(block_tables: torch.Tensor, positions: torch.Tensor, block_size: int,
                 token_rows: Optional[torch.Tensor] = None,
                 num_blocks: Optional[int] = None) -> torch.Tensor:
    """int64 slot of each token: token i at logical position positions[i] of the
    sequence whose table is block_tables[token_rows[i]] (or row i).  A negative
    position maps to -1 (skipped by the cache write).  Tensors on a CUDA device
    run the library's kernel on the current stream; CPU tensors run its host
    routine.  Returns a tensor on the inputs' device."""
    if block_tables.dtype != torch.int32 or block_tables.dim() != 2:
        raise ValueError("block_tables must be int32 [rows, max_blocks_per_seq]")
    dev = block_tables.device
    bt = block_tables.contiguous()
    pos = positions.to(device=dev, dtype=torch.int64).contiguous()
    rows = None if token_rows is None else token_rows.to(device=dev, dtype=torch.int64).contiguous()
    n = int(pos.numel())
    if rows is not None and rows.numel() != n:
        raise ValueError("token_rows must have one entry per position")
    out = torch.empty(n, dtype=torch.int64, device=dev)
    nb = _UNBOUNDED if num_blocks is None else int(num_blocks)
    args = (bt.data_ptr(), int(bt.shape[0]), int(bt.shape[1]),
            None if rows is None else rows.data_ptr(), pos.data_ptr(), n, int(block_size), nb,
            out.data_ptr())
    if dev.type == "cuda":
        st = lib().pkv_slot_mapping(*args, ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream))
        what = "pkv_slot_mapping"
    else:
        st = lib().pkv_slot_mapping_host(*args)
        what = "pkv_slot_mapping_host"
    if st != 0:
        raise PagedKVError(what, st)
    return out
