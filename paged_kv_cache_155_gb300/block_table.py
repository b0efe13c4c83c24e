"""Host-side block-table bookkeeping that produces the inputs of the cache write.

"KV Cache与PagedAttention深度解析" §5.3: the block holding logical position t of
a sequence is its table entry t // block_size, and the token sits at offset
t % block_size of that block; the flat slot the cache write takes is
block * block_size + offset.  This runs on the caller's side of the boundary
(the pages keep block tables in host memory), before the device calls.
"""
from __future__ import annotations

import torch


def slot_mapping(block_tables: torch.Tensor, positions: torch.Tensor, block_size: int) -> torch.Tensor:
    """int64 slots of positions[i] in sequence i; a negative position maps to -1 (skip)."""
    pos = positions.to(torch.int64)
    valid = pos >= 0
    safe = torch.where(valid, pos, torch.zeros_like(pos))
    blk = torch.gather(block_tables.to(torch.int64), 1, (safe // block_size).unsqueeze(1)).squeeze(1)
    slots = blk * block_size + safe % block_size
    return torch.where(valid, slots, torch.full_like(slots, -1))
