"""Python handle on the library's host block manager (pkv_bm_* in pagedkv.h).

The manager is native code; this class only marshals arguments.  It produces
the per-step inputs of the device calls: copy-on-write pairs for
``copy_blocks``, the slot mapping for ``reshape_and_cache``, and the block
tables / context lengths for ``paged_attention_decode``.
"""
from __future__ import annotations

import ctypes
from typing import Dict, List, Sequence, Tuple

import numpy as np

from ._lib import PagedKVError, lib


class OutOfBlocks(PagedKVError):
    pass


def _check(st: int, what: str):
    if st == 6:
        raise OutOfBlocks(what, st)
    if st != 0:
        raise PagedKVError(what, st)


class BlockManager:
    """Free pool + per-sequence block tables with reference-counted sharing."""

    def __init__(self, num_blocks: int, block_size: int, max_blocks_per_seq: int):
        self._lib = lib()
        self._h = self._lib.pkv_bm_create(int(num_blocks), int(block_size), int(max_blocks_per_seq))
        if not self._h:
            raise ValueError("invalid block manager sizes")
        self.num_blocks = int(num_blocks)
        self.block_size = int(block_size)
        self.max_blocks_per_seq = int(max_blocks_per_seq)

    def __del__(self):
        h, self._h = getattr(self, "_h", None), None
        if h:
            self._lib.pkv_bm_destroy(h)

    @property
    def num_free(self) -> int:
        return int(self._lib.pkv_bm_num_free(self._h))

    def refcount(self, block: int) -> int:
        return int(self._lib.pkv_bm_refcount(self._h, int(block)))

    def add_sequence(self, seq_id: int) -> None:
        _check(self._lib.pkv_bm_add_sequence(self._h, int(seq_id)), "pkv_bm_add_sequence")

    def fork(self, parent_id: int, child_id: int) -> None:
        _check(self._lib.pkv_bm_fork(self._h, int(parent_id), int(child_id)), "pkv_bm_fork")

    def share_prefix(self, src_id: int, dst_id: int, num_tokens: int) -> None:
        _check(self._lib.pkv_bm_share_prefix(self._h, int(src_id), int(dst_id), int(num_tokens)),
               "pkv_bm_share_prefix")

    def append_token(self, seq_id: int) -> Tuple[int, Tuple[int, int]]:
        """Returns (slot, (cow_src, cow_dst)); the pair is (-1, -1) when no copy is needed."""
        slot, src, dst = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
        _check(self._lib.pkv_bm_append_token(self._h, int(seq_id), ctypes.byref(slot),
                                             ctypes.byref(src), ctypes.byref(dst)),
               "pkv_bm_append_token")
        return slot.value, (src.value, dst.value)

    def free_sequence(self, seq_id: int) -> None:
        _check(self._lib.pkv_bm_free_sequence(self._h, int(seq_id)), "pkv_bm_free_sequence")

    def seq_len(self, seq_id: int) -> int:
        return int(self._lib.pkv_bm_seq_len(self._h, int(seq_id)))

    def block_table(self, seq_id: int) -> List[int]:
        buf = np.zeros(self.max_blocks_per_seq, dtype=np.int32)
        n = ctypes.c_int()
        _check(self._lib.pkv_bm_block_table(self._h, int(seq_id), buf.ctypes.data_as(ctypes.c_void_p),
                                            self.max_blocks_per_seq, ctypes.byref(n)),
               "pkv_bm_block_table")
        return buf[:n.value].tolist()

    def decode_step(self, seq_ids: Sequence[int]) -> Dict[str, np.ndarray]:
        """Append one token to each sequence; returns the step's device-call inputs
        (host arrays): slot_mapping, block_tables, context_lens, cow_pairs."""
        ids = np.ascontiguousarray(seq_ids, dtype=np.int64)
        n = int(ids.shape[0])
        slots = np.zeros(n, dtype=np.int64)
        tables = np.zeros((n, self.max_blocks_per_seq), dtype=np.int32)
        lens = np.zeros(n, dtype=np.int32)
        cow = np.zeros((max(n, 1), 2), dtype=np.int64)
        ncow = ctypes.c_int64()
        P = lambda a: a.ctypes.data_as(ctypes.c_void_p)
        _check(self._lib.pkv_bm_decode_step(self._h, P(ids), n, P(slots), P(tables), P(lens), P(cow),
                                            ctypes.byref(ncow)), "pkv_bm_decode_step")
        return {"slot_mapping": slots, "block_tables": tables, "context_lens": lens,
                "cow_pairs": cow[:ncow.value].copy()}
