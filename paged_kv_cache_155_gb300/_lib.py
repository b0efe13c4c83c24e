"""ctypes loader for libpagedkv.so: symbol signatures only, no logic.

The library is the product; nothing here computes.  If the library has not
been built, every op raises instead of falling back to anything else.
"""
from __future__ import annotations

import ctypes
import os
import threading

from ._build import LIB_PATH

_lock = threading.Lock()
_lib = None

P = ctypes.c_void_p
I64 = ctypes.c_int64
I32 = ctypes.c_int
U64 = ctypes.c_uint64
SZ = ctypes.c_size_t

# name -> (restype, argtypes); mirrors include/pagedkv.h
SIGNATURES = {
    "pkv_reshape_and_cache": (I32, [P, P, P, I64, P, P, I64, I64, I32, I32, I32, I32, P]),
    "pkv_slot_mapping": (I32, [P, I64, I32, P, P, I64, I32, I64, P, P]),
    "pkv_slot_mapping_host": (I32, [P, I64, I32, P, P, I64, I32, I64, P]),
    "pkv_decode_workspace_bytes": (SZ, [I32, I32, I32, I32, I32, I32, I32]),
    "pkv_paged_attention_decode": (I32, [P, P, P, I64, I64, P, I32, P, I32, I32, I32, I32,
                                         I32, I32, ctypes.c_float, P, P, SZ, I32, I32, P]),
    "pkv_copy_blocks": (I32, [P, P, I64, I64, I32, I32, I32, P, I64, I32, P]),
    "pkv_get_device_error": (I32, [P, ctypes.POINTER(ctypes.c_uint32)]),
    "pkv_status_string": (ctypes.c_char_p, [I32]),
    "pkv_launch_count": (U64, []),
    "pkv_decode_plan": (I32, [I32, I32, I32, I32, I32, I32, I32, I32,
                              ctypes.POINTER(I32), ctypes.POINTER(I32), ctypes.POINTER(I32),
                              ctypes.POINTER(I32)]),
    "pkv_decode_int8_plan": (I32, [I32, I32, I32, I32, I32, I32, I32, I32,
                                   ctypes.POINTER(I32), ctypes.POINTER(I32), ctypes.POINTER(I32),
                                   ctypes.POINTER(I32)]),
    "pkv_debug_wait_timeout": (I32, [U64, P]),
    "pkv_paged_attention_decode_static_scratch": (I32, [P, P, P, I64, I64, P, I32, P, I32, I32,
                                                        I32, I32, I32, I32, ctypes.c_float, P,
                                                        I32, I32, P]),
    "pkv_shared_prefix_workspace_bytes": (SZ, [I32, I32, I32, I32, I32, I32, I32, I32]),
    "pkv_paged_attention_decode_shared_prefix": (I32, [P, P, P, I64, I64, P, I32, P, I32, P, I32,
                                                       I32, I32, I32, I32, I32, ctypes.c_float,
                                                       P, P, SZ, I32, I32, P]),
    "pkv_reshape_and_cache_int8": (I32, [P, P, P, I64, P, P, I64, I64, I32, I32, I32, P, P,
                                         I32, P]),
    "pkv_decode_int8_workspace_bytes": (SZ, [I32, I32, I32, I32, I32, I32, I32]),
    "pkv_paged_attention_decode_int8": (I32, [P, P, P, P, P, I64, I64, P, I32, P, I32, I32, I32,
                                              I32, I32, I32, ctypes.c_float, P, P, SZ, I32, I32,
                                              P]),
    "pkv_prefill_workspace_bytes": (SZ, [I32, I32, I32, I32, I32, I32, I32, I32, I32]),
    "pkv_paged_attention_prefill": (I32, [P, P, P, I64, I64, P, I32, P, P, I32, I32, I32, I32,
                                          I32, I32, I32, I32, ctypes.c_float, P, P, SZ, I32, I32,
                                          P]),
    "pkv_bm_create": (P, [I64, I32, I32]),
    "pkv_bm_destroy": (None, [P]),
    "pkv_bm_num_free": (I64, [P]),
    "pkv_bm_refcount": (ctypes.c_int32, [P, I64]),
    "pkv_bm_add_sequence": (I32, [P, I64]),
    "pkv_bm_fork": (I32, [P, I64, I64]),
    "pkv_bm_share_prefix": (I32, [P, I64, I64, I64]),
    "pkv_bm_append_token": (I32, [P, I64, P, P, P]),
    "pkv_bm_free_sequence": (I32, [P, I64]),
    "pkv_bm_seq_len": (I64, [P, I64]),
    "pkv_bm_block_table": (I32, [P, I64, P, I32, ctypes.POINTER(I32)]),
    "pkv_bm_decode_step": (I32, [P, P, I32, P, P, P, P, P]),
}

STATUS = {0: "PKV_OK", 1: "PKV_ERR_INVALID_ARG", 2: "PKV_ERR_UNSUPPORTED", 3: "PKV_ERR_CUDA",
          4: "PKV_ERR_DEVICE", 5: "PKV_ERR_SCRATCH_LIMIT", 6: "PKV_ERR_OUT_OF_BLOCKS"}
DEVERR = {0x1: "slot", 0x2: "block_table", 0x4: "context_len", 0x8: "copy_pair", 0x10: "timeout"}


class PagedKVError(RuntimeError):
    def __init__(self, what: str, status: int):
        text = STATUS.get(status, str(status))
        try:
            text += f" ({lib().pkv_status_string(status).decode()})"
        except Exception:  # pragma: no cover - message decoration only
            pass
        super().__init__(f"{what} failed: {text}")
        self.status = status


def lib():
    """The loaded libpagedkv (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"libpagedkv.so is not built ({LIB_PATH}); run "
                "`python -c 'import __graft_entry__ as g; g.build()'` first. "
                "There is no fallback implementation.")
        handle = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
        return handle
