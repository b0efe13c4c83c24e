"""Thin PyTorch binding of libpagedkv: same names as the C ABI, argument
marshalling only.  Tensors supply device pointers and shapes; the current
CUDA stream of the tensors' device is passed as the stream.  Every step runs
in the library's kernels; if the library is missing the calls raise.

``prepare_*`` variants check and marshal a call's arguments once and return a
``PreparedCall``; calling it enqueues the same library call again on the
current stream (a serving loop that reuses its buffers pays the argument
checks once, not per step).

Cache tensors: ``k_cache`` / ``v_cache`` are [num_blocks, num_kv_heads,
block_size, head_dim] views sharing one block stride, normally the two
halves ``kv[:, 0]`` / ``kv[:, 1]`` of a pool ``kv`` of shape
[num_blocks, 2, num_kv_heads, block_size, head_dim] ("KV Cache与PagedAttention深度解析"
§4.3 and §5.1).
"""
from __future__ import annotations

import ctypes
import math
from typing import Optional, Tuple

import torch

from ._lib import DEVERR, PagedKVError, lib

F16, BF16, INT8 = 0, 1, 2
_workspaces = {}


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float16:
        return F16
    if t.dtype == torch.bfloat16:
        return BF16
    raise TypeError(f"unsupported dtype {t.dtype}: fp16 or bf16 expected")


_raw_stream_getter = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _raw_stream(device_index: int) -> int:
    """cudaStream_t of the device's current stream, as an integer."""
    if _raw_stream_getter is not None:
        return _raw_stream_getter(device_index)
    return torch.cuda.current_stream(device_index).cuda_stream


def _stream(t: torch.Tensor):
    return ctypes.c_void_p(_raw_stream(t.device.index if t.device.index is not None
                                       else torch.cuda.current_device()))


class PreparedCall:
    """One library call whose arguments were checked and marshalled once.

    Calling it enqueues the same call on the current stream of its device and
    returns the call's output tensor (or None).  It holds the tensors it was
    prepared with; they must keep their storage, while their contents may change
    between calls (new queries and rows, new context lengths within the bound
    given at preparation)."""
    __slots__ = ("_fn", "_args", "_dev", "_what", "_tensors", "_result")

    def __init__(self, what: str, args: tuple, device: torch.device, tensors: tuple, result=None):
        self._fn = getattr(lib(), what)
        self._args = args
        self._dev = device.index if device.index is not None else torch.cuda.current_device()
        self._what = what
        self._tensors = tensors
        self._result = result

    def __call__(self):
        st = self._fn(*self._args, _raw_stream(self._dev))
        if st != 0:
            raise PagedKVError(self._what, st)
        return self._result


def _check(status: int, what: str):
    if status != 0:
        raise PagedKVError(what, status)


def _cache_dtype_code(t: torch.Tensor) -> int:
    return INT8 if t.dtype == torch.int8 else _dtype_code(t)


def _cache_geometry(k_cache: torch.Tensor, v_cache: torch.Tensor):
    if k_cache.dim() != 4 or k_cache.shape != v_cache.shape:
        raise ValueError("k_cache/v_cache must be [num_blocks, num_kv_heads, block_size, head_dim]")
    if k_cache.stride() != v_cache.stride() or k_cache.dtype != v_cache.dtype:
        raise ValueError("k_cache and v_cache must share dtype and strides")
    nb, hkv, bs, d = k_cache.shape
    if k_cache.stride()[1:] != (bs * d, d, 1):
        raise ValueError("each block of k_cache/v_cache must be a dense [num_kv_heads, block_size, head_dim]")
    return nb, hkv, bs, d, k_cache.stride(0)


def split_pool(kv: torch.Tensor) -> Tuple[torch.Tensor, torch.Tensor]:
    """K and V halves of a pool [num_blocks, 2, num_kv_heads, block_size, head_dim]."""
    if kv.dim() != 5 or kv.shape[1] != 2 or not kv.is_contiguous():
        raise ValueError("pool must be a contiguous [num_blocks, 2, num_kv_heads, block_size, head_dim]")
    return kv[:, 0], kv[:, 1]


def reshape_and_cache(k_new: torch.Tensor, v_new: torch.Tensor, slot_mapping: torch.Tensor,
                      k_cache: torch.Tensor, v_cache: torch.Tensor) -> None:
    """Write new K/V rows [T, Hkv, d] into their slots (bit-exact); slot < 0 skips."""
    prepare_reshape_and_cache(k_new, v_new, slot_mapping, k_cache, v_cache)()


def prepare_reshape_and_cache(k_new: torch.Tensor, v_new: torch.Tensor, slot_mapping: torch.Tensor,
                              k_cache: torch.Tensor, v_cache: torch.Tensor) -> PreparedCall:
    """reshape_and_cache, checked and marshalled once (see PreparedCall)."""
    nb, hkv, bs, d, stride = _cache_geometry(k_cache, v_cache)
    t = int(k_new.shape[0])
    if k_new.shape != (t, hkv, d) or v_new.shape != k_new.shape:
        raise ValueError(f"k_new/v_new must be [T, {hkv}, {d}]")
    if not (k_new.is_contiguous() and v_new.is_contiguous() and slot_mapping.is_contiguous()):
        raise ValueError("k_new, v_new and slot_mapping must be contiguous")
    if slot_mapping.dtype != torch.int64 or slot_mapping.numel() != t:
        raise ValueError("slot_mapping must be int64 [T]")
    if k_new.dtype != k_cache.dtype or v_new.dtype != k_cache.dtype:
        raise ValueError("k_new/v_new dtype must match the cache")
    args = (k_new.data_ptr(), v_new.data_ptr(), slot_mapping.data_ptr(), t, k_cache.data_ptr(),
            v_cache.data_ptr(), nb, stride, hkv, d, bs, _dtype_code(k_cache))
    return PreparedCall("pkv_reshape_and_cache", args, k_cache.device,
                        (k_new, v_new, slot_mapping, k_cache, v_cache))


def decode_workspace_bytes(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                           max_context_len, partition_size=0) -> int:
    n = lib().pkv_decode_workspace_bytes(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                         block_size, max_context_len, partition_size)
    if n == ctypes.c_size_t(-1).value:
        raise PagedKVError("pkv_decode_workspace_bytes", 1)
    return int(n)


def _workspace(device: torch.device, nbytes: int) -> Optional[torch.Tensor]:
    if nbytes == 0:
        return None
    key = (device.type, device.index)
    buf = _workspaces.get(key)
    if buf is None or buf.numel() < nbytes:
        buf = torch.empty(nbytes, dtype=torch.uint8, device=device)
        _workspaces[key] = buf
    return buf


def paged_attention_decode(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                           block_tables: torch.Tensor, context_lens: torch.Tensor,
                           scale: Optional[float] = None, out: Optional[torch.Tensor] = None, *,
                           max_context_len: Optional[int] = None, partition_size: int = 0,
                           workspace: Optional[torch.Tensor] = None) -> torch.Tensor:
    """out[i, hq] = softmax(scale * q[i, hq] . K_i^T) V_i over the paged cache.

    q, out: [num_seqs, num_q_heads, head_dim]; block_tables int32 [num_seqs, max_blocks];
    context_lens int32 [num_seqs].  ``max_context_len`` (a host int) bounds
    context_lens; if omitted it is read back from the device (a synchronisation).
    """
    return prepare_paged_attention_decode(q, k_cache, v_cache, block_tables, context_lens, scale,
                                          out, max_context_len=max_context_len,
                                          partition_size=partition_size, workspace=workspace)()


def prepare_paged_attention_decode(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                                   block_tables: torch.Tensor, context_lens: torch.Tensor,
                                   scale: Optional[float] = None, out: Optional[torch.Tensor] = None,
                                   *, max_context_len: Optional[int] = None, partition_size: int = 0,
                                   workspace: Optional[torch.Tensor] = None) -> PreparedCall:
    """paged_attention_decode, checked and marshalled once (see PreparedCall); the
    call returns ``out``.  Later context lengths must stay within max_context_len."""
    nb, hkv, bs, d, stride = _cache_geometry(k_cache, v_cache)
    if q.dim() != 3 or q.shape[2] != d or not q.is_contiguous():
        raise ValueError(f"q must be a contiguous [num_seqs, num_q_heads, {d}]")
    b, hq = int(q.shape[0]), int(q.shape[1])
    if q.dtype != k_cache.dtype:
        raise ValueError("q dtype must match the cache")
    if block_tables.dtype != torch.int32 or block_tables.dim() != 2 or block_tables.shape[0] != b \
            or not block_tables.is_contiguous():
        raise ValueError("block_tables must be a contiguous int32 [num_seqs, max_blocks_per_seq]")
    if context_lens.dtype != torch.int32 or context_lens.numel() != b or not context_lens.is_contiguous():
        raise ValueError("context_lens must be a contiguous int32 [num_seqs]")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if max_context_len is None:
        max_context_len = int(context_lens.max().item()) if b else 0
    if out is None:
        out = torch.empty_like(q)
    elif out.shape != q.shape or out.dtype != q.dtype or not out.is_contiguous():
        raise ValueError("out must match q")
    need = decode_workspace_bytes(b, hq, hkv, d, bs, max_context_len, partition_size)
    if workspace is None:
        workspace = _workspace(q.device, need)
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    args = (q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), nb, stride, block_tables.data_ptr(),
            int(block_tables.shape[1]), context_lens.data_ptr(), int(max_context_len), b, hq, hkv, d,
            bs, float(scale), out.data_ptr(), ws_ptr, ws_bytes, int(partition_size), _dtype_code(q))
    return PreparedCall("pkv_paged_attention_decode", args, q.device,
                        (q, k_cache, v_cache, block_tables, context_lens, out, workspace), out)


def shared_prefix_workspace_bytes(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                                  prefix_len, max_context_len, partition_size=0) -> int:
    n = lib().pkv_shared_prefix_workspace_bytes(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                                block_size, prefix_len, max_context_len,
                                                partition_size)
    if n == ctypes.c_size_t(-1).value:
        raise PagedKVError("pkv_shared_prefix_workspace_bytes", 1)
    return int(n)


def paged_attention_decode_shared_prefix(q: torch.Tensor, k_cache: torch.Tensor,
                                         v_cache: torch.Tensor, prefix_block_table: torch.Tensor,
                                         prefix_len: int, block_tables: torch.Tensor,
                                         context_lens: torch.Tensor, scale: Optional[float] = None,
                                         out: Optional[torch.Tensor] = None, *,
                                         max_context_len: Optional[int] = None,
                                         partition_size: int = 0,
                                         workspace: Optional[torch.Tensor] = None) -> torch.Tensor:
    """paged_attention_decode for a batch that shares its first prefix_len tokens
    (prefix_block_table holds their blocks): the prefix is attended by all query
    rows together as dense tiles, beside each sequence's suffix, then a merge."""
    return prepare_paged_attention_decode_shared_prefix(
        q, k_cache, v_cache, prefix_block_table, prefix_len, block_tables, context_lens, scale, out,
        max_context_len=max_context_len, partition_size=partition_size, workspace=workspace)()


def prepare_paged_attention_decode_shared_prefix(
        q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
        prefix_block_table: torch.Tensor, prefix_len: int, block_tables: torch.Tensor,
        context_lens: torch.Tensor, scale: Optional[float] = None,
        out: Optional[torch.Tensor] = None, *, max_context_len: Optional[int] = None,
        partition_size: int = 0, workspace: Optional[torch.Tensor] = None) -> PreparedCall:
    """paged_attention_decode_shared_prefix, checked and marshalled once (see
    PreparedCall); the call returns ``out``."""
    nb, hkv, bs, d, stride = _cache_geometry(k_cache, v_cache)
    if q.dim() != 3 or q.shape[2] != d or not q.is_contiguous() or q.dtype != k_cache.dtype:
        raise ValueError(f"q must be a contiguous [num_seqs, num_q_heads, {d}] of the cache dtype")
    b, hq = int(q.shape[0]), int(q.shape[1])
    if prefix_block_table.dtype != torch.int32 or not prefix_block_table.is_contiguous():
        raise ValueError("prefix_block_table must be a contiguous int32 tensor")
    if block_tables.dtype != torch.int32 or block_tables.dim() != 2 or not block_tables.is_contiguous():
        raise ValueError("block_tables must be a contiguous int32 [num_seqs, max_blocks_per_seq]")
    if context_lens.dtype != torch.int32 or context_lens.numel() != b:
        raise ValueError("context_lens must be int32 [num_seqs]")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if max_context_len is None:
        max_context_len = int(context_lens.max().item())
    if out is None:
        out = torch.empty_like(q)
    need = shared_prefix_workspace_bytes(b, hq, hkv, d, bs, prefix_len, max_context_len,
                                         partition_size)
    if workspace is None:
        workspace = _workspace(q.device, need)
    args = (q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), nb, stride,
            prefix_block_table.data_ptr(), int(prefix_len), block_tables.data_ptr(),
            int(block_tables.shape[1]), context_lens.data_ptr(), int(max_context_len), b, hq, hkv, d,
            bs, float(scale), out.data_ptr(), workspace.data_ptr(),
            workspace.numel() * workspace.element_size(), int(partition_size), _dtype_code(q))
    return PreparedCall("pkv_paged_attention_decode_shared_prefix", args, q.device,
                        (q, k_cache, v_cache, prefix_block_table, block_tables, context_lens, out,
                         workspace), out)


def prefill_workspace_bytes(num_rows, num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                            max_query_len, max_context_len, kv_splits=0) -> int:
    n = lib().pkv_prefill_workspace_bytes(num_rows, num_seqs, num_q_heads, num_kv_heads, head_dim,
                                          block_size, max_query_len, max_context_len, kv_splits)
    if n == ctypes.c_size_t(-1).value:
        raise PagedKVError("pkv_prefill_workspace_bytes", 1)
    return int(n)


def paged_attention_prefill(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                            block_tables: torch.Tensor, query_start: torch.Tensor,
                            context_lens: torch.Tensor, scale: Optional[float] = None,
                            out: Optional[torch.Tensor] = None, *, max_query_len: int,
                            max_context_len: int, kv_splits: int = 0,
                            workspace: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Chunked prefill attention: q [num_rows, Hq, d] holds every sequence's chunk
    (sequence i owns rows query_start[i]:query_start[i+1], whose K/V are already in
    the cache as its last tokens); row j of chunk i attends causally to tokens
    0 .. context_lens[i] - chunk_i + j.  max_query_len / max_context_len are host bounds."""
    nb, hkv, bs, d, stride = _cache_geometry(k_cache, v_cache)
    if q.dim() != 3 or q.shape[2] != d or not q.is_contiguous() or q.dtype != k_cache.dtype:
        raise ValueError(f"q must be a contiguous [num_rows, num_q_heads, {d}] of the cache dtype")
    rows, hq = int(q.shape[0]), int(q.shape[1])
    b = int(context_lens.numel())
    if block_tables.dtype != torch.int32 or block_tables.dim() != 2 or block_tables.shape[0] != b \
            or not block_tables.is_contiguous():
        raise ValueError("block_tables must be a contiguous int32 [num_seqs, max_blocks_per_seq]")
    if query_start.dtype != torch.int32 or query_start.numel() != b + 1 \
            or not query_start.is_contiguous():
        raise ValueError("query_start must be a contiguous int32 [num_seqs + 1]")
    if context_lens.dtype != torch.int32 or not context_lens.is_contiguous():
        raise ValueError("context_lens must be a contiguous int32 [num_seqs]")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    elif out.shape != q.shape or out.dtype != q.dtype or not out.is_contiguous():
        raise ValueError("out must match q")
    need = prefill_workspace_bytes(rows, b, hq, hkv, d, bs, max_query_len, max_context_len,
                                   kv_splits)
    if workspace is None:
        workspace = _workspace(q.device, need)
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = lib().pkv_paged_attention_prefill(
        q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), nb, stride, block_tables.data_ptr(),
        int(block_tables.shape[1]), query_start.data_ptr(), context_lens.data_ptr(), rows,
        int(max_query_len), int(max_context_len), b, hq, hkv, d, bs, float(scale), out.data_ptr(),
        ws_ptr, ws_bytes, int(kv_splits), _dtype_code(q), _stream(q))
    _check(st, "pkv_paged_attention_prefill")
    return out


def copy_blocks(k_cache: torch.Tensor, v_cache: torch.Tensor, src_dst_pairs: torch.Tensor) -> None:
    """Copy K and V of block src over block dst for each row (src, dst) of an int64 [n, 2]."""
    nb, hkv, bs, d, stride = _cache_geometry(k_cache, v_cache)
    if src_dst_pairs.dtype != torch.int64 or src_dst_pairs.dim() != 2 or src_dst_pairs.shape[1] != 2 \
            or not src_dst_pairs.is_contiguous():
        raise ValueError("src_dst_pairs must be a contiguous int64 [n, 2]")
    if src_dst_pairs.device.type == "cpu":
        raise ValueError("src_dst_pairs must be on the device")
    st = lib().pkv_copy_blocks(k_cache.data_ptr(), v_cache.data_ptr(), nb, stride, hkv, d, bs,
                               src_dst_pairs.data_ptr(), int(src_dst_pairs.shape[0]),
                               _cache_dtype_code(k_cache), _stream(k_cache))
    _check(st, "pkv_copy_blocks")


# ---------------------------------------------------------------------------
# INT8 cache with per-channel scales ("KV Cache从原理到实战" §5.2)
# ---------------------------------------------------------------------------

def _check_int8_cache(k_cache, v_cache, k_scale, v_scale):
    nb, hkv, bs, d, stride = _cache_geometry(k_cache, v_cache)
    if k_cache.dtype != torch.int8:
        raise ValueError("k_cache/v_cache must be int8")
    for name, sc in (("k_scale", k_scale), ("v_scale", v_scale)):
        if sc.dtype != torch.float32 or sc.shape != (hkv, d) or not sc.is_contiguous() \
                or sc.device != k_cache.device:
            raise ValueError(f"{name} must be a contiguous float32 [{hkv}, {d}] on the cache's device")
    return nb, hkv, bs, d, stride


def reshape_and_cache_int8(k_new: torch.Tensor, v_new: torch.Tensor, slot_mapping: torch.Tensor,
                           k_cache: torch.Tensor, v_cache: torch.Tensor, k_scale: torch.Tensor,
                           v_scale: torch.Tensor) -> None:
    """Quantise new K/V rows [T, Hkv, d] (fp16/bf16) with per-channel scales [Hkv, d]
    and write the codes into their slots of an INT8 cache; slot < 0 skips."""
    prepare_reshape_and_cache_int8(k_new, v_new, slot_mapping, k_cache, v_cache, k_scale, v_scale)()


def prepare_reshape_and_cache_int8(k_new: torch.Tensor, v_new: torch.Tensor,
                                   slot_mapping: torch.Tensor, k_cache: torch.Tensor,
                                   v_cache: torch.Tensor, k_scale: torch.Tensor,
                                   v_scale: torch.Tensor) -> PreparedCall:
    """reshape_and_cache_int8, checked and marshalled once (see PreparedCall)."""
    nb, hkv, bs, d, stride = _check_int8_cache(k_cache, v_cache, k_scale, v_scale)
    t = int(k_new.shape[0])
    if k_new.shape != (t, hkv, d) or v_new.shape != k_new.shape or v_new.dtype != k_new.dtype:
        raise ValueError(f"k_new/v_new must be [T, {hkv}, {d}] of one dtype")
    if not (k_new.is_contiguous() and v_new.is_contiguous() and slot_mapping.is_contiguous()):
        raise ValueError("k_new, v_new and slot_mapping must be contiguous")
    if slot_mapping.dtype != torch.int64 or slot_mapping.numel() != t:
        raise ValueError("slot_mapping must be int64 [T]")
    args = (k_new.data_ptr(), v_new.data_ptr(), slot_mapping.data_ptr(), t, k_cache.data_ptr(),
            v_cache.data_ptr(), nb, stride, hkv, d, bs, k_scale.data_ptr(), v_scale.data_ptr(),
            _dtype_code(k_new))
    return PreparedCall("pkv_reshape_and_cache_int8", args, k_cache.device,
                        (k_new, v_new, slot_mapping, k_cache, v_cache, k_scale, v_scale))


def decode_int8_workspace_bytes(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                                max_context_len, partition_size=0) -> int:
    n = lib().pkv_decode_int8_workspace_bytes(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                              block_size, max_context_len, partition_size)
    if n == ctypes.c_size_t(-1).value:
        raise PagedKVError("pkv_decode_int8_workspace_bytes", 1)
    return int(n)


def paged_attention_decode_int8(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                                k_scale: torch.Tensor, v_scale: torch.Tensor,
                                block_tables: torch.Tensor, context_lens: torch.Tensor,
                                scale: Optional[float] = None, out: Optional[torch.Tensor] = None,
                                *, max_context_len: Optional[int] = None, partition_size: int = 0,
                                workspace: Optional[torch.Tensor] = None) -> torch.Tensor:
    """paged_attention_decode over an INT8 cache whose values are code * scale[h][channel];
    q and out fp16 or bf16."""
    return prepare_paged_attention_decode_int8(
        q, k_cache, v_cache, k_scale, v_scale, block_tables, context_lens, scale, out,
        max_context_len=max_context_len, partition_size=partition_size, workspace=workspace)()


def prepare_paged_attention_decode_int8(q: torch.Tensor, k_cache: torch.Tensor,
                                        v_cache: torch.Tensor, k_scale: torch.Tensor,
                                        v_scale: torch.Tensor, block_tables: torch.Tensor,
                                        context_lens: torch.Tensor, scale: Optional[float] = None,
                                        out: Optional[torch.Tensor] = None, *,
                                        max_context_len: Optional[int] = None,
                                        partition_size: int = 0,
                                        workspace: Optional[torch.Tensor] = None) -> PreparedCall:
    """paged_attention_decode_int8, checked and marshalled once (see PreparedCall); the
    call returns ``out``."""
    nb, hkv, bs, d, stride = _check_int8_cache(k_cache, v_cache, k_scale, v_scale)
    if q.dim() != 3 or q.shape[2] != d or not q.is_contiguous():
        raise ValueError(f"q must be a contiguous [num_seqs, num_q_heads, {d}]")
    b, hq = int(q.shape[0]), int(q.shape[1])
    if block_tables.dtype != torch.int32 or block_tables.dim() != 2 or block_tables.shape[0] != b \
            or not block_tables.is_contiguous():
        raise ValueError("block_tables must be a contiguous int32 [num_seqs, max_blocks_per_seq]")
    if context_lens.dtype != torch.int32 or context_lens.numel() != b or not context_lens.is_contiguous():
        raise ValueError("context_lens must be a contiguous int32 [num_seqs]")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if max_context_len is None:
        max_context_len = int(context_lens.max().item()) if b else 0
    if out is None:
        out = torch.empty_like(q)
    elif out.shape != q.shape or out.dtype != q.dtype or not out.is_contiguous():
        raise ValueError("out must match q")
    need = decode_int8_workspace_bytes(b, hq, hkv, d, bs, max_context_len, partition_size)
    if workspace is None:
        workspace = _workspace(q.device, need)
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    args = (q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), k_scale.data_ptr(),
            v_scale.data_ptr(), nb, stride, block_tables.data_ptr(), int(block_tables.shape[1]),
            context_lens.data_ptr(), int(max_context_len), b, hq, hkv, d, bs, float(scale),
            out.data_ptr(), ws_ptr, ws_bytes, int(partition_size), _dtype_code(q))
    return PreparedCall("pkv_paged_attention_decode_int8", args, q.device,
                        (q, k_cache, v_cache, k_scale, v_scale, block_tables, context_lens, out,
                         workspace), out)


def get_device_error(device: Optional[torch.device] = None) -> Tuple[int, list]:
    """Synchronise, read and clear the device status word: (flags, [names])."""
    dev = torch.device("cuda") if device is None else torch.device(device)
    flags = ctypes.c_uint32(0)
    with torch.cuda.device(dev):
        st = lib().pkv_get_device_error(ctypes.c_void_p(torch.cuda.current_stream().cuda_stream),
                                        ctypes.byref(flags))
    if st not in (0, 4):
        raise PagedKVError("pkv_get_device_error", st)
    names = [n for bit, n in DEVERR.items() if flags.value & bit]
    return int(flags.value), names


def launch_count() -> int:
    return int(lib().pkv_launch_count())


def decode_plan(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, max_context_len,
                partition_size, sm_count, int8=False) -> dict:
    """The library's launch decision for these arguments (pure host function): that of
    pkv_paged_attention_decode, or of the INT8-cache decode when ``int8``."""
    outs = [ctypes.c_int(0) for _ in range(4)]
    name = "pkv_decode_int8_plan" if int8 else "pkv_decode_plan"
    st = getattr(lib(), name)(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                              max_context_len, partition_size, sm_count,
                              *[ctypes.byref(o) for o in outs])
    _check(st, name)
    return {"partition_size": outs[0].value, "num_partitions": outs[1].value,
            "heads_per_block": outs[2].value, "needs_merge": bool(outs[3].value)}


def debug_wait_timeout(timeout_ns: int, device: Optional[torch.device] = None) -> None:
    """Launch the bounded-wait self test (see pkv_debug_wait_timeout)."""
    dev = torch.device("cuda") if device is None else torch.device(device)
    with torch.cuda.device(dev):
        st = lib().pkv_debug_wait_timeout(int(timeout_ns),
                                          ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    _check(st, "pkv_debug_wait_timeout")
