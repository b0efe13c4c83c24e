"""CPU oracle for paged-KV-cache decode.  TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
legs of ``bench.py`` may import this package.  The product (the CUDA library
``paged_kv_cache_155_gb300`` and its binding) never imports it, and this
package imports nothing from the product.

The arithmetic lives in ``pagedkv_oracle.c`` (fp64 throughout, exact 16-bit
decoding, libm ``exp``); this module compiles it with gcc on first use and
wraps it for numpy arrays, and adds the pages' KV-size arithmetic.

Pages cited (title and section):
  P1 = "KV Cache与PagedAttention深度解析：vLLM内存管理革命" (iopencloud.com)
  P2 = "KV Cache从原理到实战：大模型推理内存管理演进与优化" (xnwp.cn/news/16711)
  P3 = PagedAttention + prefix caching via nano-vllm (zwxr.cn/news/317362)
  P4 = "大模型 (LLM) 推理加速核心技术解析：从 KV Cache 到 PagedAttention 实战" (jsqmd.com)

Every oracle function below is pinned by tests in ``tests/test_oracle_*.py``
against closed forms, brute force, a library routine or the pages' printed
numbers; none is marked "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pagedkv_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "liboracle.so")
_lock = threading.Lock()
_lib = None

F16 = 0
BF16 = 1


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (OpenMP over (sequence, head) pairs)."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-std=c11", "-Wall",
           "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i64, i32, dbl = ctypes.c_int64, ctypes.c_int, ctypes.c_double
        lib.oracle_f16_to_f64.argtypes = [ctypes.c_uint16]
        lib.oracle_f16_to_f64.restype = dbl
        lib.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_to_f64.restype = dbl
        lib.oracle_num_threads.restype = i32
        lib.oracle_slot_for_position.argtypes = [P, i64, i32]
        lib.oracle_slot_for_position.restype = i64
        lib.oracle_blocks_needed.argtypes = [i64, i32]
        lib.oracle_blocks_needed.restype = i64
        dec = [P, P, P, i64, P, i32, P, i32, i32, i32, i32, i32, dbl, i32, P]
        lib.oracle_paged_decode.argtypes = dec
        lib.oracle_paged_decode.restype = None
        lib.oracle_paged_flash_decode.argtypes = dec
        lib.oracle_paged_flash_decode.restype = None
        lib.oracle_reshape_and_cache.argtypes = [P, P, P, i64, P, P, i64, i32, i32, i32]
        lib.oracle_reshape_and_cache.restype = None
        lib.oracle_copy_blocks.argtypes = [P, P, i64, i64, P, i64]
        lib.oracle_copy_blocks.restype = None
        f32 = ctypes.c_float
        lib.oracle_quantize_int8.argtypes = [ctypes.c_uint16, i32, f32]
        lib.oracle_quantize_int8.restype = i32
        lib.oracle_quantize_int8_array.argtypes = [P, i64, P, i64, i32, P]
        lib.oracle_quantize_int8_array.restype = None
        lib.oracle_reshape_and_cache_int8.argtypes = [P, P, P, i64, P, P, i64, i32, i32, i32,
                                                      P, P, i32]
        lib.oracle_reshape_and_cache_int8.restype = None
        lib.oracle_paged_decode_int8.argtypes = [P, P, P, P, P, i64, P, i32, P, i32, i32, i32,
                                                 i32, i32, dbl, i32, P]
        lib.oracle_paged_decode_int8.restype = None
        lib.oracle_paged_prefill.argtypes = [P, P, P, i64, P, i32, P, P, i32, i32, i32, i32, i32,
                                             dbl, i32, P]
        lib.oracle_paged_prefill.restype = None
        lib.oracle_copy_blocks_bytes.argtypes = [P, P, i64, i64, P, i64]
        lib.oracle_copy_blocks_bytes.restype = None
        _lib = lib
        return lib


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _u16(a: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype == np.float16:
        a = a.view(np.uint16)
    if a.dtype == np.int16:
        a = a.view(np.uint16)
    if a.dtype != np.uint16:
        raise TypeError(f"expected 16-bit bit patterns, got {a.dtype}")
    return a


def decode16(bits: np.ndarray, dtype: int) -> np.ndarray:
    """Exact fp64 values of 16-bit patterns, via the oracle's own decoders."""
    lib = _load()
    fn = lib.oracle_bf16_to_f64 if dtype == BF16 else lib.oracle_f16_to_f64
    flat = _u16(bits).ravel()
    table = np.array([fn(int(b)) for b in range(65536)], dtype=np.float64)
    return table[flat].reshape(np.shape(bits))


def slot_for_position(table_row: np.ndarray, t: int, block_size: int) -> int:
    """Flat slot of logical position t (P1 §5.3)."""
    row = np.ascontiguousarray(table_row, dtype=np.int32)
    return int(_load().oracle_slot_for_position(_ptr(row), int(t), int(block_size)))


def blocks_needed(t: int, block_size: int) -> int:
    """Blocks a sequence needs once it holds token t: ceil((t+1)/bs) (P1 §5.3)."""
    return int(_load().oracle_blocks_needed(int(t), int(block_size)))


def slot_mapping(block_tables: np.ndarray, positions: np.ndarray, block_size: int) -> np.ndarray:
    """Slot of positions[i] in sequence i, one oracle call per sequence."""
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    return np.array([slot_for_position(bt[i], int(p), block_size)
                     for i, p in enumerate(np.asarray(positions))], dtype=np.int64)


def _decode_call(fn_name, q, k_cache, v_cache, block_stride, block_tables, context_lens,
                 num_kv_heads, block_size, scale, dtype):
    q = _u16(q)
    kc, vc = _u16(k_cache), _u16(v_cache)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    num_seqs, num_q_heads, head_dim = q.shape
    if num_q_heads % num_kv_heads:
        raise ValueError("num_q_heads must be a multiple of num_kv_heads")
    out = np.zeros((num_seqs, num_q_heads, head_dim), dtype=np.float64)
    getattr(_load(), fn_name)(
        _ptr(q), _ptr(kc), _ptr(vc), int(block_stride), _ptr(bt), int(bt.shape[1]), _ptr(cl),
        int(num_seqs), int(num_q_heads), int(num_kv_heads), int(head_dim), int(block_size),
        float(scale), int(dtype), _ptr(out))
    return out


def paged_decode(q, k_cache, v_cache, block_stride, block_tables, context_lens,
                 num_kv_heads, block_size, scale, dtype):
    """Direct two-pass decode attention over the block tables (P1 §2.1, §4.2-4.3).

    ``q`` is [num_seqs, num_q_heads, head_dim] of 16-bit patterns; ``k_cache`` and
    ``v_cache`` are flat 16-bit arrays (the K and V halves, possibly the same
    buffer viewed twice) addressed as block*block_stride + (h*bs + off)*d + j.
    Returns fp64 [num_seqs, num_q_heads, head_dim].
    """
    return _decode_call("oracle_paged_decode", q, k_cache, v_cache, block_stride, block_tables,
                        context_lens, num_kv_heads, block_size, scale, dtype)


def paged_flash_decode(q, k_cache, v_cache, block_stride, block_tables, context_lens,
                       num_kv_heads, block_size, scale, dtype):
    """Online-softmax form of the same decode (P1 §7.2)."""
    return _decode_call("oracle_paged_flash_decode", q, k_cache, v_cache, block_stride,
                        block_tables, context_lens, num_kv_heads, block_size, scale, dtype)


def reshape_and_cache(k_new, v_new, slot_mapping_, kv_pool_bits: np.ndarray,
                      num_kv_heads: int, block_size: int, head_dim: int) -> None:
    """Byte scatter of new K/V rows into a packed pool [NB, 2, Hkv, bs, d] (in place)."""
    pool = kv_pool_bits
    assert pool.dtype == np.uint16 and pool.flags.c_contiguous
    kn, vn = _u16(k_new), _u16(v_new)
    sm = np.ascontiguousarray(slot_mapping_, dtype=np.int64)
    half = num_kv_heads * block_size * head_dim
    base = pool.ctypes.data
    _load().oracle_reshape_and_cache(
        _ptr(kn), _ptr(vn), _ptr(sm), int(sm.shape[0]), ctypes.c_void_p(base),
        ctypes.c_void_p(base + 2 * half), int(2 * half), int(num_kv_heads), int(head_dim),
        int(block_size))


def copy_blocks(kv_pool_bits: np.ndarray, src_dst: np.ndarray, num_kv_heads: int,
                block_size: int, head_dim: int) -> None:
    """Copy-on-write block copies on a packed pool [NB, 2, Hkv, bs, d] (in place)."""
    pool = kv_pool_bits
    assert pool.dtype == np.uint16 and pool.flags.c_contiguous
    pairs = np.ascontiguousarray(src_dst, dtype=np.int64).reshape(-1, 2)
    half = num_kv_heads * block_size * head_dim
    base = pool.ctypes.data
    _load().oracle_copy_blocks(ctypes.c_void_p(base), ctypes.c_void_p(base + 2 * half),
                               int(2 * half), int(half), _ptr(pairs), int(pairs.shape[0]))


def paged_prefill(q, k_cache, v_cache, block_stride, block_tables, query_start, context_lens,
                  num_kv_heads, block_size, scale, dtype):
    """Chunked prefill attention over the block tables (P4 §2 causal attention with a
    cache; P2 §2.3, §5.4).  ``q`` is [num_rows, num_q_heads, head_dim] 16-bit patterns,
    the chunks of all sequences back to back (sequence i owns rows
    query_start[i] .. query_start[i+1]-1); context_lens[i] counts the cached tokens
    including the chunk.  Row j of chunk i, at position L_i - C_i + j, attends to
    tokens 0 .. that position.  Returns fp64 [num_rows, num_q_heads, head_dim]."""
    q = _u16(q)
    kc, vc = _u16(k_cache), _u16(v_cache)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    qs = np.ascontiguousarray(query_start, dtype=np.int32)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    num_rows, num_q_heads, head_dim = q.shape
    num_seqs = int(cl.shape[0])
    if qs.shape[0] != num_seqs + 1 or int(qs[-1]) != num_rows:
        raise ValueError("query_start must hold num_seqs + 1 offsets ending at num_rows")
    if num_q_heads % num_kv_heads:
        raise ValueError("num_q_heads must be a multiple of num_kv_heads")
    if np.any(np.diff(qs) < 0) or np.any(cl < np.diff(qs)):
        raise ValueError("each chunk must be non-negative and fit in its context")
    out = np.zeros((num_rows, num_q_heads, head_dim), dtype=np.float64)
    _load().oracle_paged_prefill(
        _ptr(q), _ptr(kc), _ptr(vc), int(block_stride), _ptr(bt), int(bt.shape[1]), _ptr(qs),
        _ptr(cl), num_seqs, int(num_q_heads), int(num_kv_heads), int(head_dim), int(block_size),
        float(scale), int(dtype), _ptr(out))
    return out


# ---------------------------------------------------------------------------
# INT8 KV cache with per-channel scales (P2 §5.2).
# ---------------------------------------------------------------------------

def _f32(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float32)


def quantize_int8_scalar(bits: int, dtype: int, scale: float) -> int:
    """Code of one 16-bit value: round-half-even(clamp(x / s, -127, 127)) in fp32."""
    return int(_load().oracle_quantize_int8(int(bits) & 0xFFFF, int(dtype), float(scale)))


def quantize_int8(x_bits: np.ndarray, scales: np.ndarray, dtype: int) -> np.ndarray:
    """Codes of an array [..., heads, head_dim] of 16-bit patterns with per-channel
    scales [heads, head_dim] (broadcast over the leading axes), or one scale for all."""
    x = _u16(x_bits)
    sc = _f32(scales)
    if sc.size != 1 and x.shape[-sc.ndim:] != sc.shape:
        raise ValueError("scales must be one value or match the trailing axes of x")
    codes = np.empty(x.shape, dtype=np.int8)
    _load().oracle_quantize_int8_array(_ptr(x), int(x.size), _ptr(sc), int(sc.size), int(dtype),
                                       _ptr(codes))
    return codes


def reshape_and_cache_int8(k_new, v_new, slot_mapping_, kv_pool: np.ndarray, k_scale, v_scale,
                           num_kv_heads: int, block_size: int, head_dim: int, dtype: int) -> None:
    """Quantising cache write into a packed INT8 pool [NB, 2, Hkv, bs, d] (in place)."""
    pool = kv_pool
    assert pool.dtype == np.int8 and pool.flags.c_contiguous
    kn, vn = _u16(k_new), _u16(v_new)
    sm = np.ascontiguousarray(slot_mapping_, dtype=np.int64)
    ks, vs = _f32(k_scale), _f32(v_scale)
    half = num_kv_heads * block_size * head_dim
    base = pool.ctypes.data
    _load().oracle_reshape_and_cache_int8(
        _ptr(kn), _ptr(vn), _ptr(sm), int(sm.shape[0]), ctypes.c_void_p(base),
        ctypes.c_void_p(base + half), int(2 * half), int(num_kv_heads), int(head_dim),
        int(block_size), _ptr(ks), _ptr(vs), int(dtype))


def paged_decode_int8(q, kv_pool: np.ndarray, k_scale, v_scale, block_tables, context_lens,
                      num_kv_heads, block_size, scale, dtype):
    """Two-pass decode attention over a packed INT8 pool [NB, 2, Hkv, bs, d], each
    code dequantised as code * scale[h][channel] (P2 §5.2; P1 §2.1, §4.2-4.3).
    Returns fp64 [num_seqs, num_q_heads, head_dim]."""
    q = _u16(q)
    pool = np.ascontiguousarray(kv_pool)
    assert pool.dtype == np.int8
    ks, vs = _f32(k_scale), _f32(v_scale)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    num_seqs, num_q_heads, head_dim = q.shape
    if num_q_heads % num_kv_heads:
        raise ValueError("num_q_heads must be a multiple of num_kv_heads")
    half = num_kv_heads * block_size * head_dim
    base = pool.ctypes.data
    out = np.zeros((num_seqs, num_q_heads, head_dim), dtype=np.float64)
    _load().oracle_paged_decode_int8(
        _ptr(q), ctypes.c_void_p(base), ctypes.c_void_p(base + half), _ptr(ks), _ptr(vs),
        int(2 * half), _ptr(bt), int(bt.shape[1]), _ptr(cl), int(num_seqs), int(num_q_heads),
        int(num_kv_heads), int(head_dim), int(block_size), float(scale), int(dtype), _ptr(out))
    return out


def copy_blocks_bytes(kv_pool: np.ndarray, src_dst: np.ndarray) -> None:
    """Copy-on-write block copies on a packed pool [NB, 2, ...] of any dtype (in place)."""
    pool = kv_pool
    assert pool.flags.c_contiguous
    pairs = np.ascontiguousarray(src_dst, dtype=np.int64).reshape(-1, 2)
    block_bytes = pool[0].nbytes
    base = pool.ctypes.data
    _load().oracle_copy_blocks_bytes(ctypes.c_void_p(base), ctypes.c_void_p(base + block_bytes // 2),
                                     int(block_bytes), int(block_bytes // 2), _ptr(pairs),
                                     int(pairs.shape[0]))


# ---------------------------------------------------------------------------
# KV-size arithmetic the pages print (used as pins, not on any device path).
# ---------------------------------------------------------------------------

def kv_bytes_per_token(num_layers: int, num_kv_heads: int, head_dim: int, elem_bytes: int = 2) -> int:
    """K and V of one token over all layers: layers * 2 * kv_heads * head_dim * bytes.

    P2 §2.2 states it per layer as 2 * hidden_size * dtype_bytes (MHA, so
    hidden_size = heads * head_dim); P3 §1.2 as 2 * kv_heads * head_dim elements
    per layer under GQA; P1 §1.2 as L * 2 * d per token in fp16.
    """
    return num_layers * 2 * num_kv_heads * head_dim * elem_bytes


def kv_bytes(num_layers: int, num_kv_heads: int, head_dim: int, tokens: int,
             batch: int = 1, elem_bytes: int = 2) -> int:
    """Total KV bytes for ``batch`` sequences of ``tokens`` tokens each."""
    return kv_bytes_per_token(num_layers, num_kv_heads, head_dim, elem_bytes) * tokens * batch
