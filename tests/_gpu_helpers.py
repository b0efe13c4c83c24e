"""Helpers for the GPU parity tests: run the library's step on the device, run
the oracle on host copies of the same inputs, compare."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import paged_kv_cache_155_gb300 as pkv
from paged_kv_cache_155_gb300 import _build
from tests._paged_helpers import dtype_code, to_bits

# Acceptance for attention outputs: |got - ref| <= ATOL + RTOL * |ref| elementwise,
# against the fp64 oracle (max abs error 5e-3, relative error 1e-2).
ATOL = 5e-3
RTOL = 1e-2


def device():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    _build.build()
    return torch.device("cuda:0")


def assert_close(got: torch.Tensor, ref: np.ndarray, what: str = "decode"):
    g = got.detach().float().cpu().double().numpy()
    err = np.abs(g - ref)
    bound = ATOL + RTOL * np.abs(ref)
    bad = err > bound
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} values out of tolerance; "
                             f"max abs err {err.max():.3e}; first at {idx.tolist()}")
    assert np.isfinite(g).all()
    return float(err.max())


def check_no_device_flags(dev):
    flags, names = pkv.get_device_error(dev)
    assert flags == 0, f"device status flags raised: {names}"


def host_pool_bits(kv: torch.Tensor) -> np.ndarray:
    return to_bits(kv.cpu())


def oracle_decode(q_bits, pool_bits, tables, lens, num_kv_heads, block_size, scale, dtype):
    flat = np.ascontiguousarray(pool_bits).reshape(-1)
    half = pool_bits.shape[2] * pool_bits.shape[3] * pool_bits.shape[4]
    return oracle.paged_decode(q_bits, flat, flat[half:], 2 * half, np.asarray(tables),
                               np.asarray(lens), num_kv_heads, block_size, scale, dtype_code(dtype))


def run_step(wl, partition_size=0, tables=None):
    """The library's decode step on device: cache write of the new token at
    position len-1, then paged decode.  Returns out (device)."""
    k_cache, v_cache = pkv.split_pool(wl.kv)
    bt = wl.block_tables if tables is None else tables
    slots = pkv.slot_mapping(bt, wl.new_positions, wl.block_size, num_blocks=wl.num_blocks)
    pkv.reshape_and_cache(wl.k_new, wl.v_new, slots, k_cache, v_cache)
    return pkv.paged_attention_decode(wl.q, k_cache, v_cache, bt, wl.context_lens, wl.scale,
                                      max_context_len=int(wl.context_lens.max().item()),
                                      partition_size=partition_size)


def oracle_step_pool(wl_host_pool_bits, wl, tables=None):
    """Oracle cache write of the new tokens into a host pool copy (in place)."""
    bt = (wl.block_tables if tables is None else tables).cpu().numpy()
    slots = oracle.slot_mapping(bt, wl.new_positions.cpu().numpy(), wl.block_size)
    oracle.reshape_and_cache(to_bits(wl.k_new.cpu()), to_bits(wl.v_new.cpu()), slots,
                             wl_host_pool_bits, wl.num_kv_heads, wl.block_size, wl.head_dim)
    return slots


# ---------------------------------------------------------------- INT8 cache
def run_step_int8(wl, partition_size=0, tables=None):
    """The library's decode step over an INT8 pool: quantising cache write of the
    new token at position len-1, then paged decode.  Returns out (device)."""
    k_cache, v_cache = pkv.split_pool(wl.kv)
    bt = wl.block_tables if tables is None else tables
    slots = pkv.slot_mapping(bt, wl.new_positions, wl.block_size, num_blocks=wl.num_blocks)
    pkv.reshape_and_cache_int8(wl.k_new, wl.v_new, slots, k_cache, v_cache, wl.k_scale,
                               wl.v_scale)
    return pkv.paged_attention_decode_int8(wl.q, k_cache, v_cache, wl.k_scale, wl.v_scale, bt,
                                           wl.context_lens, wl.scale,
                                           max_context_len=int(wl.context_lens.max().item()),
                                           partition_size=partition_size)


def oracle_step_pool_int8(pool_i8: np.ndarray, wl, tables=None):
    """Oracle quantising cache write of the new tokens into a host INT8 pool copy."""
    bt = (wl.block_tables if tables is None else tables).cpu().numpy()
    slots = oracle.slot_mapping(bt, wl.new_positions.cpu().numpy(), wl.block_size)
    oracle.reshape_and_cache_int8(to_bits(wl.k_new.cpu()), to_bits(wl.v_new.cpu()), slots,
                                  pool_i8, wl.k_scale.cpu().numpy(), wl.v_scale.cpu().numpy(),
                                  wl.num_kv_heads, wl.block_size, wl.head_dim,
                                  dtype_code(wl.dtype))
    return slots


def oracle_decode_int8(wl, pool_i8, sel=None, tables=None):
    """Oracle decode of (a subset of) a workload's sequences over a host INT8 pool."""
    bt = (wl.block_tables if tables is None else tables).cpu().numpy()
    q = to_bits(wl.q.cpu())
    lens = wl.context_lens.cpu().numpy()
    if sel is not None:
        q, bt, lens = q[sel], bt[sel], lens[sel]
    return oracle.paged_decode_int8(q, pool_i8, wl.k_scale.cpu().numpy(), wl.v_scale.cpu().numpy(),
                                    bt, lens, wl.num_kv_heads, wl.block_size, wl.scale,
                                    dtype_code(wl.dtype))


# ---------------------------------------------------------------- chunked prefill
def run_prefill(wl, kv_splits=0):
    """The library's prefill step on device: the chunk rows' K/V written at their
    positions, then chunked prefill attention.  Returns out (device)."""
    k_cache, v_cache = pkv.split_pool(wl.kv)
    n = int(wl.query_start[-1])
    if n:
        slots = pkv.slot_mapping(wl.block_tables, wl.new_positions, wl.block_size,
                                 token_rows=wl.row_seq, num_blocks=wl.num_blocks)
        pkv.reshape_and_cache(wl.k_new, wl.v_new, slots, k_cache, v_cache)
    out = torch.zeros_like(wl.q)
    return pkv.paged_attention_prefill(wl.q, k_cache, v_cache, wl.block_tables, wl.query_start,
                                       wl.context_lens, wl.scale, out,
                                       max_query_len=wl.max_query_len,
                                       max_context_len=wl.max_context_len, kv_splits=kv_splits)


def oracle_prefill_step(pool_bits: np.ndarray, wl, rows=None):
    """Oracle cache write of the chunk rows into a host pool copy (in place), then the
    oracle prefill of every chunk row -- or, with rows = [(seq, j), ...], of just those
    rows (each as a one-row chunk at its own position).  Returns fp64 outputs."""
    bt = wl.block_tables.cpu().numpy()
    n = int(wl.query_start[-1])
    if n:
        slots = oracle.slot_mapping(bt[wl.row_seq.cpu().numpy()], wl.new_positions.cpu().numpy(),
                                    wl.block_size)
        oracle.reshape_and_cache(to_bits(wl.k_new.cpu()), to_bits(wl.v_new.cpu()), slots, pool_bits,
                                 wl.num_kv_heads, wl.block_size, wl.head_dim)
    flat = np.ascontiguousarray(pool_bits).reshape(-1)
    half = pool_bits.shape[2] * pool_bits.shape[3] * pool_bits.shape[4]
    q = to_bits(wl.q.cpu())
    qs = wl.query_start.cpu().numpy()
    lens = wl.context_lens.cpu().numpy()
    if rows is None:
        return oracle.paged_prefill(q[:n], flat, flat[half:], 2 * half, bt, qs, lens,
                                    wl.num_kv_heads, wl.block_size, wl.scale, dtype_code(wl.dtype))
    sel_q = np.stack([q[qs[i] + j] for i, j in rows])
    sel_bt = np.stack([bt[i] for i, _ in rows])
    sel_len = np.array([lens[i] - (qs[i + 1] - qs[i]) + j + 1 for i, j in rows], dtype=np.int32)
    return oracle.paged_prefill(sel_q, flat, flat[half:], 2 * half, sel_bt,
                                np.arange(len(rows) + 1), sel_len, wl.num_kv_heads, wl.block_size,
                                wl.scale, dtype_code(wl.dtype))


# ---------------------------------------------------------------- stale slots
# NaN, +Inf and -Inf bit patterns of each 16-bit type
_NONFINITE = {torch.float16: (0x7E00, 0x7C00, 0xFC00),
              torch.bfloat16: (0x7FC0, 0x7F80, 0xFF80)}


def poison_unused_slots(kv: torch.Tensor, tables, lens, block_size: int) -> int:
    """Overwrite every pool slot that no sequence's context covers -- the tail rows
    of each last block and every block no table reaches -- with NaN, +Inf and -Inf
    in turn, in K and V and for every KV head (a pool from torch.empty may hold
    anything there).  Attention must not read them: the result stays that of the
    covered tokens.  Returns the number of poisoned slots."""
    nb = kv.shape[0]
    covered = np.zeros((nb, block_size), dtype=bool)
    tables = np.asarray(tables.cpu() if torch.is_tensor(tables) else tables)
    lens = np.asarray(lens.cpu() if torch.is_tensor(lens) else lens)
    for i, n in enumerate(lens.tolist()):
        nblk = -(-int(n) // block_size)
        if nblk == 0:
            continue
        blocks = tables[i, :nblk]
        covered[blocks[:-1], :] = True
        covered[blocks[-1], :int(n) - (nblk - 1) * block_size] = True
    bits = to_bits(kv.cpu())
    pats = _NONFINITE[kv.dtype]
    bad = np.argwhere(~covered)
    for k, (b, o) in enumerate(bad):
        bits[b, :, :, o, :] = pats[k % 3]
    kv.copy_(torch.from_numpy(bits.view(np.int16)).view(kv.dtype).to(kv.device))
    return len(bad)
