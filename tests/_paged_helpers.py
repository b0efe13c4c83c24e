"""Test-side helpers: build paged pools from dense per-sequence K/V and call the oracle.

The block placement here is done block-wise (reshape a sequence's dense rows
into [n_blocks, bs, ...] and assign whole blocks to physical slots), which is a
different construction from the oracle's token-by-token addressing, so a dense
reference computed on the original rows checks the oracle's addressing.
"""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle


def to_bits(t: torch.Tensor) -> np.ndarray:
    """16-bit torch tensor (CPU) -> numpy uint16 bit patterns, same shape."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def from_bits(a: np.ndarray, dtype: torch.dtype) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(dtype)


def dtype_code(dtype: torch.dtype) -> int:
    return oracle.BF16 if dtype == torch.bfloat16 else oracle.F16


def random_bits(shape, dtype, gen):
    return to_bits(torch.randn(shape, generator=gen).to(dtype))


def paged_from_dense(k_dense, v_dense, block_size, num_blocks, gen, dtype):
    """Scatter dense per-sequence K/V ([L_i, Hkv, d] bit arrays) into a pool.

    Returns (pool [NB, 2, Hkv, bs, d] uint16, tables [B, MB] int32, lens [B] int32).
    Logical block j of sequence i goes to a seeded random physical block.
    """
    hkv, d = k_dense[0].shape[1], k_dense[0].shape[2]
    pool = random_bits((num_blocks, 2, hkv, block_size, d), dtype, gen)
    nblk = [math.ceil(k.shape[0] / block_size) for k in k_dense]
    assert sum(nblk) <= num_blocks
    perm = torch.randperm(num_blocks, generator=gen).numpy()
    mb = max([1] + nblk)
    tables = np.zeros((len(k_dense), mb), dtype=np.int32)
    cur = 0
    for i, (k, v) in enumerate(zip(k_dense, v_dense)):
        n = nblk[i]
        phys = perm[cur:cur + n]
        cur += n
        tables[i, :n] = phys
        for src, dst in ((k, 0), (v, 1)):
            padded = np.zeros((n * block_size, hkv, d), dtype=np.uint16)
            padded[:src.shape[0]] = src
            blocks = padded.reshape(n, block_size, hkv, d).transpose(0, 2, 1, 3)
            # leave the pool's random filler in the unused tail rows of the last block
            tail = n * block_size - src.shape[0]
            if tail:
                keep = pool[phys[-1], dst, :, block_size - tail:, :].copy()
            pool[phys, dst] = blocks
            if tail:
                pool[phys[-1], dst, :, block_size - tail:, :] = keep
    lens = np.array([k.shape[0] for k in k_dense], dtype=np.int32)
    return pool, tables, lens


def oracle_decode_pool(q_bits, pool, tables, lens, num_kv_heads, block_size, scale, dtype,
                       flash=False):
    """Call the oracle on a packed pool [NB, 2, Hkv, bs, d] (uint16)."""
    flat = np.ascontiguousarray(pool).reshape(-1)
    half = pool.shape[2] * pool.shape[3] * pool.shape[4]
    fn = oracle.paged_flash_decode if flash else oracle.paged_decode
    return fn(q_bits, flat, flat[half:], 2 * half, tables, lens, num_kv_heads, block_size, scale,
              dtype_code(dtype))


def dense_reference(q_bits, k_dense, v_dense, scale, dtype):
    """torch scaled_dot_product_attention in fp64 on the dense rows (GQA by contiguous groups)."""
    outs = []
    q = from_bits(q_bits, dtype).to(torch.float64)
    for i, (k, v) in enumerate(zip(k_dense, v_dense)):
        kt = from_bits(k, dtype).to(torch.float64).permute(1, 0, 2).unsqueeze(0)  # [1,Hkv,L,d]
        vt = from_bits(v, dtype).to(torch.float64).permute(1, 0, 2).unsqueeze(0)
        qi = q[i].unsqueeze(0).unsqueeze(2)                                      # [1,Hq,1,d]
        if kt.shape[2] == 0:
            outs.append(torch.zeros_like(q[i]))
            continue
        o = torch.nn.functional.scaled_dot_product_attention(
            qi, kt, vt, scale=scale, enable_gqa=(qi.shape[1] != kt.shape[1]))
        outs.append(o[0, :, 0, :])
    return torch.stack(outs).numpy()


def workload_bits(wl):
    """Host bit views of a workload's pool and queries."""
    return to_bits(wl.kv), to_bits(wl.q)
