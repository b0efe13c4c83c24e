"""The decode entry point that allocates nothing
(pkv_paged_attention_decode_static_scratch), called through the C ABI.

It exists for callers that cannot allocate device memory for the decode
workspace: a serving engine that reserved nearly all free device memory for
its KV block pool, or a plug-in that gets tensor pointers but no allocator.
It must give the oracle's results, and the same results as the
workspace-taking entry point, on two calls in a row (the shared scratch array
keeps the previous call's contents), and must reject plans whose scratch would
not fit its fixed array.

This file is collected last on purpose; it builds its own inputs so that it
passes alone in a fresh process as well as after the other tests.
"""
import ctypes

import numpy as np
import pytest
import torch

import paged_kv_cache_155_gb300 as pkv
from paged_kv_cache_155_gb300._lib import lib
from paged_kv_cache_155_gb300.workloads import make_decode_workload
from tests._gpu_helpers import (ATOL, RTOL, assert_close, check_no_device_flags, device,
                                host_pool_bits, oracle_decode)
from tests._paged_helpers import to_bits

SCRATCH_LIMIT = 5          # PKV_ERR_SCRATCH_LIMIT
SCRATCH_BYTES = 32 << 20   # PKV_STATIC_SCRATCH_BYTES


def _static_scratch_decode(wl, q, out, maxl, partition_size):
    k_cache, v_cache = pkv.split_pool(wl.kv)
    stream = ctypes.c_void_p(torch.cuda.current_stream(q.device).cuda_stream)
    return lib().pkv_paged_attention_decode_static_scratch(
        q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), wl.num_blocks, k_cache.stride(0),
        wl.block_tables.data_ptr(), wl.block_tables.shape[1], wl.context_lens.data_ptr(), maxl,
        wl.num_seqs, wl.num_q_heads, wl.num_kv_heads, wl.head_dim, wl.block_size, wl.scale,
        out.data_ptr(), partition_size, 0 if q.dtype == torch.float16 else 1, stream)


def _close(got, ref):
    g = got.float().cpu().double().numpy()
    r = ref.float().cpu().double().numpy()
    assert np.all(np.abs(g - r) <= ATOL + RTOL * np.abs(r))


@pytest.mark.gpu
@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16], ids=["f16", "bf16"])
def test_static_scratch_decode_matches_oracle_and_workspace_decode(dtype):
    dev = device()
    lens = [1, 700, 4096, 33, 2500, 1024, 17, 3000]
    wl = make_decode_workload(num_seqs=len(lens), num_q_heads=32, num_kv_heads=8, head_dim=128,
                              block_size=16, context_lens=lens, dtype=dtype, seed=77,
                              device=str(dev))
    maxl = max(lens)
    part = 256          # 16 partitions for the longest sequence: the scratch is used
    need = pkv.decode_workspace_bytes(wl.num_seqs, 32, 8, 128, 16, maxl, part)
    assert 0 < need <= SCRATCH_BYTES
    k_cache, v_cache = pkv.split_pool(wl.kv)
    pool = host_pool_bits(wl.kv)
    g = torch.Generator(device=dev).manual_seed(5)
    for call in range(2):                       # two calls in a row, different queries
        q = torch.randn(wl.q.shape, generator=g, device=dev).to(dtype)
        ref = pkv.paged_attention_decode(q, k_cache, v_cache, wl.block_tables, wl.context_lens,
                                         wl.scale, max_context_len=maxl, partition_size=part)
        out = torch.full_like(q, float("nan"))
        st = _static_scratch_decode(wl, q, out, maxl, part)
        assert st == 0, f"call {call}: status {st}"
        torch.cuda.synchronize()
        check_no_device_flags(dev)
        oracle_ref = oracle_decode(to_bits(q.cpu()), pool, wl.block_tables.cpu(),
                                   wl.context_lens.cpu(), wl.num_kv_heads, wl.block_size,
                                   wl.scale, dtype)
        assert_close(out, oracle_ref, what=f"static-scratch decode, call {call}")
        _close(out, ref)
    # a plan whose scratch would exceed the fixed array is refused before any launch
    big = make_decode_workload(num_seqs=64, num_q_heads=64, num_kv_heads=8, head_dim=128,
                               block_size=16, context_lens=[16] * 64, dtype=dtype, seed=1,
                               device=str(dev), max_blocks_per_seq=2048)
    need_big = pkv.decode_workspace_bytes(64, 64, 8, 128, 16, 32768, 512)
    assert need_big > SCRATCH_BYTES
    out = torch.zeros_like(big.q)
    assert _static_scratch_decode(big, big.q, out, 32768, 512) == SCRATCH_LIMIT
    assert torch.all(out == 0)
