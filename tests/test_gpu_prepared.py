"""Prepared calls (argument checks and marshalling done once, the library call
re-issued on the current stream each time): the same results as the immediate
calls, bitwise, and the oracle's results after the inputs change in place."""
import numpy as np
import pytest
import torch

import paged_kv_cache_155_gb300 as pkv
from paged_kv_cache_155_gb300.workloads import make_decode_workload
from tests._gpu_helpers import (assert_close, check_no_device_flags, device, host_pool_bits,
                                oracle_decode, oracle_step_pool)
from tests._paged_helpers import to_bits

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("hq,hkv,dtype", [(4, 4, torch.float16), (32, 8, torch.bfloat16)])
def test_prepared_step_matches_immediate_and_oracle(hq, hkv, dtype):
    dev = device()
    lens = [1, 17, 100, 33, 700, 2050]
    wl = make_decode_workload(num_seqs=len(lens), num_q_heads=hq, num_kv_heads=hkv, head_dim=128,
                              block_size=16, context_lens=lens, dtype=dtype, seed=hq + 5,
                              device=str(dev))
    k_cache, v_cache = pkv.split_pool(wl.kv)
    slots = pkv.slot_mapping(wl.block_tables, wl.new_positions, 16, num_blocks=wl.num_blocks)
    pool = host_pool_bits(wl.kv)
    out = torch.empty_like(wl.q)
    write = pkv.prepare_reshape_and_cache(wl.k_new, wl.v_new, slots, k_cache, v_cache)
    decode = pkv.prepare_paged_attention_decode(wl.q, k_cache, v_cache, wl.block_tables,
                                                wl.context_lens, wl.scale, out,
                                                max_context_len=2050, partition_size=256)
    write()
    got = decode()
    assert got is out
    torch.cuda.synchronize()
    check_no_device_flags(dev)
    oracle_step_pool(pool, wl)
    assert np.array_equal(host_pool_bits(wl.kv), pool)
    ref_now = pkv.paged_attention_decode(wl.q, k_cache, v_cache, wl.block_tables, wl.context_lens,
                                         wl.scale, max_context_len=2050, partition_size=256)
    assert torch.equal(out, ref_now)
    # new queries and a shorter context in place: the prepared call reads the new contents
    g = torch.Generator(device=dev).manual_seed(9)
    wl.q.copy_(torch.randn(wl.q.shape, generator=g, device=dev).to(dtype))
    wl.context_lens[5] = 1999
    decode()
    torch.cuda.synchronize()
    ref = oracle_decode(to_bits(wl.q.cpu()), pool, wl.block_tables.cpu(), wl.context_lens.cpu(),
                        hkv, 16, wl.scale, dtype)
    assert_close(out, ref, what="prepared decode")


def test_prepared_call_runs_on_the_current_stream():
    dev = device()
    wl = make_decode_workload(num_seqs=4, num_q_heads=8, num_kv_heads=8, head_dim=64,
                              block_size=16, context_lens=[64, 1, 200, 33], dtype=torch.float16,
                              seed=11, device=str(dev))
    k_cache, v_cache = pkv.split_pool(wl.kv)
    out = torch.zeros_like(wl.q)
    decode = pkv.prepare_paged_attention_decode(wl.q, k_cache, v_cache, wl.block_tables,
                                                wl.context_lens, wl.scale, out, max_context_len=200)
    s = torch.cuda.Stream(dev)
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        decode()
    s.synchronize()
    ref = oracle_decode(to_bits(wl.q.cpu()), host_pool_bits(wl.kv), wl.block_tables.cpu(),
                        wl.context_lens.cpu(), 8, 16, wl.scale, wl.dtype)
    assert_close(out, ref)


def test_prepared_int8_and_shared_prefix_match_immediate():
    dev = device()
    lens = [300, 1200, 33, 800]
    wl = make_decode_workload(num_seqs=4, num_q_heads=32, num_kv_heads=8, head_dim=128,
                              block_size=16, context_lens=lens, dtype=torch.float16, seed=4,
                              device=str(dev), kv_dtype=torch.int8)
    k_cache, v_cache = pkv.split_pool(wl.kv)
    out = torch.empty_like(wl.q)
    pkv.prepare_paged_attention_decode_int8(wl.q, k_cache, v_cache, wl.k_scale, wl.v_scale,
                                            wl.block_tables, wl.context_lens, wl.scale, out,
                                            max_context_len=1200)()
    now = pkv.paged_attention_decode_int8(wl.q, k_cache, v_cache, wl.k_scale, wl.v_scale,
                                          wl.block_tables, wl.context_lens, wl.scale,
                                          max_context_len=1200)
    torch.cuda.synchronize()
    assert torch.equal(out, now)
    wp = make_decode_workload(num_seqs=5, num_q_heads=32, num_kv_heads=8, head_dim=128,
                              block_size=32, context_lens=[300, 257, 500, 256, 1000],
                              dtype=torch.bfloat16, seed=10, device=str(dev),
                              shared_prefix_tokens=256)
    kc, vc = pkv.split_pool(wp.kv)
    outp = torch.empty_like(wp.q)
    pt = wp.block_tables[0, :8].contiguous()
    pkv.prepare_paged_attention_decode_shared_prefix(wp.q, kc, vc, pt, 256, wp.block_tables,
                                                     wp.context_lens, wp.scale, outp,
                                                     max_context_len=1000)()
    nowp = pkv.paged_attention_decode_shared_prefix(wp.q, kc, vc, pt, 256, wp.block_tables,
                                                    wp.context_lens, wp.scale,
                                                    max_context_len=1000)
    torch.cuda.synchronize()
    check_no_device_flags(dev)
    assert torch.equal(outp, nowp)
