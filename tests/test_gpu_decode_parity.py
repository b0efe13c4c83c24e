"""GPU parity of the decode step (cache write + paged decode) against the oracle.

Bit-exact for the cache write; attention within |got-ref| <= 5e-3 + 1e-2|ref| of
the fp64 oracle.  Shapes span several tiles, ragged tails, empty and one-token
contexts, every supported head_dim / block_size / dtype, MHA and GQA groups
(including groups that need several head subgroups), automatic and forced
split-context partitions."""
import math

import numpy as np
import pytest
import torch

import paged_kv_cache_155_gb300 as pkv
from paged_kv_cache_155_gb300.workloads import make_decode_workload
from tests._gpu_helpers import (assert_close, check_no_device_flags, device, host_pool_bits,
                                oracle_decode, oracle_step_pool, poison_unused_slots, run_step)
from tests._paged_helpers import to_bits

pytestmark = pytest.mark.gpu


def _check_step(wl_dev, partition_size=0):
    dev = wl_dev.kv.device
    pool = host_pool_bits(wl_dev.kv)                 # before the cache write
    out = run_step(wl_dev, partition_size)
    torch.cuda.synchronize()
    check_no_device_flags(dev)
    oracle_step_pool(pool, wl_dev)
    assert np.array_equal(host_pool_bits(wl_dev.kv), pool), "cache write not bit-exact"
    ref = oracle_decode(to_bits(wl_dev.q.cpu()), pool, wl_dev.block_tables.cpu(),
                        wl_dev.context_lens.cpu(), wl_dev.num_kv_heads, wl_dev.block_size,
                        wl_dev.scale, wl_dev.dtype)
    return assert_close(out, ref)


@pytest.mark.parametrize("longest", [300, 2100], ids=["short", "long"])
@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16], ids=["f16", "bf16"])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("bs", [8, 16, 32])
@pytest.mark.parametrize("hq,hkv", [(4, 4), (8, 4), (16, 4), (32, 4), (12, 4), (24, 4), (64, 4)])
def test_decode_shapes(dtype, d, bs, hq, hkv, longest):
    """Every shape, with a short and a long batch: groups of 4, 8 or 16 query heads per KV
    head run as warp-level MMAs (16 in one block at head_dim 128, as two blocks of 8 at
    head_dim 64), the others as per-lane loops."""
    dev = device()
    lens = [1, bs - 1, bs, bs + 1, 5 * bs + 3, longest, 17]
    wl = make_decode_workload(num_seqs=len(lens), num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                              block_size=bs, context_lens=lens, dtype=dtype,
                              seed=hq * 7 + d + bs, device=str(dev))
    _check_step(wl)


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16], ids=["f16", "bf16"])
@pytest.mark.parametrize("bs", [8, 16, 32])
@pytest.mark.parametrize("hq,hkv,d", [(4, 4, 128), (8, 4, 128), (16, 4, 128), (32, 4, 128),
                                      (64, 4, 128), (32, 4, 64)])
def test_decode_ignores_nonfinite_unused_slots(dtype, bs, hq, hkv, d):
    """Slots past each context (the unwritten tail of a last block) and blocks no table
    reaches hold NaN / +Inf / -Inf: the output is still the oracle's, finite, for the
    per-lane loops (groups 1, 2) and the warp-MMA forms (groups 4, 8, 16), one
    partition and several."""
    dev = device()
    lens = [1, bs - 1, bs + 1, 5 * bs + 3, 300, 17, 2 * bs]
    need = sum(-(-n // bs) for n in lens)
    wl = make_decode_workload(num_seqs=len(lens), num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                              block_size=bs, context_lens=lens, dtype=dtype, seed=hq + bs + d,
                              device=str(dev), num_blocks=need + 6)
    assert poison_unused_slots(wl.kv, wl.block_tables, wl.context_lens, bs) > 6 * bs
    _check_step(wl)
    _check_step(wl, partition_size=4 * bs)


@pytest.mark.parametrize("partition", [16, 32, 48, 256, 1024])
@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16], ids=["f16", "bf16"])
def test_decode_forced_partitions(partition, dtype):
    dev = device()
    lens = [1, 15, 16, 17, 511, 512, 513, 1500, 2049]
    wl = make_decode_workload(num_seqs=len(lens), num_q_heads=16, num_kv_heads=2, head_dim=128,
                              block_size=16, context_lens=lens, dtype=dtype, seed=partition,
                              device=str(dev))
    _check_step(wl, partition_size=partition)


@pytest.mark.parametrize("hq,hkv,dtype", [(32, 32, torch.float16), (32, 8, torch.bfloat16),
                                          (64, 8, torch.bfloat16)])
def test_decode_merge_never_reads_stale_partials(hq, hkv, dtype):
    """The merge starts behind the decode kernel and must wait for its partials: with
    the workspace filled with NaN before each call and new queries each time, every
    split-context call gives the oracle's result."""
    dev = device()
    lens = [4096, 1, 2049, 3000, 512, 4000]
    wl = make_decode_workload(num_seqs=len(lens), num_q_heads=hq, num_kv_heads=hkv, head_dim=128,
                              block_size=16, context_lens=lens, dtype=dtype, seed=hq + hkv,
                              device=str(dev))
    k_cache, v_cache = pkv.split_pool(wl.kv)
    need = pkv.decode_workspace_bytes(len(lens), hq, hkv, 128, 16, 4096, 256)
    ws = torch.empty(need, dtype=torch.uint8, device=dev)
    pool = host_pool_bits(wl.kv)
    qg = torch.Generator(device=dev).manual_seed(7)
    for call in range(4):
        q = torch.randn(wl.q.shape, generator=qg, device=dev).to(dtype)
        ws.view(torch.float32).fill_(float("nan"))
        out = pkv.paged_attention_decode(q, k_cache, v_cache, wl.block_tables, wl.context_lens,
                                         wl.scale, max_context_len=4096, partition_size=256,
                                         workspace=ws)
        torch.cuda.synchronize()
        check_no_device_flags(dev)
        ref = oracle_decode(to_bits(q.cpu()), pool, wl.block_tables.cpu(), wl.context_lens.cpu(),
                            hkv, 16, wl.scale, dtype)
        assert_close(out, ref, what=f"split decode, call {call}")


@pytest.mark.parametrize("bs", [8, 32])
def test_decode_partition_equal_to_block(bs):
    dev = device()
    lens = [3 * bs + 1, bs, 1, 7 * bs]
    wl = make_decode_workload(num_seqs=4, num_q_heads=8, num_kv_heads=8, head_dim=64,
                              block_size=bs, context_lens=lens, dtype=torch.float16, seed=bs,
                              device=str(dev))
    _check_step(wl, partition_size=bs)


def test_decode_empty_context_gives_zero_row():
    dev = device()
    wl = make_decode_workload(num_seqs=3, num_q_heads=4, num_kv_heads=2, head_dim=64,
                              block_size=16, context_lens=[5, 1, 40], dtype=torch.float16,
                              seed=3, device=str(dev))
    wl.context_lens[1] = 0
    k_cache, v_cache = pkv.split_pool(wl.kv)
    for part in (0, 16):
        out = pkv.paged_attention_decode(wl.q, k_cache, v_cache, wl.block_tables, wl.context_lens,
                                         wl.scale, max_context_len=40, partition_size=part)
        torch.cuda.synchronize()
        check_no_device_flags(dev)
        assert torch.all(out[1] == 0)
        ref = oracle_decode(to_bits(wl.q.cpu()), host_pool_bits(wl.kv), wl.block_tables.cpu(),
                            wl.context_lens.cpu(), 2, 16, wl.scale, wl.dtype)
        assert_close(out, ref)


def test_decode_full_table_and_many_sequences():
    """Contexts that fill their whole table (maximum length) and a grid of many sequences."""
    dev = device()
    n = 300
    g = torch.Generator().manual_seed(5)
    lens = torch.randint(1, 97, (n,), generator=g).tolist()
    lens[0] = 96
    wl = make_decode_workload(num_seqs=n, num_q_heads=8, num_kv_heads=1, head_dim=128,
                              block_size=32, context_lens=lens, dtype=torch.bfloat16, seed=6,
                              device=str(dev), max_blocks_per_seq=3)
    _check_step(wl)
    _check_step(wl, partition_size=32)


def test_decode_extreme_scores_stay_finite():
    """Large-magnitude q and K (scores in the hundreds) must not overflow the fp32 path."""
    dev = device()
    wl = make_decode_workload(num_seqs=4, num_q_heads=8, num_kv_heads=2, head_dim=128,
                              block_size=16, context_lens=[700, 64, 1, 333], dtype=torch.bfloat16,
                              seed=8, device=str(dev))
    wl.q.mul_(12.0)
    wl.kv[:, 0].mul_(4.0)
    _check_step(wl)
    _check_step(wl, partition_size=64)


@pytest.mark.parametrize("longest", [2047, 2100], ids=["2047", "2100"])
def test_decode_output_is_independent_of_block_placement(longest):
    """Moving every block to another physical slot leaves the output bitwise unchanged."""
    dev = device()
    wl = make_decode_workload(num_seqs=6, num_q_heads=32, num_kv_heads=8, head_dim=128,
                              block_size=16, context_lens=[1, 100, 1000, longest, 16, 555],
                              dtype=torch.float16, seed=9, device=str(dev))
    k_cache, v_cache = pkv.split_pool(wl.kv)
    outs = []
    for part in (0, 128):
        a = pkv.paged_attention_decode(wl.q, k_cache, v_cache, wl.block_tables, wl.context_lens,
                                       wl.scale, max_context_len=longest, partition_size=part)
        perm = torch.randperm(wl.num_blocks, generator=torch.Generator().manual_seed(part))
        perm = perm.to(dev)
        kv2 = torch.empty_like(wl.kv)
        kv2[perm] = wl.kv
        bt2 = perm[wl.block_tables.long()].to(torch.int32)
        k2, v2 = pkv.split_pool(kv2)
        b = pkv.paged_attention_decode(wl.q, k2, v2, bt2, wl.context_lens, wl.scale,
                                       max_context_len=longest, partition_size=part)
        torch.cuda.synchronize()
        assert torch.equal(a, b)
        outs.append(a)
    check_no_device_flags(dev)


def test_shared_prefix_reads_like_private_copies():
    """Tables pointing at one shared prefix vs private copies of it: bitwise equal."""
    dev = device()
    wl = make_decode_workload(num_seqs=5, num_q_heads=16, num_kv_heads=4, head_dim=128,
                              block_size=32, context_lens=[300, 257, 500, 256, 1000],
                              dtype=torch.bfloat16, seed=10, device=str(dev),
                              shared_prefix_tokens=256, num_blocks=200)
    k_cache, v_cache = pkv.split_pool(wl.kv)
    shared = pkv.paged_attention_decode(wl.q, k_cache, v_cache, wl.block_tables, wl.context_lens,
                                        wl.scale, max_context_len=1000)
    # give every sequence but the first private copies of the 8 prefix blocks
    used = set(wl.block_tables.cpu().flatten().tolist())
    free = [b for b in range(wl.num_blocks) if b not in used]
    pairs, tables = [], wl.block_tables.clone()
    for i in range(1, 5):
        for j in range(8):
            dst = free.pop()
            pairs.append([int(wl.block_tables[i, j]), dst])
            tables[i, j] = dst
    pkv.copy_blocks(k_cache, v_cache, torch.tensor(pairs, dtype=torch.int64, device=dev))
    private = pkv.paged_attention_decode(wl.q, k_cache, v_cache, tables, wl.context_lens,
                                         wl.scale, max_context_len=1000)
    torch.cuda.synchronize()
    check_no_device_flags(dev)
    assert torch.equal(shared, private)
    ref = oracle_decode(to_bits(wl.q.cpu()), host_pool_bits(wl.kv), tables.cpu(),
                        wl.context_lens.cpu(), 4, 32, wl.scale, wl.dtype)
    assert_close(private, ref)


def test_decode_runs_on_the_current_stream():
    dev = device()
    wl = make_decode_workload(num_seqs=4, num_q_heads=8, num_kv_heads=8, head_dim=64,
                              block_size=16, context_lens=[64, 1, 200, 33], dtype=torch.float16,
                              seed=11, device=str(dev))
    s = torch.cuda.Stream(dev)
    k_cache, v_cache = pkv.split_pool(wl.kv)
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        out = pkv.paged_attention_decode(wl.q, k_cache, v_cache, wl.block_tables,
                                         wl.context_lens, wl.scale, max_context_len=200)
    s.synchronize()
    ref = oracle_decode(to_bits(wl.q.cpu()), host_pool_bits(wl.kv), wl.block_tables.cpu(),
                        wl.context_lens.cpu(), 8, 16, wl.scale, wl.dtype)
    assert_close(out, ref)
