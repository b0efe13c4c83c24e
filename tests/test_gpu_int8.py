"""GPU parity of the INT8 KV cache (per-channel scales, "KV Cache从原理到实战" §5.2)
against the oracle: the quantising cache write is bit-exact (every fp16 and
bf16 bit pattern, ragged slot sets, padding), block copies are bit-exact, and
decode over INT8 pools matches the oracle's dequantise-then-attend definition
within |got-ref| <= 5e-3 + 1e-2|ref| for every supported shape, forced
partitions, empty contexts and the full-size INT8 workloads."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_155_gb300 as pkv
from paged_kv_cache_155_gb300 import workloads
from paged_kv_cache_155_gb300.workloads import make_decode_workload
from tests._gpu_helpers import (assert_close, check_no_device_flags, device, oracle_decode_int8,
                                oracle_step_pool_int8, run_step_int8)
from tests._paged_helpers import dtype_code, to_bits

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16], ids=["f16", "bf16"])
def test_quantiser_every_bit_pattern(dtype):
    """All 65536 16-bit patterns (NaN, inf, subnormals included) quantised with
    per-channel scales spanning 2^-20 .. 2^10: codes bit-exact vs the oracle."""
    dev = device()
    hkv, d, bs = 4, 128, 16
    per_tok = hkv * d
    t = 65536 // per_tok                                    # 128 tokens hold every pattern once
    pats = torch.randperm(65536, generator=torch.Generator().manual_seed(0)).to(torch.int32)
    rows = pats.to(torch.int16).view(dtype).reshape(t, hkv, d)
    g = torch.Generator().manual_seed(1)
    k_scale = torch.exp2(torch.empty(hkv, d).uniform_(-20, 10, generator=g)).float()
    v_scale = torch.exp2(torch.empty(hkv, d).uniform_(-4, 2, generator=g)).float()
    nb = t // bs
    kv = torch.zeros((nb, 2, hkv, bs, d), dtype=torch.int8, device=dev)
    k_cache, v_cache = pkv.split_pool(kv)
    slots = torch.arange(t, dtype=torch.int64)
    pkv.reshape_and_cache_int8(rows.to(dev), rows.flip(0).contiguous().to(dev), slots.to(dev),
                               k_cache, v_cache, k_scale.to(dev), v_scale.to(dev))
    torch.cuda.synchronize()
    check_no_device_flags(dev)
    pool = np.zeros(kv.shape, dtype=np.int8)
    oracle.reshape_and_cache_int8(to_bits(rows), to_bits(rows.flip(0)), slots.numpy(), pool,
                                  k_scale.numpy(), v_scale.numpy(), hkv, bs, d, dtype_code(dtype))
    assert np.array_equal(kv.cpu().numpy(), pool)


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16], ids=["f16", "bf16"])
@pytest.mark.parametrize("hkv,bs,d", [(4, 16, 64), (8, 16, 128), (32, 16, 128), (8, 32, 128),
                                      (2, 8, 64), (64, 8, 128)])
def test_reshape_and_cache_int8_bit_exact(dtype, hkv, bs, d):
    dev = device()
    nb, t = 40, 57
    g = torch.Generator(device=dev).manual_seed(hkv + bs)
    kv = torch.randint(-127, 128, (nb, 2, hkv, bs, d), generator=g, device=dev, dtype=torch.int8)
    k_new = torch.randn((t, hkv, d), generator=g, device=dev).to(dtype)
    v_new = (3 * torch.randn((t, hkv, d), generator=g, device=dev)).to(dtype)
    k_scale = torch.rand((hkv, d), generator=g, device=dev) * 0.05 + 0.001
    v_scale = torch.rand((hkv, d), generator=g, device=dev) * 0.05 + 0.001
    slots = torch.randperm(nb * bs, generator=torch.Generator().manual_seed(2))[:t]
    slots[::7] = -1                                     # padding tokens
    slots = slots.to(torch.int64)
    pool = kv.cpu().numpy().copy()
    k_cache, v_cache = pkv.split_pool(kv)
    pkv.reshape_and_cache_int8(k_new, v_new, slots.to(dev), k_cache, v_cache, k_scale, v_scale)
    torch.cuda.synchronize()
    check_no_device_flags(dev)
    oracle.reshape_and_cache_int8(to_bits(k_new.cpu()), to_bits(v_new.cpu()), slots.numpy(), pool,
                                  k_scale.cpu().numpy(), v_scale.cpu().numpy(), hkv, bs, d,
                                  dtype_code(dtype))
    assert np.array_equal(kv.cpu().numpy(), pool)


def test_reshape_and_cache_int8_flags_bad_slot():
    dev = device()
    kv = torch.zeros((4, 2, 2, 8, 64), dtype=torch.int8, device=dev)
    k_cache, v_cache = pkv.split_pool(kv)
    rows = torch.ones((2, 2, 64), dtype=torch.float16, device=dev)
    sc = torch.full((2, 64), 0.5, device=dev)
    pkv.reshape_and_cache_int8(rows, rows, torch.tensor([3, 32], device=dev), k_cache, v_cache,
                               sc, sc)
    flags, names = pkv.get_device_error(dev)
    assert names == ["slot"]
    assert torch.all(kv[0, :, :, 3] == 2) and int(kv.abs().sum()) == 2 * 2 * 64 * 2


def test_copy_blocks_int8_bit_exact():
    dev = device()
    g = torch.Generator(device=dev).manual_seed(4)
    kv = torch.randint(-127, 128, (30, 2, 8, 16, 128), generator=g, device=dev, dtype=torch.int8)
    pool = kv.cpu().numpy().copy()
    pairs = torch.tensor([[1, 7], [2, 9], [29, 0], [5, 6]], dtype=torch.int64)
    k_cache, v_cache = pkv.split_pool(kv)
    pkv.copy_blocks(k_cache, v_cache, pairs.to(dev))
    torch.cuda.synchronize()
    check_no_device_flags(dev)
    oracle.copy_blocks_bytes(pool, pairs.numpy())
    assert np.array_equal(kv.cpu().numpy(), pool)


def _check_step(wl, partition_size=0):
    dev = wl.kv.device
    pool = wl.kv.cpu().numpy().copy()
    out = run_step_int8(wl, partition_size)
    torch.cuda.synchronize()
    check_no_device_flags(dev)
    oracle_step_pool_int8(pool, wl)
    assert np.array_equal(wl.kv.cpu().numpy(), pool), "INT8 cache write not bit-exact"
    return assert_close(out, oracle_decode_int8(wl, pool), what="int8 decode")


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16], ids=["f16", "bf16"])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("bs", [8, 16, 32])
@pytest.mark.parametrize("hq,hkv", [(4, 4), (8, 4), (16, 4), (32, 4), (12, 4), (24, 4), (64, 4)])
def test_int8_decode_shapes(dtype, d, bs, hq, hkv):
    dev = device()
    lens = [1, bs - 1, bs, bs + 1, 5 * bs + 3, 2100, 17]
    wl = make_decode_workload(num_seqs=len(lens), num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                              block_size=bs, context_lens=lens, dtype=dtype,
                              seed=hq * 7 + d + bs, device=str(dev), kv_dtype=torch.int8)
    _check_step(wl)


@pytest.mark.parametrize("partition", [16, 32, 48, 256, 1024])
def test_int8_decode_forced_partitions(partition):
    dev = device()
    lens = [1, 15, 16, 17, 511, 512, 513, 1500, 2049]
    wl = make_decode_workload(num_seqs=len(lens), num_q_heads=16, num_kv_heads=2, head_dim=128,
                              block_size=16, context_lens=lens, dtype=torch.bfloat16,
                              seed=partition, device=str(dev), kv_dtype=torch.int8)
    _check_step(wl, partition_size=partition)


def test_int8_decode_empty_context_and_extreme_scales():
    """A zero-length context gives a zero row; large scales (scores in the hundreds)
    stay finite."""
    dev = device()
    wl = make_decode_workload(num_seqs=3, num_q_heads=8, num_kv_heads=2, head_dim=128,
                              block_size=16, context_lens=[700, 1, 333], dtype=torch.float16,
                              seed=12, device=str(dev), kv_dtype=torch.int8)
    wl.k_scale.mul_(8.0)
    wl.q.mul_(6.0)
    _check_step(wl)
    wl.context_lens[1] = 0
    k_cache, v_cache = pkv.split_pool(wl.kv)
    for part in (0, 64):
        out = pkv.paged_attention_decode_int8(wl.q, k_cache, v_cache, wl.k_scale, wl.v_scale,
                                              wl.block_tables, wl.context_lens, wl.scale,
                                              max_context_len=700, partition_size=part)
        torch.cuda.synchronize()
        check_no_device_flags(dev)
        assert torch.all(out[1] == 0)
        assert_close(out, oracle_decode_int8(wl, wl.kv.cpu().numpy()), what="int8 empty")


def test_int8_decode_is_independent_of_block_placement():
    dev = device()
    wl = make_decode_workload(num_seqs=6, num_q_heads=32, num_kv_heads=8, head_dim=128,
                              block_size=16, context_lens=[1, 100, 1000, 2100, 16, 555],
                              dtype=torch.float16, seed=9, device=str(dev), kv_dtype=torch.int8)
    k_cache, v_cache = pkv.split_pool(wl.kv)
    for part in (0, 128):
        a = pkv.paged_attention_decode_int8(wl.q, k_cache, v_cache, wl.k_scale, wl.v_scale,
                                            wl.block_tables, wl.context_lens, wl.scale,
                                            max_context_len=2100, partition_size=part)
        perm = torch.randperm(wl.num_blocks, generator=torch.Generator().manual_seed(part)).to(dev)
        kv2 = torch.empty_like(wl.kv)
        kv2[perm] = wl.kv
        bt2 = perm[wl.block_tables.long()].to(torch.int32)
        k2, v2 = pkv.split_pool(kv2)
        b = pkv.paged_attention_decode_int8(wl.q, k2, v2, wl.k_scale, wl.v_scale, bt2,
                                            wl.context_lens, wl.scale, max_context_len=2100,
                                            partition_size=part)
        torch.cuda.synchronize()
        assert torch.equal(a, b)
    check_no_device_flags(dev)


def test_int8_shared_blocks_read_like_private_copies():
    dev = device()
    wl = make_decode_workload(num_seqs=5, num_q_heads=16, num_kv_heads=4, head_dim=128,
                              block_size=32, context_lens=[300, 257, 500, 256, 1000],
                              dtype=torch.bfloat16, seed=10, device=str(dev),
                              shared_prefix_tokens=256, num_blocks=200, kv_dtype=torch.int8)
    k_cache, v_cache = pkv.split_pool(wl.kv)
    args = (wl.k_scale, wl.v_scale)
    shared = pkv.paged_attention_decode_int8(wl.q, k_cache, v_cache, *args, wl.block_tables,
                                             wl.context_lens, wl.scale, max_context_len=1000)
    used = set(wl.block_tables.cpu().flatten().tolist())
    free = [b for b in range(wl.num_blocks) if b not in used]
    pairs, tables = [], wl.block_tables.clone()
    for i in range(1, 5):
        for j in range(8):
            dst = free.pop()
            pairs.append([int(wl.block_tables[i, j]), dst])
            tables[i, j] = dst
    pkv.copy_blocks(k_cache, v_cache, torch.tensor(pairs, dtype=torch.int64, device=dev))
    private = pkv.paged_attention_decode_int8(wl.q, k_cache, v_cache, *args, tables,
                                              wl.context_lens, wl.scale, max_context_len=1000)
    torch.cuda.synchronize()
    check_no_device_flags(dev)
    assert torch.equal(shared, private)
    assert_close(private, oracle_decode_int8(wl, wl.kv.cpu().numpy(), tables=tables))


def _sample(wl):
    lens = wl.context_lens.cpu()
    return sorted({0, wl.num_seqs // 2, wl.num_seqs - 1, int(lens.argmax()), int(lens.argmin())})


@pytest.mark.parametrize("name", ["mha7b_int8", "gqa7b_int8", "long70b_int8"])
def test_int8_named_workload_full_size(name):
    dev = device()
    wl = workloads.NAMED[name](device=str(dev))
    part = workloads.DEFAULT_PARTITION[name]
    pool = wl.kv.cpu().numpy().copy()
    out = run_step_int8(wl, part)
    torch.cuda.synchronize()
    check_no_device_flags(dev)
    oracle_step_pool_int8(pool, wl)
    assert np.array_equal(wl.kv.cpu().numpy(), pool), "INT8 cache write not bit-exact"
    sel = _sample(wl)
    assert_close(out[sel], oracle_decode_int8(wl, pool, sel=sel), what=name)


@pytest.mark.parametrize("qmag", [3e4, 1e-6], ids=["large", "tiny"])
def test_int8_grouped_query_range(qmag):
    """GQA over an INT8 pool runs as warp-level fp16 MMAs with the query folded into fp16
    (q * k_scale * 2^-e per head row): queries whose q * k_scale exceeds the fp16 range,
    or sits in its subnormals, still match the oracle (scale chosen to keep scores O(1))."""
    dev = device()
    wl = make_decode_workload(num_seqs=4, num_q_heads=32, num_kv_heads=8, head_dim=128,
                              block_size=16, context_lens=[2100, 1, 700, 2500],
                              dtype=torch.bfloat16, seed=21, device=str(dev), kv_dtype=torch.int8)
    wl.q.mul_(qmag)
    wl.scale = 1.0 / (qmag * 128 ** 0.5)
    _check_step(wl)
