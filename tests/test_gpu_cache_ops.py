"""GPU parity of the byte-moving ops (bit-exact vs the oracle) and the device
status word: out-of-range device indices are skipped and flagged, a bounded
wait that runs out reports a timeout, and the context stays usable."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_155_gb300 as pkv
from tests._gpu_helpers import check_no_device_flags, device, host_pool_bits
from tests._paged_helpers import to_bits

pytestmark = pytest.mark.gpu


def _pool(dev, nb, hkv, bs, d, dtype, seed):
    g = torch.Generator(device=dev).manual_seed(seed)
    return torch.randn((nb, 2, hkv, bs, d), generator=g, device=dev).to(dtype)


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16], ids=["f16", "bf16"])
@pytest.mark.parametrize("hkv,bs,d", [(4, 16, 64), (8, 16, 128), (32, 16, 128), (8, 32, 128),
                                      (2, 8, 64), (64, 8, 128)])
def test_reshape_and_cache_bit_exact(dtype, hkv, bs, d):
    dev = device()
    nb, t = 40, 57
    kv = _pool(dev, nb, hkv, bs, d, dtype, seed=hkv + bs)
    g = torch.Generator(device=dev).manual_seed(1)
    k_new = torch.randn((t, hkv, d), generator=g, device=dev).to(dtype)
    v_new = torch.randn((t, hkv, d), generator=g, device=dev).to(dtype)
    slots = torch.randperm(nb * bs, generator=torch.Generator().manual_seed(2))[:t]
    slots[::7] = -1                                     # padding tokens
    slots = slots.to(torch.int64)
    pool = host_pool_bits(kv)
    k_cache, v_cache = pkv.split_pool(kv)
    pkv.reshape_and_cache(k_new, v_new, slots.to(dev), k_cache, v_cache)
    torch.cuda.synchronize()
    check_no_device_flags(dev)
    oracle.reshape_and_cache(to_bits(k_new.cpu()), to_bits(v_new.cpu()), slots.numpy(), pool,
                             hkv, bs, d)
    assert np.array_equal(host_pool_bits(kv), pool)


def test_reshape_and_cache_worked_example_positions():
    """Positions 0, 15, 16, 99 of the 100-token table [7,2,9,1,5,8,3] land at
    (block, offset) = (7,0), (7,15), (2,0), (3,3)."""
    dev = device()
    kv = _pool(dev, 12, 4, 16, 64, torch.float16, seed=3)
    table = torch.tensor([[7, 2, 9, 1, 5, 8, 3]] * 4, dtype=torch.int32)
    pos = torch.tensor([0, 15, 16, 99])
    slots = pkv.slot_mapping(table, pos, 16)
    k_new = torch.randn((4, 4, 64), device=dev).half()
    v_new = torch.randn((4, 4, 64), device=dev).half()
    k_cache, v_cache = pkv.split_pool(kv)
    pkv.reshape_and_cache(k_new, v_new, slots.to(dev), k_cache, v_cache)
    torch.cuda.synchronize()
    for n, (blk, off) in enumerate([(7, 0), (7, 15), (2, 0), (3, 3)]):
        assert torch.equal(kv[blk, 0, :, off], k_new[n])
        assert torch.equal(kv[blk, 1, :, off], v_new[n])


def test_slot_mapping_kernel_worked_example_and_oracle():
    """pkv_slot_mapping on the device: the worked table [7,2,9,1,5,8,3] puts positions
    0 / 15 / 16 / 99 at slots of (7,0), (7,15), (2,0), (3,3); random tables and token
    rows match the oracle's slot rule exactly; negative positions give -1."""
    dev = device()
    table = torch.tensor([[7, 2, 9, 1, 5, 8, 3]], dtype=torch.int32, device=dev)
    pos = torch.tensor([0, 15, 16, 99, -1], device=dev)
    rows = torch.zeros(5, dtype=torch.int64, device=dev)
    got = pkv.slot_mapping(table, pos, 16, token_rows=rows, num_blocks=10).cpu().tolist()
    assert got == [7 * 16, 7 * 16 + 15, 2 * 16, 3 * 16 + 3, -1]
    g = torch.Generator().manual_seed(9)
    for bs in (8, 16, 32):
        tables = torch.randint(0, 5000, (37, 64), generator=g, dtype=torch.int32)
        pos = torch.randint(-2, 64 * bs, (1000,), generator=g)
        rows = torch.randint(0, 37, (1000,), generator=g)
        got = pkv.slot_mapping(tables.to(dev), pos.to(dev), bs, token_rows=rows.to(dev),
                               num_blocks=5000)
        torch.cuda.synchronize()
        check_no_device_flags(dev)
        ref = [-1 if p < 0 else oracle.slot_for_position(tables[r].numpy(), int(p), bs)
               for r, p in zip(rows.tolist(), pos.tolist())]
        assert got.cpu().tolist() == ref
        host = pkv.slot_mapping(tables, pos, bs, token_rows=rows, num_blocks=5000)
        assert host.tolist() == ref


def test_slot_mapping_kernel_flags_bad_inputs():
    dev = device()
    tables = torch.tensor([[3, 1], [0, 2]], dtype=torch.int32, device=dev)
    for pos, rows, nb, flag in (([32, 1], None, 4, "slot"), ([1, 17], None, 2, "block_table"),
                                ([1, 1], [0, 2], 4, "slot")):
        r = None if rows is None else torch.tensor(rows, device=dev)
        got = pkv.slot_mapping(tables, torch.tensor(pos, device=dev), 16, token_rows=r,
                               num_blocks=nb)
        flags, names = pkv.get_device_error(dev)
        assert flag in names
        assert -1 in got.cpu().tolist()
    check_no_device_flags(dev)


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16], ids=["f16", "bf16"])
@pytest.mark.parametrize("hkv,bs,d", [(8, 32, 128), (4, 16, 64), (32, 16, 128), (1, 8, 64)])
def test_copy_blocks_bit_exact(dtype, hkv, bs, d):
    dev = device()
    nb = 300
    kv = _pool(dev, nb, hkv, bs, d, dtype, seed=hkv * bs)
    perm = torch.randperm(nb, generator=torch.Generator().manual_seed(4))
    src, dst = perm[:100], perm[100:228]
    pairs = torch.stack([src[torch.arange(128) % 100], dst], 1).to(torch.int64)  # sources repeat
    pool = host_pool_bits(kv)
    k_cache, v_cache = pkv.split_pool(kv)
    pkv.copy_blocks(k_cache, v_cache, pairs.to(dev))
    torch.cuda.synchronize()
    check_no_device_flags(dev)
    oracle.copy_blocks(pool, pairs.numpy(), hkv, bs, d)
    assert np.array_equal(host_pool_bits(kv), pool)


def test_bad_slot_is_flagged_and_skipped():
    dev = device()
    kv = _pool(dev, 8, 2, 16, 64, torch.float16, seed=5)
    before = kv.clone()
    k_cache, v_cache = pkv.split_pool(kv)
    kn = torch.randn((2, 2, 64), device=dev).half()
    slots = torch.tensor([8 * 16, 10**9], dtype=torch.int64, device=dev)   # both out of range
    pkv.reshape_and_cache(kn, kn, slots, k_cache, v_cache)
    flags, names = pkv.get_device_error(dev)
    assert names == ["slot"]
    assert torch.equal(kv, before)
    check_no_device_flags(dev)       # the read cleared the word


def test_bad_copy_pair_is_flagged_and_skipped():
    dev = device()
    kv = _pool(dev, 8, 2, 16, 64, torch.bfloat16, seed=6)
    before = kv.clone()
    k_cache, v_cache = pkv.split_pool(kv)
    pairs = torch.tensor([[1, 8], [-1, 2], [3, 4]], dtype=torch.int64, device=dev)
    pkv.copy_blocks(k_cache, v_cache, pairs)
    flags, names = pkv.get_device_error(dev)
    assert names == ["copy_pair"]
    after = kv.clone()
    assert torch.equal(after[4], before[3])            # the valid pair ran
    mask = torch.ones(8, dtype=torch.bool)
    mask[4] = False
    assert torch.equal(after[mask], before[mask])


def test_bad_block_table_entry_and_length_are_flagged():
    dev = device()
    kv = _pool(dev, 16, 2, 16, 64, torch.float16, seed=7)
    k_cache, v_cache = pkv.split_pool(kv)
    q = torch.randn((2, 4, 64), device=dev).half()
    tables = torch.tensor([[0, 1, 99], [2, 3, 4]], dtype=torch.int32, device=dev)
    lens = torch.tensor([40, 30], dtype=torch.int32, device=dev)
    out = pkv.paged_attention_decode(q, k_cache, v_cache, tables, lens, 0.125, max_context_len=48)
    flags, names = pkv.get_device_error(dev)
    assert names == ["block_table"]
    assert torch.isfinite(out.float()).all()
    lens2 = torch.tensor([40, 47], dtype=torch.int32, device=dev)
    pkv.paged_attention_decode(q, k_cache, v_cache, tables[1:].repeat(2, 1), lens2, 0.125,
                               max_context_len=45)
    flags, names = pkv.get_device_error(dev)
    assert names == ["context_len"]


def test_bounded_wait_times_out_and_the_context_survives():
    dev = device()
    pkv.debug_wait_timeout(50_000_000, dev)            # 50 ms on a barrier nothing completes
    flags, names = pkv.get_device_error(dev)
    assert names == ["timeout"]
    # the context is still usable
    x = torch.arange(10, device=dev)
    assert int(x.sum().item()) == 45
    check_no_device_flags(dev)
