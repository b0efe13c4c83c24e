"""The five named workloads (and the 16-head GQA shape) at full size, in the
launch configuration the benchmark times: the cache write is compared
bit-exactly over the whole pool, attention on sampled sequences against the
oracle (which computes them one by one), and the shared-prefix workload's
copy-on-write step is checked both bit-exactly and as an attention invariant
(before vs after the copies)."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_155_gb300 as pkv
from paged_kv_cache_155_gb300 import workloads
from tests._gpu_helpers import (assert_close, check_no_device_flags, device, host_pool_bits,
                                oracle_decode, oracle_step_pool, run_step)
from tests._paged_helpers import to_bits

pytestmark = pytest.mark.gpu


def _sample(wl):
    lens = wl.context_lens.cpu()
    sel = {0, wl.num_seqs // 2, wl.num_seqs - 1, int(lens.argmax()), int(lens.argmin())}
    return sorted(sel)


@pytest.mark.parametrize("name", ["tiny", "mha7b", "gqa7b", "long70b", "gqa16"])
def test_named_workload_full_size(name):
    dev = device()
    wl = workloads.NAMED[name](device=str(dev))
    part = workloads.DEFAULT_PARTITION[name]
    pool = host_pool_bits(wl.kv)
    out = run_step(wl, part)
    torch.cuda.synchronize()
    check_no_device_flags(dev)
    oracle_step_pool(pool, wl)
    assert np.array_equal(host_pool_bits(wl.kv), pool), "cache write not bit-exact"
    sel = list(range(wl.num_seqs)) if name == "tiny" else _sample(wl)
    ref = oracle_decode(to_bits(wl.q.cpu())[sel], pool, wl.block_tables.cpu()[sel],
                        wl.context_lens.cpu()[sel], wl.num_kv_heads, wl.block_size, wl.scale,
                        wl.dtype)
    assert_close(out[sel], ref, what=name)


def test_tiny_uses_the_worked_example_table():
    wl = workloads.tiny()
    assert wl.block_tables[2, :7].tolist() == [7, 2, 9, 1, 5, 8, 3]
    assert int(wl.context_lens[2]) == 100


def test_prefix_workload_copy_on_write():
    dev = device()
    wl = workloads.prefix(device=str(dev))
    k_cache, v_cache = pkv.split_pool(wl.kv)
    maxl = int(wl.context_lens.max())
    before = pkv.paged_attention_decode(wl.q, k_cache, v_cache, wl.block_tables, wl.context_lens,
                                        wl.scale, max_context_len=maxl)
    pool = host_pool_bits(wl.kv)
    pkv.copy_blocks(k_cache, v_cache, wl.cow_pairs)
    after = pkv.paged_attention_decode(wl.q, k_cache, v_cache, wl.block_tables_after_cow,
                                       wl.context_lens, wl.scale, max_context_len=maxl)
    torch.cuda.synchronize()
    check_no_device_flags(dev)
    oracle.copy_blocks(pool, wl.cow_pairs.cpu().numpy(), wl.num_kv_heads, wl.block_size,
                       wl.head_dim)
    assert np.array_equal(host_pool_bits(wl.kv), pool), "copy_blocks not bit-exact"
    assert torch.equal(before, after), "COW copies changed the attention result"
    # then the decode step proper (cache write + attention) on the post-COW tables
    out = run_step(wl, 0, tables=wl.block_tables_after_cow)
    torch.cuda.synchronize()
    check_no_device_flags(dev)
    oracle_step_pool(pool, wl, tables=wl.block_tables_after_cow)
    assert np.array_equal(host_pool_bits(wl.kv), pool)
    sel = _sample(wl)
    ref = oracle_decode(to_bits(wl.q.cpu())[sel], pool, wl.block_tables_after_cow.cpu()[sel],
                        wl.context_lens.cpu()[sel], wl.num_kv_heads, wl.block_size, wl.scale,
                        wl.dtype)
    assert_close(out[sel], ref, what="prefix")
