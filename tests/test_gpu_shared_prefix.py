"""GPU parity of the shared-prefix (cascade) decode against the oracle's plain
definition: the cascade must give the same attention as decoding each sequence
over its whole table.  Covers query-row counts that are not a multiple of 128,
prefixes that end inside a 128-token tile, MHA and GQA groups (the suffix pass
then runs per-lane loops or warp-level MMAs), both dtypes, all block sizes, forced
suffix partitions, empty suffixes, and the full shared-prefix workload."""
import numpy as np
import pytest
import torch

import paged_kv_cache_155_gb300 as pkv
from paged_kv_cache_155_gb300 import workloads
from paged_kv_cache_155_gb300.workloads import make_decode_workload
from tests._gpu_helpers import (assert_close, check_no_device_flags, device, host_pool_bits,
                                oracle_decode, poison_unused_slots)
from tests._paged_helpers import to_bits

pytestmark = pytest.mark.gpu


def _cascade_vs_oracle(wl, prefix_tokens, partition=0, sel=None):
    dev = wl.kv.device
    k_cache, v_cache = pkv.split_pool(wl.kv)
    bs = wl.block_size
    prefix_table = wl.block_tables[0, :prefix_tokens // bs].contiguous()
    maxl = int(wl.context_lens.max())
    out = pkv.paged_attention_decode_shared_prefix(
        wl.q, k_cache, v_cache, prefix_table, prefix_tokens, wl.block_tables, wl.context_lens,
        wl.scale, max_context_len=maxl, partition_size=partition)
    plain = pkv.paged_attention_decode(wl.q, k_cache, v_cache, wl.block_tables, wl.context_lens,
                                       wl.scale, max_context_len=maxl)
    torch.cuda.synchronize()
    check_no_device_flags(dev)
    sel = list(range(wl.num_seqs)) if sel is None else sel
    ref = oracle_decode(to_bits(wl.q.cpu())[sel], host_pool_bits(wl.kv), wl.block_tables.cpu()[sel],
                        wl.context_lens.cpu()[sel], wl.num_kv_heads, bs, wl.scale, wl.dtype)
    assert_close(out[sel], ref, what="shared-prefix decode")
    assert_close(out[sel], plain[sel].float().cpu().double().numpy(), what="cascade vs plain")
    return out


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16], ids=["f16", "bf16"])
@pytest.mark.parametrize("hq,hkv", [(32, 8), (16, 2), (8, 8), (12, 4)])
@pytest.mark.parametrize("bs,prefix_blocks", [(16, 13), (32, 8), (8, 40)])
def test_shared_prefix_shapes(dtype, hq, hkv, bs, prefix_blocks):
    dev = device()
    prefix = prefix_blocks * bs
    g = torch.Generator().manual_seed(hq * bs + prefix)
    n = 9
    lens = (prefix + torch.randint(0, 3 * bs + 7, (n,), generator=g)).tolist()
    lens[0] = prefix + 1
    lens[1] = prefix            # empty suffix
    wl = make_decode_workload(num_seqs=n, num_q_heads=hq, num_kv_heads=hkv, head_dim=128,
                              block_size=bs, context_lens=lens, dtype=dtype, seed=prefix + hq,
                              device=str(dev), shared_prefix_tokens=prefix)
    _cascade_vs_oracle(wl, prefix)


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16], ids=["f16", "bf16"])
@pytest.mark.parametrize("bs", [8, 16, 32])
def test_shared_prefix_ignores_nonfinite_unused_slots(dtype, bs):
    """NaN / Inf in every slot past each context and in unused blocks: the prefix tiles
    (which load whole 128-token tiles) and the suffix pass still give the oracle's result."""
    dev = device()
    prefix = 9 * bs
    lens = [prefix + 1, prefix, prefix + bs + 3, prefix + 200, prefix + 5 * bs - 1]
    need = sum(-(-n // bs) for n in lens) - 4 * (prefix // bs)
    wl = make_decode_workload(num_seqs=5, num_q_heads=32, num_kv_heads=8, head_dim=128,
                              block_size=bs, context_lens=lens, dtype=dtype, seed=bs + 40,
                              device=str(dev), shared_prefix_tokens=prefix, num_blocks=need + 5)
    poison_unused_slots(wl.kv, wl.block_tables, wl.context_lens, bs)
    _cascade_vs_oracle(wl, prefix)


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16], ids=["f16", "bf16"])
def test_shared_prefix_merge_never_reads_stale_partials(dtype):
    """The prefix tiles and the suffix pass overlap on the GPU and the merge follows
    both: with the workspace filled with NaN before each call and new queries each
    time, every call must still give the oracle's result (a merge that ran ahead of
    either producer would read NaN or the previous call's partials)."""
    dev = device()
    g = torch.Generator().manual_seed(31)
    n, prefix = 64, 1024
    lens = (prefix + torch.randint(1, 1200, (n,), generator=g)).tolist()
    wl = make_decode_workload(num_seqs=n, num_q_heads=32, num_kv_heads=8, head_dim=128,
                              block_size=16, context_lens=lens, dtype=dtype, seed=32,
                              device=str(dev), shared_prefix_tokens=prefix)
    k_cache, v_cache = pkv.split_pool(wl.kv)
    maxl = int(wl.context_lens.max())
    need = pkv.shared_prefix_workspace_bytes(n, 32, 8, 128, 16, prefix, maxl)
    ws = torch.empty(need, dtype=torch.uint8, device=dev)
    pool = host_pool_bits(wl.kv)
    qg = torch.Generator(device=dev).manual_seed(33)
    for call in range(4):
        q = torch.randn(wl.q.shape, generator=qg, device=dev).to(dtype)
        ws.view(torch.float32).fill_(float("nan"))
        out = pkv.paged_attention_decode_shared_prefix(
            q, k_cache, v_cache, wl.block_tables[0, :prefix // 16].contiguous(), prefix,
            wl.block_tables, wl.context_lens, wl.scale, max_context_len=maxl, workspace=ws)
        torch.cuda.synchronize()
        check_no_device_flags(dev)
        ref = oracle_decode(to_bits(q.cpu()), pool, wl.block_tables.cpu(), wl.context_lens.cpu(),
                            8, 16, wl.scale, dtype)
        assert_close(out, ref, what=f"shared-prefix decode, call {call}")


@pytest.mark.parametrize("partition", [0, 64, 256])
def test_shared_prefix_many_rows_and_partitions(partition):
    """B*G = 4 * 50 = 200 query rows (two row tiles, the second partial), a
    1000-token prefix (7 full 128-token tiles + a partial one), long suffixes."""
    dev = device()
    g = torch.Generator().manual_seed(partition)
    n, prefix = 50, 1000
    lens = (prefix + torch.randint(1, 700, (n,), generator=g)).tolist()
    wl = make_decode_workload(num_seqs=n, num_q_heads=32, num_kv_heads=8, head_dim=128,
                              block_size=8, context_lens=lens, dtype=torch.bfloat16, seed=7,
                              device=str(dev), shared_prefix_tokens=prefix)
    _cascade_vs_oracle(wl, prefix, partition=partition)


def test_shared_prefix_large_scores_rescale():
    """Large scores make the reference maximum move across prefix tiles."""
    dev = device()
    wl = make_decode_workload(num_seqs=6, num_q_heads=16, num_kv_heads=4, head_dim=128,
                              block_size=16, context_lens=[1030, 1100, 1025, 1500, 1024, 1300],
                              dtype=torch.bfloat16, seed=11, device=str(dev),
                              shared_prefix_tokens=1024)
    wl.q.mul_(6.0)
    # increasing key magnitudes along the prefix force repeated rescales
    ramp = torch.linspace(0.5, 3.0, 1024 // 16, device=dev).to(torch.bfloat16)
    blocks = wl.block_tables[0, :64].long()
    wl.kv[blocks, 0] = wl.kv[blocks, 0] * ramp.view(-1, 1, 1, 1)
    wl.context_lens[0] = 1024
    _cascade_vs_oracle(wl, 1024)


def test_prefix_workload_full_size():
    dev = device()
    wl = workloads.prefix(device=str(dev))
    lens = wl.context_lens.cpu()
    sel = sorted({0, 1, 63, 64, wl.num_seqs - 1, int(lens.argmax()), int(lens.argmin())})
    pre = _cascade_vs_oracle(wl, 2048, sel=sel)
    # after the copy-on-write of the last prefix block the tables differ in that block,
    # but it holds the same data: the cascade over the original prefix blocks agrees
    k_cache, v_cache = pkv.split_pool(wl.kv)
    pkv.copy_blocks(k_cache, v_cache, wl.cow_pairs)
    post = pkv.paged_attention_decode_shared_prefix(
        wl.q, k_cache, v_cache, wl.block_tables[0, :64].contiguous(), 2048,
        wl.block_tables_after_cow, wl.context_lens, wl.scale,
        max_context_len=int(lens.max()))
    torch.cuda.synchronize()
    check_no_device_flags(dev)
    assert torch.equal(pre, post)


def test_shared_prefix_flags_a_sequence_shorter_than_the_prefix():
    dev = device()
    wl = make_decode_workload(num_seqs=3, num_q_heads=8, num_kv_heads=2, head_dim=128,
                              block_size=16, context_lens=[300, 260, 400], dtype=torch.float16,
                              seed=3, device=str(dev), shared_prefix_tokens=256)
    wl.context_lens[1] = 200
    k_cache, v_cache = pkv.split_pool(wl.kv)
    pkv.paged_attention_decode_shared_prefix(wl.q, k_cache, v_cache,
                                             wl.block_tables[0, :16].contiguous(), 256,
                                             wl.block_tables, wl.context_lens, wl.scale,
                                             max_context_len=400)
    flags, names = pkv.get_device_error(dev)
    assert "context_len" in names


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16], ids=["f16", "bf16"])
def test_shared_prefix_long_suffixes(dtype):
    """Suffixes up to 2500 tokens, several suffix partitions per sequence."""
    dev = device()
    g = torch.Generator().manual_seed(21)
    n, prefix = 12, 512
    lens = (prefix + torch.randint(1, 2500, (n,), generator=g)).tolist()
    lens[3] = prefix + 2500
    wl = make_decode_workload(num_seqs=n, num_q_heads=32, num_kv_heads=8, head_dim=128,
                              block_size=16, context_lens=lens, dtype=dtype, seed=22,
                              device=str(dev), shared_prefix_tokens=prefix)
    _cascade_vs_oracle(wl, prefix)
