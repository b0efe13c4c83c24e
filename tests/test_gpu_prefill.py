"""GPU parity of chunked prefill attention against the oracle
("大模型 (LLM) 推理加速核心技术解析" §2 causal attention with a cache; "KV Cache从原理到实战"
§2.3 / §5.4): within |got-ref| <= 5e-3 + 1e-2|ref| over GQA groups 1..16, every
block size, both 16-bit types, ragged chunks (1 token, tile edges, several row
tiles), whole prompts of one length, empty caches and long cached prefixes, forced
KV splits, empty chunks, rows outside any chunk, out-of-contract lengths (flagged,
not written), and the full-size prefill workloads on sampled rows."""
import numpy as np
import pytest
import torch

import paged_kv_cache_155_gb300 as pkv
from paged_kv_cache_155_gb300 import workloads
from paged_kv_cache_155_gb300.workloads import make_prefill_workload
from tests._gpu_helpers import (assert_close, check_no_device_flags, device, host_pool_bits,
                                oracle_prefill_step, poison_unused_slots, run_prefill)

pytestmark = pytest.mark.gpu


def _check(wl, kv_splits=0):
    dev = wl.kv.device
    pool = host_pool_bits(wl.kv)
    out = run_prefill(wl, kv_splits)
    torch.cuda.synchronize()
    check_no_device_flags(dev)
    ref = oracle_prefill_step(pool, wl)
    n = int(wl.query_start[-1])
    assert np.array_equal(host_pool_bits(wl.kv), pool), "chunk K/V write not bit-exact"
    err = assert_close(out[:n], ref, what="prefill")
    if out.shape[0] > n:  # rows outside every chunk stay untouched
        assert torch.all(out[n:] == 0)
    return err


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16], ids=["f16", "bf16"])
@pytest.mark.parametrize("bs", [8, 16, 32])
@pytest.mark.parametrize("hq,hkv", [(4, 4), (8, 4), (16, 4), (32, 4), (64, 4), (12, 4)])
def test_prefill_shapes(dtype, bs, hq, hkv):
    dev = device()
    cached = [0, 5, 200, 0, 37]
    chunks = [1, 127, 129, 300, 64]
    wl = make_prefill_workload(num_q_heads=hq, num_kv_heads=hkv, head_dim=128, block_size=bs,
                               cached_lens=cached, chunk_lens=chunks, dtype=dtype,
                               seed=hq + bs, device=str(dev))
    _check(wl)


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16], ids=["f16", "bf16"])
@pytest.mark.parametrize("hq,hkv,prompt", [(8, 8, 256), (8, 8, 300), (32, 8, 512), (32, 8, 333),
                                           (48, 8, 200), (64, 8, 129)])
def test_prefill_whole_prompts_of_one_length(dtype, hq, hkv, prompt):
    """Whole prompts of one length on an empty cache (the (sequence, KV head)-major order of
    row-tile pairs): full row tiles leave through the output tensor map, a last row tile that
    reaches past its chunk row by row (prompt not a multiple of 128 / G tokens; G = 6 leaves
    rows R..127 of every tile unused)."""
    dev = device()
    wl = make_prefill_workload(num_q_heads=hq, num_kv_heads=hkv, head_dim=128, block_size=16,
                               cached_lens=[0] * 5, chunk_lens=[prompt] * 5, dtype=dtype,
                               seed=hq + prompt, device=str(dev))
    _check(wl)


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16], ids=["f16", "bf16"])
@pytest.mark.parametrize("bs", [8, 16, 32])
def test_prefill_ignores_nonfinite_unused_slots(dtype, bs):
    """NaN / Inf in every slot past each context (the chunk's K/V rows are written over
    theirs first) and in unused blocks: the output is the oracle's."""
    dev = device()
    wl = make_prefill_workload(num_q_heads=32, num_kv_heads=8, head_dim=128, block_size=bs,
                               cached_lens=[0, 5, 130, 37], chunk_lens=[1, 127, 129, 64],
                               dtype=dtype, seed=bs + 70, device=str(dev))
    poison_unused_slots(wl.kv, wl.block_tables, wl.context_lens, bs)
    _check(wl)
    _check(wl, kv_splits=2)


@pytest.mark.parametrize("splits", [1, 2, 3, 7])
def test_prefill_forced_kv_splits(splits):
    dev = device()
    wl = make_prefill_workload(num_q_heads=16, num_kv_heads=2, head_dim=128, block_size=16,
                               cached_lens=[1000, 0, 513, 2047], chunk_lens=[40, 700, 1, 130],
                               dtype=torch.bfloat16, seed=splits, device=str(dev))
    _check(wl, kv_splits=splits)


def test_prefill_one_token_chunks_match_decode():
    """Chunks of one token: the prefill call and the decode call compute the same
    attention (each checked against the oracle)."""
    dev = device()
    wl = make_prefill_workload(num_q_heads=32, num_kv_heads=8, head_dim=128, block_size=16,
                               cached_lens=[0, 99, 4095, 2000], chunk_lens=[1, 1, 1, 1],
                               dtype=torch.float16, seed=3, device=str(dev))
    out = run_prefill(wl)
    k_cache, v_cache = pkv.split_pool(wl.kv)
    dec = pkv.paged_attention_decode(wl.q, k_cache, v_cache, wl.block_tables, wl.context_lens,
                                     wl.scale, max_context_len=wl.max_context_len)
    torch.cuda.synchronize()
    check_no_device_flags(dev)
    ref = oracle_prefill_step(host_pool_bits(wl.kv), wl)  # rewrites the same rows
    assert_close(out, ref, what="prefill")
    assert_close(dec, ref, what="decode")


def test_prefill_empty_chunks_and_padding_rows():
    dev = device()
    wl = make_prefill_workload(num_q_heads=8, num_kv_heads=8, head_dim=128, block_size=8,
                               cached_lens=[10, 0, 300, 7], chunk_lens=[0, 50, 0, 3],
                               dtype=torch.float16, seed=4, device=str(dev), extra_rows=5)
    _check(wl)
    _check(wl, kv_splits=2)


def test_prefill_is_independent_of_block_placement():
    dev = device()
    wl = make_prefill_workload(num_q_heads=32, num_kv_heads=8, head_dim=128, block_size=16,
                               cached_lens=[300, 0, 1500], chunk_lens=[200, 129, 64],
                               dtype=torch.bfloat16, seed=5, device=str(dev))
    a = run_prefill(wl)
    perm = torch.randperm(wl.num_blocks, generator=torch.Generator().manual_seed(1)).to(dev)
    kv2 = torch.empty_like(wl.kv)
    kv2[perm] = wl.kv
    k2, v2 = pkv.split_pool(kv2)
    bt2 = perm[wl.block_tables.long()].to(torch.int32)
    b = pkv.paged_attention_prefill(wl.q, k2, v2, bt2, wl.query_start, wl.context_lens, wl.scale,
                                    max_query_len=wl.max_query_len,
                                    max_context_len=wl.max_context_len)
    torch.cuda.synchronize()
    check_no_device_flags(dev)
    assert torch.equal(a, b)


def test_prefill_extreme_scores_stay_finite():
    dev = device()
    wl = make_prefill_workload(num_q_heads=8, num_kv_heads=2, head_dim=128, block_size=16,
                               cached_lens=[600, 0], chunk_lens=[300, 260], dtype=torch.bfloat16,
                               seed=6, device=str(dev))
    wl.q.mul_(12.0)
    wl.kv[:, 0].mul_(4.0)
    wl.k_new.mul_(4.0)
    _check(wl)


def test_prefill_flags_out_of_contract_lengths():
    """A context shorter than its chunk and a chunk above max_query_len raise the
    context-length flag; those sequences' rows are not written, the others are."""
    dev = device()
    wl = make_prefill_workload(num_q_heads=8, num_kv_heads=4, head_dim=128, block_size=16,
                               cached_lens=[0, 100, 50], chunk_lens=[20, 30, 40],
                               dtype=torch.float16, seed=7, device=str(dev))
    k_cache, v_cache = pkv.split_pool(wl.kv)
    lens = wl.context_lens.clone()
    lens[1] = 10                                     # < its chunk of 30
    out = torch.zeros_like(wl.q)
    pkv.paged_attention_prefill(wl.q, k_cache, v_cache, wl.block_tables, wl.query_start, lens,
                                wl.scale, out, max_query_len=40,
                                max_context_len=wl.max_context_len)
    flags, names = pkv.get_device_error(dev)
    assert names == ["context_len"]
    assert torch.all(out[20:50] == 0) and not torch.all(out[:20] == 0)


def _sample_rows(wl):
    rows = []
    for i, c in enumerate(wl.chunk_lens):
        if c:
            rows += [(i, 0), (i, c // 2), (i, c - 1)]
    return rows


@pytest.mark.parametrize("name", ["prefill7b", "chunked70b"])
def test_prefill_named_workload_full_size(name):
    dev = device()
    wl = workloads.PREFILL_NAMED[name](device=str(dev))
    pool = host_pool_bits(wl.kv)
    out = run_prefill(wl)
    torch.cuda.synchronize()
    check_no_device_flags(dev)
    rows = _sample_rows(wl)
    ref = oracle_prefill_step(pool, wl, rows=rows)
    assert np.array_equal(host_pool_bits(wl.kv), pool), "chunk K/V write not bit-exact"
    qs = wl.query_start.cpu().tolist()
    got = torch.stack([out[qs[i] + j] for i, j in rows])
    assert_close(got, ref, what=name)
