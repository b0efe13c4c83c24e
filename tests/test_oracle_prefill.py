"""Pins for the oracle's chunked prefill attention.

"大模型 (LLM) 推理加速核心技术解析" §2: the new tokens' K/V join the cache and each
new query attends causally; "KV Cache从原理到实战" §2.3 / §5.4: prefill of a whole
prompt, and chunked prefill.  Pinned by:
  * a hand-computed two-token prompt (the first row sees only itself);
  * chunks of one token equal the separately pinned decode oracle;
  * a whole prompt equals torch's fp64 causal scaled_dot_product_attention on the
    dense rows; a chunk behind cached tokens equals SDPA with a boolean mask of
    the positions each row may see (checks the bottom-right alignment);
  * splitting a prompt into chunks leaves every row's output bitwise unchanged;
  * outputs do not depend on where the blocks sit in the pool.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from tests._paged_helpers import from_bits, oracle_decode_pool, paged_from_dense, to_bits


def _prefill_pool(pool, q, tables, qs, lens, hkv, bs, scale, dtype):
    flat = np.ascontiguousarray(pool).reshape(-1)
    half = pool.shape[2] * pool.shape[3] * pool.shape[4]
    code = oracle.BF16 if dtype == torch.bfloat16 else oracle.F16
    return oracle.paged_prefill(q, flat, flat[half:], 2 * half, tables, qs, lens, hkv, bs, scale,
                                code)


def _dense(lens, hkv, d, dtype, g):
    k = [to_bits(torch.randn(L, hkv, d, generator=g).to(dtype)) for L in lens]
    v = [to_bits(torch.randn(L, hkv, d, generator=g).to(dtype)) for L in lens]
    return k, v


def test_two_token_prompt_by_hand():
    # d = 2, one head; row 0 (position 0) sees only token 0 -> out = v0 exactly;
    # row 1 sees both: weights softmax(scale * [q1.k0, q1.k1]).
    g = torch.Generator().manual_seed(0)
    dtype = torch.float16
    k = to_bits(torch.tensor([[[1.0, 0.0]], [[0.0, 1.0]]], dtype=dtype))
    v = to_bits(torch.tensor([[[2.0, -1.0]], [[0.5, 4.0]]], dtype=dtype))
    q = to_bits(torch.tensor([[[1.0, 3.0]], [[2.0, 0.0]]], dtype=dtype))
    pool, tables, lens = paged_from_dense([k], [v], 4, 3, g, dtype)
    out = _prefill_pool(pool, q, tables, np.array([0, 2]), lens, 1, 4, 1.0, dtype)
    assert np.array_equal(out[0, 0], [2.0, -1.0])
    w0, w1 = math.exp(2.0), math.exp(0.0)            # q1.k0 = 2, q1.k1 = 0
    expect = (w0 * np.array([2.0, -1.0]) + w1 * np.array([0.5, 4.0])) / (w0 + w1)
    np.testing.assert_allclose(out[1, 0], expect, rtol=1e-15)


@pytest.mark.parametrize("hq,hkv", [(4, 4), (8, 2)])
def test_one_token_chunks_equal_decode(hq, hkv):
    g = torch.Generator().manual_seed(hq)
    bs, d, dtype = 8, 32, torch.bfloat16
    lens = [1, 9, 30, 64]
    k, v = _dense(lens, hkv, d, dtype, g)
    pool, tables, lens_a = paged_from_dense(k, v, bs, 40, g, dtype)
    q = to_bits(torch.randn(len(lens), hq, d, generator=g).to(dtype))
    qs = np.arange(len(lens) + 1)
    got = _prefill_pool(pool, q, tables, qs, lens_a, hkv, bs, 0.2, dtype)
    ref = oracle_decode_pool(q, pool, tables, lens_a, hkv, bs, 0.2, dtype)
    np.testing.assert_allclose(got, ref, rtol=1e-14, atol=1e-15)


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16], ids=["f16", "bf16"])
def test_whole_prompt_equals_causal_sdpa(dtype):
    g = torch.Generator().manual_seed(3)
    hq, hkv, bs, d = 8, 2, 16, 64
    lens = [1, 17, 50]
    k, v = _dense(lens, hkv, d, dtype, g)
    pool, tables, lens_a = paged_from_dense(k, v, bs, 20, g, dtype)
    qs = np.concatenate([[0], np.cumsum(lens)])
    q = to_bits(torch.randn(int(qs[-1]), hq, d, generator=g).to(dtype))
    scale = 1 / math.sqrt(d)
    got = _prefill_pool(pool, q, tables, qs, lens_a, hkv, bs, scale, dtype)
    qd = from_bits(q, dtype).to(torch.float64)
    for i, L in enumerate(lens):
        qi = qd[qs[i]:qs[i + 1]].permute(1, 0, 2).unsqueeze(0)              # [1, Hq, L, d]
        kt = from_bits(k[i], dtype).to(torch.float64).permute(1, 0, 2).unsqueeze(0)
        vt = from_bits(v[i], dtype).to(torch.float64).permute(1, 0, 2).unsqueeze(0)
        o = torch.nn.functional.scaled_dot_product_attention(qi, kt, vt, scale=scale, is_causal=True,
                                                             enable_gqa=True)
        np.testing.assert_allclose(got[qs[i]:qs[i + 1]], o[0].permute(1, 0, 2).numpy(),
                                   rtol=1e-10, atol=1e-12)


def test_chunk_behind_cached_tokens_equals_masked_sdpa():
    g = torch.Generator().manual_seed(4)
    hq, hkv, bs, d, dtype = 4, 4, 8, 32, torch.float16
    lens = [40, 23, 9]
    chunks = [7, 23, 1]                                   # cached prefix of 33, 0 and 8 tokens
    k, v = _dense(lens, hkv, d, dtype, g)
    pool, tables, lens_a = paged_from_dense(k, v, bs, 20, g, dtype)
    qs = np.concatenate([[0], np.cumsum(chunks)])
    q = to_bits(torch.randn(int(qs[-1]), hq, d, generator=g).to(dtype))
    got = _prefill_pool(pool, q, tables, qs, lens_a, hkv, bs, 0.3, dtype)
    qd = from_bits(q, dtype).to(torch.float64)
    for i, (L, C) in enumerate(zip(lens, chunks)):
        qi = qd[qs[i]:qs[i + 1]].permute(1, 0, 2).unsqueeze(0)
        kt = from_bits(k[i], dtype).to(torch.float64).permute(1, 0, 2).unsqueeze(0)
        vt = from_bits(v[i], dtype).to(torch.float64).permute(1, 0, 2).unsqueeze(0)
        rows_pos = torch.arange(L - C, L).unsqueeze(1)
        mask = torch.arange(L).unsqueeze(0) <= rows_pos    # [C, L]
        o = torch.nn.functional.scaled_dot_product_attention(qi, kt, vt, attn_mask=mask, scale=0.3)
        np.testing.assert_allclose(got[qs[i]:qs[i + 1]], o[0].permute(1, 0, 2).numpy(),
                                   rtol=1e-10, atol=1e-12)


def test_chunking_does_not_change_rows():
    g = torch.Generator().manual_seed(5)
    hq, hkv, bs, d, dtype = 8, 4, 16, 64, torch.bfloat16
    L = 70
    k, v = _dense([L], hkv, d, dtype, g)
    pool, tables, _ = paged_from_dense(k, v, bs, 10, g, dtype)
    q = to_bits(torch.randn(L, hq, d, generator=g).to(dtype))
    whole = _prefill_pool(pool, q, tables, np.array([0, L]), np.array([L]), hkv, bs, 0.125, dtype)
    pieces = []
    for lo, hi in [(0, 1), (1, 33), (33, 64), (64, 70)]:
        pieces.append(_prefill_pool(pool, q[lo:hi], tables, np.array([0, hi - lo]), np.array([hi]),
                                    hkv, bs, 0.125, dtype))
    assert np.array_equal(np.concatenate(pieces), whole)


def test_prefill_is_independent_of_block_placement():
    g = torch.Generator().manual_seed(6)
    hq, hkv, bs, d, dtype = 4, 2, 8, 32, torch.float16
    lens = [12, 30]
    chunks = [12, 5]
    k, v = _dense(lens, hkv, d, dtype, g)
    pool, tables, lens_a = paged_from_dense(k, v, bs, 12, g, dtype)
    qs = np.concatenate([[0], np.cumsum(chunks)])
    q = to_bits(torch.randn(int(qs[-1]), hq, d, generator=g).to(dtype))
    a = _prefill_pool(pool, q, tables, qs, lens_a, hkv, bs, 0.2, dtype)
    perm = torch.randperm(12, generator=g).numpy()
    pool2 = np.empty_like(pool)
    pool2[perm] = pool
    b = _prefill_pool(pool2, q, perm[tables].astype(np.int32), qs, lens_a, hkv, bs, 0.2, dtype)
    assert np.array_equal(a, b)
