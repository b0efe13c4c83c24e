"""Pins for the CPU oracle: each test checks it against something other than itself.

Pins used (no GPU needed):
  * 16-bit decoders vs numpy's float16 and torch's bfloat16 casts, all 65536 patterns;
  * closed forms (one token, equal keys, zero query, one dominant key);
  * a hand-computed two-token case;
  * torch's fp64 scaled_dot_product_attention on dense rows that were scattered into
    the pool block-wise (checks block-table addressing, GQA grouping, scale, masking);
  * the online-softmax form of "KV Cache与PagedAttention深度解析" §7.2 against the direct form;
  * invariants the pages fix: physical placement, block size, shared vs private blocks;
  * the worked block-table example (§4.2) and the slot rule (§5.3) of the same page;
  * the pages' KV-size arithmetic (tests/golden/kv_size_arithmetic.txt).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from tests._paged_helpers import (dense_reference, from_bits, oracle_decode_pool,
                                  paged_from_dense, random_bits, to_bits)
from tests.conftest import read_golden


# ---------------------------------------------------------------- decoders
def test_f16_decoder_matches_numpy_all_patterns():
    bits = np.arange(65536, dtype=np.uint16)
    got = oracle.decode16(bits, oracle.F16)
    ref = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    # signed zeros keep their sign
    assert math.copysign(1.0, got[0x8000]) == -1.0


def test_bf16_decoder_matches_torch_all_patterns():
    bits = np.arange(65536, dtype=np.uint16)
    got = oracle.decode16(bits, oracle.BF16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


# ---------------------------------------------------------------- closed forms
def _single_seq(k_rows, v_rows, q_row, dtype=torch.float16, bs=4, scale=None, seed=0):
    """One sequence, one head: rows are float lists; returns (oracle out, exact inputs)."""
    g = torch.Generator().manual_seed(seed)
    k = to_bits(torch.tensor(k_rows, dtype=torch.float32).to(dtype)).reshape(len(k_rows), 1, -1)
    v = to_bits(torch.tensor(v_rows, dtype=torch.float32).to(dtype)).reshape(len(v_rows), 1, -1)
    q = to_bits(torch.tensor([q_row], dtype=torch.float32).to(dtype)).reshape(1, 1, -1)
    nb = math.ceil(len(k_rows) / bs) + 3
    pool, tables, lens = paged_from_dense([k], [v], bs, nb, g, dtype)
    d = q.shape[-1]
    sc = 1.0 / math.sqrt(d) if scale is None else scale
    out = oracle_decode_pool(q, pool, tables, lens, 1, bs, sc, dtype)
    return out[0, 0], from_bits(v, dtype).double().numpy()[:, 0, :]


def test_single_token_returns_its_value_exactly():
    out, v = _single_seq([[0.5, -1.0, 2.0, 3.0]], [[1.25, -7.5, 0.0, 3.0]], [9.0, 1.0, -2.0, 4.0])
    assert np.array_equal(out, v[0])


def test_equal_keys_give_mean_of_values():
    rows_k = [[1.0, 2.0, -1.0, 0.5]] * 6
    rows_v = [[float(i), -2.0 * i, 0.25 * i, 1.0] for i in range(6)]
    out, v = _single_seq(rows_k, rows_v, [3.0, -1.0, 2.0, 0.5])
    np.testing.assert_allclose(out, v.mean(axis=0), rtol=0, atol=1e-14)


def test_zero_query_gives_mean_of_values():
    g = torch.Generator().manual_seed(5)
    k = torch.randn(11, 8, generator=g).tolist()
    v = torch.randn(11, 8, generator=g).tolist()
    out, vv = _single_seq(k, v, [0.0] * 8, bs=4)
    np.testing.assert_allclose(out, vv.mean(axis=0), rtol=0, atol=1e-14)


def test_one_dominant_key_selects_its_value():
    k = [[0.0, 0.0], [0.0, 0.0], [64.0, 0.0], [0.0, 0.0], [0.0, 0.0]]
    v = [[1.0, 2.0], [3.0, 4.0], [-5.0, 6.5], [7.0, 8.0], [9.0, 10.0]]
    out, vv = _single_seq(k, v, [64.0, 0.0], bs=2, scale=1.0)
    # scores 4096 vs 0: the other weights are exp(-4096) == 0 in fp64
    assert np.array_equal(out, vv[2])


def test_two_token_hand_computed():
    # scale 1: scores q.k0 = 0 and q.k1 = 1, weights 1/(1+e) and e/(1+e)
    out, _ = _single_seq([[0.0, 0.0], [1.0, 0.0]], [[2.0, -4.0], [6.0, 8.0]], [1.0, 3.0],
                         bs=2, scale=1.0)
    e = math.e
    ref = np.array([(2.0 + 6.0 * e) / (1 + e), (-4.0 + 8.0 * e) / (1 + e)])
    np.testing.assert_allclose(out, ref, rtol=1e-15, atol=0)


def test_scale_enters_the_exponent():
    # scores 0 and 2*scale with scale=0.5: weights 1/(1+e), e/(1+e)
    out, _ = _single_seq([[0.0, 0.0], [2.0, 0.0]], [[1.0, 0.0], [0.0, 1.0]], [1.0, 0.0],
                         bs=2, scale=0.5)
    e = math.e
    np.testing.assert_allclose(out, [1 / (1 + e), e / (1 + e)], rtol=1e-15)


# ---------------------------------------------------------------- dense cross-check
@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("hq,hkv,d,bs", [(4, 4, 64, 16), (8, 2, 64, 8), (16, 2, 128, 32),
                                         (6, 3, 32, 16)])
def test_oracle_matches_dense_sdpa(dtype, hq, hkv, d, bs):
    g = torch.Generator().manual_seed(hq * 131 + d + bs)
    lens = [1, bs - 1, bs, bs + 1, 3 * bs + 5, 0, 77]
    k = [random_bits((n, hkv, d), dtype, g) for n in lens]
    v = [random_bits((n, hkv, d), dtype, g) for n in lens]
    q = random_bits((len(lens), hq, d), dtype, g)
    nb = sum(math.ceil(n / bs) for n in lens) + 5
    pool, tables, cl = paged_from_dense(k, v, bs, nb, g, dtype)
    scale = 1.0 / math.sqrt(d)
    got = oracle_decode_pool(q, pool, tables, cl, hkv, bs, scale, dtype)
    ref = dense_reference(q, k, v, scale, dtype)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-13)
    # the empty sequence gives a zero row
    assert np.all(got[lens.index(0)] == 0.0)


def test_dense_check_catches_a_wrong_gqa_mapping():
    """Guard that the dense pin can tell the contiguous grouping from an interleaved one."""
    dtype = torch.float16
    g = torch.Generator().manual_seed(9)
    k = [random_bits((40, 2, 16), dtype, g)]
    v = [random_bits((40, 2, 16), dtype, g)]
    q = random_bits((1, 4, 16), dtype, g)
    ref = dense_reference(q, k, v, 0.25, dtype)
    # interleaved mapping hq -> hq % Hkv would swap heads 1 and 2
    swapped = dense_reference(q[:, [0, 2, 1, 3]], k, v, 0.25, dtype)[:, [0, 2, 1, 3]]
    assert not np.allclose(ref, swapped)


# ---------------------------------------------------------------- online form
@pytest.mark.parametrize("bs", [8, 16, 32])
def test_online_form_equals_direct_form(bs):
    dtype = torch.bfloat16
    g = torch.Generator().manual_seed(bs)
    lens = [1, 5, bs, 2 * bs + 3, 200]
    k = [random_bits((n, 2, 64), dtype, g) for n in lens]
    v = [random_bits((n, 2, 64), dtype, g) for n in lens]
    q = random_bits((len(lens), 8, 64), dtype, g)
    pool, tables, cl = paged_from_dense(k, v, bs, 64, g, dtype)
    a = oracle_decode_pool(q, pool, tables, cl, 2, bs, 0.125, dtype)
    b = oracle_decode_pool(q, pool, tables, cl, 2, bs, 0.125, dtype, flash=True)
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-14)


def test_per_block_softmax_of_the_naive_loop_is_not_the_definition():
    """§4.3's first loop normalises each block on its own; the result differs from
    softmax over the whole context, which is why the oracle follows §2.1 / §7.2."""
    dtype = torch.float16
    g = torch.Generator().manual_seed(3)
    n, bs, d = 48, 16, 32
    k = random_bits((n, 1, d), dtype, g)
    v = random_bits((n, 1, d), dtype, g)
    q = random_bits((1, 1, d), dtype, g)
    ref = dense_reference(q, [k], [v], 1 / math.sqrt(d), dtype)[0, 0]
    kd = from_bits(k, dtype).double()[:, 0]
    vd = from_bits(v, dtype).double()[:, 0]
    qd = from_bits(q, dtype).double()[0, 0]
    naive = torch.zeros(d, dtype=torch.float64)
    for b in range(n // bs):
        s = (kd[b * bs:(b + 1) * bs] @ qd) / math.sqrt(d)
        naive += torch.softmax(s, 0) @ vd[b * bs:(b + 1) * bs]
    assert not np.allclose(naive.numpy(), ref, atol=1e-3)


# ---------------------------------------------------------------- invariants
def _relabel(pool, tables, lens, bs, gen):
    """Move every used block to a new random physical slot (same logical content)."""
    nb = pool.shape[0]
    perm = torch.randperm(nb, generator=gen).numpy()
    new_pool = np.empty_like(pool)
    new_pool[perm] = pool
    new_tables = tables.copy()
    for i in range(tables.shape[0]):
        n = math.ceil(lens[i] / bs)
        new_tables[i, :n] = perm[tables[i, :n]]
    return new_pool, new_tables


def test_physical_placement_does_not_change_result_bitwise():
    dtype = torch.float16
    g = torch.Generator().manual_seed(11)
    lens = [33, 100, 1, 64]
    k = [random_bits((n, 4, 64), dtype, g) for n in lens]
    v = [random_bits((n, 4, 64), dtype, g) for n in lens]
    q = random_bits((4, 8, 64), dtype, g)
    pool, tables, cl = paged_from_dense(k, v, 16, 40, g, dtype)
    a = oracle_decode_pool(q, pool, tables, cl, 4, 16, 0.125, dtype)
    pool2, tables2 = _relabel(pool, tables, cl, 16, g)
    b = oracle_decode_pool(q, pool2, tables2, cl, 4, 16, 0.125, dtype)
    assert np.array_equal(a, b)


def test_block_size_is_a_free_parameter():
    dtype = torch.bfloat16
    g = torch.Generator().manual_seed(12)
    lens = [1, 31, 64, 95]
    k = [random_bits((n, 2, 64), dtype, g) for n in lens]
    v = [random_bits((n, 2, 64), dtype, g) for n in lens]
    q = random_bits((4, 4, 64), dtype, g)
    outs = []
    for bs in (8, 16, 32):
        pool, tables, cl = paged_from_dense(k, v, bs, 64, g, dtype)
        outs.append(oracle_decode_pool(q, pool, tables, cl, 2, bs, 0.125, dtype))
    np.testing.assert_allclose(outs[0], outs[1], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(outs[0], outs[2], rtol=1e-12, atol=1e-14)


def test_shared_blocks_read_like_private_copies():
    """Two sequences with the same prefix: shared physical blocks vs private copies."""
    dtype = torch.float16
    g = torch.Generator().manual_seed(13)
    bs, d = 16, 64
    pref_k = random_bits((48, 2, d), dtype, g)
    pref_v = random_bits((48, 2, d), dtype, g)
    tails_k = [random_bits((n, 2, d), dtype, g) for n in (7, 20)]
    tails_v = [random_bits((n, 2, d), dtype, g) for n in (7, 20)]
    k = [np.concatenate([pref_k, t]) for t in tails_k]
    v = [np.concatenate([pref_v, t]) for t in tails_v]
    q = random_bits((2, 4, d), dtype, g)
    pool, tables, cl = paged_from_dense(k, v, bs, 32, g, dtype)
    private = oracle_decode_pool(q, pool, tables, cl, 2, bs, 0.125, dtype)
    shared_tables = tables.copy()
    shared_tables[1, :3] = tables[0, :3]            # sequence 1 now points at sequence 0's prefix
    shared = oracle_decode_pool(q, pool, shared_tables, cl, 2, bs, 0.125, dtype)
    assert np.array_equal(private, shared)


# ---------------------------------------------------------------- slot rule and worked example
def test_worked_example_block_table():
    gold = read_golden("worked_example_block_table.txt")
    table = np.array([int(x) for x in gold["block_table"].split()], dtype=np.int32)
    bs = int(gold["block_size"])
    n = int(gold["context_len"])
    assert oracle.blocks_needed(n - 1, bs) == int(gold["num_blocks"]) == len(table)
    assert n - (len(table) - 1) * bs == int(gold["last_block_tokens"])
    for key, val in gold.items():
        if key.startswith("token_"):
            t = int(key.split("_")[1])
            blk, off = (int(x) for x in val.split())
            assert oracle.slot_for_position(table, t, bs) == blk * bs + off


def test_blocks_needed_grows_at_block_boundaries():
    # a new block is needed exactly when the token index crosses a multiple of bs
    for bs in (8, 16, 32):
        counts = [oracle.blocks_needed(t, bs) for t in range(4 * bs)]
        assert counts[0] == 1
        for t in range(1, 4 * bs):
            assert counts[t] - counts[t - 1] == (1 if t % bs == 0 else 0)


def test_kv_size_arithmetic_matches_the_pages():
    gold = {k: int(v) for k, v in read_golden("kv_size_arithmetic.txt").items()}
    # 7B MHA (32 heads x 128 = hidden 4096), 32 layers, fp16
    assert oracle.kv_bytes_per_token(1, 32, 128) == gold["mha7b_per_layer_per_token"]
    assert oracle.kv_bytes_per_token(32, 32, 128) == gold["mha7b_per_token"]
    assert oracle.kv_bytes(32, 32, 128, 4096, batch=16) == gold["mha7b_4096_tokens_batch16"]
    assert oracle.kv_bytes(32, 32, 128, 128 * 1024) == gold["mha7b_128k_tokens"]
    # 7B GQA (8 KV heads of 128)
    assert oracle.kv_bytes_per_token(1, 8, 128) == gold["gqa7b_per_layer_per_token"]
    assert oracle.kv_bytes_per_token(32, 8, 128) == gold["gqa7b_per_token"]
    assert oracle.kv_bytes(32, 8, 128, 4096) == gold["gqa7b_4096_tokens"]
    assert oracle.kv_bytes(32, 8, 128, 4096, batch=32) == gold["gqa7b_4096_tokens_batch32"]
    assert (oracle.kv_bytes_per_token(32, 32, 128) // oracle.kv_bytes_per_token(32, 8, 128)
            == gold["mha_over_gqa_ratio"])
    # 70B taken as MHA with d = 8192 (64 heads x 128), 80 layers, 4096 tokens
    assert oracle.kv_bytes(80, 64, 128, 4096) == gold["llama70b_mha_formula_4096"]
    assert gold["llama70b_page_printed_misprint"] != gold["llama70b_mha_formula_4096"]


# ---------------------------------------------------------------- cache write and block copy
def test_reshape_and_cache_lands_at_block_and_offset():
    hkv, bs, d, nb = 3, 16, 64, 12
    g = torch.Generator().manual_seed(21)
    pool = random_bits((nb, 2, hkv, bs, d), torch.float16, g)
    before = pool.copy()
    table = np.array([7, 2, 9, 1, 5, 8, 3], dtype=np.int32)
    positions = [0, 15, 16, 99]
    kn = random_bits((4, hkv, d), torch.float16, g)
    vn = random_bits((4, hkv, d), torch.float16, g)
    slots = np.array([oracle.slot_for_position(table, t, bs) for t in positions] , dtype=np.int64)
    oracle.reshape_and_cache(kn, vn, slots, pool, hkv, bs, d)
    expect = {0: (7, 0), 15: (7, 15), 16: (2, 0), 99: (3, 3)}
    touched = np.zeros(pool.shape[:4], dtype=bool)
    for n, t in enumerate(positions):
        blk, off = expect[t]
        assert np.array_equal(pool[blk, 0, :, off, :], kn[n])
        assert np.array_equal(pool[blk, 1, :, off, :], vn[n])
        touched[blk, :, :, off] = True
    assert np.array_equal(pool[~touched], before[~touched])


def test_reshape_and_cache_skips_negative_slots():
    g = torch.Generator().manual_seed(22)
    pool = random_bits((4, 2, 2, 8, 64), torch.bfloat16, g)
    before = pool.copy()
    kn = random_bits((2, 2, 64), torch.bfloat16, g)
    vn = random_bits((2, 2, 64), torch.bfloat16, g)
    oracle.reshape_and_cache(kn, vn, np.array([-1, -5], dtype=np.int64), pool, 2, 8, 64)
    assert np.array_equal(pool, before)


def test_copy_blocks_copies_k_and_v_and_leaves_sources():
    g = torch.Generator().manual_seed(23)
    pool = random_bits((10, 2, 2, 32, 64), torch.bfloat16, g)
    before = pool.copy()
    pairs = np.array([[3, 7], [3, 8], [1, 0]], dtype=np.int64)
    oracle.copy_blocks(pool, pairs, 2, 32, 64)
    for s, dst in pairs:
        assert np.array_equal(pool[dst], before[s])
    untouched = [b for b in range(10) if b not in (7, 8, 0)]
    assert np.array_equal(pool[untouched], before[untouched])
