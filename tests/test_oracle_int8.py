"""Pins for the oracle's INT8 KV cache (per-channel scales).

"KV Cache从原理到实战" §5.2: an INT8 cache halves the bytes; scales per channel,
separately for K and V.  The quantiser's rounding is a reading (round to nearest,
ties to even, symmetric range [-127, 127], single-precision division); the pins
below fix every part of it by properties that do not restate its formula:

  * exact multiples of a power-of-two scale give their multiplier back;
  * half-way values go to the even neighbour, symmetrically in sign;
  * values beyond the range saturate at +-127;
  * every code is within half a step of x / s (nearest-integer bound) and the
    codes are monotone in x, over all finite fp16 patterns;
  * the cache write lands codes only at the slots of the slot rule;
  * decode over codes whose dequantised values are exact fp16 numbers equals the
    (separately pinned) 16-bit oracle on those numbers, and decode over random
    codes and scales equals torch's fp64 attention on the dequantised rows.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from tests._paged_helpers import from_bits, oracle_decode_pool, to_bits


def _f16_bits(values):
    return np.asarray(values, dtype=np.float16).view(np.uint16)


# ---------------------------------------------------------------- quantiser
@pytest.mark.parametrize("scale_exp", [-7, -4, 0, 3])
def test_exact_multiples_round_trip(scale_exp):
    s = 2.0 ** scale_exp
    ks = np.arange(-127, 128)
    codes = oracle.quantize_int8(_f16_bits(ks * s), np.float32([s]), oracle.F16)
    assert np.array_equal(codes.astype(np.int64), ks)


def test_ties_go_to_even():
    s = 0.25
    # x / s = k + 1/2 exactly
    halves = np.array([0.5, 1.5, 2.5, 3.5, 4.5, 125.5, 126.5])
    expect = np.array([0, 2, 2, 4, 4, 126, 126])
    got = oracle.quantize_int8(_f16_bits(halves * s), np.float32([s]), oracle.F16).astype(int)
    assert np.array_equal(got, expect)
    got_neg = oracle.quantize_int8(_f16_bits(-halves * s), np.float32([s]), oracle.F16).astype(int)
    assert np.array_equal(got_neg, -expect)


def test_saturation():
    s = 1.0 / 64
    vals = [127.4 * s, 127.5 * s, 128 * s, 1000 * s, -127.6 * s, -1000 * s, np.inf, -np.inf]
    got = oracle.quantize_int8(_f16_bits(vals), np.float32([s]), oracle.F16).astype(int).tolist()
    assert got == [127, 127, 127, 127, -127, -127, 127, -127]


@pytest.mark.parametrize("dtype", [oracle.F16, oracle.BF16], ids=["f16", "bf16"])
@pytest.mark.parametrize("scale", [0.0173, 0.5, 3.1])
def test_nearest_integer_bound_and_monotone_all_patterns(dtype, scale):
    bits = np.arange(65536, dtype=np.uint16)
    x = oracle.decode16(bits, dtype)
    finite = np.isfinite(x)
    bits, x = bits[finite], x[finite]
    codes = oracle.quantize_int8(bits, np.float32([scale]), dtype).astype(np.float64)
    s = float(np.float32(scale))
    r = x / s
    inside = np.abs(r) <= 127
    # nearest integer: |r - code| <= 1/2 (plus the single-precision quotient's rounding)
    assert np.all(np.abs(r[inside] - codes[inside]) <= 0.5 + 1e-5 * np.maximum(1, np.abs(r[inside])))
    assert np.all(codes[~inside] == np.sign(r[~inside]) * 127)
    order = np.argsort(x, kind="stable")
    assert np.all(np.diff(codes[order]) >= 0)
    # odd symmetry: code(-x) = -code(x)
    neg = oracle.quantize_int8(bits ^ 0x8000, np.float32([scale]), dtype).astype(np.float64)
    assert np.array_equal(neg, -codes)


def test_per_channel_scale_is_taken_per_head_and_channel():
    hkv, d = 3, 8
    scales = 2.0 ** (-(np.arange(hkv * d) % 7)).reshape(hkv, d).astype(np.float32)
    ks = (np.arange(2 * hkv * d).reshape(2, hkv, d) % 255) - 127
    x = _f16_bits(ks * scales[None])
    codes = oracle.quantize_int8(x, scales, oracle.F16).astype(int)
    assert np.array_equal(codes, ks)


# ---------------------------------------------------------------- cache ops
def _int8_pool(nb, hkv, bs, d, gen):
    return torch.randint(-127, 128, (nb, 2, hkv, bs, d), generator=gen, dtype=torch.int8).numpy()


def test_cache_write_places_codes_at_slots_only():
    g = torch.Generator().manual_seed(1)
    nb, hkv, bs, d = 6, 2, 8, 16
    pool = _int8_pool(nb, hkv, bs, d, g)
    before = pool.copy()
    ks = np.float32(2.0 ** -3)
    vs = np.float32(2.0 ** -5)
    k_scale = np.full((hkv, d), ks, np.float32)
    v_scale = np.full((hkv, d), vs, np.float32)
    slots = np.array([0, 13, -1, 47], dtype=np.int64)
    kc = (np.arange(4 * hkv * d).reshape(4, hkv, d) % 200) - 100
    vc = -kc // 2
    oracle.reshape_and_cache_int8(_f16_bits(kc * ks), _f16_bits(vc * vs), slots, pool, k_scale,
                                  v_scale, hkv, bs, d, oracle.F16)
    expect = before.copy()
    for n, s in enumerate(slots):
        if s < 0:
            continue
        expect[s // bs, 0, :, s % bs, :] = kc[n]
        expect[s // bs, 1, :, s % bs, :] = np.clip(vc[n], -127, 127)
    assert np.array_equal(pool, expect)


def test_copy_blocks_bytes_copies_whole_blocks():
    g = torch.Generator().manual_seed(2)
    pool = _int8_pool(5, 2, 8, 16, g)
    before = pool.copy()
    oracle.copy_blocks_bytes(pool, np.array([[1, 3], [4, 0]]))
    expect = before.copy()
    expect[3] = before[1]
    expect[0] = before[4]
    assert np.array_equal(pool, expect)


# ---------------------------------------------------------------- decode
def _pool_tables(lens, bs, nb, gen):
    nblk = [math.ceil(L / bs) for L in lens]
    perm = torch.randperm(nb, generator=gen).numpy()
    tables = np.zeros((len(lens), max(nblk + [1])), dtype=np.int32)
    cur = 0
    for i, n in enumerate(nblk):
        tables[i, :n] = perm[cur:cur + n]
        cur += n
    return tables


@pytest.mark.parametrize("hq,hkv", [(4, 4), (8, 2)])
def test_decode_equals_16bit_oracle_on_exact_dequantised_values(hq, hkv):
    """Scales 2^-e per channel: code * s is an exact fp16 number, so the INT8 oracle
    must equal the pinned 16-bit oracle run on a pool holding those numbers."""
    g = torch.Generator().manual_seed(hq + hkv)
    bs, d, nb = 8, 32, 40
    lens = [1, 7, 8, 9, 60]
    pool = _int8_pool(nb, hkv, bs, d, g)
    exps = torch.randint(3, 9, (2, hkv, d), generator=g).numpy()
    k_scale = (2.0 ** -exps[0]).astype(np.float32)
    v_scale = (2.0 ** -exps[1]).astype(np.float32)
    deq = pool.astype(np.float64)
    deq[:, 0] *= k_scale[None, :, None, :]
    deq[:, 1] *= v_scale[None, :, None, :]
    pool16 = deq.astype(np.float16)
    assert np.array_equal(pool16.astype(np.float64), deq)  # exact
    tables = _pool_tables(lens, bs, nb, g)
    q = to_bits(torch.randn(len(lens), hq, d, generator=g).to(torch.float16))
    lens_a = np.array(lens, dtype=np.int32)
    got = oracle.paged_decode_int8(q, pool, k_scale, v_scale, tables, lens_a, hkv, bs,
                                   1 / math.sqrt(d), oracle.F16)
    ref = oracle_decode_pool(q, pool16.view(np.uint16), tables, lens_a, hkv, bs,
                             1 / math.sqrt(d), torch.float16)
    np.testing.assert_allclose(got, ref, rtol=1e-13, atol=1e-15)


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16], ids=["f16", "bf16"])
def test_decode_matches_dense_sdpa_on_dequantised_rows(dtype):
    g = torch.Generator().manual_seed(5)
    hq, hkv, bs, d, nb = 8, 2, 16, 64, 64
    lens = [1, 15, 16, 17, 200, 0]
    pool = _int8_pool(nb, hkv, bs, d, g)
    k_scale = torch.empty(hkv, d).uniform_(0.005, 0.05, generator=g).numpy().astype(np.float32)
    v_scale = torch.empty(hkv, d).uniform_(0.005, 0.05, generator=g).numpy().astype(np.float32)
    tables = _pool_tables(lens, bs, nb, g)
    q = to_bits(torch.randn(len(lens), hq, d, generator=g).to(dtype))
    scale = 1 / math.sqrt(d)
    got = oracle.paged_decode_int8(q, pool, k_scale, v_scale, tables, np.array(lens, np.int32),
                                   hkv, bs, scale, 0 if dtype == torch.float16 else 1)
    qd = from_bits(q, dtype).to(torch.float64)
    for i, L in enumerate(lens):
        if L == 0:
            assert np.all(got[i] == 0)
            continue
        rows = [(tables[i, t // bs], t % bs) for t in range(L)]
        k = np.stack([pool[b, 0, :, o, :] for b, o in rows]).astype(np.float64) * k_scale
        v = np.stack([pool[b, 1, :, o, :] for b, o in rows]).astype(np.float64) * v_scale
        kt = torch.from_numpy(k).permute(1, 0, 2).unsqueeze(0)
        vt = torch.from_numpy(v).permute(1, 0, 2).unsqueeze(0)
        o = torch.nn.functional.scaled_dot_product_attention(
            qd[i].unsqueeze(0).unsqueeze(2), kt, vt, scale=scale, enable_gqa=True)
        np.testing.assert_allclose(got[i], o[0, :, 0, :].numpy(), rtol=1e-10, atol=1e-12)


def test_decode_is_independent_of_block_placement():
    g = torch.Generator().manual_seed(9)
    hq, hkv, bs, d, nb = 4, 2, 8, 16, 30
    lens = [5, 40, 17]
    pool = _int8_pool(nb, hkv, bs, d, g)
    ks = np.full((hkv, d), 0.03, np.float32)
    vs = np.full((hkv, d), 0.07, np.float32)
    tables = _pool_tables(lens, bs, nb, g)
    q = to_bits(torch.randn(3, hq, d, generator=g).to(torch.float16))
    lens_a = np.array(lens, np.int32)
    a = oracle.paged_decode_int8(q, pool, ks, vs, tables, lens_a, hkv, bs, 0.25, oracle.F16)
    perm = torch.randperm(nb, generator=g).numpy()
    pool2 = np.empty_like(pool)
    pool2[perm] = pool
    b = oracle.paged_decode_int8(q, pool2, ks, vs, perm[tables].astype(np.int32), lens_a, hkv, bs,
                                 0.25, oracle.F16)
    assert np.array_equal(a, b)
