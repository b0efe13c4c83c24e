"""The C-ABI library without a GPU: it loads, exports every symbol the header
declares, rejects out-of-contract arguments on the host before touching CUDA,
and its launch planner behaves as documented.  Also checks the product's host
slot helper against the oracle's slot rule."""
import ctypes
import os
import re
import subprocess

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_155_gb300 import _build, block_table
from tests.conftest import ROOT

INVALID, UNSUPPORTED = 1, 2


@pytest.fixture(scope="module")
def lib():
    _build.build()
    from paged_kv_cache_155_gb300._lib import lib as load
    return load()


def header_symbols():
    text = open(os.path.join(ROOT, "include", "pagedkv.h")).read()
    return sorted(set(re.findall(r"PKV_API\s+[\w\s\*]+?\b(pkv_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    syms = header_symbols()
    for name in ("pkv_reshape_and_cache", "pkv_paged_attention_decode", "pkv_copy_blocks",
                 "pkv_decode_workspace_bytes", "pkv_get_device_error", "pkv_status_string"):
        assert name in syms


def test_library_exports_every_declared_symbol(lib):
    syms = header_symbols()
    out = subprocess.run(["nm", "-D", "--defined-only", _build.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT\s+(\w+)$", out, flags=re.M))
    missing = [s for s in syms if s not in exported]
    assert not missing, f"declared but not exported: {missing}"
    for s in syms:
        assert getattr(lib, s) is not None
    # nothing else leaks out under the pkv_ prefix that the header does not declare
    extra = sorted(s for s in exported if s.startswith("pkv_") and s not in syms)
    assert not extra, f"exported but undeclared: {extra}"


def test_status_strings(lib):
    for code in range(5):
        assert lib.pkv_status_string(code)
    assert b"unknown" in lib.pkv_status_string(99)


def _dec(lib, **kw):
    a = dict(q=16, k=16, v=16, nb=64, stride=2 * 4 * 16 * 64, bt=16, mb=8, cl=16, maxl=100,
             b=4, hq=4, hkv=4, d=64, bs=16, scale=0.125, out=16, ws=None, wsb=0, part=0, dt=0)
    a.update(kw)
    return lib.pkv_paged_attention_decode(a["q"], a["k"], a["v"], a["nb"], a["stride"], a["bt"],
                                          a["mb"], a["cl"], a["maxl"], a["b"], a["hq"], a["hkv"],
                                          a["d"], a["bs"], a["scale"], a["out"], a["ws"], a["wsb"],
                                          a["part"], a["dt"], None)


def test_decode_rejects_bad_arguments_on_host(lib):
    assert _dec(lib, d=96) == UNSUPPORTED
    assert _dec(lib, bs=64) == UNSUPPORTED
    assert _dec(lib, dt=7) == UNSUPPORTED
    assert _dec(lib, hq=6, hkv=4) == INVALID          # not a multiple
    assert _dec(lib, maxl=8 * 16 + 1) == INVALID      # beyond max_blocks_per_seq * bs
    assert _dec(lib, stride=100) == INVALID           # smaller than one half block
    assert _dec(lib, stride=2 * 4 * 16 * 64 + 4) == INVALID  # not 16-byte aligned
    assert _dec(lib, k=8) == INVALID                  # misaligned cache pointer
    assert _dec(lib, q=0) == INVALID                  # null q
    assert _dec(lib, scale=float("nan")) == INVALID
    assert _dec(lib, part=24) == INVALID              # not a multiple of block_size
    assert _dec(lib, nb=0) == INVALID
    assert _dec(lib, b=-1) == INVALID


def test_cache_ops_reject_bad_arguments_on_host(lib):
    r = lib.pkv_reshape_and_cache
    good = dict(kn=16, vn=16, sm=16, t=4, kc=16, vc=16, nb=8, stride=2 * 2 * 16 * 64, hkv=2, d=64, bs=16, dt=0)

    def call(**kw):
        a = dict(good)
        a.update(kw)
        return r(a["kn"], a["vn"], a["sm"], a["t"], a["kc"], a["vc"], a["nb"], a["stride"],
                 a["hkv"], a["d"], a["bs"], a["dt"], None)

    assert call(d=80) == UNSUPPORTED
    assert call(t=-1) == INVALID
    assert call(kn=0) == INVALID
    assert call(sm=12) == INVALID          # int64 slots must be 8-byte aligned
    assert call(stride=10) == INVALID
    assert call(t=0, kn=0, vn=0, sm=0) == 0  # empty: no-op, nothing dereferenced
    c = lib.pkv_copy_blocks
    assert c(16, 16, 8, 2 * 2 * 16 * 64, 2, 64, 16, 0, 3, 0, None) == INVALID   # null pairs
    assert c(16, 16, 8, 2 * 2 * 16 * 64, 2, 64, 16, 0, 0, 0, None) == 0         # empty
    assert c(16, 16, 8, 2 * 2 * 16 * 64, 2, 64, 12, 16, 1, 0, None) == UNSUPPORTED
    assert lib.pkv_debug_wait_timeout(0, None) == INVALID


def test_int8_entry_points_reject_bad_arguments_on_host(lib):
    def dec(**kw):
        a = dict(q=16, k=16, v=16, ks=16, vs=16, nb=64, stride=2 * 4 * 16 * 64, bt=16, mb=8, cl=16,
                 maxl=100, b=4, hq=4, hkv=4, d=64, bs=16, scale=0.125, out=16, ws=None, wsb=0,
                 part=0, dt=0)
        a.update(kw)
        return lib.pkv_paged_attention_decode_int8(
            a["q"], a["k"], a["v"], a["ks"], a["vs"], a["nb"], a["stride"], a["bt"], a["mb"],
            a["cl"], a["maxl"], a["b"], a["hq"], a["hkv"], a["d"], a["bs"], a["scale"], a["out"],
            a["ws"], a["wsb"], a["part"], a["dt"], None)

    assert dec(dt=2) == UNSUPPORTED                    # q is fp16 or bf16, not INT8
    assert dec(d=96) == UNSUPPORTED
    assert dec(ks=0) == INVALID                        # scales required
    assert dec(vs=8) == INVALID                        # scales 16-byte aligned
    assert dec(stride=2 * 4 * 16 * 64 + 8) == INVALID  # INT8 block stride: multiple of 16
    assert dec(hq=6) == INVALID
    assert dec(part=24) == INVALID
    assert dec(b=0) == 0                               # empty batch: nothing to do

    def rc(**kw):
        a = dict(kn=16, vn=16, sm=16, t=4, kc=16, vc=16, nb=8, stride=2 * 2 * 16 * 64, hkv=2, d=64,
                 bs=16, ks=16, vs=16, dt=0)
        a.update(kw)
        return lib.pkv_reshape_and_cache_int8(a["kn"], a["vn"], a["sm"], a["t"], a["kc"], a["vc"],
                                              a["nb"], a["stride"], a["hkv"], a["d"], a["bs"],
                                              a["ks"], a["vs"], a["dt"], None)

    assert rc(dt=2) == UNSUPPORTED                     # the new rows are fp16 or bf16
    assert rc(d=80) == UNSUPPORTED
    assert rc(ks=0) == INVALID
    assert rc(vs=4) == INVALID
    assert rc(stride=2 * 2 * 16 * 64 + 8) == INVALID
    assert rc(t=0, kn=0, vn=0, sm=0, ks=0, vs=0) == 0  # empty: no-op
    c = lib.pkv_copy_blocks
    assert c(16, 16, 8, 2 * 2 * 16 * 64, 2, 64, 16, 0, 0, 2, None) == 0          # INT8, empty
    assert c(16, 16, 8, 2 * 2 * 16 * 64 + 8, 2, 64, 16, 16, 1, 2, None) == INVALID  # 8-byte stride
    assert c(16, 16, 8, 2 * 2 * 16 * 64, 2, 64, 16, 16, 1, 3, None) == UNSUPPORTED
    # explicit partitions: the INT8 workspace is partials of (d + 2) floats per slot
    ws = lib.pkv_decode_int8_workspace_bytes(4, 32, 8, 128, 16, 4096, 512)
    assert ws == 4 * 32 * 8 * (128 + 2) * 4
    assert lib.pkv_decode_int8_workspace_bytes(4, 32, 8, 128, 16, 500, 512) == 0


def test_prefill_rejects_bad_arguments_on_host(lib):
    def pf(**kw):
        a = dict(q=16, k=16, v=16, nb=64, stride=2 * 4 * 16 * 128, bt=16, mb=8, qs=16, cl=16,
                 rows=100, mq=50, mc=100, b=4, hq=8, hkv=4, d=128, bs=16, scale=0.125, out=16,
                 ws=None, wsb=0, splits=1, dt=0)
        a.update(kw)
        return lib.pkv_paged_attention_prefill(
            a["q"], a["k"], a["v"], a["nb"], a["stride"], a["bt"], a["mb"], a["qs"], a["cl"],
            a["rows"], a["mq"], a["mc"], a["b"], a["hq"], a["hkv"], a["d"], a["bs"], a["scale"],
            a["out"], a["ws"], a["wsb"], a["splits"], a["dt"], None)

    assert pf(d=64) == UNSUPPORTED                   # head_dim 128 only
    assert pf(bs=64) == UNSUPPORTED
    assert pf(dt=2) == UNSUPPORTED
    assert pf(hq=6) == INVALID
    assert pf(mc=40) == INVALID                      # context bound below the chunk bound
    assert pf(mc=8 * 16 + 1, mq=1) == INVALID        # beyond the tables
    assert pf(splits=-1) == INVALID
    assert pf(scale=float("inf")) == INVALID
    assert pf(qs=0) == INVALID
    assert pf(stride=2 * 4 * 16 * 128 + 4) == INVALID
    assert pf(splits=2, mc=1000, mb=100) == INVALID  # a split plan needs a workspace
    assert pf(b=0) == 0 and pf(rows=0) == 0 and pf(mq=0) == 0   # nothing to do
    # explicit splits: whole 128-token tiles, partials of (d + 2) floats per row and split
    ws = lib.pkv_prefill_workspace_bytes(100, 4, 8, 4, 128, 16, 50, 1000, 3)
    assert ws == 100 * 8 * 3 * (128 + 2) * 4
    assert lib.pkv_prefill_workspace_bytes(100, 4, 8, 4, 128, 16, 50, 1000, 1) == 0
    assert lib.pkv_prefill_workspace_bytes(100, 4, 8, 4, 128, 16, 50, 100, 5) == 0  # one tile
    assert lib.pkv_prefill_workspace_bytes(100, 4, 8, 4, 64, 16, 50, 100, 1) == ctypes.c_size_t(-1).value


def plan(lib, b, hq, hkv, d, bs, maxl, part, sm=152):
    outs = [ctypes.c_int() for _ in range(4)]
    st = lib.pkv_decode_plan(b, hq, hkv, d, bs, maxl, part, sm, *[ctypes.byref(o) for o in outs])
    return st, [o.value for o in outs]


def test_plan_explicit_partition(lib):
    st, (p, n, gh, merge) = plan(lib, 16, 64, 8, 128, 16, 32768, 512)
    assert st == 0 and p == 512 and n == 64 and gh == 8 and merge == 1


def test_plan_heads_per_block_follows_the_group(lib):
    # a block serves the largest of 16 (16-bit caches at head_dim 128), 8, 4, 2, 1 query
    # heads dividing the group, whatever the context length; a group of 16 takes one block
    # of 16 at head_dim 128 and two blocks of 8 at head_dim 64 or over an INT8 cache
    for hq, hkv, want in [(32, 32, 1), (32, 16, 2), (32, 8, 4), (64, 8, 8), (24, 8, 1),
                          (48, 8, 2), (128, 8, 16), (256, 8, 16)]:
        for d, maxl in [(128, 4000), (128, 1000), (64, 4000)]:
            st, (_, _, gh, _) = plan(lib, 4, hq, hkv, d, 16, maxl, 0)
            assert st == 0 and gh == (8 if want == 16 and d == 64 else want), (hq, hkv, d, maxl)
            st, (_, _, gh8, _) = plan_int8(lib, 4, hq, hkv, d, 16, maxl, 0)
            assert st == 0 and gh8 == min(want, 8), (hq, hkv, d, maxl)


def test_plan_gqa_partitions_cover_the_context(lib):
    for maxl in (2048, 4096, 8192, 32768):
        st, (p, n, gh, _) = plan(lib, 64, 32, 8, 128, 16, maxl, 0)
        assert st == 0 and gh == 4 and p % 16 == 0 and p >= 256 and (n - 1) * p < maxl <= n * p


def test_plan_auto_split_fills_the_gpu_and_respects_limits(lib):
    # tiny: never split below the minimum partition
    st, (p, n, _, merge) = plan(lib, 4, 4, 4, 64, 16, 100, 0)
    assert st == 0 and n == 1 and merge == 0 and p % 16 == 0
    # few long sequences: split into several partitions, each a multiple of bs
    st, (p, n, _, merge) = plan(lib, 16, 64, 8, 128, 16, 32768, 0)
    assert st == 0 and n > 1 and merge == 1 and p % 16 == 0 and (n - 1) * p < 32768 <= n * p
    # empty batch of contexts
    st, (p, n, _, merge) = plan(lib, 4, 4, 4, 64, 16, 0, 0)
    assert st == 0 and n == 1 and merge == 0
    # partition too long for the table slice
    st, _ = plan(lib, 1, 8, 8, 128, 16, 1 << 20, 1024 * 16 + 16)
    assert st == INVALID


def plan_int8(lib, b, hq, hkv, d, bs, maxl, part, sm=152):
    outs = [ctypes.c_int() for _ in range(4)]
    st = lib.pkv_decode_int8_plan(b, hq, hkv, d, bs, maxl, part, sm, *[ctypes.byref(o) for o in outs])
    return st, [o.value for o in outs]


def test_plan_auto_split_per_kernel_form(lib):
    # partition_size 0: eight waves of the form's resident blocks per SM (16-bit per-lane
    # 2, 16-bit warp MMAs 3 or 2 with sixteen heads per block, INT8 per-lane 6, INT8 warp
    # MMAs 4), partitions of at least 256 tokens, a multiple of the block size, whose K/V
    # bytes are at least 32x their partial outputs (GH rows of head_dim + 2 floats,
    # written and read back).  Forms with two resident blocks per SM that the floors
    # leave short of eight waves take the fewest partitions in [n / 2, n] whose blocks
    # fill whole waves within 0.15 of the best count there.
    def expect(b, hq, hkv, d, bs, maxl, resident, kv_bytes, sm=152):
        g = hq // hkv
        gh = 16 if (kv_bytes == 2 and d == 128 and g % 16 == 0) else next(x for x in (8, 4, 2, 1) if g % x == 0)
        units = b * hkv * (g // gh)
        slots = sm * resident
        want = max(1, -(-(slots * 8) // units))
        p = max(-(-maxl // want), 256, -(-(32 * 2 * gh * (d + 2) * 4) // (2 * d * kv_bytes)))
        p = -(-p // bs) * bs
        n = -(-maxl // p)
        if resident == 2 and n > 1 and units * n < slots * 8:
            def fill(k):
                blocks = units * k
                return blocks / (-(-blocks // slots) * slots)
            def part(k):
                return -(-(-(-maxl // k)) // bs) * bs
            ks = range((n + 1) // 2, n)
            best = max([fill(n)] + [fill(-(-maxl // part(k))) for k in ks])
            for k in ks:
                if fill(-(-maxl // part(k))) >= best - 0.15:
                    return part(k)
        return p
    cases = [  # (plan, b, hq, hkv, d, bs, maxl, resident, kv bytes per value)
        (plan, 32, 32, 32, 128, 16, 4096, 2, 2),        # MHA 7B: 1376-token partitions
        (plan, 64, 32, 8, 128, 16, 8192, 3, 2),         # GQA 7B, warp MMAs
        (plan, 16, 64, 8, 128, 16, 32768, 3, 2),        # 70B long context
        (plan, 16, 128, 8, 128, 16, 8192, 2, 2),        # 16 heads per block: 4 partitions of 2048
        (plan, 8, 128, 8, 128, 16, 32768, 2, 2),        # ... 17 partitions of 1936
        (plan, 32, 64, 4, 128, 16, 4096, 2, 2),         # ... 2 partitions of 2048
        (plan_int8, 64, 32, 8, 128, 16, 8192, 4, 1),    # INT8 GQA 7B
        (plan_int8, 16, 64, 8, 128, 16, 32768, 4, 1),   # INT8 70B: the partial-bytes floor
        (plan_int8, 32, 32, 32, 128, 16, 4096, 6, 1),   # INT8 MHA 7B, per-lane loops
        (plan_int8, 4, 4, 4, 64, 16, 100, 6, 1),        # tiny: one partition
    ]
    got = {}
    for fn, b, hq, hkv, d, bs, maxl, resident, eb in cases:
        st, (p, n, _, merge) = fn(lib, b, hq, hkv, d, bs, maxl, 0)
        assert st == 0 and p == expect(b, hq, hkv, d, bs, maxl, resident, eb), (fn.__name__, b, hq, hkv, maxl, p)
        assert (n - 1) * p < max(maxl, 1) <= n * p and merge == (n > 1)
        got[(fn.__name__, b, hq, hkv, maxl)] = p
    assert got[("plan", 32, 32, 32, 4096)] == 1376
    assert got[("plan_int8", 64, 32, 8, 8192)] == 832
    assert got[("plan_int8", 16, 64, 8, 32768)] == 1040
    assert got[("plan_int8", 32, 32, 32, 4096)] == 512
    assert got[("plan", 16, 128, 8, 8192)] == 2048
    assert got[("plan", 8, 128, 8, 32768)] == 1936


def test_int8_and_16bit_decode_share_explicit_partitions(lib):
    # with an explicit partition the INT8 and 16-bit calls split alike, so the two
    # workspace queries agree for every shape (explicit partitions: no device query)
    for b, hq, hkv, d, bs, maxl, part in [(4, 32, 8, 128, 16, 4096, 512), (16, 64, 8, 128, 16, 32768, 1024),
                                          (3, 4, 4, 64, 8, 100, 16), (7, 48, 8, 128, 32, 2000, 256)]:
        a = lib.pkv_decode_workspace_bytes(b, hq, hkv, d, bs, maxl, part)
        i8 = lib.pkv_decode_int8_workspace_bytes(b, hq, hkv, d, bs, maxl, part)
        assert a == i8 and a == (0 if maxl <= part else b * hq * -(-maxl // part) * (d + 2) * 4)


def test_workspace_bytes_explicit_partition(lib):
    n = lib.pkv_decode_workspace_bytes(16, 64, 8, 128, 16, 32768, 512)
    assert n == 16 * 64 * 64 * (128 + 2) * 4
    assert lib.pkv_decode_workspace_bytes(4, 4, 4, 64, 16, 100, 256) == 0
    assert lib.pkv_decode_workspace_bytes(4, 4, 4, 64, 16, 100, 24) == ctypes.c_size_t(-1).value


def test_host_slot_helper_matches_oracle_slot_rule():
    g = torch.Generator().manual_seed(0)
    for bs in (8, 16, 32):
        tables = torch.randint(0, 1000, (9, 40), generator=g, dtype=torch.int32)
        pos = torch.randint(0, 40 * bs, (9,), generator=g)
        pos[3] = -1
        got = block_table.slot_mapping(tables, pos, bs).numpy()
        for i in range(9):
            if pos[i] < 0:
                assert got[i] == -1
            else:
                assert got[i] == oracle.slot_for_position(tables[i].numpy(), int(pos[i]), bs)


def _host_slots(lib, tables, pos, bs, rows=None, num_blocks=1 << 40):
    bt = np.ascontiguousarray(tables, dtype=np.int32)
    p = np.ascontiguousarray(pos, dtype=np.int64)
    r = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    out = np.full(p.shape[0], 12345, dtype=np.int64)
    st = lib.pkv_slot_mapping_host(bt.ctypes.data, bt.shape[0], bt.shape[1],
                                   None if r is None else r.ctypes.data, p.ctypes.data,
                                   p.shape[0], bs, num_blocks, out.ctypes.data)
    return st, out


def test_slot_mapping_host_worked_example(lib):
    """The worked table of "KV Cache与PagedAttention深度解析" §4.2 through the C ABI:
    positions 0 / 15 / 16 / 47 / 95 / 96 / 99 land where the page's table puts them,
    and a negative position is padding."""
    from tests.conftest import read_golden
    gold = read_golden("worked_example_block_table.txt")
    table = [int(x) for x in gold["block_table"].split()]
    bs = int(gold["block_size"])
    pos = [0, 15, 16, 47, 95, 96, 99, -1]
    st, out = _host_slots(lib, [table] * len(pos), pos, bs)
    assert st == 0
    for t, slot in zip(pos, out):
        if t < 0:
            assert slot == -1
            continue
        blk, off = (int(x) for x in gold[f"token_{t}"].split())
        assert (slot // bs, slot % bs) == (blk, off)
    # one table row shared by every token through token_rows
    st, out2 = _host_slots(lib, [table], pos, bs, rows=[0] * len(pos))
    assert st == 0 and np.array_equal(out, out2)


def test_slot_mapping_host_matches_oracle_and_flags_bad_inputs(lib):
    g = np.random.default_rng(3)
    for bs in (8, 16, 32):
        tables = g.integers(0, 1000, (9, 40)).astype(np.int32)
        pos = g.integers(0, 40 * bs, 9)
        pos[4] = -3
        rows = g.integers(0, 9, 9)
        st, out = _host_slots(lib, tables, pos, bs, rows=rows, num_blocks=1000)
        assert st == 0
        ref = [-1 if p < 0 else oracle.slot_for_position(tables[r], int(p), bs)
               for r, p in zip(rows, pos)]
        assert out.tolist() == ref
    tables = np.array([[3, 1], [0, 2]], dtype=np.int32)
    # a position past the table, a table entry past the pool, a token row past the table
    for pos, rows, nb in (([32, 1], None, 4), ([1, 17], None, 2), ([1, 1], [0, 2], 4)):
        st, out = _host_slots(lib, tables, pos, 16, rows=rows, num_blocks=nb)
        assert st == INVALID
        assert -1 in out.tolist() and 12345 not in out.tolist()
    st, _ = _host_slots(lib, tables[:1], [0, 1], 16)   # fewer rows than tokens, no token_rows
    assert st == INVALID


def test_package_import_does_not_need_a_gpu():
    import paged_kv_cache_155_gb300 as pkv
    assert callable(pkv.paged_attention_decode)


def test_shared_prefix_decode_rejects_bad_arguments_on_host(lib):
    def call(**kw):
        a = dict(q=16, k=16, v=16, nb=64, stride=2 * 2 * 16 * 128, pt=16, plen=256, bt=16, mb=32,
                 cl=16, maxl=400, b=4, hq=8, hkv=2, d=128, bs=16, out=16, ws=16, wsb=1 << 20,
                 part=0, dt=1)
        a.update(kw)
        return lib.pkv_paged_attention_decode_shared_prefix(
            a["q"], a["k"], a["v"], a["nb"], a["stride"], a["pt"], a["plen"], a["bt"], a["mb"],
            a["cl"], a["maxl"], a["b"], a["hq"], a["hkv"], a["d"], a["bs"], 0.088, a["out"],
            a["ws"], a["wsb"], a["part"], a["dt"], None)
    assert call(d=64) == UNSUPPORTED              # the prefix tiles are built for head_dim 128
    assert call(plen=250) == INVALID              # not a multiple of block_size
    assert call(plen=0) == INVALID
    assert call(plen=512) == INVALID              # longer than max_context_len
    assert call(pt=0) == INVALID                  # no prefix table
    assert call(ws=0) == INVALID                  # the workspace is required
    assert call(hq=6, hkv=4) == INVALID
