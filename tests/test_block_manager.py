"""Host block manager (native, no GPU): block-table growth, slot rule, sharing,
copy-on-write and the free pool, checked against the oracle's slot rule and byte
operations and against the pages' worked example."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_155_gb300.block_manager import BlockManager, OutOfBlocks
from tests._paged_helpers import random_bits
from tests.conftest import read_golden


def _grow(bm, seq, n):
    slots = []
    for _ in range(n):
        slot, cow = bm.append_token(seq)
        assert cow == (-1, -1)
        slots.append(slot)
    return slots


def test_worked_example_growth_and_slots():
    gold = read_golden("worked_example_block_table.txt")
    bs, n = int(gold["block_size"]), int(gold["context_len"])
    bm = BlockManager(num_blocks=20, block_size=bs, max_blocks_per_seq=16)
    bm.add_sequence(0)
    slots = _grow(bm, 0, n)
    table = bm.block_table(0)
    assert len(table) == int(gold["num_blocks"])
    assert n - (len(table) - 1) * bs == int(gold["last_block_tokens"])
    for t, s in enumerate(slots):
        assert s == oracle.slot_for_position(np.array(table, dtype=np.int32), t, bs)
    assert bm.num_free == 20 - 7


def test_table_grows_exactly_when_a_new_block_is_needed():
    for bs in (8, 16, 32):
        bm = BlockManager(64, bs, 64)
        bm.add_sequence(7)
        for t in range(5 * bs):
            bm.append_token(7)
            assert len(bm.block_table(7)) == oracle.blocks_needed(t, bs)
            assert bm.seq_len(7) == t + 1


def test_fork_shares_blocks_and_copy_on_write_gives_private_copies():
    bm = BlockManager(32, 16, 16)
    bm.add_sequence(0)
    _grow(bm, 0, 30)                         # blocks b0 (full) and b1 (14 tokens)
    b0, b1 = bm.block_table(0)
    bm.fork(0, 1)                            # a beam-search branch at token 30
    assert bm.refcount(b0) == 2 and bm.refcount(b1) == 2
    slot, cow = bm.append_token(1)           # the branch writes into the shared last block
    assert cow[0] == b1 and cow[1] not in (b0, b1)
    assert bm.block_table(1) == [b0, cow[1]]
    assert slot == cow[1] * 16 + 14
    assert bm.refcount(b1) == 1 and bm.refcount(cow[1]) == 1 and bm.refcount(b0) == 2
    slot, cow = bm.append_token(0)           # the parent now owns b1 alone: no copy
    assert cow == (-1, -1) and slot == b1 * 16 + 14
    bm.free_sequence(0)
    bm.free_sequence(1)
    assert bm.num_free == 32                 # every reference count returned to zero
    assert all(bm.refcount(b) == 0 for b in range(32))


def test_share_prefix_reuses_full_blocks():
    bm = BlockManager(16, 8, 8)
    bm.add_sequence(0)
    _grow(bm, 0, 20)
    bm.add_sequence(1)
    bm.share_prefix(0, 1, 16)
    assert bm.block_table(1) == bm.block_table(0)[:2]
    assert bm.seq_len(1) == 16
    slot, cow = bm.append_token(1)           # position 16 starts a fresh private block
    assert cow == (-1, -1) and bm.block_table(1)[2] not in bm.block_table(0)
    with pytest.raises(Exception):
        bm.share_prefix(0, 1, 8)             # destination not empty


def test_out_of_blocks_raises_and_changes_nothing():
    bm = BlockManager(2, 4, 8)
    bm.add_sequence(0)
    _grow(bm, 0, 8)
    assert bm.num_free == 0
    with pytest.raises(OutOfBlocks):
        bm.append_token(0)
    assert bm.seq_len(0) == 8 and len(bm.block_table(0)) == 2
    bm.add_sequence(1)
    with pytest.raises(OutOfBlocks):
        bm.decode_step([1])
    assert bm.seq_len(1) == 0


def test_decode_step_capacity_is_exact_for_forked_sequences():
    # two branches share a partial last block; one free block suffices (one copy, one in place)
    bm = BlockManager(3, 4, 8)
    bm.add_sequence(0)
    _grow(bm, 0, 6)                          # two blocks, one free left
    bm.fork(0, 1)
    step = bm.decode_step([0, 1])
    assert len(step["cow_pairs"]) == 1
    assert bm.num_free == 0
    assert step["context_lens"].tolist() == [7, 7]


def test_decode_step_matches_single_appends_and_rejects_duplicates():
    bm = BlockManager(64, 16, 8)
    for s in range(3):
        bm.add_sequence(s)
        _grow(bm, s, 5 + 13 * s)
    step = bm.decode_step([2, 0, 1])
    for row, s in enumerate([2, 0, 1]):
        table = bm.block_table(s)
        assert step["block_tables"][row, :len(table)].tolist() == table
        assert step["context_lens"][row] == bm.seq_len(s)
        t = bm.seq_len(s) - 1
        assert step["slot_mapping"][row] == oracle.slot_for_position(np.array(table, np.int32), t, 16)
    with pytest.raises(Exception):
        bm.decode_step([0, 0])


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_random_serving_history_never_mixes_sequences(seed):
    """Random appends, forks (beam branches), prefix shares and frees.  Applying
    the manager's copy-on-write pairs and slots with the oracle's byte ops to a
    host pool, every live sequence must read back exactly its own token history."""
    rng = np.random.default_rng(seed)
    hkv, bs, d = 2, 8, 64
    nb, mb = 96, 16
    bm = BlockManager(nb, bs, mb)
    pool = random_bits((nb, 2, hkv, bs, d), torch.float16, torch.Generator().manual_seed(seed))
    history = {}          # seq id -> list of (k row, v row) bit arrays, one per token
    next_id = 0
    for _ in range(400):
        op = rng.random()
        live = sorted(history)
        if not live or op < 0.08:
            bm.add_sequence(next_id)
            history[next_id] = []
            next_id += 1
        elif op < 0.14:
            parent = live[rng.integers(len(live))]
            bm.fork(parent, next_id)
            history[next_id] = list(history[parent])
            next_id += 1
        elif op < 0.18:
            src = live[rng.integers(len(live))]
            n_full = (len(history[src]) // bs) * bs
            if n_full:
                bm.add_sequence(next_id)
                bm.share_prefix(src, next_id, n_full)
                history[next_id] = list(history[src][:n_full])
                next_id += 1
        elif op < 0.24 and len(live) > 1:
            victim = live[rng.integers(len(live))]
            bm.free_sequence(victim)
            del history[victim]
        else:
            batch = [s for s in live if len(history[s]) < mb * bs]
            batch = list(rng.permutation(batch))[:5]
            if not batch:
                continue
            try:
                step = bm.decode_step(batch)
            except OutOfBlocks:
                continue
            oracle.copy_blocks(pool, step["cow_pairs"], hkv, bs, d)
            kn = rng.integers(0, 65536, (len(batch), hkv, d), dtype=np.uint16) & 0x3bff
            vn = rng.integers(0, 65536, (len(batch), hkv, d), dtype=np.uint16) & 0x3bff
            oracle.reshape_and_cache(kn, vn, step["slot_mapping"], pool, hkv, bs, d)
            for row, s in enumerate(batch):
                history[s].append((kn[row], vn[row]))
        # invariant: each live sequence reads its own history through its table
        for s, hist in history.items():
            table = bm.block_table(s)
            assert len(table) == (len(hist) + bs - 1) // bs
            for t, (k, v) in enumerate(hist):
                blk, off = table[t // bs], t % bs
                assert np.array_equal(pool[blk, 0, :, off, :], k)
                assert np.array_equal(pool[blk, 1, :, off, :], v)
    # reference counts equal the number of tables naming each block
    counts = np.zeros(nb, dtype=np.int64)
    for s in history:
        for b in bm.block_table(s):
            counts[b] += 1
    assert [bm.refcount(b) for b in range(nb)] == counts.tolist()
    assert bm.num_free == int((counts == 0).sum())
