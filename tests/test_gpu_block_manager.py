"""A small serving loop on the GPU driven by the native block manager:
prefill, decode steps over a batch, beam-style forks (copy-on-write) and frees.
Each step's device calls (copy_blocks, reshape_and_cache, paged_attention_decode)
take exactly the manager's outputs; the same outputs drive the oracle's byte ops
on a host pool, and the decode output is compared with the oracle every step."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_155_gb300 as pkv
from paged_kv_cache_155_gb300.block_manager import BlockManager
from tests._gpu_helpers import assert_close, check_no_device_flags, device
from tests._paged_helpers import dtype_code, to_bits

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("hq,hkv,d,bs,dtype", [(32, 8, 128, 16, torch.bfloat16),
                                               (8, 8, 64, 8, torch.float16)])
def test_serving_loop_with_forks(hq, hkv, d, bs, dtype):
    dev = device()
    g = torch.Generator(device=dev).manual_seed(hq + d)
    nb, mb = 256, 64
    bm = BlockManager(nb, bs, mb)
    kv = torch.randn((nb, 2, hkv, bs, d), generator=g, device=dev).to(dtype)
    k_cache, v_cache = pkv.split_pool(kv)
    host = to_bits(kv.cpu())
    rng = np.random.default_rng(0)

    # prefill three sequences with 40..200 tokens in one cache write
    seqs = [0, 1, 2]
    slots = []
    for s, n in zip(seqs, (40, 131, 200)):
        bm.add_sequence(s)
        for _ in range(n):
            slot, cow = bm.append_token(s)
            slots.append(slot)
    kn = torch.randn((len(slots), hkv, d), generator=g, device=dev).to(dtype)
    vn = torch.randn((len(slots), hkv, d), generator=g, device=dev).to(dtype)
    sm = torch.tensor(slots, dtype=torch.int64)
    pkv.reshape_and_cache(kn, vn, sm.to(dev), k_cache, v_cache)
    oracle.reshape_and_cache(to_bits(kn.cpu()), to_bits(vn.cpu()), sm.numpy(), host, hkv, bs, d)

    next_id = 3
    for step_no in range(24):
        if step_no % 6 == 2:                       # a beam branch off a random live sequence
            bm.fork(int(rng.choice(seqs)), next_id)
            seqs.append(next_id)
            next_id += 1
        if step_no == 15:                          # one request finishes
            bm.free_sequence(seqs.pop(0))
        st = bm.decode_step(seqs)
        b = len(seqs)
        cow = torch.from_numpy(st["cow_pairs"])
        if len(cow):
            pkv.copy_blocks(k_cache, v_cache, cow.to(dev))
            oracle.copy_blocks(host, cow.numpy(), hkv, bs, d)
        kn = torch.randn((b, hkv, d), generator=g, device=dev).to(dtype)
        vn = torch.randn((b, hkv, d), generator=g, device=dev).to(dtype)
        pkv.reshape_and_cache(kn, vn, torch.from_numpy(st["slot_mapping"]).to(dev), k_cache, v_cache)
        oracle.reshape_and_cache(to_bits(kn.cpu()), to_bits(vn.cpu()), st["slot_mapping"], host,
                                 hkv, bs, d)
        q = torch.randn((b, hq, d), generator=g, device=dev).to(dtype)
        tables = torch.from_numpy(st["block_tables"]).to(dev)
        lens = torch.from_numpy(st["context_lens"]).to(dev)
        out = pkv.paged_attention_decode(q, k_cache, v_cache, tables, lens, 1.0 / d ** 0.5,
                                         max_context_len=int(st["context_lens"].max()))
        torch.cuda.synchronize()
        check_no_device_flags(dev)
        flat = host.reshape(-1)
        half = hkv * bs * d
        ref = oracle.paged_decode(to_bits(q.cpu()), flat, flat[half:], 2 * half, st["block_tables"],
                                  st["context_lens"], hkv, bs, 1.0 / d ** 0.5, dtype_code(dtype))
        assert_close(out, ref, what=f"step {step_no}")
    # the device pool and the oracle's pool went through the same writes and copies
    assert np.array_equal(to_bits(kv.cpu()), host)
