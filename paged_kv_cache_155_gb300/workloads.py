"""Seeded synthetic decode workloads (inputs only).

This module draws the inputs that both the CUDA path and the CPU oracle
consume: the physical KV pool, the queries, the block tables (a seeded random
placement of each sequence's logical blocks in the pool), the context lengths,
the new token's K/V rows and, for the shared-prefix workload, the
copy-on-write pairs.  It holds none of the method's arithmetic: no slot
addressing, no attention.  Each side derives slot mappings itself.

Every tensor is drawn from ``torch.Generator`` seeds, values N(0, 1) in the
stated 16-bit dtype.  The whole pool is filled (unused blocks included) so
that a read of a stale or wrong block shows up as a wrong result.

The five named workloads follow the shapes the pages discuss:
  tiny    -- 4 sequences, context lengths {1, 17, 100, 33}, MHA 4 heads,
             head_dim 64, block_size 16, 64-block pool; the 100-token
             sequence uses the block table [7, 2, 9, 1, 5, 8, 3] of the worked
             example in "KV Cache与PagedAttention深度解析" §4.2.
  mha7b   -- Llama-2-7B-shaped MHA layer: 32 heads, head_dim 128, bs 16,
             32 sequences of 4096 tokens, 8192-block pool fully used.
  gqa7b   -- 7B GQA layer: 32 q / 8 kv heads, 64 sequences, lengths U[128, 8192].
  prefix  -- shared 2048-token prefix (64 blocks of 32) in every table plus a
             private suffix U[64, 1024]; bf16; 128 copy-on-write pairs.
  long70b -- Llama-2-70B-shaped GQA: 64 q / 8 kv heads, 16 sequences of 32768.

An extra decode shape, outside the pages' configurations, exercises groups of 16
query heads per KV head (one 16-head block per KV head):
  gqa16   -- 128 q / 8 kv heads, head_dim 128, bs 16, 16 sequences of 8192, bf16.

Chunked-prefill workloads (prefill7b, chunked70b) are described at
make_prefill_workload below.

INT8-cache variants (``kv_dtype=torch.int8``; "KV Cache从原理到实战" §5.2):
the pool holds codes drawn as round(32 * N(0, 1)) clipped to [-127, 127] (the
codes a Gaussian channel quantised with its maximum near 4 sigma would have),
and every (KV head, channel) gets a K and a V scale sigma_c / 32 with
sigma_c ~ U[0.5, 1.5], so dequantised values are N(0, sigma_c^2).  The new
token's rows stay 16-bit (the cache write quantises them).  mha7b_int8,
gqa7b_int8 and long70b_int8 are the named shapes above over such a pool.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional, Sequence

import torch

WORKED_EXAMPLE_TABLE = [7, 2, 9, 1, 5, 8, 3]


@dataclass
class DecodeWorkload:
    name: str
    dtype: torch.dtype
    num_seqs: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    kv: torch.Tensor                 # [num_blocks, 2, Hkv, bs, d] pool
    q: torch.Tensor                  # [B, Hq, d]
    block_tables: torch.Tensor       # [B, max_blocks_per_seq] int32 (unused entries = 0)
    context_lens: torch.Tensor       # [B] int32, counting the new token
    k_new: torch.Tensor              # [B, Hkv, d] the new token's K row per sequence
    v_new: torch.Tensor              # [B, Hkv, d]
    new_positions: torch.Tensor      # [B] int64 logical position of the new token (= len - 1)
    scale: float
    k_scale: Optional[torch.Tensor] = None            # INT8 pool: [Hkv, d] float32
    v_scale: Optional[torch.Tensor] = None
    cow_pairs: Optional[torch.Tensor] = None          # [n, 2] int64 (src, dst)
    block_tables_after_cow: Optional[torch.Tensor] = None
    shared_prefix_blocks: int = 0
    meta: dict = field(default_factory=dict)

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def max_context_len(self) -> int:
        return int(self.context_lens.max().item()) if self.num_seqs else 0

    @property
    def k_cache(self) -> torch.Tensor:
        return self.kv[:, 0]

    @property
    def v_cache(self) -> torch.Tensor:
        return self.kv[:, 1]

    def to(self, device) -> "DecodeWorkload":
        moved = {}
        for name in ("kv", "q", "block_tables", "context_lens", "k_new", "v_new",
                     "new_positions", "k_scale", "v_scale", "cow_pairs", "block_tables_after_cow"):
            t = getattr(self, name)
            moved[name] = None if t is None else t.to(device)
        return DecodeWorkload(
            name=self.name, dtype=self.dtype, num_seqs=self.num_seqs,
            num_q_heads=self.num_q_heads, num_kv_heads=self.num_kv_heads,
            head_dim=self.head_dim, block_size=self.block_size, num_blocks=self.num_blocks,
            scale=self.scale, shared_prefix_blocks=self.shared_prefix_blocks,
            meta=dict(self.meta), **moved)


def _randn(shape, dtype, gen, device):
    return torch.randn(shape, generator=gen, device=device, dtype=torch.float32).to(dtype)


def make_decode_workload(*, name: str = "custom", num_seqs: int, num_q_heads: int,
                         num_kv_heads: int, head_dim: int, block_size: int,
                         context_lens: Sequence[int], num_blocks: Optional[int] = None,
                         dtype: torch.dtype = torch.float16, seed: int = 0,
                         device: str = "cpu", shared_prefix_tokens: int = 0,
                         fixed_tables: Optional[dict] = None, cow_last_prefix_block: bool = False,
                         max_blocks_per_seq: Optional[int] = None,
                         kv_dtype: Optional[torch.dtype] = None) -> DecodeWorkload:
    """Build a seeded workload.

    ``context_lens`` are the per-sequence lengths (the new token included).
    With ``shared_prefix_tokens`` > 0 (a multiple of block_size) every table
    starts with the same prefix blocks.  ``fixed_tables`` maps a sequence index
    to an explicit list of physical blocks.  ``cow_last_prefix_block`` adds one
    copy-on-write pair per sequence: the last shared prefix block to a fresh
    private block, and the tables that point at the copies.  ``kv_dtype=torch.int8``
    draws an INT8 pool and per-channel scales (module docstring); ``dtype`` stays
    the type of the queries and of the new rows.
    """
    lens = [int(x) for x in context_lens]
    assert len(lens) == num_seqs and num_q_heads % num_kv_heads == 0
    bs = block_size
    gen_cpu = torch.Generator().manual_seed(seed)
    if shared_prefix_tokens:
        assert shared_prefix_tokens % bs == 0
        assert all(n >= shared_prefix_tokens for n in lens)
    prefix_blocks = shared_prefix_tokens // bs
    need = [math.ceil(n / bs) for n in lens]
    private = [need[i] - prefix_blocks for i in range(num_seqs)]
    fixed_tables = fixed_tables or {}
    total = prefix_blocks + sum(private[i] for i in range(num_seqs) if i not in fixed_tables)
    total_fixed = sum(len(v) for v in fixed_tables.values())
    n_cow = num_seqs if (cow_last_prefix_block and prefix_blocks) else 0
    if num_blocks is None:
        num_blocks = total + total_fixed + n_cow
    mb = max_blocks_per_seq or max([1] + need)
    assert mb >= max([0] + need)

    # seeded random placement of logical blocks in the pool
    reserved = set()
    for v in fixed_tables.values():
        reserved.update(int(b) for b in v)
    perm = [int(b) for b in torch.randperm(num_blocks, generator=gen_cpu).tolist() if b not in reserved]
    assert len(perm) >= total + n_cow, "pool too small for the requested lengths"
    cursor = 0
    prefix = perm[cursor:cursor + prefix_blocks]
    cursor += prefix_blocks
    tables = torch.zeros((num_seqs, mb), dtype=torch.int32)
    for i in range(num_seqs):
        if i in fixed_tables:
            row = [int(b) for b in fixed_tables[i]]
            assert len(row) == need[i]
        else:
            row = prefix + perm[cursor:cursor + private[i]]
            cursor += private[i]
        if row:
            tables[i, :len(row)] = torch.tensor(row, dtype=torch.int32)

    cow_pairs = tables_after = None
    if n_cow:
        fresh = perm[cursor:cursor + n_cow]
        cursor += n_cow
        src = prefix[-1]
        cow_pairs = torch.tensor([[src, fresh[i]] for i in range(num_seqs)], dtype=torch.int64)
        tables_after = tables.clone()
        tables_after[:, prefix_blocks - 1] = torch.tensor(fresh, dtype=torch.int32)

    gen = torch.Generator(device=device).manual_seed(seed + 1)
    k_scale = v_scale = None
    if kv_dtype == torch.int8:
        kv = torch.randn((num_blocks, 2, num_kv_heads, bs, head_dim), generator=gen,
                         device=device).mul_(32).round_().clamp_(-127, 127).to(torch.int8)
        sig = torch.rand((2, num_kv_heads, head_dim), generator=gen, device=device) + 0.5
        k_scale, v_scale = (sig[0] / 32).contiguous(), (sig[1] / 32).contiguous()
    else:
        assert kv_dtype in (None, dtype)
        kv = _randn((num_blocks, 2, num_kv_heads, bs, head_dim), dtype, gen, device)
    q = _randn((num_seqs, num_q_heads, head_dim), dtype, gen, device)
    k_new = _randn((num_seqs, num_kv_heads, head_dim), dtype, gen, device)
    v_new = _randn((num_seqs, num_kv_heads, head_dim), dtype, gen, device)
    ctx = torch.tensor(lens, dtype=torch.int32)
    pos = (ctx.to(torch.int64) - 1)
    return DecodeWorkload(
        name=name, dtype=dtype, num_seqs=num_seqs, num_q_heads=num_q_heads,
        num_kv_heads=num_kv_heads, head_dim=head_dim, block_size=bs, num_blocks=num_blocks,
        kv=kv, q=q, block_tables=tables.to(device), context_lens=ctx.to(device),
        k_new=k_new, v_new=v_new, new_positions=pos.to(device),
        scale=1.0 / math.sqrt(head_dim), k_scale=k_scale, v_scale=v_scale,
        cow_pairs=None if cow_pairs is None else cow_pairs.to(device),
        block_tables_after_cow=None if tables_after is None else tables_after.to(device),
        shared_prefix_blocks=prefix_blocks, meta={"seed": seed})


def _uniform_lens(n, lo, hi, seed):
    g = torch.Generator().manual_seed(seed + 1000)
    return torch.randint(lo, hi + 1, (n,), generator=g).tolist()


# Named workloads.  ``scale_seqs`` shrinks the batch (same per-sequence shape)
# so the parity tests can run a small copy that the oracle finishes quickly.
def tiny(device="cpu", seed=0):
    return make_decode_workload(
        name="tiny", num_seqs=4, num_q_heads=4, num_kv_heads=4, head_dim=64, block_size=16,
        context_lens=[1, 17, 100, 33], num_blocks=64, dtype=torch.float16, seed=seed,
        device=device, fixed_tables={2: WORKED_EXAMPLE_TABLE})


def mha7b(device="cpu", seed=1, num_seqs=32, context_len=4096, num_blocks=None, kv_dtype=None):
    nb = num_blocks if num_blocks is not None else num_seqs * math.ceil(context_len / 16)
    return make_decode_workload(
        name="mha7b" + ("_int8" if kv_dtype == torch.int8 else ""), num_seqs=num_seqs,
        num_q_heads=32, num_kv_heads=32, head_dim=128, block_size=16,
        context_lens=[context_len] * num_seqs, num_blocks=nb, dtype=torch.float16, seed=seed,
        device=device, kv_dtype=kv_dtype)


def gqa7b(device="cpu", seed=2, num_seqs=64, lo=128, hi=8192, num_blocks=32768, kv_dtype=None):
    lens = _uniform_lens(num_seqs, lo, hi, seed)
    nb = max(num_blocks, sum(math.ceil(n / 16) for n in lens))
    return make_decode_workload(
        name="gqa7b" + ("_int8" if kv_dtype == torch.int8 else ""), num_seqs=num_seqs,
        num_q_heads=32, num_kv_heads=8, head_dim=128, block_size=16, context_lens=lens,
        num_blocks=nb, dtype=torch.float16, seed=seed, device=device,
        max_blocks_per_seq=math.ceil(hi / 16), kv_dtype=kv_dtype)


def prefix(device="cpu", seed=3, num_seqs=128, prefix_tokens=2048, lo=64, hi=1024,
           num_blocks=8192):
    suffix = _uniform_lens(num_seqs, lo, hi, seed)
    lens = [prefix_tokens + s for s in suffix]
    return make_decode_workload(
        name="prefix", num_seqs=num_seqs, num_q_heads=32, num_kv_heads=8, head_dim=128,
        block_size=32, context_lens=lens, num_blocks=num_blocks, dtype=torch.bfloat16,
        seed=seed, device=device, shared_prefix_tokens=prefix_tokens,
        cow_last_prefix_block=True, max_blocks_per_seq=(prefix_tokens + hi + 31) // 32)


def long70b(device="cpu", seed=4, num_seqs=16, context_len=32768, num_blocks=None,
            kv_dtype=None):
    nb = num_blocks if num_blocks is not None else num_seqs * math.ceil(context_len / 16)
    return make_decode_workload(
        name="long70b" + ("_int8" if kv_dtype == torch.int8 else ""), num_seqs=num_seqs,
        num_q_heads=64, num_kv_heads=8, head_dim=128, block_size=16,
        context_lens=[context_len] * num_seqs, num_blocks=nb, dtype=torch.bfloat16, seed=seed,
        device=device, kv_dtype=kv_dtype)


def gqa16(device="cpu", seed=8, num_seqs=16, context_len=8192, num_blocks=None):
    nb = num_blocks if num_blocks is not None else num_seqs * math.ceil(context_len / 16)
    return make_decode_workload(
        name="gqa16", num_seqs=num_seqs, num_q_heads=128, num_kv_heads=8, head_dim=128,
        block_size=16, context_lens=[context_len] * num_seqs, num_blocks=nb,
        dtype=torch.bfloat16, seed=seed, device=device)


def mha7b_int8(device="cpu", seed=1, **kw):
    return mha7b(device=device, seed=seed, kv_dtype=torch.int8, **kw)


def gqa7b_int8(device="cpu", seed=2, **kw):
    return gqa7b(device=device, seed=seed, kv_dtype=torch.int8, **kw)


def long70b_int8(device="cpu", seed=4, **kw):
    return long70b(device=device, seed=seed, kv_dtype=torch.int8, **kw)


# ---------------------------------------------------------------------------
# Chunked prefill workloads ("大模型 (LLM) 推理加速核心技术解析" §2; "KV Cache从原理到实战"
# §2.3 / §5.4): each sequence has ``cached`` tokens already in the cache and a
# chunk of ``chunk`` new tokens whose K/V rows are written at the positions
# that follow; every chunk row is a query.
# ---------------------------------------------------------------------------
@dataclass
class PrefillWorkload:
    name: str
    dtype: torch.dtype
    num_seqs: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    kv: torch.Tensor                 # [num_blocks, 2, Hkv, bs, d]
    q: torch.Tensor                  # [num_rows, Hq, d], the chunks back to back
    k_new: torch.Tensor              # [num_rows, Hkv, d]
    v_new: torch.Tensor
    new_positions: torch.Tensor      # [num_rows] int64, absolute position of each chunk row
    row_seq: torch.Tensor            # [num_rows] int64, the sequence of each chunk row
    block_tables: torch.Tensor       # [B, max_blocks_per_seq] int32
    query_start: torch.Tensor        # [B + 1] int32
    context_lens: torch.Tensor       # [B] int32, chunk included
    chunk_lens: list
    scale: float
    meta: dict = field(default_factory=dict)

    @property
    def num_rows(self) -> int:
        return int(self.q.shape[0])

    @property
    def max_query_len(self) -> int:
        return max([0] + list(self.chunk_lens))

    @property
    def max_context_len(self) -> int:
        return int(self.context_lens.max().item()) if self.num_seqs else 0


def make_prefill_workload(*, name: str = "prefill", num_q_heads: int, num_kv_heads: int,
                          head_dim: int, block_size: int, cached_lens: Sequence[int],
                          chunk_lens: Sequence[int], dtype: torch.dtype = torch.float16,
                          seed: int = 0, device: str = "cpu", num_blocks: Optional[int] = None,
                          extra_rows: int = 0) -> PrefillWorkload:
    """Seeded chunked-prefill inputs.  ``extra_rows`` appends query rows that belong
    to no sequence (the call must leave their output untouched)."""
    cached = [int(x) for x in cached_lens]
    chunks = [int(x) for x in chunk_lens]
    assert len(cached) == len(chunks)
    b, bs = len(chunks), block_size
    lens = [c + n for c, n in zip(cached, chunks)]
    need = [math.ceil(n / bs) for n in lens]
    total = sum(need)
    nb = num_blocks if num_blocks is not None else total + 8
    assert nb >= total
    gen_cpu = torch.Generator().manual_seed(seed)
    perm = torch.randperm(nb, generator=gen_cpu).tolist()
    mb = max([1] + need)
    tables = torch.zeros((b, mb), dtype=torch.int32)
    cur = 0
    for i, n in enumerate(need):
        if n:
            tables[i, :n] = torch.tensor(perm[cur:cur + n], dtype=torch.int32)
        cur += n
    qs = [0]
    for n in chunks:
        qs.append(qs[-1] + n)
    rows = qs[-1] + extra_rows
    pos, seq_of = [], []
    for i, (c, n) in enumerate(zip(cached, chunks)):
        pos += list(range(c, c + n))
        seq_of += [i] * n
    gen = torch.Generator(device=device).manual_seed(seed + 1)
    kv = _randn((nb, 2, num_kv_heads, bs, head_dim), dtype, gen, device)
    q = _randn((rows, num_q_heads, head_dim), dtype, gen, device)
    k_new = _randn((qs[-1], num_kv_heads, head_dim), dtype, gen, device)
    v_new = _randn((qs[-1], num_kv_heads, head_dim), dtype, gen, device)
    return PrefillWorkload(
        name=name, dtype=dtype, num_seqs=b, num_q_heads=num_q_heads, num_kv_heads=num_kv_heads,
        head_dim=head_dim, block_size=bs, num_blocks=nb, kv=kv, q=q, k_new=k_new, v_new=v_new,
        new_positions=torch.tensor(pos, dtype=torch.int64).to(device),
        row_seq=torch.tensor(seq_of, dtype=torch.int64).to(device),
        block_tables=tables.to(device), query_start=torch.tensor(qs, dtype=torch.int32).to(device),
        context_lens=torch.tensor(lens, dtype=torch.int32).to(device), chunk_lens=chunks,
        scale=1.0 / math.sqrt(head_dim), meta={"seed": seed, "cached": cached})


def prefill7b(device="cpu", seed=5, num_seqs=4, prompt=2048):
    """Whole prompts: 4 sequences of 2048 new tokens on an empty cache, Llama-2-7B MHA
    layer (32 heads of 128), block 16, fp16."""
    return make_prefill_workload(
        name="prefill7b", num_q_heads=32, num_kv_heads=32, head_dim=128, block_size=16,
        cached_lens=[0] * num_seqs, chunk_lens=[prompt] * num_seqs, dtype=torch.float16,
        seed=seed, device=device)


def chunked70b(device="cpu", seed=6, num_seqs=8, chunk=512, hi=7680):
    """Chunked prefill behind long contexts: 8 sequences, each a 512-token chunk after
    U[0, 7680] cached tokens, Llama-2-70B GQA layer (64 q / 8 kv heads), block 16, bf16."""
    cached = _uniform_lens(num_seqs, 0, hi, seed)
    return make_prefill_workload(
        name="chunked70b", num_q_heads=64, num_kv_heads=8, head_dim=128, block_size=16,
        cached_lens=cached, chunk_lens=[chunk] * num_seqs, dtype=torch.bfloat16, seed=seed,
        device=device)


PREFILL_NAMED = {"prefill7b": prefill7b, "chunked70b": chunked70b}


NAMED = {"tiny": tiny, "mha7b": mha7b, "gqa7b": gqa7b, "prefix": prefix, "long70b": long70b,
         "mha7b_int8": mha7b_int8, "gqa7b_int8": gqa7b_int8, "long70b_int8": long70b_int8,
         "gqa16": gqa16}

# The default partition size each named workload is run with (0 = library's choice).
DEFAULT_PARTITION = {"tiny": 0, "mha7b": 0, "gqa7b": 0, "prefix": 0, "long70b": 512,
                     "mha7b_int8": 0, "gqa7b_int8": 0, "long70b_int8": 0, "gqa16": 0}
