"""Benchmark of the paged decode step on GB300.

A step is one pass of the hot path over one batch: the cache write of each
sequence's new token (reshape_and_cache) followed by paged decode attention
(plus the split-context merge when the plan splits).  The default workload is
the Llama-2-7B-shaped MHA decode layer (32 sequences x 4096 tokens, 32 heads of
128, block 16, fp16, 2 GiB pool -- larger than L2, so no flush is needed).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload mha7b|gqa7b|prefix|long70b|tiny|mha7b_int8|gqa7b_int8|long70b_int8|gqa16]
                    [--partition P]

Prints one JSON line (rank 0).  `value` is decode tokens/s (one token per
sequence per step) over all ranks, device-timed with inputs resident in HBM;
`e2e` is the same metric through the Python API (calls prepared once on their
buffers, re-issued each step) with each step's inputs copied
from pinned host memory and its output copied back inside the timed region, as a
serving loop runs it: two sets of device buffers, the copies on their own
streams, so step i's copies overlap step i-1's kernels (`e2e.serial_value` is
the same loop with every copy on the compute stream).
`roofline` reports the decode kernel's algorithmic KV+q+out bytes per launch
over its CUDA-event time against the measured HBM copy bandwidth.
`--impl reference` times the CPU oracle (the reference arm of this build) on
bounded samples of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import tempfile
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged decode attn tokens/s and KV-read GB/s (% of GB300 HBM peak)"
FALLBACK_HBM_GBS = 6800.0


# --------------------------------------------------------------------------- helpers
def _dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(value, device, world):
    """The largest of every rank's value (the slowest rank's time), or value at N=1."""
    if world <= 1:
        return float(value)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tokens_per_s(world, num_seqs, ms_per_step):
    """Decode tokens/s of all ranks: each rank decodes one token for each of its own
    num_seqs sequences per step (weak scaling), timed by the slowest rank."""
    return world * num_seqs / (ms_per_step / 1000.0)


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def _kernel_source_hash():
    h = hashlib.sha256()
    for name in ("decode_kernel.cuh", "pkv_device.cuh"):
        with open(os.path.join(ROOT, "paged_kv_cache_155_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def _profiled_traffic(workload):
    """DRAM bytes per decode launch from the committed ncu summary, if it was
    taken on the current kernel source (else None)."""
    path = os.path.join(ROOT, "profiles", f"paged_decode_{workload}.md")
    if not os.path.exists(path):
        return None
    text = open(path).read()
    src = re.search(r"kernel_source_hash:\s*([0-9a-f]+)", text)
    val = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
    if not src or not val or src.group(1) != _kernel_source_hash():
        return None
    return float(val.group(1))


class ClockSampler:
    """nvidia-smi clock / throttle-reason sampling during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid=None):
        self.proc = None
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "200"]
        if uuid:
            cmd += ["-i", uuid]
        try:
            self.proc = subprocess.Popen(cmd, stdout=self.file, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.file.flush()
        rows = []
        with open(self.file.name) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    rows.append((float(parts[1]), float(parts[2]), parts[5:9]))
                except ValueError:
                    continue
        os.unlink(self.file.name)
        if not rows:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, r in rows for i in range(4) if r[i].lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows),
                "sm_max_mhz": max(r[1] for r in rows), "reasons": reasons, "samples": len(rows)}


def _algorithmic_bytes(wl):
    """K+V of every context token per KV head (once per GQA group) + q + out
    (+ the per-channel scales of an INT8 cache)."""
    e = wl.kv.element_size()
    tokens = sum(int(x) for x in wl.context_lens.cpu().tolist())
    kv = tokens * 2 * wl.num_kv_heads * wl.head_dim * e
    qo = 2 * wl.num_seqs * wl.num_q_heads * wl.head_dim * wl.q.element_size()
    scales = 2 * wl.num_kv_heads * wl.head_dim * 4 if wl.k_scale is not None else 0
    return kv + qo + scales


def _unique_bytes(wl):
    """Bytes a decode must read at least once: K+V of every distinct context token
    (a prefix shared by every table counted once) + q + out (+ INT8 scales).  Equal
    to the algorithmic bytes except for the shared-prefix workload."""
    if not wl.shared_prefix_blocks:
        return _algorithmic_bytes(wl)
    e = wl.kv.element_size()
    pre = wl.shared_prefix_blocks * wl.block_size
    tokens = pre + sum(int(x) - pre for x in wl.context_lens.cpu().tolist())
    qo = 2 * wl.num_seqs * wl.num_q_heads * wl.head_dim * wl.q.element_size()
    return tokens * 2 * wl.num_kv_heads * wl.head_dim * e + qo


# The pages' five configurations, by workload name.
CONFIG_WORKLOADS = {"1": "tiny", "2": "mha7b", "3": "gqa7b", "4": "prefix", "5": "long70b"}


def _config_summary(main, line, others):
    """Compact per-configuration figures (kept short: the last key of the line)."""
    r3 = lambda x: None if x is None else round(float(x), 3)
    out = {}
    for key, name in CONFIG_WORKLOADS.items():
        if name == main:
            e = {"workload": name, "tokens_per_s": round(line["value"]),
                 "kv_read_gbps": round(line["kv_read_gbps"]),
                 "hbm_frac": r3(line["hbm_frac_of_measured"]),
                 "decode_us": round(line["roofline"]["launch_ms"] * 1e3, 1)}
        else:
            w = others.get(name)
            if w is None:
                continue
            e = {"workload": name, "tokens_per_s": round(w["tokens_per_s"]),
                 "kv_read_gbps": round(w["kv_read_gbps"]), "hbm_frac": r3(w["hbm_frac_of_measured"]),
                 "decode_us": round(w["decode_ms"] * 1e3, 1)}
            if name == "tiny":
                e.update({"eager_us_per_step": round(w["ms_per_step"] * 1e3, 1),
                          "graph_us_per_step": round(w["graph_us_per_step"], 1)})
                e.pop("kv_read_gbps"), e.pop("hbm_frac")
            if name == "prefix":
                c = w["shared_prefix_decode"]
                e = {"workload": "prefix, shared-prefix decode",
                     "tokens_per_s": round(c["tokens_per_s"]), "unique_gbps": round(c["unique_gbps"]),
                     "hbm_frac_unique": r3(c["unique_frac_of_measured"]),
                     "hbm_frac_unique_l2_flushed":
                         r3(c["l2_flushed"]["shared_prefix_unique_frac_of_measured"]),
                     "decode_us": round(c["decode_ms"] * 1e3, 1),
                     "plain_decode_hbm_frac_unique": r3(w["hbm_frac_of_measured"])}
        out[key] = e
    for name in ("mha7b_int8", "gqa7b_int8", "long70b_int8", "gqa16"):
        w = others.get(name)
        if w is not None:
            out[name] = {"hbm_frac": r3(w["hbm_frac_of_measured"]),
                         "decode_us": round(w["decode_ms"] * 1e3, 1)}
    for name in ("prefill7b", "chunked70b"):
        w = others.get(name)
        if w is not None:
            out[name] = {"tflops": round(w["tflops"]), "frac": r3(w["tensor_frac_of_measured_bf16"]),
                         "attention_us": round(w["attention_ms"] * 1e3, 1)}
    return out


def _step_calls(pkv, wl, k_cache, v_cache, out, maxl, part, k_new, v_new, slots, q, bt, cl):
    """(cache write, decode) of one step through the public API, for a 16-bit or an
    INT8 pool, each prepared once on the given buffers (a serving loop reuses its
    buffers; only the library calls are re-issued per step)."""
    if wl.kv.dtype == __import__("torch").int8:
        write = pkv.prepare_reshape_and_cache_int8(k_new, v_new, slots, k_cache, v_cache, wl.k_scale,
                                                   wl.v_scale)
        decode = pkv.prepare_paged_attention_decode_int8(q, k_cache, v_cache, wl.k_scale, wl.v_scale,
                                                         bt, cl, wl.scale, out, max_context_len=maxl,
                                                         partition_size=part)
    else:
        write = pkv.prepare_reshape_and_cache(k_new, v_new, slots, k_cache, v_cache)
        decode = pkv.prepare_paged_attention_decode(q, k_cache, v_cache, bt, cl, wl.scale, out,
                                                    max_context_len=maxl, partition_size=part)
    return write, decode


def _make_workload(name, device, seed, num_seqs=None):
    from paged_kv_cache_155_gb300 import workloads
    kw = {"num_seqs": num_seqs} if (num_seqs and name != "tiny") else {}
    return workloads.NAMED[name](device=device, seed=seed, **kw)


def _workload_config(wl, name, plan, partition):
    lens = wl.context_lens.cpu()
    return {"workload": name, "num_seqs": wl.num_seqs, "num_q_heads": wl.num_q_heads,
            "num_kv_heads": wl.num_kv_heads, "head_dim": wl.head_dim,
            "block_size": wl.block_size, "num_blocks": wl.num_blocks,
            "context_len_min": int(lens.min()), "context_len_max": int(lens.max()),
            "context_tokens": int(lens.sum()), "partition_size": plan["partition_size"],
            "num_partitions": plan["num_partitions"], "partition_arg": partition,
            "kv_dtype": str(wl.kv.dtype).replace("torch.", ""),
            "l2": f"no flush: pool of {wl.kv.numel() * wl.kv.element_size() / 2**30:.2f} GiB "
                  "> 129 MB L2"}


# --------------------------------------------------------------------------- oracle legs
def _oracle_units(wl_host, pool_bits, units, q_bits):
    """Run the oracle on (sequence, KV head) units; returns seconds.  Units of one
    KV head go to the oracle in one call so its OpenMP loop over (sequence,
    query head) pairs can use every core."""
    import numpy as np
    import oracle
    g = wl_host.num_q_heads // wl_host.num_kv_heads
    flat = pool_bits.reshape(-1)
    half = wl_host.num_kv_heads * wl_host.block_size * wl_host.head_dim
    row_off = wl_host.block_size * wl_host.head_dim
    tables = wl_host.block_tables.numpy()
    lens = wl_host.context_lens.numpy()
    code = oracle.BF16 if str(wl_host.dtype).endswith("bfloat16") else oracle.F16
    by_head = {}
    for (i, h) in units:
        by_head.setdefault(h, []).append(i)
    t0 = time.perf_counter()
    for h, seqs in by_head.items():
        sel = np.array(seqs)
        # KV head h alone: shift the K/V bases to head h's rows of block 0
        oracle.paged_decode(q_bits[sel, h * g:(h + 1) * g], flat[h * row_off:],
                            flat[half + h * row_off:], 2 * half, tables[sel], lens[sel],
                            1, wl_host.block_size, wl_host.scale, code)
    return time.perf_counter() - t0


def _oracle_int8_seqs(wl_host, pool_i8, seqs, q_bits):
    """The INT8 oracle on whole sequences (every KV head); returns seconds."""
    import numpy as np
    import oracle
    code = oracle.BF16 if str(wl_host.dtype).endswith("bfloat16") else oracle.F16
    sel = np.array(seqs)
    t0 = time.perf_counter()
    oracle.paged_decode_int8(q_bits[sel], pool_i8, wl_host.k_scale.numpy(), wl_host.v_scale.numpy(),
                             wl_host.block_tables.numpy()[sel], wl_host.context_lens.numpy()[sel],
                             wl_host.num_kv_heads, wl_host.block_size, wl_host.scale, code)
    return time.perf_counter() - t0


def _oracle_sample(wl_host, pool, qb, n, start):
    """The oracle on n work units from `start` on: (sequence, KV head) units of a 16-bit
    pool, whole sequences of an INT8 one.  Returns (seconds, decode tokens done)."""
    if wl_host.k_scale is not None:
        seqs = [(start + k) % wl_host.num_seqs for k in range(n)]
        return _oracle_int8_seqs(wl_host, pool, seqs, qb), float(n)
    return _oracle_units(wl_host, pool, _unit_list(wl_host, n, start), qb), n / wl_host.num_kv_heads


def _pool_host(wl_host):
    """Host pool in the oracle's form: 16-bit patterns, or the INT8 codes."""
    import torch
    if wl_host.kv.dtype == torch.int8:
        return wl_host.kv.contiguous().numpy()
    return _bits(wl_host.kv)


def _unit_list(wl_host, n, start=0):
    total = wl_host.num_seqs * wl_host.num_kv_heads
    out = []
    for k in range(start, start + n):
        k %= total
        out.append((k % wl_host.num_seqs, k // wl_host.num_seqs))
    return out


def _bits(t):
    import numpy as np
    import torch
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def cpu_baseline(wl_dev, budget_s=12.0):
    """The oracle on a bounded sample of the workload, on this host's cores."""
    import oracle
    wl_host = wl_dev.to("cpu")
    pool = _pool_host(wl_host)
    qb = _bits(wl_host.q)
    i8 = wl_host.k_scale is not None
    t1, _ = _oracle_sample(wl_host, pool, qb, 1, 0)
    total = wl_host.num_seqs * (1 if i8 else wl_host.num_kv_heads)
    n = max(1, min(64 * total, int(budget_s / max(t1, 1e-6))))   # whole steps repeat if cheap
    t, tokens = _oracle_sample(wl_host, pool, qb, n, 1)
    unit = "whole sequences" if i8 else "(sequence, KV head) units"
    return {"value": tokens / t, "unit": "tokens/s", "cores": oracle.num_threads(),
            "kind": "oracle",
            "sample": f"{n} {unit} of {wl_host.num_seqs}x{wl_host.num_kv_heads}"
                      f" ({n / total:.3f} steps' worth),"
                      f" {t:.1f} s, fp64 C oracle, OpenMP over query heads"}


def run_reference(args):
    world, rank, _ = _dist_env()
    if rank != 0:
        return 0
    import torch
    import oracle
    oracle.build()
    wl = _make_workload(args.workload, "cpu", 1234, args.num_seqs)
    pool, qb = _pool_host(wl), _bits(wl.q)
    i8 = wl.k_scale is not None
    per_step_budget = max(0.002, 150.0 / max(1, args.steps + args.warmup))
    t1, _ = _oracle_sample(wl, pool, qb, 1, 0)
    n = max(1, min(wl.num_seqs * (1 if i8 else wl.num_kv_heads), int(per_step_budget / max(t1, 1e-6))))
    cursor = 1
    for _ in range(args.warmup):
        _oracle_sample(wl, pool, qb, n, cursor)
        cursor += n
    total, tokens = 0.0, 0.0
    for _ in range(args.steps):
        dt, tk = _oracle_sample(wl, pool, qb, n, cursor)
        total += dt
        tokens += tk
        cursor += n
    value = tokens / total
    ms_full = 1000.0 * wl.num_seqs / value
    unit = "whole sequences" if i8 else "(sequence, KV head) units"
    sample = f"each step {n} {unit} of {wl.num_seqs}x{wl.num_kv_heads}; fp64 C oracle"
    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_full,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "impl": "reference",
            "config": {"workload": args.workload, "num_seqs": wl.num_seqs,
                       "num_q_heads": wl.num_q_heads, "num_kv_heads": wl.num_kv_heads,
                       "head_dim": wl.head_dim, "block_size": wl.block_size},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": oracle.num_threads(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# --------------------------------------------------------------------------- our arm
def measure_workload(pkv, name, dev, steps, peak, partition=None):
    """Device-timed decode step of one named workload (eager launches), the
    decode call's share, and the per-step latency when the step is replayed
    from a CUDA graph (no host launch cost; what a serving loop that captures
    its decode step sees)."""
    import torch
    from paged_kv_cache_155_gb300 import workloads
    wl = _make_workload(name, str(dev), 1234)
    k_cache, v_cache = pkv.split_pool(wl.kv)
    maxl = int(wl.context_lens.max())
    part = workloads.DEFAULT_PARTITION[name] if partition is None else partition
    slots = pkv.slot_mapping(wl.block_tables, wl.new_positions, wl.block_size,
                             num_blocks=wl.num_blocks)
    out = torch.empty_like(wl.q)
    stream = torch.cuda.current_stream(dev)
    write, decode = _step_calls(pkv, wl, k_cache, v_cache, out, maxl, part, wl.k_new, wl.v_new,
                                slots, wl.q, wl.block_tables, wl.context_lens)

    def step():
        write()
        decode()

    for _ in range(5):
        step()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for k in range(steps):
        write()
        ev[k][0].record(stream)
        decode()
        ev[k][1].record(stream)
    t1.record(stream)
    torch.cuda.synchronize()
    ms_step = t0.elapsed_time(t1) / steps
    dec_times = [a.elapsed_time(b) for a, b in ev]
    dec_ms = statistics.median(dec_times)
    nbytes = _algorithmic_bytes(wl)
    unique = _unique_bytes(wl)
    # CUDA-graph replay of `reps` steps
    reps = 50
    side = torch.cuda.Stream(dev)
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        for _ in range(3):
            step()
    stream.wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for _ in range(reps):
            step()
    graph.replay()
    torch.cuda.synchronize()
    g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    g0.record(stream)
    for _ in range(4):
        graph.replay()
    g1.record(stream)
    torch.cuda.synchronize()
    graph_ms = g0.elapsed_time(g1) / (4 * reps)
    flags, names = pkv.get_device_error(dev)
    if flags:
        raise RuntimeError(f"device flags on {name}: {names}")
    result = {"tokens_per_s": wl.num_seqs / (ms_step / 1e3), "ms_per_step": ms_step,
              "decode_ms": dec_ms, "decode_ms_mean": statistics.mean(dec_times),
              "kv_read_gbps": unique / (dec_ms / 1e3) / 1e9,
              "hbm_frac_of_measured": unique / (dec_ms / 1e3) / 1e9 / peak,
              "graph_us_per_step": graph_ms * 1e3,
              "graph_tokens_per_s": wl.num_seqs / (graph_ms / 1e3),
              "algorithmic_bytes": nbytes, "num_seqs": wl.num_seqs,
              "partition_size": part, "kv_dtype": str(wl.kv.dtype).replace("torch.", "")}
    if name == "prefix":
        result["effective_gbps"] = nbytes / (dec_ms / 1e3) / 1e9
        result["note"] = ("kv_read_gbps and hbm_frac count unique bytes (the shared prefix "
                          "once); effective_gbps counts every sequence's prefix reads (logical "
                          "bytes), which after the first touch come from L2")
        # copy-on-write of the last shared prefix block into one private block per sequence
        pairs = wl.cow_pairs
        blk_bytes = 2 * wl.num_kv_heads * wl.block_size * wl.head_dim * 2
        for _ in range(3):
            pkv.copy_blocks(k_cache, v_cache, pairs)
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        c0.record(stream)
        for _ in range(50):
            pkv.copy_blocks(k_cache, v_cache, pairs)
        c1.record(stream)
        torch.cuda.synchronize()
        cms = c0.elapsed_time(c1) / 50
        moved = 2 * pairs.shape[0] * blk_bytes  # read + write
        result["copy_blocks"] = {"pairs": int(pairs.shape[0]), "us": cms * 1e3,
                                 "gbps_read_plus_write": moved / (cms / 1e3) / 1e9}
        # the same step with the shared-prefix (cascade) decode: the 2048-token prefix is
        # attended by all query rows together and read once per 128 rows
        pre_tokens = wl.shared_prefix_blocks * wl.block_size
        pre_table = wl.block_tables[0, :wl.shared_prefix_blocks].contiguous()

        cascade = pkv.prepare_paged_attention_decode_shared_prefix(
            wl.q, k_cache, v_cache, pre_table, pre_tokens, wl.block_tables, wl.context_lens,
            wl.scale, out, max_context_len=maxl)
        for _ in range(5):
            write()
            cascade()
        torch.cuda.synchronize()
        ev2 = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(steps)]
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s0.record(stream)
        for k in range(steps):
            write()
            ev2[k][0].record(stream)
            cascade()
            ev2[k][1].record(stream)
        s1.record(stream)
        torch.cuda.synchronize()
        flags, names = pkv.get_device_error(dev)
        if flags:
            raise RuntimeError(f"device flags on the shared-prefix decode: {names}")
        c_step = s0.elapsed_time(s1) / steps
        c_dec = statistics.median(a.elapsed_time(b) for a, b in ev2)

        # the same two decodes with L2 flushed before every call (a 256 MiB write,
        # outside the timed region): the shared prefix is then read from HBM each time
        flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

        def flushed_ms(call, n=50):
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(n)]
            for a, b in evs:
                flush.fill_(1)
                a.record(stream)
                call()
                b.record(stream)
            torch.cuda.synchronize()
            return statistics.median(a.elapsed_time(b) for a, b in evs)

        plain_flushed = flushed_ms(decode)
        cascade_flushed = flushed_ms(cascade)
        del flush
        result["shared_prefix_decode"] = {
            "tokens_per_s": wl.num_seqs / (c_step / 1e3), "ms_per_step": c_step,
            "decode_ms": c_dec, "speedup_vs_plain_decode": dec_ms / c_dec,
            "unique_bytes": unique, "unique_gbps": unique / (c_dec / 1e3) / 1e9,
            "unique_frac_of_measured": unique / (c_dec / 1e3) / 1e9 / peak,
            "logical_gbps": nbytes / (c_dec / 1e3) / 1e9,
            "l2_flushed": {"plain_decode_ms": plain_flushed, "shared_prefix_decode_ms": cascade_flushed,
                           "plain_unique_gbps": unique / (plain_flushed / 1e3) / 1e9,
                           "shared_prefix_unique_gbps": unique / (cascade_flushed / 1e3) / 1e9,
                           "shared_prefix_unique_frac_of_measured":
                               unique / (cascade_flushed / 1e3) / 1e9 / peak,
                           "note": "256 MiB written before each call, outside the timed region"}}
    del wl, k_cache, v_cache, out, graph
    torch.cuda.empty_cache()
    return result


def _tensor_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        return 1900.0, "fallback"


def measure_prefill(pkv, name, dev, steps):
    """Device-timed chunked-prefill step of one named prefill workload: the chunk
    rows' cache write, then the prefill attention.  Causal FLOPs count 2 * 2 * d
    per (query head, visible token) pair (QK^T and PV)."""
    import torch
    from paged_kv_cache_155_gb300 import workloads
    wl = workloads.PREFILL_NAMED[name](device=str(dev))
    k_cache, v_cache = pkv.split_pool(wl.kv)
    slots = pkv.slot_mapping(wl.block_tables, wl.new_positions, wl.block_size,
                             token_rows=wl.row_seq, num_blocks=wl.num_blocks)
    out = torch.empty_like(wl.q)
    stream = torch.cuda.current_stream(dev)
    mq, mc = wl.max_query_len, wl.max_context_len

    def attn():
        pkv.paged_attention_prefill(wl.q, k_cache, v_cache, wl.block_tables, wl.query_start,
                                    wl.context_lens, wl.scale, out, max_query_len=mq,
                                    max_context_len=mc)

    for _ in range(5):
        pkv.reshape_and_cache(wl.k_new, wl.v_new, slots, k_cache, v_cache)
        attn()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for k in range(steps):
        pkv.reshape_and_cache(wl.k_new, wl.v_new, slots, k_cache, v_cache)
        ev[k][0].record(stream)
        attn()
        ev[k][1].record(stream)
    t1.record(stream)
    torch.cuda.synchronize()
    flags, names = pkv.get_device_error(dev)
    if flags:
        raise RuntimeError(f"device flags on {name}: {names}")
    ms_step = t0.elapsed_time(t1) / steps
    attn_ms = statistics.median(a.elapsed_time(b) for a, b in ev)
    visible = int((wl.new_positions.cpu() + 1).sum())
    flops = 4 * wl.head_dim * wl.num_q_heads * visible
    peak, kind = _tensor_peak()
    tflops = flops / (attn_ms / 1e3) / 1e12
    result = {"tokens_per_s": wl.num_rows / (ms_step / 1e3), "ms_per_step": ms_step,
              "attention_ms": attn_ms, "causal_flops": flops, "tflops": tflops,
              "tensor_frac_of_measured_bf16": tflops / peak, "peak_source": f"{kind} bf16_tflops",
              "num_seqs": wl.num_seqs, "query_rows": wl.num_rows,
              "context_len_max": mc, "chunk_len_max": mq}
    del wl, k_cache, v_cache, out
    torch.cuda.empty_cache()
    return result


def run_ours(args):
    import torch
    import torch.distributed as dist

    world, rank, local = _dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)

    from paged_kv_cache_155_gb300 import _build
    _build.build()
    import paged_kv_cache_155_gb300 as pkv

    wl = _make_workload(args.workload, str(dev), 1234 + rank, args.num_seqs)
    k_cache, v_cache = pkv.split_pool(wl.kv)
    maxl = int(wl.context_lens.max())
    part = args.partition
    sm = torch.cuda.get_device_properties(dev).multi_processor_count
    plan = pkv.decode_plan(wl.num_seqs, wl.num_q_heads, wl.num_kv_heads, wl.head_dim,
                           wl.block_size, maxl, part, sm, int8=wl.kv.dtype == torch.int8)
    slots = pkv.slot_mapping(wl.block_tables, wl.new_positions, wl.block_size,
                             num_blocks=wl.num_blocks)
    out = torch.empty_like(wl.q)
    stream = torch.cuda.current_stream(dev)
    write, decode = _step_calls(pkv, wl, k_cache, v_cache, out, maxl, part, wl.k_new, wl.v_new,
                                slots, wl.q, wl.block_tables, wl.context_lens)

    def step():
        write()
        decode()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    flags, names = pkv.get_device_error(dev)
    if flags:
        raise RuntimeError(f"device flags during warm-up: {names}")

    # ---- device-timed region
    dec_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.steps)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    sampler = ClockSampler(uuid) if rank == 0 else None
    time.sleep(0.25 if sampler else 0)
    launches0 = pkv.launch_count()
    t_start.record(stream)
    for k in range(args.steps):
        write()
        dec_ev[k][0].record(stream)
        decode()
        dec_ev[k][1].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize()
    launches = pkv.launch_count() - launches0
    clocks = sampler.stop() if sampler else None
    if world > 1:
        dist.barrier()
    ms_total = t_start.elapsed_time(t_end)
    dec_times = [a.elapsed_time(b) for a, b in dec_ev]
    dec_ms = statistics.median(dec_times)
    ms_total = max_over_ranks(ms_total, dev, world)
    ms_step = ms_total / args.steps
    value = whole_job_tokens_per_s(world, wl.num_seqs, ms_step)
    flags, names = pkv.get_device_error(dev)
    if flags:
        raise RuntimeError(f"device flags during the timed region: {names}")

    # ---- end to end through the API with host buffers
    pin = lambda t: t.detach().cpu().pin_memory()
    h_q, h_k, h_v = pin(wl.q), pin(wl.k_new), pin(wl.v_new)
    h_slots, h_bt, h_cl = pin(slots), pin(wl.block_tables), pin(wl.context_lens)
    h_out = torch.empty(wl.q.shape, dtype=wl.q.dtype, pin_memory=True)
    d_q, d_k, d_v = torch.empty_like(wl.q), torch.empty_like(wl.k_new), torch.empty_like(wl.v_new)
    d_slots, d_bt, d_cl = torch.empty_like(slots), torch.empty_like(wl.block_tables), \
        torch.empty_like(wl.context_lens)
    h2d = sum(t.numel() * t.element_size() for t in (h_q, h_k, h_v, h_slots, h_bt, h_cl))
    d2h = h_out.numel() * h_out.element_size()
    write_e, decode_e = _step_calls(pkv, wl, k_cache, v_cache, out, maxl, part, d_k, d_v, d_slots,
                                    d_q, d_bt, d_cl)

    def e2e_step():
        for d, h in ((d_q, h_q), (d_k, h_k), (d_v, h_v), (d_slots, h_slots), (d_bt, h_bt),
                     (d_cl, h_cl)):
            d.copy_(h, non_blocking=True)
        write_e()
        decode_e()
        h_out.copy_(out, non_blocking=True)

    def time_loop(one_step, n, tail=None):
        if world > 1:
            dist.barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(n):
            one_step(i)
        if tail is not None:
            tail()
        e1.record(stream)
        torch.cuda.synchronize()
        return max_over_ranks(e0.elapsed_time(e1) / n, dev, world)

    e2e_steps = max(3, args.steps // 2)
    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    serial_ms = time_loop(lambda i: e2e_step(), e2e_steps)

    # the serving-loop form: buffer set i % 2 per step, inputs in on stream cs_in,
    # results out on stream cs_out (one copy stream would queue step i's inputs
    # behind step i-1's result, which waits for step i-1's kernels)
    cs_in, cs_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    sets = []
    for _ in range(2):
        d_in = tuple(torch.empty_like(t) for t in (wl.q, wl.k_new, wl.v_new, slots,
                                                   wl.block_tables, wl.context_lens))
        d_res = torch.empty_like(wl.q)
        h_res = torch.empty(wl.q.shape, dtype=wl.q.dtype, pin_memory=True)
        q_, k_, v_, sl_, bt_, cl_ = d_in
        w_b, dec_b = _step_calls(pkv, wl, k_cache, v_cache, d_res, maxl, part, k_, v_, sl_, q_, bt_,
                                 cl_)
        sets.append({"in": d_in, "res": d_res, "h_res": h_res, "write": w_b, "decode": dec_b,
                     "copied_in": torch.cuda.Event(), "computed": torch.cuda.Event(),
                     "copied_out": torch.cuda.Event()})
    hosts = (h_q, h_k, h_v, h_slots, h_bt, h_cl)

    def pipelined_step(i):
        b = sets[i % 2]
        with torch.cuda.stream(cs_in):
            cs_in.wait_event(b["computed"])     # step i-2's kernels are done with the inputs
            for d, h in zip(b["in"], hosts):
                d.copy_(h, non_blocking=True)
            b["copied_in"].record(cs_in)
        stream.wait_event(b["copied_in"])
        stream.wait_event(b["copied_out"])      # step i-2's result has left this buffer
        b["write"]()
        b["decode"]()
        b["computed"].record(stream)
        with torch.cuda.stream(cs_out):
            cs_out.wait_event(b["computed"])
            b["h_res"].copy_(b["res"], non_blocking=True)
            b["copied_out"].record(cs_out)

    def drain():
        for b in sets:
            stream.wait_event(b["copied_out"])  # the last results are in host memory

    for i in range(4):
        pipelined_step(i)
    torch.cuda.synchronize()
    start_gate = torch.cuda.Event()
    start_gate.record(stream)
    cs_in.wait_event(start_gate)                # the copy streams start inside the timed region
    cs_out.wait_event(start_gate)
    e2e_ms = time_loop(pipelined_step, e2e_steps, drain)
    e2e_value = whole_job_tokens_per_s(world, wl.num_seqs, e2e_ms)
    serial_value = whole_job_tokens_per_s(world, wl.num_seqs, serial_ms)

    # ---- roofline of the decode kernel(s)
    peak, peak_kind = _peaks()
    bytes_launch = _unique_bytes(wl)
    achieved = bytes_launch / (dec_ms / 1000.0) / 1e9
    roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
            "frac": achieved / peak, "traffic": _profiled_traffic(args.workload),
            "peak_source": f"{peak_kind} hbm_gbs",
            "kernel": "paged_decode_kernel" + ("+merge" if plan["needs_merge"] else ""),
            "algorithmic_bytes_per_launch": bytes_launch, "launch_ms": dec_ms,
            "launch_ms_is": f"median of {len(dec_times)} CUDA-event-timed calls in the timed "
                            "region", "launch_ms_mean": statistics.mean(dec_times)}

    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f16" if wl.dtype == torch.float16 else "bf16", "data": "synthetic",
            "config": _workload_config(wl, args.workload, plan, part),
            "kv_read_gbps": achieved, "hbm_frac_of_measured": achieved / peak,
            "hbm_frac_of_nominal_8000": achieved / 8000.0,
            "clocks": clocks, "gpu_launches": launches,
            "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                    "copies": "double-buffered; inputs and results on two copy streams, "
                              "overlapping the previous step's kernels",
                    "serial_value": serial_value, "serial_ms_per_step": serial_ms},
            "roofline": roof}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl)
    if world == 1 and not args.no_other_workloads:
        others = {}
        for name in ("tiny", "mha7b", "gqa7b", "prefix", "long70b", "mha7b_int8", "gqa7b_int8",
                     "long70b_int8", "gqa16"):
            if name == args.workload:
                continue
            others[name] = measure_workload(pkv, name, dev, 300, peak)
        for name in ("prefill7b", "chunked70b"):
            others[name] = measure_prefill(pkv, name, dev, 50)
        line["other_workloads"] = others
        line["configs"] = _config_summary(args.workload, line, others)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="mha7b",
                    choices=["tiny", "mha7b", "gqa7b", "prefix", "long70b", "mha7b_int8",
                             "gqa7b_int8", "long70b_int8", "gqa16"])
    ap.add_argument("--partition", type=int, default=-1,
                    help="tokens per split-context partition (0 = library's choice; "
                         "default: the workload's own setting)")
    ap.add_argument("--num-seqs", type=int, default=0,
                    help="override the workload's batch (profiling on a smaller case)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-other-workloads", action="store_true",
                    help="skip the device-timed lines of the other named workloads")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.partition < 0:
        from paged_kv_cache_155_gb300.workloads import DEFAULT_PARTITION
        args.partition = DEFAULT_PARTITION[args.workload]
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
