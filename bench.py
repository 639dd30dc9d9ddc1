#!/usr/bin/env python
"""Benchmark of the paged KV attention hot path on one GB300 (or N, as independent replicas).

One step = one decode step of the memory-bound workload: 64 sequences x 4096 cached tokens,
32 query / 8 KV heads, head_dim 128, block 16, bf16 (1,073,741,824 bytes of K+V):
  1. pa_reshape_and_cache writes the step's 64 new key/value rows into the pools;
  2. pa_paged_attention_decode (split-KV kernel + log-sum-exp combine) answers the 64 queries.
The two calls are captured as one CUDA graph, replayed once per timed step.
The headline value is decode HBM throughput: algorithmic bytes (the K/V of every cached
position read once, q, out, the used block-table entries, the new rows) per second.
A second leg times causal prefill of 4 x 8192 tokens (block 64): the prompt's cache write
plus pa_paged_attention_varlen, reported in TFLOP/s of causal attention.

The inputs (1.07 GB of cache per step, 0.4 GB for prefill) exceed the 129 MB L2, so no
flush is needed between timed steps.

--impl reference times the float64 CPU oracle (the only reference this method has) on a
bounded sample of the same workload and prints the same metric.
"""

from __future__ import annotations

import argparse
import functools
import json
import os
import statistics
import subprocess
import tempfile
import sys
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "paged decode attn HBM GB/s (% of peak) at 64x4096; prefill TFLOP/s"
DECODE_WORKLOAD = "decode_64x4096_bf16"
PREFILL_WORKLOAD = "prefill_4x8192_bf16"
CASCADE_WORKLOAD = "cascade_64x4000_bf16"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ----------------------------------------------------------------------------- accounting
def kv_bytes_per_token(num_kv_heads: int, head_dim: int, elem_bytes: int) -> int:
    """Bytes of one cached position of one layer: a key and a value row per KV head."""
    return 2 * num_kv_heads * head_dim * elem_bytes


def decode_call_bytes(context_lens, num_q_heads, num_kv_heads, head_dim, block_size, elem_bytes) -> int:
    """Algorithmic bytes of one decode call: every cached position's K and V once, the
    queries, the outputs, the used block-table entries and the lengths."""
    kv = sum(int(L) for L in context_lens) * kv_bytes_per_token(num_kv_heads, head_dim, elem_bytes)
    S = len(context_lens)
    qo = 2 * S * num_q_heads * head_dim * elem_bytes
    tables = sum(-(-int(L) // block_size) for L in context_lens) * 4 + S * 4
    return kv + qo + tables


def cache_write_bytes(num_tokens, num_kv_heads, head_dim, elem_bytes) -> int:
    """reshape_and_cache: read and write each new key and value row, read the slot."""
    return 2 * num_tokens * kv_bytes_per_token(num_kv_heads, head_dim, elem_bytes) + 4 * num_tokens


def causal_flops(q_lens, seq_lens, num_q_heads, head_dim, causal=True) -> float:
    """4 * D flops (q.k and p.v) per visible (query, key) pair per query head."""
    pairs = 0
    for ql, L in zip(q_lens, seq_lens):
        ql, L = int(ql), int(L)
        if causal:
            prior = L - ql
            pairs += ql * prior + ql * (ql + 1) // 2
        else:
            pairs += ql * L
    return 4.0 * head_dim * num_q_heads * pairs


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"]))}, "measured"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def load_traffic():
    """Per-launch DRAM bytes of the dominant kernels from the committed ncu summaries, for each
    kernel whose source file is unchanged since the capture (its hash is recorded)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return {}
    out = {}
    for name, k in d.get("kernels", {}).items():
        if k.get("source_hash") == source_hash(k.get("source", "")):
            out[name] = k.get("bytes_per_launch")
    return out


def source_hash(source: str) -> str:
    """Hash of one kernel source file plus the shared device headers it includes."""
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "paged_kv_attention_gb300", "csrc")
    for name in (source, "pa_common.cuh", "tc_common.cuh", "decode_common.cuh"):
        try:
            with open(os.path.join(csrc, name), "rb") as f:
                h.update(name.encode() + f.read())
        except OSError:
            return ""
    return h.hexdigest()[:16]


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,utilization.gpu")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.gpu = gpu_index
        # the raw samples go to PA_BENCH_LOG_DIR when set (the summary is in the JSON line)
        log_dir = os.environ.get("PA_BENCH_LOG_DIR") or tempfile.gettempdir()
        self.path = os.path.join(log_dir, f"clocks_bench_{os.getpid()}.csv")

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) != 10:
                    continue
                try:
                    util = float(parts[9])
                except ValueError:
                    util = 0.0
                try:
                    rows.append((float(parts[1]), float(parts[2]), float(parts[3]), parts[5:9], util))
                except ValueError:
                    continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        seen = set()
        for r in rows:
            for n, v in zip(names, r[3]):
                if v.lower().startswith("active"):
                    seen.add(n)
        # a sample is under load when a kernel ran for at least half of its 100 ms period
        under = [r for r in rows if r[4] >= 50.0]
        loaded = under or rows
        return {"sm_mhz": statistics.median(r[0] for r in loaded), "sm_max_mhz": max(r[1] for r in rows),
                "power_w_max": max(r[2] for r in rows), "reasons": sorted(seen), "samples": len(rows),
                "samples_under_load": len(under),
                "sm_mhz_min_under_load": min((r[0] for r in under), default=None)}


# ----------------------------------------------------------------------------- distributed
def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def barrier(world):
    if world > 1:
        torch.distributed.barrier()


def max_over_ranks(x: float, world: int) -> float:
    """The slowest rank's time: every rank's work is counted against it."""
    if world == 1:
        return x
    dev = "cuda" if torch.distributed.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_step_per_rank: float, steps: int, max_ms: float, world: int) -> float:
    """Units per second over all ranks: every rank processes its own batch (weak scaling),
    timed by the slowest rank."""
    return world * units_per_step_per_rank * steps / (max_ms / 1e3)


# ----------------------------------------------------------------------------- oracle timing
def packed_buffers(tensors, dev, align=256):
    """One pinned host buffer holding `tensors` back to back (each at a 256-byte aligned
    offset), a device buffer of the same layout, and device views shaped like the tensors."""
    offs, total = [], 0
    for t in tensors:
        offs.append(total)
        total += -(-t.numel() * t.element_size() // align) * align
    hin = torch.zeros(total, dtype=torch.uint8).pin_memory()
    din = torch.empty(total, dtype=torch.uint8, device=dev)
    views = []
    for t, o in zip(tensors, offs):
        n = t.numel() * t.element_size()
        hin[o:o + n].copy_(t.contiguous().view(-1).view(torch.uint8))
        views.append(din[o:o + n].view(t.dtype).view(t.shape))
    din.copy_(hin)
    return hin, din, views


def time_oracle_decode(case, ko, vo, budget_s: float = 12.0, max_seqs: int | None = None):
    """Time the float64 oracle on whole sequences of the decode workload, as many as fit
    ~budget_s (at least one). Returns (GB/s of algorithmic bytes, seconds, seqs, threads)."""
    import oracle
    S = case.num_reqs
    lens = case.seq_lens.tolist()
    t0 = time.perf_counter()
    oracle.paged_attention_decode(case.q, ko, vo, case.block_tables, case.seq_lens, case.scale, seqs=[0])
    one = max(time.perf_counter() - t0, 1e-3)
    n = max(1, min(S if max_seqs is None else max_seqs, int(budget_s / one)))
    seqs = list(range(n))
    t0 = time.perf_counter()
    oracle.paged_attention_decode(case.q, ko, vo, case.block_tables, case.seq_lens, case.scale, seqs=seqs)
    dt = time.perf_counter() - t0
    nbytes = decode_call_bytes([lens[s] for s in seqs], case.num_q_heads, case.num_kv_heads, case.head_dim,
                               case.block_size, case.q.element_size())
    return nbytes / dt / 1e9, dt, n, torch.get_num_threads()


def oracle_pools(case):
    import oracle
    kc, vc = case.empty_pools()
    oracle.reshape_and_cache(case.key, case.value, kc, vc, case.slot_mapping)
    return kc, vc


def run_reference(args, world, rank):
    """--impl reference: the float64 CPU oracle, timed as it stands on the host cores, on
    bounded samples of the decode workload (rank 0 only)."""
    if rank != 0:
        return
    import workloads
    case = workloads.NAMED[DECODE_WORKLOAD]()
    ko, vo = oracle_pools(case)
    import oracle
    lens = case.seq_lens.tolist()
    per_step = 2  # sequences per timed step: a bounded sample of the 64
    seqs_of = lambda i: [(i * per_step + j) % case.num_reqs for j in range(per_step)]  # noqa: E731
    for i in range(args.warmup):
        oracle.paged_attention_decode(case.q, ko, vo, case.block_tables, case.seq_lens, case.scale, seqs=seqs_of(i))
    total_bytes, t0 = 0, time.perf_counter()
    for i in range(args.steps):
        s = seqs_of(args.warmup + i)
        oracle.paged_attention_decode(case.q, ko, vo, case.block_tables, case.seq_lens, case.scale, seqs=s)
        total_bytes += decode_call_bytes([lens[j] for j in s], case.num_q_heads, case.num_kv_heads, case.head_dim,
                                         case.block_size, 2)
    dt = time.perf_counter() - t0
    value = total_bytes / dt / 1e9
    sample = f"{per_step} of 64 sequences per step (all heads, full 4096-token contexts)"
    line = {"metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(dt / max(args.steps, 1) * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": DECODE_WORKLOAD, "num_seqs": 64, "context_len": 4096, "num_q_heads": 32,
                       "num_kv_heads": 8, "head_dim": 128, "block_size": 16, "sample": sample},
            "impl": "reference",
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": torch.get_num_threads(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- GPU legs
def decode_leg(args, world, rank, dev):
    import paged_kv_attention_gb300 as pa
    import workloads
    case = workloads.NAMED[DECODE_WORKLOAD]()
    if args.decode_seqs != case.num_reqs:  # a smaller batch of the same workload (profiling)
        case = workloads.decode_case(f"decode_{args.decode_seqs}x4096_bf16", 1003, [4096] * args.decode_seqs,
                                     num_q_heads=32, num_kv_heads=8, head_dim=128, block_size=16,
                                     dtype=torch.bfloat16)
    S, Hq, Hkv, D, bs = case.num_reqs, case.num_q_heads, case.num_kv_heads, case.head_dim, case.block_size
    lens = case.seq_lens.tolist()
    kc, vc = (t.to(dev) for t in case.empty_pools())
    pa.reshape_and_cache(case.key.to(dev), case.value.to(dev), kc, vc, case.slot_mapping.to(dev))
    # the step's new rows: the last cached position of every sequence
    offs = torch.cumsum(case.seq_lens.long(), 0) - 1
    new_k, new_v = case.key[offs].contiguous(), case.value[offs].contiguous()
    new_slots = case.slot_mapping[offs].contiguous()
    # the step's inputs (q, the new rows, their slots, the lengths) live in one device buffer laid
    # out like one pinned host buffer, so the end-to-end leg moves them with a single copy
    host_inputs = [case.q, new_k, new_v, new_slots, case.seq_lens]
    hin, din, (q, nk, nv, ns, ctx) = packed_buffers(host_inputs, dev)
    tables = case.block_tables.to(dev)
    out = torch.empty_like(q)
    splits = pa.decode_auto_splits(S, Hq, Hkv, D, bs, tables.shape[1], case.dtype)
    ws = torch.empty(max(pa.decode_workspace_bytes(S, Hq, D, tables.shape[1], bs, splits), 16),
                     dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def step(qd, kd, vd, sd, ld, od):
        pa.reshape_and_cache(kd, vd, kc, vc, sd)
        pa.paged_attention_decode(qd, kc, vc, tables, ld, case.scale, num_splits=splits, out=od, workspace=ws)

    for _ in range(args.warmup):
        step(q, nk, nv, ns, ctx, out)
    torch.cuda.synchronize()

    def write_call():
        pa.reshape_and_cache(nk, nv, kc, vc, ns)

    def decode_call():
        pa.paged_attention_decode(q, kc, vc, tables, ctx, case.scale, num_splits=splits, out=out, workspace=ws)

    def step_calls():
        write_call()
        decode_call()

    if args.no_graph:
        run_write, run_call, run_step = write_call, decode_call, step_calls
    else:
        # the step (both calls) captured once as one graph and replayed, as a serving loop runs
        # it; each call also captured alone, for the per-call times (launch shapes depend only on
        # host sizes; lengths and positions are read from device buffers at every replay)
        graphs = []
        for fn in (write_call, decode_call, step_calls):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                fn()
            graphs.append(g)
        run_write, run_call, run_step = graphs[0].replay, graphs[1].replay, graphs[2].replay
        for _ in range(3):
            run_write()
            run_call()
            run_step()
        torch.cuda.synchronize()
    # per-call times: each call's graph between events, over enough replays (call_reps) that the
    # clock sampler sees the GPU under load while they run
    n_rep = max(args.steps, args.call_reps)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(n_rep)]
    torch.cuda.synchronize()
    for i in range(n_rep):
        ev[i][0].record(stream)
        run_write()
        ev[i][1].record(stream)
        run_call()
        ev[i][2].record(stream)
    torch.cuda.synchronize()
    write_ms = sum(e[0].elapsed_time(e[1]) for e in ev) / n_rep
    call_ms = sum(e[1].elapsed_time(e[2]) for e in ev) / n_rep
    # the timed steps
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for i in range(args.steps):
        run_step()
    end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    wall = time.perf_counter() - t0
    total_ms = start.elapsed_time(end)
    total_ms = max_over_ranks(total_ms, world)

    call_bytes = decode_call_bytes(lens, Hq, Hkv, D, bs, 2)
    step_bytes = call_bytes + cache_write_bytes(S, Hkv, D, 2)
    value = whole_job_rate(step_bytes, args.steps, total_ms, world) / 1e9

    if args.no_e2e:
        return dict(case=case, splits=splits, total_ms=total_ms, wall=wall, write_ms=write_ms, call_ms=call_ms,
                    call_reps=n_rep, call_bytes=call_bytes, step_bytes=step_bytes, value=value, e2e_value=None,
                    h2d=0, d2h=0, launches=args.steps * (2 + (1 if splits > 1 else 0)), out=out.cpu())
    # End to end: every step's inputs copied in from one pinned host buffer (one copy), the same
    # two calls, every step's output read back to pinned host memory, all inside the timed
    # region. As a serving loop runs it: two sets of device buffers, the copy-in of step i + 1
    # (on its own stream) overlapping step i, and the read-back of step i (on a third stream)
    # overlapping step i + 1. Each step's graph starts once its inputs have landed, and a buffer
    # set is refilled only after the step before last has finished with it.
    hout = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    sets = [(din, out)]
    views2 = []
    din2 = torch.empty_like(din)
    for t, v in zip(host_inputs, (q, nk, nv, ns, ctx)):
        off = v.data_ptr() - din.data_ptr()
        n = t.numel() * t.element_size()
        views2.append(din2[off:off + n].view(t.dtype).view(t.shape))
    sets.append((din2, torch.empty_like(out)))
    step_graphs = []
    for bi, (dbuf, obuf) in enumerate(sets):
        qv, kv_, vv, sv, lv = (q, nk, nv, ns, ctx) if bi == 0 else views2
        if args.no_graph:
            step_graphs.append(functools.partial(step, qv, kv_, vv, sv, lv, obuf))
        else:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                step(qv, kv_, vv, sv, lv, obuf)
            step_graphs.append(g.replay)
    h2d_stream, d2h_stream = torch.cuda.Stream(), torch.cuda.Stream()

    def e2e_steps(n):
        landed = [torch.cuda.Event() for _ in range(2)]
        done = [None, None]   # step finished with buffer set b
        read = [None, None]   # read-back of set b's output finished
        with torch.cuda.stream(h2d_stream):
            sets[0][0].copy_(hin, non_blocking=True)
            landed[0].record(h2d_stream)
        for i in range(n):
            b = i % 2
            stream.wait_event(landed[b])
            if read[b] is not None:
                stream.wait_event(read[b])
            step_graphs[b]()
            done[b] = torch.cuda.Event()
            done[b].record(stream)
            if i + 1 < n:
                nb = (i + 1) % 2
                with torch.cuda.stream(h2d_stream):
                    if done[nb] is not None:
                        h2d_stream.wait_event(done[nb])
                    sets[nb][0].copy_(hin, non_blocking=True)
                    landed[nb] = torch.cuda.Event()
                    landed[nb].record(h2d_stream)
            with torch.cuda.stream(d2h_stream):
                d2h_stream.wait_event(done[b])
                hout.copy_(sets[b][1], non_blocking=True)
                read[b] = torch.cuda.Event()
                read[b].record(d2h_stream)
        for r in read:
            if r is not None:
                stream.wait_event(r)

    def serial_steps(n):  # the same, one step after another on one stream (no overlap)
        for _ in range(n):
            din.copy_(hin, non_blocking=True)
            step_graphs[0]()
            hout.copy_(out, non_blocking=True)

    serial_steps(max(3, args.warmup // 4))
    torch.cuda.synchronize()
    barrier(world)
    s_start, s_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s_start.record(stream)
    serial_steps(args.steps)
    s_end.record(stream)
    torch.cuda.synchronize()
    serial_ms = max_over_ranks(s_start.elapsed_time(s_end), world)
    e2e_steps(max(3, args.warmup // 4))
    torch.cuda.synchronize()
    barrier(world)
    e2e_start = torch.cuda.Event(enable_timing=True)
    e2e_end = torch.cuda.Event(enable_timing=True)
    e2e_start.record(stream)
    e2e_steps(args.steps)
    e2e_end.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e2e_start.elapsed_time(e2e_end), world)
    h2d = hin.numel()
    d2h = hout.numel() * hout.element_size()
    e2e_value = whole_job_rate(step_bytes, args.steps, e2e_ms, world) / 1e9
    e2e_serial = whole_job_rate(step_bytes, args.steps, serial_ms, world) / 1e9
    return dict(e2e_serial=e2e_serial, e2e_ms_per_step=e2e_ms / args.steps, serial_ms_per_step=serial_ms / args.steps,
                case=case, splits=splits, total_ms=total_ms, wall=wall, write_ms=write_ms, call_ms=call_ms,
                call_reps=n_rep, call_bytes=call_bytes, step_bytes=step_bytes, value=value, e2e_value=e2e_value,
                h2d=h2d, d2h=d2h, launches=args.steps * (2 + (1 if splits > 1 else 0)), out=hout.clone())


def decode_int8_leg(args, dev, code_dtype=torch.int8):
    """The same 64x4096 decode over an 8-bit cache (int8 or fp8 E4M3 codes + one fp32 scale per
    (slot, KV head)), quantised by the library's own write; the decode call replayed as a CUDA
    graph."""
    import paged_kv_attention_gb300 as pa
    import workloads
    case = workloads.NAMED[DECODE_WORKLOAD]()
    if args.decode_seqs != case.num_reqs:  # a smaller batch of the same workload (profiling)
        case = workloads.decode_case(f"decode_{args.decode_seqs}x4096_bf16", 1003, [4096] * args.decode_seqs,
                                     num_q_heads=32, num_kv_heads=8, head_dim=128, block_size=16,
                                     dtype=torch.bfloat16)
    S, Hq, Hkv, D, bs = case.num_reqs, case.num_q_heads, case.num_kv_heads, case.head_dim, case.block_size
    shape = (case.num_blocks, bs, Hkv, D)
    kc = torch.empty(shape, dtype=code_dtype, device=dev)
    vc = torch.empty(shape, dtype=code_dtype, device=dev)
    ks = torch.empty(shape[:3], dtype=torch.float32, device=dev)
    vs = torch.empty(shape[:3], dtype=torch.float32, device=dev)
    pa.reshape_and_cache_quant(case.key.to(dev), case.value.to(dev), kc, vc, ks, vs, case.slot_mapping.to(dev))
    q, tables, ctx = case.q.to(dev), case.block_tables.to(dev), case.seq_lens.to(dev)
    out = torch.empty_like(q)
    splits = pa.decode_auto_splits(S, Hq, Hkv, D, bs, tables.shape[1], torch.bfloat16)
    ws = torch.empty(max(pa.decode_workspace_bytes(S, Hq, D, tables.shape[1], bs, 0), 16), dtype=torch.uint8,
                     device=dev)

    def call():
        pa.paged_attention_decode_quant(q, kc, vc, ks, vs, tables, ctx, case.scale, out=out, workspace=ws)

    for _ in range(3):
        call()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    for _ in range(3):
        g.replay()
    stream = torch.cuda.current_stream()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    n_rep = max(args.steps, args.call_reps)
    start.record(stream)
    for _ in range(n_rep):
        g.replay()
    end.record(stream)
    torch.cuda.synchronize()
    ms = start.elapsed_time(end) / n_rep
    lens = case.seq_lens.tolist()
    positions = sum(int(L) for L in lens)
    nbytes = positions * Hkv * (2 * D * 1 + 2 * 4) + 2 * S * Hq * D * 2 + \
        sum(-(-int(L) // bs) for L in lens) * 4 + S * 4
    return dict(ms=ms, bytes=nbytes, gbs=nbytes / (ms / 1e3) / 1e9, reps=n_rep)


def cascade_leg(args, dev):
    """64 sequences behind one shared 4,000-token prefix: the cascade decode (prefix read once,
    suffixes split-KV, one combine) against the plain decode over each sequence's full table
    (prefix pages + its own), both replayed as CUDA graphs. The working set of the cascade
    (about 50 MB) fits in L2, so a 256 MB buffer is rewritten (then another read, leaving clean
    lines) between timed calls and only the calls are timed."""
    import paged_kv_attention_gb300 as pa
    import workloads
    case = workloads.NAMED[CASCADE_WORKLOAD]()
    kc, vc = (t.to(dev) for t in case.empty_pools())
    pa.reshape_and_cache(case.key.to(dev), case.value.to(dev), kc, vc, case.slot_mapping.to(dev))
    S, Hq, Hkv, D, bs = case.num_reqs - 1, case.num_q_heads, case.num_kv_heads, case.head_dim, case.block_size
    P = int(case.seq_lens[0])
    suffix = case.seq_lens[1:]
    width = -(-int(suffix.max()) // bs)
    q = case.q.to(dev)
    ptable = case.block_tables[0].to(dev)
    plen = torch.tensor([P], dtype=torch.int32, device=dev)
    stables = case.block_tables[1:, :width].contiguous().to(dev)
    slens = suffix.to(dev)
    n_pre = -(-P // bs)
    assert P % bs == 0, "the plain-decode comparison concatenates whole prefix pages"
    full_tables = torch.cat([case.block_tables[0, :n_pre].expand(S, -1), case.block_tables[1:, :width]],
                            dim=1).contiguous().to(dev)
    full_lens = (suffix + P).to(dev)
    out_c, out_p = torch.empty_like(q), torch.empty_like(q)
    ws_c = torch.empty(pa._lib.load().pa_cascade_workspace_bytes(S, Hq, D, bs, ptable.numel(), width),
                       dtype=torch.uint8, device=dev)
    ws_p = torch.empty(max(pa.decode_workspace_bytes(S, Hq, D, full_tables.shape[1], bs, 0), 16),
                       dtype=torch.uint8, device=dev)

    def cascade():
        pa.cascade_decode(q, kc, vc, ptable, plen, stables, slens, case.scale, out=out_c, workspace=ws_c)

    def plain():
        pa.paged_attention_decode(q, kc, vc, full_tables, full_lens, case.scale, out=out_p, workspace=ws_p)

    # between timed calls: rewrite 256 MB (> L2), then read another 256 MB so that the lines the
    # call evicts are clean (the write-backs of the flush stay outside the timed region)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    flush_read = torch.zeros(64 << 20, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    result = {}
    for name, fn in (("cascade", cascade), ("plain", plain)):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        for _ in range(3):
            g.replay()
        n = max(50, args.config_calls)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        torch.cuda.synchronize()
        for i in range(n):
            flush.fill_(i & 255)
            flush_read.sum()
            ev[i][0].record(stream)
            g.replay()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        result[name] = sum(a.elapsed_time(b) for a, b in ev) / n
    diff = (out_c.float() - out_p.float()).abs().max().item()
    row = Hkv * D * 2 * 2
    unique = (P + int(suffix.sum())) * row
    logical = (S * P + int(suffix.sum())) * row
    return dict(case=case, cascade_ms=result["cascade"], plain_ms=result["plain"], unique=unique, logical=logical,
                max_diff=diff, launches=3 * n)


def prefill_leg(args, dev, steps, workload=PREFILL_WORKLOAD, code_dtype=None):
    import paged_kv_attention_gb300 as pa
    import workloads
    case = workloads.NAMED[workload]()
    if args.prefill_seqs != case.num_reqs and workload == PREFILL_WORKLOAD:  # a smaller batch of the same workload (profiling)
        case = workloads.make_case(f"prefill_{args.prefill_seqs}x8192_bf16", 1005, [8192] * args.prefill_seqs,
                                   [8192] * args.prefill_seqs, num_q_heads=32, num_kv_heads=8, head_dim=128,
                                   block_size=64, dtype=torch.bfloat16)
    kc, vc = (t.to(dev) for t in case.empty_pools())
    q = case.q.to(dev)
    key, value, slots = case.key.to(dev), case.value.to(dev), case.slot_mapping.to(dev)
    qsl, sl, tables = case.query_start_loc.to(dev), case.seq_lens.to(dev), case.block_tables.to(dev)
    out = torch.empty_like(q)
    stream = torch.cuda.current_stream()
    if code_dtype is not None:  # an 8-bit cache (codes + one fp32 scale per slot and KV head)
        kc = torch.empty(kc.shape, dtype=code_dtype, device=dev)
        vc = torch.empty(vc.shape, dtype=code_dtype, device=dev)
        ks = torch.empty(kc.shape[:3], dtype=torch.float32, device=dev)
        vs = torch.empty(kc.shape[:3], dtype=torch.float32, device=dev)

        def write():
            pa.reshape_and_cache_quant(key, value, kc, vc, ks, vs, slots)

        def attend():
            pa.paged_attention_varlen_quant(q, kc, vc, ks, vs, qsl, sl, tables, case.max_query_len, True,
                                            case.scale, out=out)
    else:
        def write():
            pa.reshape_and_cache(key, value, kc, vc, slots)

        def attend():
            pa.paged_attention_varlen(q, kc, vc, qsl, sl, tables, case.max_query_len, True, case.scale, out=out)

    def step():
        write()
        attend()

    for _ in range(max(2, min(args.warmup, 3))):
        step()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for i in range(steps):
        ev[i][0].record(stream)
        write()
        ev[i][1].record(stream)
        attend()
        ev[i][2].record(stream)
    torch.cuda.synchronize()
    write_ms = sum(e[0].elapsed_time(e[1]) for e in ev) / steps
    attn_ms = sum(e[1].elapsed_time(e[2]) for e in ev) / steps
    ql = (case.query_start_loc[1:] - case.query_start_loc[:-1]).tolist()
    flops = causal_flops(ql, case.seq_lens.tolist(), case.num_q_heads, case.head_dim)
    return dict(case=case, write_ms=write_ms, attn_ms=attn_ms, flops=flops, tflops=flops / (attn_ms / 1e3) / 1e12,
                launches=2 * steps, out=out.cpu())


def configs_leg(args, dev, peaks):
    """The other workloads of the hot path (the parity configurations): the fp32 latency case,
    the ragged bf16 decode, the head_dim-256 decode and the mixed varlen batch (on the default
    grid, on a host-planned grid, and with its short requests on the split-KV decode). Each call
    is captured in a CUDA graph and replayed; before every timed call 256 MB are rewritten and
    re-read so that no input stays in L2 (the fp32 case, whose 0.2 MB live in L2 between steps
    of a real decode loop, is also timed warm); CUDA events on the call's stream; median and
    minimum of `n` calls. The two small decodes are also launched eagerly. Returns the timings
    and, per workload, the case, the GPU output of the timed call and how to run the oracle on
    it (the parity check itself runs with the CPU baseline, outside every timed region)."""
    import paged_kv_attention_gb300 as pa
    import workloads
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    rd = torch.zeros(64 << 20, device=dev)
    n_calls = max(50, args.config_calls)

    def timed(fn, n=n_calls, graph=True, cold=True):
        for _ in range(5):
            fn()
        torch.cuda.synchronize()
        run = fn
        if graph:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                fn()
            for _ in range(3):
                g.replay()
            run = g.replay
        events = []
        for _ in range(n):
            if cold:
                flush.fill_(1)
                rd.sum()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            run()
            e1.record()
            events.append((e0, e1))
        torch.cuda.synchronize()
        us = sorted(a.elapsed_time(b) * 1e3 for a, b in events)
        return statistics.median(us), us[0]

    hbm, tf = peaks["hbm_gbs"], peaks["bf16_tflops"]
    res, outputs = {}, {}
    launches = 0
    for name in ("decode_1seq_fp32", "decode_ragged32_bf16", "decode_64x4096_bf16_d256"):
        case = workloads.NAMED[name]()
        kc, vc = (t.to(dev) for t in case.empty_pools())
        pa.reshape_and_cache(case.key.to(dev), case.value.to(dev), kc, vc, case.slot_mapping.to(dev))
        q, t, lens = case.q.to(dev), case.block_tables.to(dev), case.seq_lens.to(dev)
        o = torch.empty_like(q)
        S, Hq, Hkv, D, bs = case.num_reqs, case.num_q_heads, case.num_kv_heads, case.head_dim, case.block_size
        splits = pa.decode_auto_splits(S, Hq, Hkv, D, bs, t.shape[1], case.dtype)
        ws = torch.empty(max(pa.decode_workspace_bytes(S, Hq, D, t.shape[1], bs, splits), 16), dtype=torch.uint8,
                         device=dev)

        def call():
            pa.paged_attention_decode(q, kc, vc, t, lens, case.scale, out=o, workspace=ws)

        med, mn = timed(call)
        per_call = 2 if splits > 1 else 1
        launches += n_calls * per_call
        elt = 4 if case.dtype == torch.float32 else 2
        nbytes = decode_call_bytes(case.seq_lens.tolist(), Hq, Hkv, D, bs, elt)
        entry = {"us_median": round(med, 2), "us_min": round(mn, 2), "splits": splits, "calls": n_calls,
                 "algorithmic_bytes": nbytes, "queries_per_s": round(S / (med * 1e-6)),
                 "GBps": round(nbytes / med / 1e3, 1), "frac_of_hbm_peak": round(nbytes / med / 1e3 / hbm, 4)}
        if name != "decode_64x4096_bf16_d256":
            emed, emn = timed(call, graph=False)
            launches += n_calls * per_call
            entry["eager_us_median"], entry["eager_us_min"] = round(emed, 2), round(emn, 2)
        if name == "decode_1seq_fp32":
            wmed, wmn = timed(call, cold=False)
            launches += n_calls * per_call
            entry["warm_us_median"], entry["warm_us_min"] = round(wmed, 2), round(wmn, 2)
            ewmed, ewmn = timed(call, graph=False, cold=False)
            launches += n_calls * per_call
            entry["warm_eager_us_median"], entry["warm_eager_us_min"] = round(ewmed, 2), round(ewmn, 2)
            entry.pop("GBps")
            entry.pop("frac_of_hbm_peak")
            entry["bound"] = "latency (0.2 MB: no bandwidth claim)"
        res[name] = entry
        outputs[name] = (case, "decode", {}, o.cpu())
        del kc, vc
    case = workloads.NAMED["varlen_mixed_bf16"]()
    kc, vc = (t.to(dev) for t in case.empty_pools())
    pa.reshape_and_cache(case.key.to(dev), case.value.to(dev), kc, vc, case.slot_mapping.to(dev))
    q = case.q.to(dev)
    a = (kc, vc, case.query_start_loc.to(dev), case.seq_lens.to(dev), case.block_tables.to(dev), case.max_query_len,
         True, case.scale)
    qls = (case.query_start_loc[1:] - case.query_start_loc[:-1]).tolist()
    sls = case.seq_lens.tolist()
    flops = causal_flops(qls, sls, case.num_q_heads, case.head_dim)
    nbytes = sum(sls) * kv_bytes_per_token(case.num_kv_heads, case.head_dim, 2) + \
        2 * case.num_tokens * case.num_q_heads * case.head_dim * 2
    variants = [("varlen_mixed_bf16", dict(), "default grid: every tile pair up to max_query_len, heaviest first")]
    items = pa.varlen_plan(case.query_start_loc, case.seq_lens, case.max_query_len, case.num_q_heads,
                           case.num_kv_heads, True).to(dev)
    variants.append(("varlen_mixed_bf16_planned", dict(work_items=items),
                     "host-planned grid (pa_varlen_plan, outside the timed call): only the pairs the batch has"))
    ws = torch.empty(max(pa._lib.load().pa_varlen_workspace_bytes(case.num_reqs, case.num_q_heads, case.head_dim,
                                                                   case.block_tables.shape[1], case.block_size), 16),
                     dtype=torch.uint8, device=dev)
    variants.append(("varlen_mixed_bf16_device_plan", dict(workspace=ws, schedule="tensor"),
                     "grid planned on the device by a one-CTA kernel in the call (graph-safe), every request on "
                     "the tensor-core kernel"))
    variants.append(("varlen_mixed_bf16_split_decodes", dict(workspace=ws, schedule="split"),
                     "device-planned grid; requests of <= 8 queries on the split-KV decode, launched to fill the "
                     "tensor-core grid's tail"))
    variants.append(("varlen_mixed_bf16_auto", dict(workspace=ws, schedule="auto"),
                     "pa_paged_attention_varlen_ws: device-planned grid, short requests routed by the batch's "
                     "shape (here: the tensor-core kernel)"))
    for vname, kw, desc in variants:
        o = torch.empty_like(q)
        med, mn = timed(lambda: pa.paged_attention_varlen(q, *a, out=o, **kw))
        sched = kw.get("schedule")
        launches += n_calls * (4 if sched == "split" else 2 if sched in ("tensor", "auto") else 1)
        res[vname] = {
            "grid": desc, "us_median": round(med, 2), "us_min": round(mn, 2), "calls": n_calls,
            "causal_flops": flops, "algorithmic_bytes": nbytes,
            "queries_per_s": round(case.num_tokens / (med * 1e-6)),
            "TFLOPs": round(flops / med / 1e6, 1), "GBps": round(nbytes / med / 1e3, 1),
            "frac_of_tensor_peak": round(flops / med / 1e6 / tf, 4),
            "frac_of_hbm_peak": round(nbytes / med / 1e3 / hbm, 4),
            "floor_us": round(max(flops / tf / 1e6, nbytes / hbm / 1e3), 1)}
        if "work_items" in kw:
            res[vname]["items"] = int(items.numel())
        outputs[vname] = (case, "varlen", {}, o.cpu())
    return res, outputs, launches


def config_parity(outputs):
    """Max and mean |GPU - oracle| of each configuration's timed call (float64 oracle, every row;
    run with the CPU baseline, outside every timed region)."""
    import oracle
    pools = {}
    res = {}
    for name, (case, kind, kw, got) in outputs.items():
        if case.name not in pools:
            pools[case.name] = oracle_pools(case)
        ko, vo = pools[case.name]
        if kind == "decode":
            want = oracle.paged_attention_decode(case.q, ko, vo, case.block_tables, case.seq_lens, case.scale)
        else:
            want = oracle.paged_attention_varlen(case.q, ko, vo, case.query_start_loc, case.seq_lens,
                                                 case.block_tables, True, case.scale)
        d = (got.double() - want).abs()
        res[name] = {"max_abs": float(d.max()), "mean_abs": float(d.mean()), "rows": int(got.shape[0])}
    return res


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--prefill-steps", type=int, default=150,
                    help="timed prefill calls (each 4 x 8192 call is ~1.6 ms)")
    ap.add_argument("--call-reps", type=int, default=2000,
                    help="replays behind each per-call time (decode call, 8-bit decodes)")
    ap.add_argument("--config-calls", type=int, default=200,
                    help="timed calls per parity configuration and for the cascade")
    ap.add_argument("--no-configs", action="store_true", help="skip the parity-configuration legs")
    ap.add_argument("--no-prefill", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--only", choices=["all", "decode", "prefill", "int8", "cascade", "configs"], default="all",
                    help="run one leg only (profiling runs); 'configs' times the parity configurations")
    ap.add_argument("--decode-seqs", type=int, default=64, help="sequences of 4096 tokens in the decode leg")
    ap.add_argument("--prefill-seqs", type=int, default=4, help="prompts of 8192 tokens in the prefill leg")
    ap.add_argument("--prefill-dim", type=int, choices=[64, 128, 256], default=128,
                    help="head_dim of the prefill leg run by --only prefill (profiling)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-graph", action="store_true", help="launch the decode step eagerly, not as CUDA graphs")
    ap.add_argument("--no-int8", action="store_true", help="skip the 8-bit-cache decode legs (int8, fp8 E4M3)")
    ap.add_argument("--no-cascade", action="store_true", help="skip the shared-prefix (cascade) decode leg")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, world, rank)
        return
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=dev)
    peaks, peak_src = load_peaks()
    traffic = load_traffic()

    if args.only == "configs":
        r, _, _ = configs_leg(args, dev, peaks)
        if rank == 0:
            print(json.dumps({"configs": r, "peak_source": peak_src, "l2": "256 MB rewritten and re-read before "
                              "every timed call"}), flush=True)
        return
    if args.only == "cascade":
        c = cascade_leg(args, dev)
        if rank == 0:
            print(json.dumps({"cascade_only": True, "cascade_us": round(c["cascade_ms"] * 1e3, 2),
                              "plain_us": round(c["plain_ms"] * 1e3, 2),
                              "saving": round(c["plain_ms"] / c["cascade_ms"], 3), "max_diff": c["max_diff"]}),
                  flush=True)
        return
    if args.only == "int8":
        q8 = decode_int8_leg(args, dev)
        if rank == 0:
            print(json.dumps({"int8_only": True, "value": round(q8["gbs"], 2), "unit": "GB/s",
                              "call_ms": round(q8["ms"], 5)}), flush=True)
        return
    with ClockSampler(local) as clocks:
        d = None if args.only == "prefill" else decode_leg(args, world, rank, dev)
        pre_wl = PREFILL_WORKLOAD if args.prefill_dim == 128 else f"{PREFILL_WORKLOAD}_d{args.prefill_dim}"
        p = None if (args.no_prefill or args.only == "decode") else prefill_leg(args, dev, args.prefill_steps, pre_wl)
        p_dims = {} if (args.no_prefill or args.only != "all") else {
            d: prefill_leg(args, dev, max(1, args.prefill_steps // 2), f"{PREFILL_WORKLOAD}_d{d}") for d in (256, 64)}
        p_q8 = None if (args.no_prefill or args.no_int8 or args.only != "all") else \
            prefill_leg(args, dev, max(1, args.prefill_steps // 2), code_dtype=torch.int8)
        q8 = None if (args.no_int8 or args.only != "all") else decode_int8_leg(args, dev)
        f8 = None if (args.no_int8 or args.only != "all") else decode_int8_leg(args, dev, torch.float8_e4m3fn)
        cz = None if (args.no_cascade or args.only != "all") else cascade_leg(args, dev)
        cf = None if (args.no_configs or args.only != "all") else configs_leg(args, dev, peaks)
    clk = clocks.summary()
    if d is None:
        if rank == 0 and p is not None:
            pc = p["case"]
            wbytes = cache_write_bytes(pc.num_tokens, pc.num_kv_heads, pc.head_dim, 2)
            print(json.dumps({"prefill_only": True, "workload": pc.name, "value": round(p["tflops"], 2),
                              "unit": "TFLOP/s", "attn_ms": round(p["attn_ms"], 4),
                              "cache_write_ms": round(p["write_ms"], 4),
                              "cache_write_GBps": round(wbytes / (p["write_ms"] * 1e-3) / 1e9, 1),
                              "clocks": clk}), flush=True)
        return

    case = d["case"]
    dec_achieved = d["call_bytes"] / (d["call_ms"] / 1e3) / 1e9
    hbm = peaks["hbm_gbs"]
    line = {
        "metric": METRIC,
        "value": round(d["value"], 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(d["total_ms"] / args.steps, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": case.name, "num_seqs": case.num_reqs, "context_len": 4096,
                   "num_q_heads": case.num_q_heads, "num_kv_heads": case.num_kv_heads, "head_dim": case.head_dim,
                   "block_size": case.block_size, "num_splits": d["splits"],
                   "step": "reshape_and_cache(64 new rows) + decode(split-KV + combine)",
                   "launch": "eager" if args.no_graph else "one CUDA graph per step (write + decode), replayed; per-call times from one graph per call",
                   "l2": "no flush: 1.07 GB of K/V per step > 129 MB L2",
                   "parallelism": "replicas" if world == 1 else f"dp{world} (independent batches per GPU)"},
        "hbm_frac_of_peak": round(d["value"] / world / hbm, 4),
        "roofline": {"bound": "hbm", "kernel": "decode call (decode_bf16_kernel + combine_kernel)",
                     "achieved": round(dec_achieved, 2), "peak": hbm, "unit": "GB/s",
                     "frac": round(dec_achieved / hbm, 4), "peak_source": peak_src,
                     "algorithmic_bytes_per_launch": d["call_bytes"], "launch_ms": round(d["call_ms"], 5),
                     "traffic": traffic.get("decode_bf16_kernel")},
        "cache_write_ms": round(d["write_ms"], 5),
        "e2e": None if d["e2e_value"] is None else {
            "value": round(d["e2e_value"], 2), "unit": "GB/s", "h2d_bytes_per_step": d["h2d"],
            "d2h_bytes_per_step": d["d2h"], "ms_per_step": round(d["e2e_ms_per_step"], 5),
            "copies": "every step's inputs copied in from pinned host memory and its output read back to "
                      "pinned host memory inside the timed region; the copy-in of step i + 1 and the read-back "
                      "of step i overlap step i (two device buffer sets, two copy streams), as a serving loop "
                      "runs them",
            "serial": {"value": round(d["e2e_serial"], 2), "unit": "GB/s",
                       "ms_per_step": round(d["serial_ms_per_step"], 5),
                       "note": "the same steps with copy-in, step and read-back one after another on one stream"}},
        "gpu_launches": d["launches"],
        "decode_queries_per_s": round(world * case.num_reqs / (d["call_ms"] * 1e-3)),
        "clocks": clk,
    }
    if p is not None:
        tf_peak = peaks["bf16_tflops"]
        line["prefill"] = {
            "workload": PREFILL_WORKLOAD, "value": round(p["tflops"], 2), "unit": "TFLOP/s",
            "attn_ms": round(p["attn_ms"], 4), "cache_write_ms": round(p["write_ms"], 4),
            "causal_flops": p["flops"], "steps": args.prefill_steps, "gpu_launches": p["launches"],
            "roofline": {"bound": "tensor", "kernel": "varlen attention", "achieved": round(p["tflops"], 2),
                         "peak": tf_peak, "unit": "TFLOP/s", "frac": round(p["tflops"] / tf_peak, 4),
                         "peak_source": peak_src, "traffic": traffic.get("varlen_kernel")},
        }
        # the prompts' cache write (reshape_and_cache of all 32,768 rows), HBM-bound
        pc = p["case"]
        wbytes = cache_write_bytes(pc.num_tokens, pc.num_kv_heads, pc.head_dim, 2)
        wgbs = wbytes / (p["write_ms"] * 1e-3) / 1e9
        line["prefill"]["cache_write"] = {"algorithmic_bytes": wbytes, "GBps": round(wgbs, 1),
                                          "frac_of_hbm_peak": round(wgbs / peaks["hbm_gbs"], 4),
                                          "kernel": "reshape_and_cache_kernel"}
    for dim, pd in p_dims.items():
        tf_peak = peaks["bf16_tflops"]
        line[f"prefill_d{dim}"] = {
            "workload": pd["case"].name + f" ({pd['case'].num_q_heads} q / {pd['case'].num_kv_heads} KV heads, "
                                         f"head_dim {dim}, block 64, causal)",
            "value": round(pd["tflops"], 2), "unit": "TFLOP/s", "attn_ms": round(pd["attn_ms"], 4),
            "causal_flops": pd["flops"], "steps": max(1, args.prefill_steps // 2), "gpu_launches": pd["launches"],
            "frac_of_tensor_peak": round(pd["tflops"] / tf_peak, 4), "peak_source": peak_src,
            "traffic": traffic.get("varlen_tc256_kernel") if dim == 256 else None}
    if p_q8 is not None:
        line["prefill_int8"] = {
            "workload": "prefill_4x8192_int8 (the 4 x 8192 prompts over an int8 cache: codes + fp32 scales, "
                        "dequantised to bf16 tiles in shared memory)",
            "value": round(p_q8["tflops"], 2), "unit": "TFLOP/s", "attn_ms": round(p_q8["attn_ms"], 4),
            "causal_flops": p_q8["flops"], "steps": max(1, args.prefill_steps // 2),
            "gpu_launches": p_q8["launches"], "frac_of_tensor_peak": round(p_q8["tflops"] / peaks["bf16_tflops"], 4),
            "peak_source": peak_src}
    if q8 is not None:
        line["decode_int8"] = {
            "workload": "decode_64x4096_int8 (same queries and tokens, int8 codes + fp32 scales)",
            "value": round(q8["gbs"], 2), "unit": "GB/s", "call_ms": round(q8["ms"], 5),
            "algorithmic_bytes_per_launch": q8["bytes"], "frac_of_hbm_peak": round(q8["gbs"] / hbm, 4),
            "speedup_vs_bf16_call": round(d["call_ms"] / q8["ms"], 3), "traffic": traffic.get("decode_seg_kernel"),
            "kernel": "decode_seg_kernel<int8> + combine_seg_kernel (balanced segments)"}
    if f8 is not None:
        line["decode_fp8"] = {
            "workload": "decode_64x4096_fp8_e4m3 (same queries and tokens, E4M3 codes + fp32 scales)",
            "value": round(f8["gbs"], 2), "unit": "GB/s", "call_ms": round(f8["ms"], 5),
            "algorithmic_bytes_per_launch": f8["bytes"], "frac_of_hbm_peak": round(f8["gbs"] / hbm, 4),
            "speedup_vs_bf16_call": round(d["call_ms"] / f8["ms"], 3)}
    if cz is not None:
        cms = cz["cascade_ms"]
        line["cascade"] = {
            "workload": CASCADE_WORKLOAD + " (64 sequences, shared 4,000-token prefix, own suffixes of 1-256)",
            "cascade_us": round(cms * 1e3, 2), "plain_decode_us": round(cz["plain_ms"] * 1e3, 2),
            "saving": round(cz["plain_ms"] / cms, 3),
            "logical_kv_bytes": cz["logical"], "unique_kv_bytes": cz["unique"],
            "effective_GBps": round(cz["logical"] / (cms / 1e3) / 1e9, 1),
            "unique_GBps": round(cz["unique"] / (cms / 1e3) / 1e9, 1),
            "max_abs_diff_vs_plain": cz["max_diff"],
            "l2": "256 MB rewritten, then 256 MB read, between timed calls",
            "gpu_launches": cz["launches"]}
    if cf is not None:
        line["configs"] = cf[0]
        line["configs_note"] = ("parity configurations, each call a CUDA graph replay with 256 MB rewritten and "
                                "re-read before it (L2 cold); median of the calls; gpu_launches counts their "
                                "kernel launches")
        line["configs_gpu_launches"] = cf[2]
    if rank == 0 and world == 1 and not args.no_cpu_baseline and case.num_reqs == 64:
        _, ko_vo = None, oracle_pools(case)
        v, dt, n, threads = time_oracle_decode(case, *ko_vo)
        line["cpu_baseline"] = {"value": round(v, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                                "sample": f"{n} of 64 sequences (full 4096-token contexts, all 32 heads), "
                                          f"{dt:.1f} s"}
        # the same oracle on one host thread (a bounded sample of a few sequences)
        torch.set_num_threads(1)
        try:
            v1, dt1, n1, _ = time_oracle_decode(case, *ko_vo, budget_s=4.0, max_seqs=4)
        finally:
            torch.set_num_threads(threads)
        line["cpu_baseline"]["one_thread"] = {"value": round(v1, 4), "unit": "GB/s",
                                              "sample": f"{n1} sequences, {dt1:.1f} s"}
        # parity of the timed calls against the same oracle, every row (outside every timed region)
        import oracle
        want = oracle.paged_attention_decode(case.q, *ko_vo, case.block_tables, case.seq_lens, case.scale)
        diff = (d["out"].double() - want).abs()
        parity = {case.name: {"max_abs": float(diff.max()), "mean_abs": float(diff.mean()),
                              "rows": int(want.shape[0])}}
        if cf is not None:
            parity.update(config_parity(cf[1]))
        for pp in [p] + list(p_dims.values()):
            if pp is None:
                continue
            # a prefill: a sample of rows (the first and last 128 of every prompt and every 97th)
            pc = pp["case"]
            qsl = pc.query_start_loc.tolist()
            rows = sorted({t for r in range(pc.num_reqs) for t in
                           list(range(qsl[r], qsl[r] + 128)) + list(range(qsl[r + 1] - 128, qsl[r + 1])) +
                           list(range(qsl[r], qsl[r + 1], 97))})
            idx = torch.tensor(rows)
            pko, pvo = oracle_pools(pc)
            want = oracle.paged_attention_varlen(pc.q, pko, pvo, pc.query_start_loc, pc.seq_lens, pc.block_tables,
                                                 True, pc.scale, tokens=idx)
            diff = (pp["out"][idx].double() - want[idx]).abs()
            parity[pc.name] = {"max_abs": float(diff.max()), "mean_abs": float(diff.mean()), "rows": len(rows),
                               "rows_of": int(pc.num_tokens)}
        if p_q8 is not None:
            # the int8-cache prefill against the oracle over the oracle's own quantised cache, same rows
            from oracle import quant
            pc = p_q8["case"]
            shape = (pc.num_blocks, pc.block_size, pc.num_kv_heads, pc.head_dim)
            ko8, vo8 = torch.zeros(shape, dtype=torch.int8), torch.zeros(shape, dtype=torch.int8)
            kso, vso = torch.zeros(shape[:3]), torch.zeros(shape[:3])
            quant.reshape_and_cache_quant(pc.key, pc.value, ko8, vo8, kso, vso, pc.slot_mapping, "int8")
            want = quant.paged_attention_varlen_quant(pc.q, ko8, vo8, kso, vso, pc.query_start_loc, pc.seq_lens,
                                                      pc.block_tables, True, pc.scale, tokens=idx)
            diff = (p_q8["out"][idx].double() - want[idx]).abs()
            parity["prefill_4x8192_int8"] = {"max_abs": float(diff.max()), "mean_abs": float(diff.mean()),
                                             "rows": len(rows), "rows_of": int(pc.num_tokens)}
        line["parity_vs_oracle"] = parity
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
