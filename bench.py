"""Benchmark of the paged-KV attention hot path on GB300.

One step = one pass of the path over one batch of the llama7b-decode workload
(8 sequences, context ~ U[512, 2048], 32 heads, head_dim 128, block_size 16,
8192-block pool, bf16): write each sequence's new token into the pool through
slot_mapping, then paged decode over the whole context (split-KV plus the
log-sum-exp merge) -- one pa_decode_write call, the public entry point for a
decode step.  The headline value is the K/V bytes the step
must read from HBM divided by the step's device time, with L2 flushed between
timed steps.  The same line carries five secondary measurements (the
packed-prefill workload in TFLOP/s, the long-context decode workload in GB/s,
the headline decode over INT8 and over FP8 pools in GB/s, and copy-on-write
block copies in GB/s), the roofline of the dominant kernel, the oracle's CPU
time, and an end-to-end figure through host buffers.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

With --gpus N > 1 (launched by torchrun) every rank runs its own batch on its
own GPU (the decode batch shards by sequence: weak scaling, no data-path
collective); the value is all ranks' bytes over the slowest rank's time.
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
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

HEADLINE = "llama7b-decode"
METRIC = "paged-decode KV-read GB/s (% of HBM peak); varlen prefill TFLOP/s"
L2_FLUSH_BYTES = 512 << 20  # > 129 MB L2
HOST_LEAD_CYCLES = 1_000_000  # ~0.5 ms of device spin ahead of each timed step


# ---------------------------------------------------------------------------
# algorithmic work
# ---------------------------------------------------------------------------
def kv_read_bytes(x) -> int:
    """K and V bytes decode must read: every context position, every KV head."""
    return int(x.context_lens.sum().item()) * x.num_kv_heads * x.head_dim * 2 * 2


def decode_bytes(x) -> int:
    """All HBM bytes the decode launch needs: K/V, q in, out, the block-table
    entries it walks, context_lens."""
    s, hq, d, bs = x.num_seqs, x.num_q_heads, x.head_dim, x.block_size
    blocks = int(((x.context_lens + bs - 1) // bs).sum().item())
    return kv_read_bytes(x) + 2 * s * hq * d * 2 + blocks * 4 + s * 4


def write_bytes(x) -> int:
    n = int(x.slot_mapping.numel())
    return 2 * n * x.num_kv_heads * x.head_dim * 2 * 2 + n * 8


def prefill_flops(x) -> int:
    """4 * Hq * D per visible (query, key) pair (QK^T and PV), causal
    bottom-right: row i of a sequence with q queries, L keys sees L-q+i+1."""
    q = x.q_lens.long()
    L = x.context_lens.long()
    if x.causal:
        pairs = (q * (L - q) + q * (q + 1) // 2).sum().item()
    else:
        pairs = (q * L).sum().item()
    return int(4 * x.num_q_heads * x.head_dim * pairs)


# ---------------------------------------------------------------------------
# device-side helpers
# ---------------------------------------------------------------------------
class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=5)

    def summary(self):
        mhz, maxmhz, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [c.strip() for c in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                mhz.append(float(f[1]))
                maxmhz = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(mhz) if mhz else None, "sm_max_mhz": maxmhz,
                "reasons": sorted(reasons), "samples": len(mhz)}


def flush_l2(buf):
    """Write a buffer larger than L2, then read a second one: the write
    evicts every useful line, the read evicts the write's dirty lines, so their
    write-back happens here (untimed) and not inside the next timed step."""
    buf[0].add_(1)
    buf[1].sum()


def settle(step, seconds: float = 0.25):
    """Untimed back-to-back steps for a fixed wall time after the warm-up
    steps, so the timed region does not start while the GPU's clocks are
    still ramping up from idle."""
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < seconds:
        for _ in range(20):
            step()
        torch.cuda.synchronize()


# seconds of untimed steps before each timed loop (0 in the --only profiling
# mode, whose launch counts must be fixed)
SETTLE_S = 0.25


def time_steps(step, k, flush_buf, stream):
    """Per-step device time (ms) with CUDA events on the launching stream, L2
    flushed (untimed) before each step."""
    if SETTLE_S > 0:
        settle(step, SETTLE_S)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(k)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(k)]
    for e in starts + ends:  # create the events now, not inside the timed loop
        e.record(stream)
    torch.cuda.synchronize()
    for i in range(k):
        flush_l2(flush_buf)
        # a short device-side spin before the start event, so the host has
        # enqueued the step by the time the GPU reaches it: the interval then
        # holds the step's device time, not the host's launch latency
        torch.cuda._sleep(HOST_LEAD_CYCLES)
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize()
    return [s.elapsed_time(e) for s, e in zip(starts, ends)]


def source_hash(*names) -> str:
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "paged_kv_cache_34_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str, src_hash: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current source of the kernel."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path):
        return None
    for line in open(path):
        m = re.match(r"\s*(\S+)\s+(\S+)\s+src=(\w+)\s+dram_bytes_per_launch=(\d+)", line)
        if m and m.group(1) == kernel and m.group(2) == workload and m.group(3) == src_hash:
            return int(m.group(4))
    return None


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return d["hbm_gbs"], d["bf16_tflops"], d.get("bf16_tflops_sustained"), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


# ---------------------------------------------------------------------------
# the steps
# ---------------------------------------------------------------------------
def decode_step_fn(pa, x, out, ws, stream):
    """One decode step through the public API: pa_decode_write (this step's
    cache write, then the decode, as one call)."""
    def step():
        pa.pa_decode_write(out, x.q, x.k_new, x.v_new, x.k_pool, x.v_pool, x.slot_mapping,
                           x.block_table, x.context_lens, scale=x.scale,
                           max_context_len=x.max_context_len, partition_size=x.partition_size,
                           workspace=ws, stream=stream)
    return step


def decode_workspace(pa, x):
    """Workspace for the plan pa_decode uses, and the plan: partition size
    (0 = balanced split across the grid's workers) and partitions of the
    longest context (None for the balanced split, whose pieces depend on
    the device-side lengths)."""
    part, need = pa.pa_decode_plan(x.num_seqs, x.num_q_heads, x.num_kv_heads, x.head_dim,
                                   x.max_context_len, x.partition_size)
    ws = torch.empty(max(need, 256), dtype=torch.uint8, device="cuda") if need else None
    if part == 0:
        nparts = None
    else:
        nparts = math.ceil(x.max_context_len / part) if x.max_context_len else 1
    return ws, part, nparts


def bench_decode(pa, W, name, steps, warmup, flush_buf, stream, seed=None, overrides=None):
    x = W.make_inputs(name, seed=seed, device="cuda", **(overrides or {}))
    out = torch.empty_like(x.q)
    ws, part, nparts = decode_workspace(pa, x)
    step = decode_step_fn(pa, x, out, ws, stream)
    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    t_step = time_steps(step, steps, flush_buf, stream)
    # the decode launch alone (for its roofline), same conditions
    def dec():
        pa.pa_decode(out, x.q, x.k_pool, x.v_pool, x.block_table, x.context_lens,
                     scale=x.scale, max_context_len=x.max_context_len,
                     partition_size=x.partition_size, workspace=ws, stream=stream)
    t_dec = time_steps(dec, steps, flush_buf, stream)
    return x, out, ws, part, nparts, t_step, t_dec


def bench_decode_kv8(pa, W, name, steps, warmup, flush_buf, stream, fmt="int8"):
    """The decode workload over 8-bit pools (fmt "int8" or "fp8").  The
    16-bit pools are quantised once, whole, by the library's 8-bit write under
    per-KV-head absmax / (largest code) scales; a step is the one-call 8-bit
    step (this step's new tokens written, then the decode).  Returns the
    inputs, the plan, the step times and the times of the decode call alone."""
    x = W.make_inputs(name, device="cuda")
    hkv, d = x.num_kv_heads, x.head_dim
    top = 127.0 if fmt == "int8" else 448.0
    write = pa.pa_reshape_and_cache_int8 if fmt == "int8" else pa.pa_reshape_and_cache_fp8
    decode = pa.pa_decode_int8 if fmt == "int8" else pa.pa_decode_fp8
    step_call = pa.pa_decode_write_int8 if fmt == "int8" else pa.pa_decode_write_fp8

    def absmax_scale(pool):
        # unwritten pool slots hold NaN: they quantise to 0 and set no scale
        a = pool.reshape(-1, hkv, d).float().nan_to_num(0.0, 0.0, 0.0).abs().amax(dim=(0, 2))
        return (a / top).clamp_min(1e-6).contiguous()
    ks, vs = absmax_scale(x.k_pool), absmax_scale(x.v_pool)
    code = torch.int8 if fmt == "int8" else torch.uint8
    kc = torch.empty(x.k_pool.shape, dtype=code, device="cuda")
    vc = torch.empty_like(kc)
    slots = torch.arange(x.k_pool.shape[0] * x.block_size, dtype=torch.int64, device="cuda")
    write(x.k_pool.reshape(-1, hkv, d), x.v_pool.reshape(-1, hkv, d), kc, vc, slots, ks, vs,
          stream=stream)
    x.k_pool = x.v_pool = None  # the 16-bit pools are not read again
    del slots
    out = torch.empty_like(x.q)
    ws, part, nparts = decode_workspace(pa, x)

    def dec():
        decode(out, x.q, kc, vc, x.block_table, x.context_lens, ks, vs, scale=x.scale,
               max_context_len=x.max_context_len, partition_size=x.partition_size,
               workspace=ws, stream=stream)

    def step():
        step_call(out, x.q, x.k_new, x.v_new, kc, vc, x.slot_mapping, x.block_table,
                  x.context_lens, ks, vs, scale=x.scale, max_context_len=x.max_context_len,
                  partition_size=x.partition_size, workspace=ws, stream=stream)
    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    t_step = time_steps(step, steps, flush_buf, stream)
    t_dec = time_steps(dec, steps, flush_buf, stream)
    return x, part, nparts, t_step, t_dec


COPY_PAIRS = 1024


def bench_copy_blocks(pa, steps, warmup, flush_buf, stream):
    """Copy-on-write of whole blocks on pools shaped like llama7b-decode's
    (8192 blocks of 16 tokens x 32 KV heads x 128, bf16: 128 KB per block and
    pool): each call copies 1024 blocks to 1024 others in both pools.
    Returns the bytes one call moves (read + written) and the call times."""
    nb = 8192
    g = torch.Generator(device="cuda").manual_seed(1234)
    k = torch.randn(nb, 16, 32, 128, generator=g, device="cuda").to(torch.bfloat16)
    v = torch.randn(nb, 16, 32, 128, generator=g, device="cuda").to(torch.bfloat16)
    ids = torch.randperm(nb, generator=g, device="cuda")
    mapping = torch.stack([ids[:COPY_PAIRS], ids[COPY_PAIRS:2 * COPY_PAIRS]], dim=1).contiguous()

    def call():
        pa.pa_copy_blocks(k, v, mapping, stream=stream)
    for _ in range(warmup):
        call()
    torch.cuda.synchronize()
    t = time_steps(call, steps, flush_buf, stream)
    moved = 2 * 2 * COPY_PAIRS * k[0].numel() * k.element_size()  # K+V, read+written
    return moved, t


def bench_prefill(pa, W, steps, warmup, flush_buf, stream, name="packed-prefill",
                  overrides=None):
    """A prefill step (this step's K/V rows written, then causal attention of
    the packed queries against the paged cache), and the prefill call alone."""
    x = W.make_inputs(name, device="cuda", **(overrides or {}))
    out = torch.empty_like(x.q)

    def pre():
        pa.pa_prefill_varlen(out, x.q, x.k_pool, x.v_pool, x.block_table, x.cu_seqlens_q,
                             x.context_lens, scale=x.scale, max_seqlen_q=x.max_seqlen_q,
                             max_context_len=x.max_context_len, causal=True, stream=stream)

    def step():
        pa.pa_reshape_and_cache(x.k_new, x.v_new, x.k_pool, x.v_pool, x.slot_mapping,
                                stream=stream)
        pre()
    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    t_step = time_steps(step, steps, flush_buf, stream)
    t_pre = time_steps(pre, steps, flush_buf, stream)
    return x, t_step, t_pre


def e2e_decode(pa, W, name, steps, warmup, stream):
    """Through host buffers: each step uploads its inputs (q, the new K/V rows,
    slot_mapping, context_lens, block_table) from one pinned staging buffer in
    one copy, runs write + decode (pa_decode_write) and copies the output back.
    The step is captured once as a CUDA graph and replayed (eager launches if
    capture is unavailable); host wall clock around each replay."""
    x = W.make_inputs(name, device="cuda")
    names = ("q", "k_new", "v_new", "slot_mapping", "context_lens", "block_table")
    offs, total = {}, 0
    for k in names:
        t = getattr(x, k)
        offs[k] = total
        total = (total + t.numel() * t.element_size() + 255) // 256 * 256
    host = torch.zeros(total, dtype=torch.uint8).pin_memory()
    dev = torch.empty(total, dtype=torch.uint8, device="cuda")
    views = {}
    for k in names:
        t = getattr(x, k).contiguous()
        n = t.numel() * t.element_size()
        host[offs[k]:offs[k] + n].copy_(t.cpu().view(torch.uint8).reshape(-1))
        views[k] = dev[offs[k]:offs[k] + n].view(t.dtype).view(t.shape)
    out_h = torch.empty(x.q.shape, dtype=x.q.dtype).pin_memory()
    out_d = torch.empty_like(x.q)
    ws, _, _ = decode_workspace(pa, x)
    h2d = total
    d2h = out_h.numel() * out_h.element_size()

    def step(s):
        with torch.cuda.stream(s):
            dev.copy_(host, non_blocking=True)
            pa.pa_decode_write(out_d, views["q"], views["k_new"], views["v_new"], x.k_pool,
                               x.v_pool, views["slot_mapping"], views["block_table"],
                               views["context_lens"], scale=x.scale,
                               max_context_len=x.max_context_len,
                               partition_size=x.partition_size, workspace=ws, stream=s)
            out_h.copy_(out_d, non_blocking=True)
    for _ in range(warmup):
        step(stream)
    torch.cuda.synchronize()
    run, method = (lambda: step(stream)), "eager launches"
    try:
        graph = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream()
        with torch.cuda.graph(graph, stream=cap):
            step(cap)
        graph.replay()
        torch.cuda.synchronize()
        run, method = graph.replay, "CUDA graph replay"
    except Exception as e:  # noqa: BLE001 - report how the step was run
        print(f"e2e: graph capture unavailable ({e}); timing eager launches", file=sys.stderr)
        torch.cuda.synchronize()
    for _ in range(warmup):
        run()
    torch.cuda.synchronize()
    flush = torch.zeros(2, L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
    times = []
    for _ in range(steps):
        flush_l2(flush)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        run()
        torch.cuda.synchronize()
        times.append((time.perf_counter() - t0) * 1e3)
    want = out_d.clone()
    step(stream)
    torch.cuda.synchronize()
    if not torch.equal(out_h.cuda(), want):
        raise RuntimeError("e2e: the replayed step's output differs from an eager step's")
    return kv_read_bytes(x), times, h2d, d2h, method


# ---------------------------------------------------------------------------
# CPU baseline: the oracle on the host cores
# ---------------------------------------------------------------------------
def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo), for the record."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith(("model name", "cpu part")):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def oracle_decode_rate(x_dev, budget_s: float, max_calls: int | None = None,
                       threads: int | None = None):
    """The oracle's write + decode over sequences of the workload, repeated
    until ~budget_s of CPU time (on `threads` OpenMP threads, default all);
    returns (GB/s of K/V read, calls, threads, seconds)."""
    import oracle
    x = x_dev.to("cpu")
    kp = oracle._u16(x.k_pool)
    vp = oracle._u16(x.v_pool)
    lib = oracle.load()
    oracle.set_threads(threads or os.cpu_count() or 1, lib=lib)
    threads = oracle.max_threads(lib)
    kv_per_seq = (x.context_lens.long() * x.num_kv_heads * x.head_dim * 4).tolist()
    # one call = one sequence's write + decode (all heads); cycle through them
    nbytes, calls, t0 = 0, 0, time.perf_counter()
    cu = 0
    slots = x.slot_mapping
    while True:
        b = calls % x.num_seqs
        n_new = int(x.new_lens[b])
        if n_new:
            oracle.write(kp, vp, x.k_new[cu:cu + n_new], x.v_new[cu:cu + n_new],
                         slots[cu:cu + n_new], x.block_size, lib=lib)
        cu = (cu + n_new) % max(1, slots.numel())
        oracle.decode(x.q[b:b + 1], kp, vp, x.block_table[b:b + 1], x.context_lens[b:b + 1],
                      x.num_kv_heads, x.block_size, x.scale, lib=lib)
        nbytes += kv_per_seq[b]
        calls += 1
        el = time.perf_counter() - t0
        if el >= budget_s or (max_calls and calls >= max_calls):
            break
    return nbytes / el / 1e9, calls, threads, el


def oracle_prefill_rate(x_dev, budget_s: float, rows_per_seq: int = 8):
    """The oracle's prefill on a sample of query rows (the last rows_per_seq
    of every sequence: the rows with the most visible keys), repeated until
    ~budget_s; returns (TFLOP/s of visible pairs, calls, threads, seconds)."""
    import oracle
    x = x_dev.to("cpu")
    lib = oracle.load()
    oracle.set_threads(os.cpu_count() or 1, lib=lib)
    threads = oracle.max_threads(lib)
    kp, vp = oracle._u16(x.k_pool), oracle._u16(x.v_pool)
    # the step's write first (the sample then reads this step's rows too)
    oracle.write(kp, vp, x.k_new, x.v_new, x.slot_mapping, x.block_size, lib=lib)
    cu, q, L = x.cu_seqlens_q.tolist(), x.q_lens.tolist(), x.context_lens.tolist()
    rows, pairs = [], 0
    for b in range(x.num_seqs):
        for i in range(max(0, q[b] - rows_per_seq), q[b]):
            rows.append(cu[b] + i)
            pairs += L[b] - q[b] + i + 1
    rows = np.asarray(rows, dtype=np.int64)
    flops = 4 * x.num_q_heads * x.head_dim * pairs
    calls, t0 = 0, time.perf_counter()
    while True:
        oracle.prefill(x.q, kp, vp, x.block_table, x.cu_seqlens_q, x.context_lens,
                       x.num_kv_heads, x.block_size, x.scale, causal=x.causal, rows=rows,
                       lib=lib)
        calls += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    return flops * calls / el / 1e12, calls, threads, el


def headline_config(x, world: int) -> dict:
    """The headline workload's description, the same in both arms."""
    return {"workload": HEADLINE, "sequences_per_gpu": x.num_seqs, "context": "U[512,2048]",
            "heads": f"{x.num_q_heads}/{x.num_kv_heads}", "head_dim": x.head_dim,
            "block_size": x.block_size, "pool_blocks": x.num_blocks,
            "step": "one decode step: cache write of each sequence's new token, then "
                    "attention over its whole context",
            "l2": "flushed before every timed GPU step (512 MB write, then 512 MB read)",
            "parallelism": f"replica x{world}" if world > 1 else "single GPU"}


# ---------------------------------------------------------------------------
def dist_setup(gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
        rank = dist.get_rank()
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", rank)))
        return dist, rank, world
    torch.cuda.set_device(0)
    return None, 0, 1


def _reduce(dist, v: float, op) -> float:
    """All-reduce one number over the ranks (a CPU tensor under gloo)."""
    if dist is None:
        return v
    dev = "cpu" if dist.get_backend() == "gloo" else "cuda"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=op)
    return float(t.item())


def reduce_max(dist, v: float) -> float:
    return v if dist is None else _reduce(dist, v, dist.ReduceOp.MAX)


def reduce_sum(dist, v: float) -> float:
    return v if dist is None else _reduce(dist, v, dist.ReduceOp.SUM)


def rank_seed(W, rank: int) -> int:
    """Each rank draws its own batch of the headline workload (weak scaling:
    the work per GPU is fixed, the job grows with the ranks)."""
    return W.default_seed(HEADLINE) + 7919 * rank


def whole_job_gbs(dist, bytes_this_rank: int, ms_this_rank: float) -> tuple[float, float]:
    """(GB/s of the whole job, slowest rank's ms): every rank's bytes over the
    slowest rank's time."""
    ms_max = reduce_max(dist, ms_this_rank)
    return reduce_sum(dist, bytes_this_rank) / (ms_max * 1e-3) / 1e9, ms_max


def run_reference(args):
    """The oracle (the path's plain fp64 CPU statement) timed on the host
    cores on bounded samples of the same workload and metric."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from paged_kv_cache_34_gb300 import workloads as W
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    x = W.make_inputs(HEADLINE, device=dev)
    per_step = max(0.02, min(2.0, 60.0 / max(1, args.steps + args.warmup)))
    oracle_decode_rate(x, per_step * args.warmup, max_calls=max(1, args.warmup))
    rates, calls_total, secs = [], 0, 0.0
    threads = 1
    for _ in range(args.steps):
        r, calls, threads, el = oracle_decode_rate(x, per_step)
        rates.append(r)
        calls_total += calls
        secs += el
    value = calls_total and sum(rates) / len(rates)
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(secs * 1e3 / max(1, args.steps), 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": headline_config(x, args.gpus),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads,
                         "kind": "oracle", "cpu_model": cpu_model(),
                         "sample": f"{calls_total} single-sequence write+decode oracle calls "
                                   f"(~{per_step:.2f} s per step) cycling the 8 sequences"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def run_only(pa, W, args, flush_buf, stream):
    """One kernel's workload alone, without the e2e, secondary and CPU legs,
    and with a fixed number of launches (a profiling target): W warm-up steps,
    K timed steps, then K calls of the kernel alone."""
    global SETTLE_S
    SETTLE_S = 0.0
    decode_only = {"decode": (HEADLINE, None), "long-context": ("long-context-decode", None),
                   "continuous-batching": ("continuous-batching", None),
                   "continuous-batching-g16": ("continuous-batching", {"num_q_heads": 128}),
                   "tiny-decode": ("tiny-decode", None)}
    if args.only in decode_only:
        name, over = decode_only[args.only]
        x, _, _, part, nparts, _, t = bench_decode(pa, W, name, args.steps, args.warmup,
                                                   flush_buf, stream, overrides=over)
        ms = statistics.fmean(t)
        print(json.dumps({"only": args.only, "workload": name, "ms": round(ms, 5),
                          "GBps": round(decode_bytes(x) / (ms * 1e-3) / 1e9, 1),
                          "partition_size": part, "partitions": nparts}))
    elif args.only in ("decode-int8", "decode-fp8"):
        x, part, nparts, _, t = bench_decode_kv8(pa, W, HEADLINE, args.steps, args.warmup,
                                                 flush_buf, stream, args.only[7:])
        ms = statistics.fmean(t)
        kv8 = kv_read_bytes(x) // 2
        print(json.dumps({"only": args.only, "workload": HEADLINE, "ms": round(ms, 5),
                          "GBps": round((kv8 + decode_bytes(x) - kv_read_bytes(x))
                                        / (ms * 1e-3) / 1e9, 1),
                          "partition_size": part, "partitions": nparts}))
    elif args.only == "copy-blocks":
        moved, t = bench_copy_blocks(pa, args.steps, args.warmup, flush_buf, stream)
        ms = statistics.fmean(t)
        print(json.dumps({"only": "copy-blocks", "pairs": COPY_PAIRS, "ms": round(ms, 5),
                          "GBps": round(moved / (ms * 1e-3) / 1e9, 1)}))
    else:
        name = "chunked-prefill" if args.only == "chunked-prefill" else "packed-prefill"
        over = {"num_kv_heads": 8} if args.only == "prefill-gqa4" else None
        x, _, t = bench_prefill(pa, W, args.steps, args.warmup, flush_buf, stream, name, over)
        ms = statistics.fmean(t)
        print(json.dumps({"only": args.only, "workload": name, "ms": round(ms, 5),
                          "TFLOPs": round(prefill_flops(x) / (ms * 1e-3) / 1e12, 1),
                          "KV_GBps": round(kv_read_bytes(x) / (ms * 1e-3) / 1e9, 1)}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-secondary", action="store_true",
                    help="skip the packed-prefill, long-context, 8-bit pool and copy-blocks "
                         "measurements")
    ap.add_argument("--cpu-budget", type=float, default=15.0,
                    help="seconds of oracle time for the CPU baseline")
    ap.add_argument("--only",
                    choices=["decode", "long-context", "continuous-batching",
                             "continuous-batching-g16", "tiny-decode", "decode-int8",
                             "decode-fp8", "copy-blocks", "prefill", "chunked-prefill",
                             "prefill-gqa4"],
                    help="time one kernel's workload alone (a small profiling target)")
    args = ap.parse_args()
    if args.impl == "reference":
        run_reference(args)
        return
    assert args.warmup >= 3, "at least 3 warm-up steps"

    import paged_kv_cache_34_gb300 as pa
    from paged_kv_cache_34_gb300 import build as pabuild
    from paged_kv_cache_34_gb300 import workloads as W
    if not pabuild.up_to_date():
        pabuild.build()
    dist, rank, world = dist_setup(args.gpus)
    stream = torch.cuda.current_stream()
    flush_buf = torch.zeros(2, L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
    hbm_peak, tf_peak, tf_sustained, peak_kind = measured_peaks()
    if args.only:
        run_only(pa, W, args, flush_buf, stream)
        return

    # ---- headline: write + decode on the llama7b-decode workload ----------
    seed = rank_seed(W, rank)  # each rank its own batch
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    with ClockSampler(torch.cuda.current_device()) as clocks:
        x, out, ws, part, nparts, t_step, t_dec = bench_decode(
            pa, W, HEADLINE, args.steps, args.warmup, flush_buf, stream, seed=seed)
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    if dist is not None:
        dist.barrier()
    ms_step = statistics.fmean(t_step)
    kv = kv_read_bytes(x)
    value, ms_step_max = whole_job_gbs(dist, kv, ms_step)  # every rank's own batch
    merge = nparts is None or nparts > 1  # the merge kernel runs
    # 16-bit pools with the balanced split write inside the decode launch;
    # otherwise the write is a launch of its own
    separate_write = x.slot_mapping.numel() > 0 and part != 0
    launches_per_step = (1 if separate_write else 0) + 1 + (1 if merge else 0)

    ms_dec = statistics.fmean(t_dec)
    dec_achieved = decode_bytes(x) / (ms_dec * 1e-3) / 1e9
    dec_hash = source_hash("decode_kernel.cuh", "decode.cu", "pa_device.cuh")
    traffic = recorded_traffic("pa_decode", HEADLINE, dec_hash)

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step_max, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": headline_config(x, world),
        "step_detail": {"call": "pa_decode_write (the cache write inside the decode launch)"
                                if not separate_write else "pa_decode_write",
                        "split_kv": "balanced across workers" if part == 0 else
                                    f"fixed partitions of {part} tokens ({nparts} for the longest)",
                        "kv_bytes_per_step": kv, "wall_s_timed_region": round(wall, 3),
                        "pct_of_hbm_peak": round(100 * value / world / hbm_peak, 2)},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks.summary(),
        "roofline": {"kernel": "pa_decode (split-KV decode + merge launches)", "bound": "hbm",
                     "achieved": round(dec_achieved, 1), "peak": hbm_peak,
                     "peak_kind": peak_kind, "unit": "GB/s",
                     "frac": round(dec_achieved / hbm_peak, 4), "traffic": traffic,
                     "algorithmic_bytes_per_launch": decode_bytes(x),
                     "ms_per_launch": round(ms_dec, 5)},
    }

    if rank == 0:
        # ---- e2e through host buffers ----------------------------------
        kv_e2e, t_e2e, h2d, d2h, e2e_method = e2e_decode(pa, W, HEADLINE, max(20, args.steps // 4),
                                             args.warmup, stream)
        line["e2e"] = {"value": round(kv_e2e / (statistics.fmean(t_e2e) * 1e-3) / 1e9, 2),
                       "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                       "ms_per_step": round(statistics.fmean(t_e2e), 5),
                       "method": e2e_method + " of [one H2D copy of the packed inputs, "
                                 "pa_decode_write, one D2H copy of the output], host wall "
                                 "clock, L2 flushed before each step"}

        ob = max(1.0, args.cpu_budget / 6)  # oracle seconds per secondary workload
        if not args.no_secondary:
            sec = {}
            pre_hash = source_hash("prefill.cu", "pa_tcgen05.cuh", "pa_device.cuh")
            # ---- prefill: packed (q = L; also with 32 query heads over 8 KV
            # heads, packed four to a tile) and chunked / multi-token (q < L)
            for pname, over in (("packed-prefill", None), ("chunked-prefill", None),
                                ("packed-prefill", {"num_kv_heads": 8})):
                key = pname + ("-gqa4" if over else "")
                xp, t_pstep, t_pre = bench_prefill(pa, W, max(10, args.steps // 10), args.warmup,
                                                   flush_buf, stream, pname, over)
                fl = prefill_flops(xp)
                ms_pre = statistics.fmean(t_pre)
                tf = fl / (ms_pre * 1e-3) / 1e12
                kvb = kv_read_bytes(xp)
                entry = {
                    "value": round(tf, 2), "unit": "TFLOP/s", "flops": fl,
                    "kv_bytes": kvb, "ms_prefill": round(ms_pre, 5),
                    "ms_write_plus_prefill": round(statistics.fmean(t_pstep), 5),
                    "q_lens": "q = L" if pname == "packed-prefill" else "1, 4, 64 cycling",
                    "heads": f"{xp.num_q_heads}/{xp.num_kv_heads}"}
                if pname == "packed-prefill":
                    entry["write_GBps"] = round(write_bytes(xp) / ((statistics.fmean(t_pstep)
                                                                    - ms_pre) * 1e-3) / 1e9, 1)
                    entry["roofline"] = {
                        "bound": "tensor", "achieved": round(tf, 1), "peak": tf_peak,
                        "peak_kind": f"{peak_kind} bf16 burst", "unit": "TFLOP/s",
                        "frac": round(tf / tf_peak, 4),
                        "traffic": recorded_traffic("pa_prefill_varlen", key, pre_hash)}
                else:
                    # a few queries per sequence against long contexts: the
                    # K/V bytes, not the flops, set the bound
                    gbp = kvb / (ms_pre * 1e-3) / 1e9
                    entry["roofline"] = {
                        "bound": "hbm", "achieved": round(gbp, 1), "peak": hbm_peak,
                        "unit": "GB/s", "frac": round(gbp / hbm_peak, 4),
                        "traffic": recorded_traffic("pa_prefill_varlen", key, pre_hash)}
                r, calls, th, el = oracle_prefill_rate(xp, ob)
                entry["cpu_baseline"] = {"value": round(r, 6), "unit": "TFLOP/s", "cores": th,
                                         "kind": "oracle",
                                         "sample": f"{calls} oracle prefill calls on the last "
                                                   f"8 query rows of each sequence ({el:.1f} s)"}
                sec[key] = entry
                del xp
            # ---- 16-bit decodes: the other decode workloads (and a 16-query-
            # head group over the continuous-batching batch)
            for dname, over, note in (
                    ("tiny-decode", {}, "launch-bound (132 KB of K/V): no roofline claim"),
                    ("continuous-batching", {}, None),
                    ("continuous-batching", {"num_q_heads": 128},
                     "128 query heads over 8 KV heads (16 per KV head, one K/V read)"),
                    ("long-context-decode", {}, None)):
                key = dname if not over else f"{dname}-g{over['num_q_heads'] // 8}"
                xd, _, _, partd, npd, _, t_d = bench_decode(
                    pa, W, dname, max(10, args.steps // 10), args.warmup, flush_buf, stream,
                    overrides=over)
                ms_d = statistics.fmean(t_d)
                gbd = decode_bytes(xd) / (ms_d * 1e-3) / 1e9
                entry = {"value": round(kv_read_bytes(xd) / (ms_d * 1e-3) / 1e9, 1),
                         "unit": "GB/s", "ms_decode": round(ms_d, 5),
                         "heads": f"{xd.num_q_heads}/{xd.num_kv_heads}",
                         "partition_size": partd, "partitions": npd}
                if note:
                    entry["note"] = note
                entry["roofline"] = None if dname == "tiny-decode" else {
                    "bound": "hbm", "achieved": round(gbd, 1), "peak": hbm_peak,
                    "unit": "GB/s", "frac": round(gbd / hbm_peak, 4),
                    "traffic": recorded_traffic("pa_decode", key, dec_hash)}
                r, calls, th, el = oracle_decode_rate(xd, ob)
                entry["cpu_baseline"] = {"value": round(r, 4), "unit": "GB/s", "cores": th,
                                         "kind": "oracle",
                                         "sample": f"{calls} single-sequence oracle decode "
                                                   f"calls ({el:.1f} s)"}
                sec[key] = entry
                del xd
            for fmt, pools in (("int8", "int8 codes"), ("fp8", "FP8 E4M3 codes")):
                xi, parti, npi, t_istep, t_idec = bench_decode_kv8(
                    pa, W, HEADLINE, max(20, args.steps // 4), args.warmup, flush_buf, stream,
                    fmt)
                ms_i = statistics.fmean(t_idec)
                kv8 = kv_read_bytes(xi) // 2  # one byte per element
                gb8 = (kv8 + decode_bytes(xi) - kv_read_bytes(xi)) / (ms_i * 1e-3) / 1e9
                sec[f"llama7b-decode-{fmt}"] = {
                    "value": round(kv8 / (ms_i * 1e-3) / 1e9, 1), "unit": "GB/s",
                    "pools": f"{pools}, per-KV-head fp32 scales (absmax / largest code)",
                    "ms_decode": round(ms_i, 5),
                    "ms_write_plus_decode": round(statistics.fmean(t_istep), 5),
                    "speedup_vs_16bit_decode": round(ms_dec / ms_i, 3),
                    "partition_size": parti, "partitions": npi,
                    "roofline": {"bound": "hbm", "achieved": round(gb8, 1), "peak": hbm_peak,
                                 "unit": "GB/s", "frac": round(gb8 / hbm_peak, 4),
                                 "traffic": recorded_traffic(f"pa_decode_{fmt}", HEADLINE,
                                                             dec_hash)}}
                del xi
            moved, t_cp = bench_copy_blocks(pa, max(20, args.steps // 4), args.warmup,
                                            flush_buf, stream)
            ms_cp = statistics.fmean(t_cp)
            gb_cp = moved / (ms_cp * 1e-3) / 1e9
            sec["copy-blocks"] = {
                "value": round(gb_cp, 1), "unit": "GB/s (read + written)",
                "pairs": COPY_PAIRS, "bytes_per_call": moved, "ms_call": round(ms_cp, 5),
                "workload": "1024 of 8192 llama7b-shaped blocks (128 KB per block and pool) "
                            "copied in both pools",
                "roofline": {"bound": "hbm", "achieved": round(gb_cp, 1), "peak": hbm_peak,
                             "unit": "GB/s", "frac": round(gb_cp / hbm_peak, 4),
                             "traffic": recorded_traffic(
                                 "pa_copy_blocks", "copy-blocks",
                                 source_hash("copy_blocks.cu", "pa_device.cuh"))}}
            line["secondary"] = sec

        # ---- the oracle on the host cores: all of them, then one --------
        r, calls, threads, el = oracle_decode_rate(x, args.cpu_budget)
        r1, calls1, _, el1 = oracle_decode_rate(x, max(1.0, args.cpu_budget / 3), threads=1)
        line["cpu_baseline"] = {"value": round(r, 4), "unit": "GB/s", "cores": threads,
                                "kind": "oracle", "cpu_model": cpu_model(),
                                "value_single_thread": round(r1, 4),
                                "sample": f"{calls} single-sequence write+decode oracle calls "
                                          f"({el:.1f} s) cycling the workload's 8 sequences on "
                                          f"{threads} threads; {calls1} calls ({el1:.1f} s) on "
                                          "one thread"}
        print(json.dumps(line))
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
