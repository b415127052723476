"""Benchmark of the compressed-KV decode step on GB300.

A step is one decode step of the whole stack: for every layer,
quantize-append of the new token, fused-dequant paged decode attention with
H2O score accumulation, sink/recent/top-k selection and compaction.  The
workload is the Qwen2.5-14B-shaped stack (48 layers, batch 32, 40 query / 8 KV
heads, head_dim 128, context 8192, INT4 per-token codes with bf16 sinks, H2O
budget 2457 = 4 sinks + 512 recent + 1941 heavy hitters), synthetic seeded
inputs.  Every step starts from the same pre-step state: a device snapshot of
all layers' caches is copied back before each step, outside the timed region;
that 14 GB copy also flushes the 129 MB L2, so each timed step reads its KV
from HBM.

Metric: KV bytes the decode attention must read per step (codes + fp32 scales
of every pool slot, bf16 sinks) divided by the step time, GB/s; also
sequence-steps per second.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
"""
from __future__ import annotations

import argparse
import json
import math
import os
import subprocess
import tempfile
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

WORKLOAD = "qwen14b_b32_gqa5_t8192_int4_h2o_48l"
METRIC = "decode-attention KV bytes read GB/s (% of GB300 HBM peak); seq·steps/s"


def kv_read_bytes_per_step(w, slots_per_head: int, layers: int, batch: int | None = None) -> int:
    """Algorithmic KV bytes the attention reads in one step: per (sequence, KV
    head) every pool slot's K and V codes and fp32 scales, plus the 4 bf16
    sinks' K and V."""
    per_slot = 2 * (128 * w.bits // 8) + 2 * 4
    sinks = 4 * 2 * 128 * 2
    return layers * (w.batch if batch is None else batch) * w.num_kv_heads * (slots_per_head * per_slot + sinks)


# ---------------------------------------------------------------------------
# distributed helpers (one process per GPU; independent replicas, no
# collective on the data path)
# ---------------------------------------------------------------------------

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def copy_groups(layers: int) -> tuple[list, list]:
    """The end-to-end step's copy groups, as (first, end) layer ranges: inputs
    [0, 1), [1, 3), [3, 7), ... (doubling, so each group is copied long before
    its first layer runs) and outputs ..., [L-4, L-2), [L-2, L-1), [L-1, L)
    (halving toward the end, so only the last layer's output is copied after
    the last layer)."""
    in_groups, a = [], 0
    while a < layers:
        in_groups.append((a, min(layers, 2 * a + 1)))
        a = 2 * a + 1
    out_groups, b = [], layers
    while b > 0:
        out_groups.insert(0, (max(0, layers - 2 * (layers - b) - 1), b))
        b = out_groups[0][0]
    return in_groups, out_groups


def shard_range(total: int, world: int, rank: int) -> tuple[int, int]:
    """Contiguous slice [begin, end) of `total` units for `rank`."""
    base, extra = divmod(total, world)
    begin = rank * base + min(rank, extra)
    return begin, begin + base + (1 if rank < extra else 0)


def reduce_max(value: float, world: int, device=None) -> float:
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = os.path.join(tempfile.gettempdir(), f"kvc_clocks_bench_{os.getpid()}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx = max(mx, float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        sm.sort()
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# CPU oracle leg (bounded sample of the same workload)
# ---------------------------------------------------------------------------

def oracle_sample(n_seq: int = 1, reps: int = 1, layer: int = 0, barrier=None, span=None):
    """Time the oracle's decode step on `n_seq` sequences x 8 KV heads of one
    layer at full context.  Returns (seconds, kv_bytes_read, description).
    With `barrier`, waits on it once the inputs are built, and appends the
    (start, end) of the timed loop, on the monotonic clock, to `span`."""
    import copy

    import numpy as np

    from compressed_kv_cache_kvc_gb300 import workloads as W
    from oracle import kvc_oracle as O
    w = W.WORKLOADS[WORKLOAD]
    d = W.gen_layer(w, layer, batch=n_seq)
    f = O.bf16_bits_to_f32
    base = O.OracleCache(n_seq, w.num_q_heads, w.num_kv_heads, w.bits)
    for b in range(n_seq):
        base.append(b, f(d["k"][b]), f(d["v"][b]))
    total = 0.0
    if barrier is not None:
        barrier.wait()
    t_begin = time.perf_counter()
    for _ in range(reps):
        c = copy.deepcopy(base)
        t0 = time.perf_counter()
        for b in range(n_seq):
            c.append(b, f(d["k_new"][b]), f(d["v_new"][b]))
            c.attend(b, f(d["q"][b]))
            c.evict(b, c.keep_masks(b, "h2o", budget=w.budget, recent=w.recent))
        total += time.perf_counter() - t0
    if span is not None:
        span.extend([t_begin, time.perf_counter()])
    slots = w.context + 1 - 4
    per_seq = kv_read_bytes_per_step(w, slots, 1) // w.batch
    desc = (f"oracle decode step (append, fp64 attention + H2O, select, evict) of {n_seq} sequence(s) x "
            f"{w.num_kv_heads} KV heads of one layer at context {w.context}, {reps} rep(s), 1 thread")
    return total, per_seq * n_seq * reps, desc


def run_oracle_child(n_seq: int, reps: int):
    """Run oracle_sample in a fresh single-threaded process."""
    env = dict(os.environ)
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        env[k] = "1"
    p = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-child", str(n_seq), str(reps)],
                       capture_output=True, text=True, env=env, timeout=1800)
    if p.returncode != 0:
        raise RuntimeError(p.stderr[-2000:])
    return json.loads(p.stdout.strip().splitlines()[-1])


def oracle_workload_sample(name: str, evict: str, retention: float, bf16_window: int, codes: str,
                           reps: int) -> tuple[float, int, str]:
    """The oracle's first decode step after the prompt (append, fp64
    attention with H2O scores, selection, eviction) of one sequence x every
    KV head of layer 0 of workload `name`, in the report's eviction mode,
    bf16 window and codes; timed over `reps` repetitions from the same state.
    Returns (seconds, KV bytes the attention reads, description)."""
    import copy

    from compressed_kv_cache_kvc_gb300 import workloads as W
    from oracle import kvc_oracle as O
    w = W.WORKLOADS[name]
    d = W.gen_layer(w, 0, batch=1)
    f = O.bf16_bits_to_f32
    n = int(d["lengths"][0])
    base = O.OracleCache(1, w.num_q_heads, w.num_kv_heads, w.bits, bf16_window=bf16_window, codes=codes)
    base.append(0, f(d["k"][0][:, :n]), f(d["v"][0][:, :n]))
    if evict == "block":
        kw = dict(mode="block", recent=w.recent, retention=retention)
    else:
        kw = dict(mode=w.mode, budget=w.budget, recent=w.recent, window=w.window)
    total = 0.0
    for _ in range(reps):
        c = copy.deepcopy(base)
        t0 = time.perf_counter()
        c.append(0, f(d["k_new"][0]), f(d["v_new"][0]))
        c.attend(0, f(d["q"][0]))
        c.evict(0, c.keep_masks(0, **kw))
        total += time.perf_counter() - t0
    per_slot = 2 * (128 * w.bits // 8) + 2 * 4
    ring = min(bf16_window, max(0, n + 1 - 4))
    pool = n + 1 - 4 - ring
    nbytes = (pool * per_slot + (ring + 4) * 2 * 128 * 2) * w.num_kv_heads * reps
    desc = (f"oracle decode step (append, fp64 attention + H2O, select, evict; {kw['mode']}) of 1 sequence x "
            f"{w.num_kv_heads} KV heads at context {n}, {reps} rep(s), 1 thread")
    return total, nbytes, desc


def run_oracle_workload_child(name: str, evict: str, retention: float, bf16_window: int, codes: str,
                              reps: int) -> tuple[float, int, str]:
    """oracle_workload_sample in a fresh single-threaded process."""
    env = dict(os.environ)
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        env[k] = "1"
    spec = json.dumps([name, evict, retention, bf16_window, codes, reps])
    p = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-workload-child", spec],
                       capture_output=True, text=True, env=env, timeout=1800)
    if p.returncode != 0:
        raise RuntimeError(p.stderr[-2000:])
    r = json.loads(p.stdout.strip().splitlines()[-1])
    return r["seconds"], r["bytes"], r["desc"]


def oracle_context_sample(name: str, n1: int, bf16_window: int, codes: str) -> tuple[float, float, str]:
    """The oracle's prompt over context (prefill_chunk: append the prompt,
    each prompt query attends to the held tokens in their stored form, H2O
    scores) of one sequence of workload `name` at its full context, timed
    (the context's own appends untimed).  Returns (seconds, flops, desc)."""
    import numpy as np

    from compressed_kv_cache_kvc_gb300 import workloads as W
    from oracle import kvc_oracle as O
    w = W.WORKLOADS[name]
    rng = np.random.default_rng(78)
    ctx, hq, hkv = w.context, w.num_q_heads, w.num_kv_heads
    c = O.OracleCache(1, hq, hkv, w.bits, bf16_window=bf16_window, codes=codes)
    c.append(0, rng.standard_normal((hkv, ctx, 128)).astype(np.float32),
             rng.standard_normal((hkv, ctx, 128)).astype(np.float32))
    q = rng.standard_normal((hq, n1, 128)).astype(np.float32)
    k = rng.standard_normal((hkv, n1, 128)).astype(np.float32)
    v = rng.standard_normal((hkv, n1, 128)).astype(np.float32)
    t0 = time.perf_counter()
    c.prefill_chunk(0, q, k, v)
    secs = time.perf_counter() - t0
    flops = 4.0 * 128 * sum(ctx + i + 1 for i in range(n1)) * hq
    return secs, flops, (f"oracle prefill_chunk of a {n1}-token prompt over {ctx} tokens of context, one sequence x "
                         f"{hkv} KV heads, 1 thread")


def oracle_prefill_sample(n: int) -> tuple[float, str]:
    """The oracle's prefill attention (fp64 causal attention and column sums)
    of one query head over its KV head at prompt length n, timed; seeded
    inputs of the workload's distribution."""
    import numpy as np

    from oracle import kvc_oracle as O
    rng = np.random.default_rng(77)
    q = rng.standard_normal((1, n, 128)).astype(np.float32)
    k = rng.standard_normal((1, n, 128)).astype(np.float32)
    v = rng.standard_normal((1, n, 128)).astype(np.float32)
    t0 = time.perf_counter()
    O.prefill_attention(q, k, v)
    return time.perf_counter() - t0, f"oracle prefill_attention of one query head at prompt length {n}, 1 thread"


def run_oracle_prefill_child(n: int) -> tuple[float, str]:
    """oracle_prefill_sample in a fresh single-threaded process."""
    env = dict(os.environ)
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        env[k] = "1"
    p = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-prefill-child", str(n)],
                       capture_output=True, text=True, env=env, timeout=1800)
    if p.returncode != 0:
        raise RuntimeError(p.stderr[-2000:])
    r = json.loads(p.stdout.strip().splitlines()[-1])
    return r["seconds"], r["desc"]


def _oracle_proc(n_seq: int, reps: int, layer: int, barrier, queue):
    span = []
    secs, nbytes, desc = oracle_sample(n_seq, reps, layer, barrier, span)
    queue.put({"seconds": secs, "bytes": nbytes, "desc": desc, "span": span})


def run_oracle_all_cores(n_seq: int, reps: int, n_proc: int | None = None):
    """The same sample on every host core at once: one single-threaded
    spawned process per core, each on its own layer's inputs, all starting
    their timed loops together (a barrier after the inputs are built).
    Throughput = all processes' bytes / (last end - first start)."""
    import multiprocessing as mp
    n_proc = n_proc or os.cpu_count() or 1
    ctx = mp.get_context("spawn")
    saved = {k: os.environ.get(k) for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")}
    for k in saved:
        os.environ[k] = "1"
    try:
        barrier = ctx.Barrier(n_proc)
        queue = ctx.Queue()
        procs = [ctx.Process(target=_oracle_proc, args=(n_seq, reps, i, barrier, queue)) for i in range(n_proc)]
        for p in procs:
            p.start()
        res = [queue.get(timeout=1800) for _ in procs]
        for p in procs:
            p.join()
    finally:
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    t0 = min(r["span"][0] for r in res)
    t1 = max(r["span"][1] for r in res)
    nbytes = sum(r["bytes"] for r in res)
    return {"seconds": t1 - t0, "bytes": nbytes, "cores": n_proc, "desc": res[0]["desc"]}


def reference_arm(args):
    """--impl reference: the oracle timed on the host cores, same metric."""
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    from compressed_kv_cache_kvc_gb300 import workloads as W
    w = W.WORKLOADS[WORKLOAD]
    n_seq, reps = 1, 2
    for _ in range(args.warmup):
        run_oracle_all_cores(n_seq, 1)
    secs, nbytes, cores = 0.0, 0, 1
    desc = ""
    for _ in range(args.steps):
        r = run_oracle_all_cores(n_seq, reps)
        secs += r["seconds"]
        nbytes += r["bytes"]
        cores = r["cores"]
        desc = (f"{cores} single-threaded processes at once, each: "
                + r["desc"].replace(", 1 thread", ""))
    gbs = nbytes / secs / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": secs / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": WORKLOAD, "batch": w.batch, "num_q_heads": w.num_q_heads,
                                            "num_kv_heads": w.num_kv_heads, "head_dim": 128,
                                            "context": w.context, "layers": w.layers, "bits": w.bits,
                                            "budget": w.budget, "recent": w.recent,
                                            "parallelism": "host cores", "sample": desc},
            "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": desc},
            "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

def gpu_arm(args):
    import numpy as np
    import torch

    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", torch.cuda.current_device())

    from compressed_kv_cache_kvc_gb300 import workloads as W
    from compressed_kv_cache_kvc_gb300.build import build_library
    build_library()
    from compressed_kv_cache_kvc_gb300.cache import KVCache

    w = W.WORKLOADS[WORKLOAD]
    layers = args.layers or w.layers
    Hq, Hkv, T = w.num_q_heads, w.num_kv_heads, w.context
    # replicas: every rank runs the whole workload on its own draws (weak
    # scaling); batch: the workload's sequences are divided over the ranks,
    # each rank drawing the single-GPU workload and keeping its slice
    # (strong scaling, the union of the ranks' work is the one-GPU job)
    b0, b1 = shard_range(w.batch, ws, rank) if args.split == "batch" else (0, w.batch)
    B = b1 - b0
    mbps = (T + 1 + 15) // 16 + 1
    nblocks = B * mbps
    caches, snaps, inputs = [], [], []
    for l in range(layers):
        c = KVCache(Hq, Hkv, w.bits, nblocks, B, mbps, device=dev)
        if args.split == "batch":
            q, k, v, kn, vn = (x[b0:b1].contiguous() for x in W.gen_layer_torch(w, l, dev))
        else:
            q, k, v, kn, vn = W.gen_layer_torch(w, l + 1000 * rank, dev)
        c.quantize_append(k, v)
        del k, v
        torch.cuda.synchronize()
        caches.append(c)
        snaps.append(c.state_view.clone())
        inputs.append((q, kn, vn))
    torch.cuda.synchronize()
    # the one-call step shares one workspace; the overlapped step gives each
    # layer its own (a layer's eviction still reads it while the next attends)
    ws_buf = caches[0].workspace(B)
    for c in caches:
        c._ws[ws_buf.numel()] = ws_buf
    wss = [ws_buf] + [torch.empty_like(ws_buf) for _ in range(layers - 1)]
    evict_stream = torch.cuda.Stream(device=dev)
    outs = [torch.empty(B, Hq, 128, dtype=torch.bfloat16, device=dev) for _ in range(layers)]
    slots0 = caches[0].lengths(0)[0]  # pool slots before the step's append
    kv_bytes = kv_read_bytes_per_step(w, slots0 + 1, layers, batch=B)  # this rank's

    # a read of 512 MB after each restore (untimed): the restore's copy
    # leaves L2 full of dirty lines, which would otherwise be written back
    # while the first layer runs
    flush_buf = torch.ones(128 * 1024 * 1024, dtype=torch.float32, device=dev)
    flush_out = torch.empty((), dtype=torch.float32, device=dev)

    def restore():
        for c, s in zip(caches, snaps):
            c.state_view.copy_(s, non_blocking=True)
        torch.sum(flush_buf, dim=0, out=flush_out)

    def step(stream=None, overlap=not args.serial):
        # one library call per layer.  Overlapped (the default): append,
        # split-K attention and merge on `stream`; the layer's eviction (H2O
        # scores, selection, compaction lists, row moves) on a second stream,
        # running while the next layer attends; the eviction stream joins
        # `stream` after the last layer.  Serial: kvc_decode_step, append,
        # split-K attention, then the fused merge + scores + selection +
        # compaction kernel, all on `stream`.
        n = 0
        s = stream if stream is not None else torch.cuda.current_stream()
        for l, c in enumerate(caches):
            q, kn, vn = inputs[l]
            if overlap:
                c.decode_step_overlap(q, kn, vn, evict_stream, mode="h2o", budget=w.budget, recent=w.recent,
                                      out=outs[l], workspace=wss[l], stream=s)
            else:
                c.decode_step(q, kn, vn, mode="h2o", budget=w.budget, recent=w.recent, out=outs[l],
                              workspace=ws_buf, stream=s)
            n += c.last_launch_count()
        if overlap:
            s.wait_stream(evict_stream)
        return n

    def resync():
        for c in caches:
            c.sync_host()

    # trace events around every layer's split-K attention kernel
    tr = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(layers)]
    for a, b in tr:
        a.record()
        b.record()  # creates the underlying CUDA events

    def set_tracing(on: bool):
        for c, (a, b) in zip(caches, tr):
            if on:
                c.set_trace_events(a, b)
            else:
                c.set_trace_events(None, None)

    stream = torch.cuda.Stream(device=dev)
    # eager warm-up (sets kernel attributes), then capture one step
    launches = 0
    for _ in range(max(1, args.warmup)):
        restore()
        torch.cuda.synchronize()
        resync()
        with torch.cuda.stream(stream):
            launches = step()
        torch.cuda.synchronize()
    # graphs of the step: the plain one is what the step time is taken from;
    # the traced ones have an event pair around every layer's split-K launch
    # (event nodes add gaps between the kernels, so their step times are not
    # used): with the eviction in line the split kernel has the GPU to itself
    # (the roofline), overlapped it shares the GPU with the previous layer's
    # eviction (its duration inside the step, reported beside)
    graph = traced = traced_in_step = None
    if not args.eager:
        for on, ov in ((False, not args.serial), (True, False), (True, True)):
            if on and ov and args.serial:
                continue
            set_tracing(on)
            restore()
            torch.cuda.synchronize()
            resync()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                step(overlap=ov)
            torch.cuda.synchronize()
            for _ in range(args.warmup):
                restore()
                torch.cuda.synchronize()
                g.replay()
            torch.cuda.synchronize()
            if not on:
                graph = g
            elif not ov:
                traced = g
            else:
                traced_in_step = g
        set_tracing(False)
    else:
        set_tracing(True)

    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(dev.index) if rank == 0 else None
    barrier(ws)
    torch.cuda.synchronize()
    if sampler:
        sampler.start()
    step_ms, attn_ms, attn_in_step_ms = [], [], []
    with torch.cuda.stream(stream):
        for _ in range(args.steps):
            restore()
            if graph is None:
                torch.cuda.synchronize()
                resync()
            ev0.record(stream)
            if graph is not None:
                graph.replay()
            else:
                step()
            ev1.record(stream)
            ev1.synchronize()
            step_ms.append(ev0.elapsed_time(ev1))
            if graph is None:
                attn_ms.extend(a.elapsed_time(b) for a, b in tr)
        # the split kernel's launches, timed by the event nodes of the traced
        # graph over as many steps
        for _ in range(args.steps if traced is not None else 0):
            restore()
            traced.replay()
            torch.cuda.synchronize()
            attn_ms.extend(a.elapsed_time(b) for a, b in tr)
        for _ in range(args.steps if traced_in_step is not None else 0):
            restore()
            traced_in_step.replay()
            torch.cuda.synchronize()
            attn_in_step_ms.extend(a.elapsed_time(b) for a, b in tr)
    torch.cuda.synchronize()
    # for context: the same step with the eviction in line (kvc_decode_step)
    serial_ms, launches_serial = [], 0
    if graph is not None and not args.serial:
        restore()
        torch.cuda.synchronize()
        resync()
        g_serial = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_serial, stream=stream):
            launches_serial = step(overlap=False)
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            for _ in range(args.steps):
                restore()
                ev0.record(stream)
                g_serial.replay()
                ev1.record(stream)
                ev1.synchronize()
                serial_ms.append(ev0.elapsed_time(ev1))
        del g_serial
    barrier(ws)
    clocks = sampler.stop() if sampler else None
    total_ms = sum(step_ms)
    total_ms_max = reduce_max(total_ms, ws, dev)
    ms_per_step = total_ms_max / args.steps
    # bytes and sequences of all ranks (with a batch split the ranks' slices
    # add up to the one-GPU workload)
    kv_bytes_all = kv_read_bytes_per_step(w, slots0 + 1, layers) if args.split == "batch" else kv_bytes * ws
    value = kv_bytes_all / (ms_per_step * 1e-3) / 1e9
    seq_steps = (w.batch if args.split == "batch" else B * ws) / (ms_per_step * 1e-3)
    attn_avg_ms = sum(attn_ms) / len(attn_ms)
    attn_bytes = kv_bytes // layers
    peaks = {}
    try:
        peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except (OSError, ValueError):
        pass
    peak = float(peaks.get("hbm_gbs", 6800.0))
    achieved = attn_bytes / (attn_avg_ms * 1e-3) / 1e9

    # e2e through the public API with host buffers: per step, the H2D copy of
    # every layer's query and new K/V from pinned memory, the step, the D2H
    # copy of every layer's output.  The copies run on a copy stream,
    # pipelined with the layers as a serving loop would, in groups of layers
    # that double in size: inputs [0, 1), [1, 3), [3, 7), ... (a layer waits
    # only for its group, long copied by the time the layers before it have
    # run), outputs ..., [L-4, L-2), [L-2, L-1), [L-1, L) (each group goes
    # back once the attention stream has written it, so after the last layer
    # only its own output is still to copy); the step ends when the last
    # output has landed.
    shapes = [tuple(t.shape) for t in inputs[0]]
    sizes = [math.prod(sh) for sh in shapes]
    per_layer = sum(sizes)
    h_in_all = torch.empty(layers * per_layer, dtype=torch.bfloat16).pin_memory()
    d_in_all = torch.empty(layers * per_layer, dtype=torch.bfloat16, device=dev)
    d_in = []
    for l in range(layers):
        off, views = l * per_layer, []
        for t, sh, n in zip(inputs[l], shapes, sizes):
            h_in_all[off:off + n].copy_(t.reshape(-1).cpu())
            views.append(d_in_all[off:off + n].view(sh))
            off += n
        d_in.append(tuple(views))
    d_out_all = torch.empty(layers, B, Hq, 128, dtype=torch.bfloat16, device=dev)
    h_out_all = torch.empty(layers, B, Hq, 128, dtype=torch.bfloat16).pin_memory()
    h2d = h_in_all.numel() * h_in_all.element_size()
    d2h = h_out_all.numel() * h_out_all.element_size()

    copy_stream = torch.cuda.Stream(device=dev)
    in_groups, out_groups = copy_groups(layers)
    in_first = {g[0]: (i, g) for i, g in enumerate(in_groups)}
    out_last = {g[1] - 1: g for g in out_groups}
    in_ready = [torch.cuda.Event() for _ in in_groups]
    out_ready = [torch.cuda.Event() for _ in out_groups]

    def e2e_step_calls():
        s = torch.cuda.current_stream()
        copy_stream.wait_stream(s)
        with torch.cuda.stream(copy_stream):
            for (l0, l1), ev in zip(in_groups, in_ready):
                seg = slice(l0 * per_layer, l1 * per_layer)
                d_in_all[seg].copy_(h_in_all[seg], non_blocking=True)
                ev.record(copy_stream)
        no = 0
        for l, c in enumerate(caches):
            q, kn, vn = d_in[l]
            if l in in_first:
                s.wait_event(in_ready[in_first[l][0]])
            if args.serial:
                c.decode_step(q, kn, vn, mode="h2o", budget=w.budget, recent=w.recent, out=d_out_all[l],
                              workspace=ws_buf, stream=s)
            else:
                c.decode_step_overlap(q, kn, vn, evict_stream, mode="h2o", budget=w.budget, recent=w.recent,
                                      out=d_out_all[l], workspace=wss[l], stream=s)
            if l in out_last:
                # the outputs are written on `s` (the merge, or the in-line post kernel)
                l0, l1 = out_last[l]
                out_ready[no].record(s)
                copy_stream.wait_event(out_ready[no])
                no += 1
                with torch.cuda.stream(copy_stream):
                    h_out_all[l0:l1].copy_(d_out_all[l0:l1], non_blocking=True)
        if not args.serial:
            s.wait_stream(evict_stream)
        s.wait_stream(copy_stream)

    e_steps = max(1, min(args.steps, 10))
    # (a) each call launched as the user makes it
    e2e_eager_ms = []
    with torch.cuda.stream(stream):
        for _ in range(e_steps):
            restore()
            torch.cuda.synchronize()
            resync()
            ev0.record(stream)
            e2e_step_calls()
            ev1.record(stream)
            ev1.synchronize()
            e2e_eager_ms.append(ev0.elapsed_time(ev1))
    # (b) the same calls captured once into a CUDA graph, as a serving loop
    # would: every replay copies the pinned host inputs in and the outputs out
    e2e_ms = []
    if graph is not None:
        restore()
        torch.cuda.synchronize()
        resync()
        e2e_graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(e2e_graph, stream=stream):
            e2e_step_calls()
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            for _ in range(e_steps):
                restore()
                torch.cuda.synchronize()
                ev0.record(stream)
                e2e_graph.replay()
                ev1.record(stream)
                ev1.synchronize()
                e2e_ms.append(ev0.elapsed_time(ev1))
    else:
        e2e_ms = e2e_eager_ms
    e2e_step = reduce_max(sum(e2e_ms), ws, dev) / e_steps
    e2e_value = kv_bytes_all / (e2e_step * 1e-3) / 1e9
    e2e_eager_step = reduce_max(sum(e2e_eager_ms), ws, dev) / e_steps
    for c in caches:
        st = c.read_status()
        if st:
            raise RuntimeError(f"device status {st:#x}")

    if rank != 0:
        return
    cpu = None
    if not args.no_cpu_baseline and ws == 1:
        r1 = run_oracle_child(4, 60)
        ra = run_oracle_all_cores(4, 12)
        cpu = {"value": ra["bytes"] / ra["seconds"] / 1e9, "unit": "GB/s", "cores": ra["cores"], "kind": "oracle",
               "sample": (f"{ra['cores']} single-threaded processes at once, each: "
                          + ra["desc"].replace("60 rep(s)", "12 rep(s)").replace(", 1 thread", "")),
               "seconds": ra["seconds"],
               "single_thread": {"value": r1["bytes"] / r1["seconds"] / 1e9, "unit": "GB/s", "cores": 1,
                                 "sample": r1["desc"], "seconds": r1["seconds"]}}
    traffic = None
    tpath = os.path.join(ROOT, "profiles", "attn_split_int4_traffic.json")
    if os.path.exists(tpath):
        try:
            tj = json.load(open(tpath))
            traffic = tj.get("dram_bytes_per_launch")
        except (OSError, ValueError):
            traffic = None
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "strong" if args.split == "batch" else "weak",
        "vs_baseline": None, "dtype": "int4-codes/f16-mma/f32-accum", "data": "synthetic",
        "config": {"workload": WORKLOAD, "batch": B, "num_q_heads": Hq, "num_kv_heads": Hkv, "head_dim": 128,
                   "context": T, "layers": layers, "bits": w.bits, "budget": w.budget, "recent": w.recent,
                   "parallelism": f"batch-split{ws}" if args.split == "batch" else f"replicas{ws}",
                   "l2": "state restore copy (>L2), then a 512 MB read, between timed steps",
                   "cuda_graph": graph is not None,
                   "eviction": ("in line (kvc_decode_step)" if args.serial else
                                "on a second stream (kvc_decode_step_overlap), overlapping the next layer")},
        "seq_steps_per_s": seq_steps,
        "kv_bytes_per_step": kv_bytes,
        "frac_of_hbm_peak": value / peak,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": traffic, "kernel": "attn_split_kernel<4>", "bytes_per_launch": attn_bytes,
                     "avg_launch_ms": attn_avg_ms, "peak_source": "MEASURED_PEAKS.json hbm_gbs (measured)",
                     "timed_in": ("the one-call step (eviction in line): the kernel has the GPU to itself"
                                  if traced is not None else "the timed steps"),
                     "avg_launch_ms_in_overlapped_step": (sum(attn_in_step_ms) / len(attn_in_step_ms)
                                                          if attn_in_step_ms else None)},
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_value, "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_step,
                "path": (("H2D copies of the layers' inputs from pinned host memory and D2H copies of their "
                          "outputs in groups of layers on a copy stream, pipelined with %s per layer; captured "
                          "once into a CUDA graph and replayed every step"
                          if graph is not None else
                          "H2D and D2H copies in groups of layers on a copy stream, pipelined with %s per "
                          "layer, eager")
                         % ("KVCache.decode_step" if args.serial
                            else "KVCache.decode_step_overlap (eviction on a second stream)")),
                "eager": {"value": kv_bytes * ws / (e2e_eager_step * 1e-3) / 1e9, "ms_per_step": e2e_eager_step,
                          "path": "the same calls launched one by one"}},
        "one_call_step": ({"ms_per_step": sum(serial_ms) / len(serial_ms),
                           "value": kv_bytes_all / (sum(serial_ms) / len(serial_ms) * 1e-3) / 1e9,
                           "path": "kvc_decode_step per layer (eviction in line), CUDA graph"}
                          if serial_ms else None),
        "gpu_launches": launches * args.steps + (launches_serial or launches) * len(serial_ms)
        + ((launches_serial or launches) * args.steps if traced is not None else 0)
        + (launches * args.steps if traced_in_step is not None else 0),
        "clocks": clocks,
    }
    print(json.dumps(line))


# ---------------------------------------------------------------------------
# per-workload report (not the bench line): every synthetic workload through
# the same one-call step, as absolute numbers and fractions of the HBM peak
# ---------------------------------------------------------------------------

def prefill_report(args, name: str):
    """Time one layer's prefill (kvc_prefill_attention: append, causal
    attention, H2O scores) on workload `name`'s shape, every sequence a fresh
    prompt of the workload's context length; inputs seeded, resident on the
    device.  Prints one JSON line with the attention's algorithmic TFLOP/s
    against the measured bf16 tensor peak."""
    import numpy as np
    import torch

    from compressed_kv_cache_kvc_gb300 import workloads as W
    from compressed_kv_cache_kvc_gb300.build import build_library
    build_library()
    from compressed_kv_cache_kvc_gb300.cache import KVCache

    dev = torch.device("cuda", torch.cuda.current_device())
    w = W.WORKLOADS[name]
    B, Hq, Hkv, n = w.batch, w.num_q_heads, w.num_kv_heads, w.context
    mbps = (n + 15) // 16 + 1
    c = KVCache(Hq, Hkv, w.bits, B * mbps, B, mbps, device=dev, bf16_window=args.bf16_window)
    g = torch.Generator(device=dev)
    g.manual_seed(1234)
    q = torch.randn(B, Hq, n, 128, device=dev, generator=g).to(torch.bfloat16)
    k = torch.randn(B, Hkv, n, 128, device=dev, generator=g).to(torch.bfloat16)
    v = torch.randn(B, Hkv, n, 128, device=dev, generator=g).to(torch.bfloat16)
    out = torch.empty_like(q)
    nbytes = c.lib.kvc_prefill_workspace_bytes(c.handle, B, n)
    raw = torch.empty(nbytes + 256, dtype=torch.uint8, device=dev)
    ws = raw[(-raw.data_ptr()) % 256:][:nbytes]
    stream = torch.cuda.Stream(device=dev)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    tr0, tr1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    tr0.record()
    tr1.record()  # creates the underlying CUDA events
    c.set_trace_events(tr0, tr1)  # around the attention kernel inside the call

    def run(scores):
        ms, ms_kernel = [], []
        for i in range(max(1, args.warmup) + args.steps):
            c.reset(stream=stream)
            with torch.cuda.stream(stream):
                ev0.record(stream)
                c.prefill(q, k, v, out=out, workspace=ws, accumulate_h2o=scores, stream=stream)
                ev1.record(stream)
            ev1.synchronize()
            if i >= max(1, args.warmup):
                ms.append(ev0.elapsed_time(ev1))
                ms_kernel.append(tr0.elapsed_time(tr1))
        return float(np.median(ms)), float(np.median(ms_kernel))

    ms_all, _ = run(True)
    ms_attn, ms_fwd = run(False)
    c.set_trace_events(None, None)
    # the append alone (the first part of every call above): bf16 K and V in,
    # codes, scales, positions and zeroed scores out
    ms_app = []
    for i in range(max(1, args.warmup) + args.steps):
        c.reset(stream=stream)
        with torch.cuda.stream(stream):
            ev0.record(stream)
            c.quantize_append(k, v, stream=stream)
            ev1.record(stream)
        ev1.synchronize()
        if i >= max(1, args.warmup):
            ms_app.append(ev0.elapsed_time(ev1))
    ms_app = float(np.median(ms_app))
    n_pool = max(n - args.bf16_window - 4, 0)  # quantised tokens; the rest are sinks or in the bf16 window
    app_bytes = (2 * B * Hkv * n * 256  # bf16 K and V rows in
                 + 2 * B * Hkv * n_pool * (128 * w.bits // 8 + 4) + B * Hkv * n_pool * 8  # codes, scales, pos, score
                 + 2 * B * Hkv * (n - n_pool) * 256 + B * Hkv * (n - n_pool) * 4)  # bf16 rows, score
    st = c.read_status()
    if st:
        raise RuntimeError(f"device status {st:#x}")
    pairs = n * (n + 1) / 2  # (query, key <= query) pairs per query head
    attn_flop = 4.0 * 128 * pairs * Hq * B  # QK^T and PV
    score_flop = 2.0 * 128 * pairs * Hq * B  # QK^T again, for the column sums
    peaks = {}
    try:
        peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except (OSError, ValueError):
        pass
    peak = float(peaks.get("bf16_tflops", 1900.0))
    hbm = float(peaks.get("hbm_gbs", 6800.0))
    cpu = None
    if not args.no_cpu_baseline:
        secs, desc = run_oracle_prefill_child(n)
        head_flop = 4.0 * 128 * pairs  # one query head's attention
        cpu = {"value": head_flop / secs / 1e12, "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
               "sample": desc}
    line = {"workload": name, "prefill": True, "batch": B, "n": n, "q_heads": Hq, "kv_heads": Hkv,
            "bits": w.bits, "bf16_window": args.bf16_window,
            "ms_with_scores": ms_all, "ms_without_scores": ms_attn,
            "attention_tflops": attn_flop / (ms_attn * 1e-3) / 1e12,
            "attention_frac_of_bf16_peak": attn_flop / (ms_attn * 1e-3) / 1e12 / peak,
            "forward_kernel_ms": ms_fwd, "forward_kernel_tflops": attn_flop / (ms_fwd * 1e-3) / 1e12,
            "forward_kernel_frac_of_bf16_peak": attn_flop / (ms_fwd * 1e-3) / 1e12 / peak,
            "scores_tflops": score_flop / ((ms_all - ms_attn) * 1e-3) / 1e12 if ms_all > ms_attn else None,
            "append_ms": ms_app, "append_gbs": app_bytes / (ms_app * 1e-3) / 1e9,
            "append_frac_of_hbm_peak": app_bytes / (ms_app * 1e-3) / 1e9 / hbm, "peak_hbm_gbs": hbm,
            "prompt_tokens_per_s": B * n / (ms_all * 1e-3), "peak_bf16_tflops": peak, "steps_timed": args.steps,
            "cpu_baseline": cpu,
            "note": "ms_* and attention_tflops include the append of the prompt (quantisation into the "
                    "pool); forward_kernel_* is the attention kernel alone (CUDA events around it inside the call)"}
    print(json.dumps(line), flush=True)


def prefill_context_report(args, name: str):
    """Time one layer's prompt of args.prefill_context tokens on sequences
    that hold the workload's context in the compressed cache
    (kvc_prefill_context: the append, then the multi-query attention over
    the pool (and the bf16 window with --bf16-window) in two passes, with H2O
    scores); the state is restored before every timed call; inputs seeded,
    resident on the device.  Prints one JSON line with the attention's
    algorithmic rate (4 x 128 flops per visible (query row, key) pair: QK and
    PV) and the pool bytes one pass reads per second."""
    import numpy as np
    import torch

    from compressed_kv_cache_kvc_gb300 import workloads as W
    from compressed_kv_cache_kvc_gb300.build import build_library
    build_library()
    from compressed_kv_cache_kvc_gb300.cache import KVCache

    dev = torch.device("cuda", torch.cuda.current_device())
    w = W.WORKLOADS[name]
    B, Hq, Hkv, ctx, n1 = w.batch, w.num_q_heads, w.num_kv_heads, w.context, args.prefill_context
    G = Hq // Hkv
    mbps = (ctx + n1 + 15) // 16 + 2
    c = KVCache(Hq, Hkv, w.bits, B * mbps, B, mbps, device=dev, codes=args.codes, bf16_window=args.bf16_window)
    g = torch.Generator(device=dev)
    g.manual_seed(1234)
    k0 = torch.randn(B, Hkv, ctx, 128, device=dev, generator=g).to(torch.bfloat16)
    v0 = torch.randn(B, Hkv, ctx, 128, device=dev, generator=g).to(torch.bfloat16)
    q1 = torch.randn(B, Hq, n1, 128, device=dev, generator=g).to(torch.bfloat16)
    k1 = torch.randn(B, Hkv, n1, 128, device=dev, generator=g).to(torch.bfloat16)
    v1 = torch.randn(B, Hkv, n1, 128, device=dev, generator=g).to(torch.bfloat16)
    c.quantize_append(k0, v0)
    torch.cuda.synchronize()
    snap = c.state_view.clone()
    out = torch.empty_like(q1)
    ws = c.prefill_context_workspace(B, n1)
    stream = torch.cuda.Stream(device=dev)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ms = []
    for i in range(max(1, args.warmup) + args.steps):
        c.state_view.copy_(snap)
        torch.cuda.synchronize()
        c.sync_host()
        with torch.cuda.stream(stream):
            ev0.record(stream)
            c.prefill_context(q1, k1, v1, out=out, workspace=ws, stream=stream)
            ev1.record(stream)
        ev1.synchronize()
        if i >= max(1, args.warmup):
            ms.append(ev0.elapsed_time(ev1))
    st = c.read_status()
    if st:
        raise RuntimeError(f"device status {st:#x}")
    launches = c.last_launch_count()
    t = float(np.median(ms))
    # query i (position ctx + i) sees ctx + i + 1 keys (sinks, pool, window)
    pairs = sum(ctx + i + 1 for i in range(n1)) * G * Hkv * B
    flops = 4 * 128 * pairs
    per_slot = 2 * (128 * w.bits // 8) + 2 * 4
    pool_slots = max(0, ctx + n1 - 4 - args.bf16_window)
    pool_bytes = pool_slots * per_slot * Hkv * B
    peaks = {}
    try:
        peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except (OSError, ValueError):
        pass
    line = {"workload": name, "prefill_context": n1, "batch": B, "context": ctx, "q_heads": Hq, "kv_heads": Hkv,
            "bits": w.bits, "codes": args.codes, "bf16_window": args.bf16_window, "ms_per_call": t,
            "prompt_tokens_per_s": B * n1 / (t * 1e-3),
            "attention_tflops": flops / (t * 1e-3) / 1e12,
            "attention_frac_of_bf16_peak": flops / (t * 1e-3) / 1e12 / float(peaks.get("bf16_tflops", 1900.0)),
            "pool_bytes_one_pass": pool_bytes, "pool_gbs_one_pass": pool_bytes / (t * 1e-3) / 1e9,
            "launches_per_call": launches, "steps_timed": args.steps,
            "note": "append + two passes of the multi-query attention (row statistics; outputs and column sums); "
                    "the time includes the append"}
    if not args.no_cpu_baseline:
        env = dict(os.environ)
        for k_ in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
            env[k_] = "1"
        spec = json.dumps([name, n1, args.bf16_window, args.codes])
        p = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-context-child", spec],
                           capture_output=True, text=True, env=env, timeout=1800)
        if p.returncode != 0:
            raise RuntimeError(p.stderr[-2000:])
        r = json.loads(p.stdout.strip().splitlines()[-1])
        line["cpu_baseline"] = {"value": r["flops"] / r["seconds"] / 1e12, "unit": "TFLOP/s", "cores": 1,
                                "kind": "oracle", "sample": r["desc"]}
    print(json.dumps(line), flush=True)


def workload_report(args, name: str):
    """Time the decode step of workload `name` on one GPU: all its layers,
    one `decode_step` per layer, replayed from a CUDA graph; the state is
    restored before every timed step (first step after the prefill), and for
    multi-step workloads the consecutive steps are also timed without
    restoring.  Prints one JSON line."""
    import numpy as np
    import torch

    from compressed_kv_cache_kvc_gb300 import workloads as W
    from compressed_kv_cache_kvc_gb300.build import build_library
    build_library()
    from compressed_kv_cache_kvc_gb300.cache import KVCache

    dev = torch.device("cuda", torch.cuda.current_device())
    w = W.WORKLOADS[name]
    layers = args.layers or w.layers
    B, Hq, Hkv, T = w.batch, w.num_q_heads, w.num_kv_heads, w.context
    mbps = (T + w.steps + 15) // 16 + 1
    nblocks = B * mbps
    lengths = W.context_lengths(w)
    order = W.block_order(w, nblocks) if w.shuffled_blocks else None
    per_slot = 2 * (128 * w.bits // 8) + 2 * 4
    caches, inputs = [], []
    for l in range(layers):
        c = KVCache(Hq, Hkv, w.bits, nblocks, B, mbps, block_order=order, device=dev,
                    bf16_window=args.bf16_window, codes=args.codes)
        q, k, v, kn, vn = W.gen_layer_torch(w, l, dev)
        if np.all(lengths == T):
            c.quantize_append(k, v)
        else:
            for b in range(B):
                n = int(lengths[b])
                c.quantize_append(k[b:b + 1, :, :n].contiguous(), v[b:b + 1, :, :n].contiguous(), seq_begin=b)
        del k, v
        caches.append(c)
        inputs.append((q, kn, vn))
    torch.cuda.synchronize()  # the prefill ran on the default stream; the steps run on their own
    ws_buf = caches[0].workspace(B)
    # overlapped eviction (the default): one workspace per layer
    wss = [ws_buf] + ([torch.empty_like(ws_buf) for _ in range(layers - 1)] if not args.serial else [])
    evict_stream = torch.cuda.Stream(device=dev)
    outs = [torch.empty(B, Hq, 128, dtype=torch.bfloat16, device=dev) for _ in range(layers)]
    budgets = [w.budget] * layers
    if args.schedule and w.mode == "h2o":
        from compressed_kv_cache_kvc_gb300.budgets import pyramid_budgets
        if args.schedule == "linear":
            budgets = pyramid_budgets(layers, "linear", recent=w.recent, base=w.budget)
        else:
            budgets = pyramid_budgets(layers, "quadratic", recent=w.recent, context=w.context,
                                      base_ratio=w.budget / w.context)

    def step(stream=None, overlap=not args.serial):
        # overlapped: each layer's eviction on a second stream (joined after
        # the last layer); serial: kvc_decode_step, all on `stream`
        s = stream if stream is not None else torch.cuda.current_stream()
        for l, c in enumerate(caches):
            q, kn, vn = inputs[l]
            if args.evict == "block":
                kw = dict(mode="block", recent=w.recent, retention=args.retention, out=outs[l])
            else:
                kw = dict(mode=w.mode, budget=budgets[l], recent=w.recent, window=w.window, out=outs[l])
            if overlap:
                c.decode_step_overlap(q, kn, vn, evict_stream, workspace=wss[l], stream=s, **kw)
            else:
                c.decode_step(q, kn, vn, workspace=ws_buf, stream=s, **kw)
        if overlap:
            s.wait_stream(evict_stream)

    stream = torch.cuda.Stream(device=dev)
    if w.mode == "streaming":
        # one untimed step: the timed steps see the steady window
        with torch.cuda.stream(stream):
            step()
        torch.cuda.synchronize()
    snaps = [c.state_view.clone() for c in caches]
    def step_kv_bytes(pool_only=False):
        """What the step's attention reads: the pool after the append (one
        more slot per sequence: the new token, or with a bf16 window the
        token leaving it), the bf16 sinks and the bf16 window (the split-K
        kernel reads the pool and the sinks, the window kernel the window)."""
        tot = 0
        for c in caches:
            for b in range(B):
                S, P = c.lengths(b)
                pool = S + (1 if P + 1 - args.bf16_window > 4 else 0) if args.bf16_window else S + 1
                ring = 0 if pool_only else min(args.bf16_window, max(0, P + 1 - 4))
                tot += (pool * per_slot + (ring + 4) * 2 * 128 * 2) * Hkv
        return tot

    kv_bytes = step_kv_bytes()
    split_bytes = step_kv_bytes(pool_only=True)

    flush_buf = torch.ones(128 * 1024 * 1024, dtype=torch.float32, device=dev)
    flush_out = torch.empty((), dtype=torch.float32, device=dev)

    def restore():
        for c, sn in zip(caches, snaps):
            c.state_view.copy_(sn, non_blocking=True)
        torch.sum(flush_buf, dim=0, out=flush_out)  # L2: clean lines (see gpu_arm)
        torch.cuda.synchronize()
        for c in caches:
            c.sync_host()

    tr = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(layers)]
    for a, b in tr:
        a.record()
        b.record()

    def set_tracing(on: bool):
        for c, (a, b) in zip(caches, tr):
            if on:
                c.set_trace_events(a, b)
            else:
                c.set_trace_events(None, None)

    for _ in range(max(1, args.warmup)):
        restore()
        with torch.cuda.stream(stream):
            step()
        torch.cuda.synchronize()
    # the step time from a plain graph, the split kernel's launch durations
    # from a graph of the step with the eviction in line and event nodes
    # around the split launches (which add gaps to the step)
    graphs = {}
    for on in (False, True):
        set_tracing(on)
        restore()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            step(overlap=(not args.serial) and not on)
        torch.cuda.synchronize()
        graphs[on] = g
    set_tracing(False)
    graph = graphs[False]
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    step_ms, attn_ms = [], []
    for _ in range(args.steps):
        restore()
        with torch.cuda.stream(stream):
            ev0.record(stream)
            graph.replay()
            ev1.record(stream)
        ev1.synchronize()
        step_ms.append(ev0.elapsed_time(ev1))
    for _ in range(args.steps):
        restore()
        with torch.cuda.stream(stream):
            graphs[True].replay()
        torch.cuda.synchronize()
        attn_ms.extend(a.elapsed_time(b) for a, b in tr)
    for c in caches:
        st = c.read_status()
        if st:
            raise RuntimeError(f"device status {st:#x}")
    peaks = {}
    try:
        peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except (OSError, ValueError):
        pass
    peak = float(peaks.get("hbm_gbs", 6800.0))
    ms = float(np.median(step_ms))
    attn = float(np.median(attn_ms))
    line = {"workload": name, "layers": layers, "batch": B, "bits": w.bits,
            "mode": ("block, retention %g" % args.retention) if args.evict == "block" else w.mode,
            "bf16_window": args.bf16_window, "codes": args.codes,
            "budgets": ({"schedule": args.schedule, "first": budgets[0], "middle": budgets[layers // 2],
                         "last": budgets[-1]} if args.schedule and w.mode == "h2o" else budgets[0]),
            "first_step": {"ms": ms, "kv_bytes": kv_bytes, "step_gbs": kv_bytes / (ms * 1e-3) / 1e9,
                           "step_frac_of_peak": kv_bytes / (ms * 1e-3) / 1e9 / peak,
                           "seq_steps_per_s": B / (ms * 1e-3),
                           "split_us_per_layer": attn * 1e3,
                           "split_gbs": split_bytes / layers / (attn * 1e-3) / 1e9,
                           "split_frac_of_peak": split_bytes / layers / (attn * 1e-3) / 1e9 / peak},
            "peak_gbs": peak, "steps_timed": args.steps,
            "eviction": "in line" if args.serial else "on a second stream, overlapping the next layer"}
    if w.steps > 1:
        # the workload's consecutive steps from the prefill, without restoring
        restore()
        per_step = []
        total_bytes = 0
        for _ in range(w.steps):
            total_bytes += step_kv_bytes()
            with torch.cuda.stream(stream):
                ev0.record(stream)
                step()
                ev1.record(stream)
            ev1.synchronize()
            per_step.append(ev0.elapsed_time(ev1))
        tot = sum(per_step)
        line["consecutive_steps_eager"] = {"steps": w.steps, "launch": "eager", "ms_total": tot,
                                           "kv_bytes": total_bytes, "gbs": total_bytes / (tot * 1e-3) / 1e9,
                                           "ms_first": per_step[0],
                                           "ms_median_later": float(np.median(per_step[1:])),
                                           "seq_steps_per_s": B * w.steps / (tot * 1e-3)}
        # the same steps from CUDA graphs: the first step (hundreds of rows
        # move per pair) replays the first-step graph, then one graph captured
        # at the steady state (one token evicted and at most one row moved per
        # pair: no move kernel) is replayed for the remaining steps, all
        # back to back between two events
        restore()
        with torch.cuda.stream(stream):
            step()  # step 1 eagerly, so the steady graph is captured at step-2 lengths
        torch.cuda.synchronize()
        steady = torch.cuda.CUDAGraph()
        with torch.cuda.graph(steady, stream=stream):
            step()
        torch.cuda.synchronize()
        launches_steady = sum(c.last_launch_count() for c in caches)
        reps = []
        for _ in range(max(1, min(args.steps, 5))):
            restore()
            with torch.cuda.stream(stream):
                ev0.record(stream)
                graph.replay()
                ev_mid = torch.cuda.Event(enable_timing=True)
                ev_mid.record(stream)
                for _ in range(w.steps - 1):
                    steady.replay()
                ev1.record(stream)
            ev1.synchronize()
            reps.append((ev0.elapsed_time(ev1), ev_mid.elapsed_time(ev1)))
        for c in caches:
            c.sync_host()
        tot_g = float(np.median([r[0] for r in reps]))
        later = float(np.median([r[1] for r in reps]))
        line["consecutive_steps"] = {"steps": w.steps, "launch": "cuda graphs", "ms_total": tot_g,
                                     "kv_bytes": total_bytes, "gbs": total_bytes / (tot_g * 1e-3) / 1e9,
                                     "frac_of_peak": total_bytes / (tot_g * 1e-3) / 1e9 / peak,
                                     "ms_later_steps": later,
                                     "us_per_layer_steady": later * 1e3 / ((w.steps - 1) * layers),
                                     "launches_per_layer_steady": launches_steady / layers,
                                     "seq_steps_per_s": B * w.steps / (tot_g * 1e-3), "repetitions": len(reps)}
        for c in caches:
            st = c.read_status()
            if st:
                raise RuntimeError(f"device status {st:#x}")
    if not args.no_cpu_baseline:
        # the oracle beside it: the same first step on one sequence of layer 0
        secs, nbytes, desc = run_oracle_workload_child(name, args.evict, args.retention, args.bf16_window,
                                                       args.codes, 3)
        line["cpu_baseline"] = {"value": nbytes / secs / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
                                "sample": desc}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--layers", type=int, default=0, help="override the layer count (profiling only)")
    ap.add_argument("--eager", action="store_true", help="launch each call instead of replaying a CUDA graph")
    ap.add_argument("--serial", action="store_true",
                    help="the one-call step with the eviction in line (default: the eviction on a second stream)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload", default=None,
                    help="report mode: time this workload (or 'all') instead of printing the bench line")
    ap.add_argument("--schedule", default=None, choices=["linear", "quadratic"],
                    help="report mode: per-layer H2O budgets (PyramidKV-style schedule)")
    ap.add_argument("--evict", default=None, choices=["block"],
                    help="report mode: block-granular eviction instead of the workload's mode")
    ap.add_argument("--retention", type=float, default=0.25, help="report mode, --evict block: pages kept")
    ap.add_argument("--codes", default="int", choices=["int", "e4m3"],
                    help="report mode: code format (e4m3: FP8 codes, 8-bit workloads)")
    ap.add_argument("--prefill", action="store_true",
                    help="report mode: time one layer's prefill (fresh prompts of the workload's context)")
    ap.add_argument("--prefill-context", type=int, default=0,
                    help="report mode: time a prompt of this many tokens over the workload's context")
    ap.add_argument("--bf16-window", type=int, default=0,
                    help="report mode: hybrid precision, the last W positions kept in bf16 (W <= recent)")
    ap.add_argument("--split", default="replicas", choices=["replicas", "batch"],
                    help="N > 1: independent replicas (weak scaling) or the batch divided over the GPUs (strong)")
    ap.add_argument("--oracle-child", nargs=2, type=int, default=None, help=argparse.SUPPRESS)
    ap.add_argument("--oracle-prefill-child", type=int, default=None, help=argparse.SUPPRESS)
    ap.add_argument("--oracle-workload-child", default=None, help=argparse.SUPPRESS)
    ap.add_argument("--oracle-context-child", default=None, help=argparse.SUPPRESS)
    args = ap.parse_args()
    if args.oracle_context_child is not None:
        secs, flops, desc = oracle_context_sample(*json.loads(args.oracle_context_child))
        print(json.dumps({"seconds": secs, "flops": flops, "desc": desc}))
        return
    if args.oracle_workload_child is not None:
        secs, nbytes, desc = oracle_workload_sample(*json.loads(args.oracle_workload_child))
        print(json.dumps({"seconds": secs, "bytes": nbytes, "desc": desc}))
        return
    if args.oracle_prefill_child is not None:
        secs, desc = oracle_prefill_sample(args.oracle_prefill_child)
        print(json.dumps({"seconds": secs, "desc": desc}))
        return
    if args.oracle_child is not None:
        secs, nbytes, desc = oracle_sample(args.oracle_child[0], args.oracle_child[1])
        print(json.dumps({"seconds": secs, "bytes": nbytes, "desc": desc}))
        return
    if args.impl == "reference":
        reference_arm(args)
        return
    if args.workload:
        from compressed_kv_cache_kvc_gb300 import workloads as W
        for name in (list(W.WORKLOADS) if args.workload == "all" else [args.workload]):
            if args.prefill_context:
                prefill_context_report(args, name)
            else:
                (prefill_report if args.prefill else workload_report)(args, name)
        return
    gpu_arm(args)


if __name__ == "__main__":
    main()
