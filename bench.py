#!/usr/bin/env python3
"""Benchmark of the compressed-sparse-attention decode path on GB300.

One step = one pass of the whole hot path over the 64K-context decode batch
(B = 32 sequences of 65536 tokens, C4 N = 16384 compressed entries, H = 64,
Hi = 64, top-512 + a 128-token window): window indices -> indexer logits ->
top-k -> sparse attention (+ split merge), every step in libdsv4sa kernels,
called through the C ABI.

Timing: CUDA events on the launching stream around each step; before every
step (outside the events) a 512 MB buffer is written and a second 512 MB
buffer is read, so L2 holds none of the step's data and no dirty lines whose
write-back would compete with the step; then a GPU sleep lets the host
enqueue the whole step, so the events see device time.
The timed region is bracketed by a barrier and a synchronize on both sides;
the slowest rank sets the time.  Under torchrun each rank runs its own batch
of 32 sequences (weak scaling; no collective on the data path).

``--impl reference`` times the fp64 CPU oracle on the host cores instead (the
reference arm of this benchmark): each step is one query row of the same
workload.
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

METRIC = "sparse-attn decode query-tokens/s (H=64, top-512, 64K ctx); % of roofline"
UNIT = "query-tokens/s"
WORKLOAD = ("decode64k: B=32 sequences x 65536 tokens (C4 N=16384 entries), H=64 query heads, "
            "Hi=64 indexer heads, top-512 + 128-token window, FP8/BF16 paged cache (64-slot pages, shuffled)")
L2_FLUSH_BYTES = 512 << 20   # written, then a second buffer is read: L2 ends cold and clean
SLEEP_CYCLES = 2_000_000
KV_ROW_BYTES = 604        # 448 e4m3 + 64 bf16 + 7 fp32 scales
KEY_ROW_BYTES = 136       # 128 e4m3 + 2 fp32 scales


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--batch", type=int, default=32, help="sequences per GPU (profiling only)")
    ap.add_argument("--profile", action="store_true",
                    help="profiling driver for ncu: the path only, no L2 flush buffer, no e2e / CPU legs")
    ap.add_argument("--profile-feeders", action="store_true",
                    help="profiling driver for ncu: the KV-cache writer and compressor cases once each, no step")
    ap.add_argument("--cpu-child", type=int, default=0, help=argparse.SUPPRESS)
    return ap.parse_args()


# ---------------------------------------------------------------- multi-rank host logic

def rank_env():
    """(rank, world, local_rank) from the torchrun environment (1 process = 1 GPU)."""
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def shard_seed(rank: int) -> int:
    """Each rank decodes its own batch of independent sequences (weak scaling)."""
    from compressed_sparse_attention_c4_gb300 import workloads as W
    return W.SEEDS["decode"] + 1000 * rank


def reduce_max(x: float, dist, device) -> float:
    """The slowest rank sets the job time."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world: int, queries_per_rank: int, ms_per_step: float) -> float:
    """Whole-job query-tokens/s: every rank's queries over the slowest rank's step time."""
    return world * queries_per_rank / (ms_per_step / 1e3)


# ---------------------------------------------------------------- peaks, clocks, profiles

def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


def profiled_traffic(kernel_src: str, profile_md: str):
    """DRAM bytes per launch recorded by an ncu capture, if the kernel source is
    unchanged since (the summary stores the source's sha256)."""
    try:
        src = open(os.path.join(ROOT, kernel_src), "rb").read()
        text = open(os.path.join(ROOT, profile_md)).read()
    except OSError:
        return None
    sha = hashlib.sha256(src).hexdigest()
    m_sha = re.search(r"source_sha256:\s*([0-9a-f]{64})", text)
    m_b = re.search(r"dram_bytes_per_full_launch:\s*([0-9.eE+]+)", text)
    if not m_sha or not m_b or m_sha.group(1) != sha:
        return None
    return float(m_b.group(1))


class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.skip = 0

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None
            return self
        t0 = time.time()     # the timed region starts once the sampler reports
        while not self.lines and time.time() - t0 < 3.0 and self.proc.poll() is None:
            time.sleep(0.01)
        self.skip = len(self.lines)
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

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines[self.skip:]:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------- algorithmic work

def algorithmic_work(w, idx_c, idx_w):
    """Bytes the method must move and FLOPs it must do for one step (logits excluded)."""
    import numpy as np
    nvis = np.where(w.c128, 0, w.n_vis).astype(np.int64)
    valid = (idx_c >= 0).sum(axis=1) + (idx_w >= 0).sum(axis=1)
    idx_bytes = int(nvis.sum()) * KEY_ROW_BYTES + w.T * w.Hi * (128 + 8 + 4)
    attn_bytes = int(valid.sum()) * KV_ROW_BYTES + 2 * w.T * w.H * 512 * 2 + w.T * (w.kc + w.kw) * 4
    misc = w.T * w.k * 4 + w.T * w.kw * 4
    fp8_flops = 2 * w.Hi * 128 * int(nvis.sum())
    bf16_flops = 4 * w.H * 512 * int(valid.sum())
    return idx_bytes, attn_bytes + misc + idx_bytes, fp8_flops, bf16_flops


def measure_inverse_rope(L, torch, d, w, stream, kernels, flush_l2, reps=50):
    """The step with the inverse rotary embedding of the output fused into the
    attention (a (cos, sin) table of random angles, one row per position) against
    the same step without it: both as CUDA graphs, replayed alternately after an
    L2 flush and a GPU sleep, event-timed on the launching stream."""
    rows = int(d.pos.max().item()) + 1
    g = torch.Generator(device=d.pos.device).manual_seed(11)
    ang = torch.rand((rows, 32), generator=g, device=d.pos.device, dtype=torch.float64) * (2 * math.pi)
    cs = torch.stack([torch.cos(ang), torch.sin(ang)], dim=-1).to(torch.float32).contiguous()
    n_max = max(1, int(w.n_max))

    def rope_step():
        for name, fn in kernels[:-1]:
            fn()
        kernels[-1][1](rope_cs=cs, rope_pos=d.pos)

    def plain_step():
        for name, fn in kernels:
            fn()

    graphs = []
    for fn in (plain_step, rope_step):
        fn()
        stream.synchronize()
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=stream):
            fn()
        stream.synchronize()
        graphs.append(gr)
    ms = [[], []]
    for k in range(2 * (reps + 3)):
        flush_l2()
        torch.cuda._sleep(SLEEP_CYCLES)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        graphs[k % 2].replay()
        e1.record(stream)
        if k >= 6:
            ms[k % 2].append((e0, e1))
    torch.cuda.synchronize()
    st, bits = L.dsv4sa_check_errors()
    if st != 0:
        raise RuntimeError(f"device error word after the inverse-rope steps: {st} ({bits})")
    t = [statistics.mean(a.elapsed_time(b) for a, b in m) * 1e3 for m in ms]
    return {"step_us_with": t[1], "step_us_without": t[0], "extra_us": t[1] - t[0],
            "note": "dsv4sa_attn_args.rope_cs / rope_pos: the last 64 dims of every output rotated back by the "
                    "query's table row inside the attention's output write; same graph-timed step otherwise"}


def measure_compressor(L, torch, dev, stream, flush_l2, hbm_gbs, reps=20):
    """The KV compressor on a prefill chunk (4096 tokens -> 1024 C4 entries with
    the overlap transform), a decode step (32 sequences completing a C4 window)
    and an online C128 decode step (32 tokens folded into 32 states): each call
    a one-launch CUDA graph, replayed after an L2 flush and a GPU sleep,
    event-timed.  Bytes: BF16 kv and score rows read, BF16 entries written."""
    g = torch.Generator(device=dev).manual_seed(13)
    rows = 1 << 16
    ang = torch.rand((rows, 32), generator=g, device=dev, dtype=torch.float64) * (2 * math.pi)
    cs = torch.stack([torch.cos(ang), torch.sin(ang)], dim=-1).to(torch.float32).contiguous()
    w = (torch.rand(512, generator=g, device=dev) + 0.5).contiguous()

    def timed(fn):
        fn()
        stream.synchronize()
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=stream):
            fn()
        stream.synchronize()
        ms = []
        for k in range(reps + 3):
            flush_l2()
            torch.cuda._sleep(SLEEP_CYCLES)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            gr.replay()
            e1.record(stream)
            if k >= 3:
                ms.append((e0, e1))
        torch.cuda.synchronize()
        return statistics.mean(a.elapsed_time(b) for a, b in ms) * 1e3

    out = {}
    for name, n_tok, n, first_fn in (("c4_prefill_4096", 4096, 1024, lambda n: torch.arange(n) * 4),
                                     ("c4_decode_32", 32 * 8, 32, lambda n: torch.arange(n) * 8 + 4)):
        kv = torch.randn((n_tok, 1024), generator=g, device=dev).to(torch.bfloat16)
        sc = torch.randn((n_tok, 1024), generator=g, device=dev).to(torch.bfloat16)
        ape = (torch.randn((4, 1024), generator=g, device=dev) * 0.3).contiguous()
        first = first_fn(n).to(torch.int32).to(dev)
        prev = torch.where(first >= 4, first - 4, torch.full_like(first, -1))
        pos = (torch.arange(n, device=dev, dtype=torch.int32) * 4 + 4) % rows
        o = torch.empty((n, 512), dtype=torch.bfloat16, device=dev)
        us = timed(lambda: L.dsv4sa_compress_windows(kv, sc, first, prev, pos, 4, True, ape, w, cs, o, stream=stream))
        nbytes = (n_tok if name.startswith("c4_prefill") else 8 * n) * 1024 * 2 * 2 + n * 1024
        out[name] = {"entries": n, "us": us, "bytes": nbytes, "achieved_gbs": nbytes / us / 1e3,
                     "frac_of_hbm": nbytes / us / 1e3 / hbm_gbs}
    B = 32
    kv = torch.randn((B, 512), generator=g, device=dev).to(torch.bfloat16)
    sc = torch.randn((B, 512), generator=g, device=dev).to(torch.bfloat16)
    ape = (torch.randn((128, 512), generator=g, device=dev) * 0.3).contiguous()
    state, count = L.online_c128_state(B, dev)
    idx = torch.arange(B, dtype=torch.int32, device=dev)
    o = torch.empty((B, 512), dtype=torch.bfloat16, device=dev)
    done = torch.empty(B, dtype=torch.int32, device=dev)
    us = timed(lambda: L.dsv4sa_compress_online_c128(kv, sc, idx, state, count, idx * 0, ape, w, cs, o, done,
                                                     stream=stream))
    out["c128_online_decode_32"] = {"tokens": B, "us": us}
    st, bits = L.dsv4sa_check_errors()
    if st != 0:
        raise RuntimeError(f"device error word after the compressor: {st} ({bits})")
    out["note"] = ("dsv4sa_compress_windows / dsv4sa_compress_online_c128, one-launch CUDA graphs after an L2 flush; "
                   "bytes = BF16 kv and score rows read + BF16 entries written")
    return out


def measure_cache_writer(L, torch, dev, stream, flush_l2, hbm_gbs, reps=20):
    """The KV-cache writer on a decode step (32 new KV rows + 32 indexer keys),
    a prefill chunk (4096 + 4096) and a bulk write (65536 + 65536): the two
    launches captured as one CUDA graph, replayed after an L2 flush and a GPU
    sleep that covers the host's enqueue, event-timed on the launching stream.
    A graph of one empty kernel, timed the same way, gives the fixed part."""

    def timed(graph):
        ms = []
        for k in range(reps + 3):
            flush_l2()
            torch.cuda._sleep(SLEEP_CYCLES)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            graph.replay()
            e1.record(stream)
            if k >= 3:
                ms.append((e0, e1))
        torch.cuda.synchronize()
        return statistics.mean(a.elapsed_time(b) for a, b in ms)

    empty = torch.cuda.CUDAGraph()
    with torch.cuda.graph(empty, stream=stream):
        torch.cuda._sleep(0)
    out = {"empty_graph_us": timed(empty) * 1e3}
    for name, n in (("decode_32", 32), ("prefill_4096", 4096), ("bulk_65536", 65536)):
        pages = (n + 63) // 64
        kv_buf = L._alloc_pool(L.POOL_KV, pages, dev)           # 1024-byte aligned pool
        kv = L.dsv4sa_pool_desc_init(L.POOL_KV, kv_buf, pages)
        key_buf = L._alloc_pool(L.POOL_IDXK, pages, dev)
        keys = L.dsv4sa_pool_desc_init(L.POOL_IDXK, key_buf, pages)
        pt = torch.randperm(pages, dtype=torch.int32, device=dev).view(1, pages)
        seq = torch.zeros(n, dtype=torch.int32, device=dev)
        ent = torch.arange(n, dtype=torch.int32, device=dev)
        g = torch.Generator(device=dev).manual_seed(7)
        rows = torch.randn((n, 512), generator=g, device=dev).to(torch.bfloat16)
        krows = torch.randn((n, 128), generator=g, device=dev).to(torch.bfloat16)

        def write():
            L.dsv4sa_cache_write(kv, pt, seq, ent, rows, stream)
            L.dsv4sa_cache_write(keys, pt, seq, ent, krows, stream)

        torch.cuda.synchronize()
        write()
        stream.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            write()
        stream.synchronize()
        t = timed(graph)
        nbytes = n * (1024 + KV_ROW_BYTES) + n * (256 + KEY_ROW_BYTES)
        out[name] = {"rows": n, "us": t * 1e3, "bytes": nbytes, "achieved_gbs": nbytes / (t / 1e3) / 1e9,
                     "frac_of_hbm": nbytes / (t / 1e3) / 1e9 / hbm_gbs}
        if name == "bulk_65536":
            # the same keys into an FP4 indexer-key pool (E2M1 two per byte + E8M0 per 32), alone
            f_buf = L._alloc_pool(L.POOL_IDXK_FP4, pages, dev)
            fkeys = L.dsv4sa_pool_desc_init(L.POOL_IDXK_FP4, f_buf, pages)
            L.dsv4sa_cache_write(fkeys, pt, seq, ent, krows, stream)
            stream.synchronize()
            fgraph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(fgraph, stream=stream):
                L.dsv4sa_cache_write(fkeys, pt, seq, ent, krows, stream)
            stream.synchronize()
            tf = timed(fgraph)
            fbytes = n * (256 + 68)
            out["fp4_keys_65536"] = {"rows": n, "us": tf * 1e3, "bytes": fbytes,
                                     "achieved_gbs": fbytes / (tf / 1e3) / 1e9,
                                     "frac_of_hbm": fbytes / (tf / 1e3) / 1e9 / hbm_gbs}
    st, bits = L.dsv4sa_check_errors()
    if st != 0:
        raise RuntimeError(f"device error word after the writer: {st} ({bits})")
    return out


# ---------------------------------------------------------------- CPU oracle (baseline / reference arm)

def cpu_child(rows: int):
    """Runs in a single-threaded subprocess: the oracle over `rows` query rows of
    the decode workload (same per-sequence shapes, fewer sequences)."""
    import numpy as np
    import oracle
    from compressed_sparse_attention_c4_gb300 import workloads as W
    w = W.make("decode", B=rows)
    work = w.as_dict()
    t0 = time.perf_counter()
    done = 0
    while True:
        for t in range(rows):
            oracle.decode_step(work, rows=[t], k=w.k)
            done += 1
        if time.perf_counter() - t0 >= 10.0:
            break
    dt = time.perf_counter() - t0
    print(json.dumps({"rows": done, "seconds": dt, "value": done / dt}))


def run_cpu_baseline(rows=4):
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-child", str(rows)], env=env,
                       capture_output=True, text=True, timeout=900)
    line = [x for x in r.stdout.splitlines() if x.startswith("{")]
    if r.returncode != 0 or not line:
        return {"value": None, "unit": UNIT, "cores": 1, "kind": "oracle", "error": r.stderr[-300:]}
    d = json.loads(line[-1])
    return {"value": d["value"], "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"{d['rows']} decode query rows (the oracle's indexer, top-k and attention per row; "
                      f"sequences of 65536 tokens, H=64, Hi=64), {d['seconds']:.1f} s single-threaded numpy fp64"}


def reference_arm(args):
    rank, _, _ = rank_env()
    if rank != 0:
        return
    import oracle
    from compressed_sparse_attention_c4_gb300 import workloads as W
    w = W.make("decode", B=4)
    work = w.as_dict()
    for i in range(args.warmup):
        oracle.decode_step(work, rows=[i % w.T], k=w.k)
    t0 = time.perf_counter()
    for i in range(args.steps):
        oracle.decode_step(work, rows=[i % w.T], k=w.k)
    dt = time.perf_counter() - t0
    value = args.steps / dt
    threads = os.cpu_count()
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * dt / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "step": "one query row of the decode batch through the fp64 oracle"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": f"{args.steps} query rows, one per step, numpy fp64 with default BLAS threads"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}))


# ---------------------------------------------------------------- GPU arm

def gpu_arm(args):
    import numpy as np
    import torch
    from compressed_sparse_attention_c4_gb300 import dsv4sa as L
    from compressed_sparse_attention_c4_gb300 import workloads as W

    rank, world, local = rank_env()
    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())
    if not os.path.exists(L.LIB_PATH):
        raise RuntimeError("libdsv4sa.so missing: run __graft_entry__.build() first")

    if args.profile_feeders:
        # the writer's and the compressor's bench cases, each graph replayed 4 times
        stream = torch.cuda.Stream(device=dev)
        torch.cuda.set_stream(stream)
        flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

        def flush_l2():
            flush.zero_()
        hbm, _, _ = measured_peaks()
        writer = measure_cache_writer(L, torch, dev, stream, flush_l2, hbm, reps=1)
        compressor = measure_compressor(L, torch, dev, stream, flush_l2, hbm, reps=1)
        st, bits = L.dsv4sa_check_errors()
        print(json.dumps({"profile_feeders": True, "status": st, "bits": bits, "writer": writer,
                          "compressor": compressor}))
        if st != 0:
            raise SystemExit(1)
        return
    if args.profile:
        w = W.make("decode", B=args.batch)
        d = L.upload(w, dev)
    else:
        w = W.make("decode", seed=shard_seed(rank))
        d = L.upload(w, dev)
        flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
        clean = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

        def flush_l2():
            flush.zero_()
            clean.sum()
    n_max = max(1, int(w.n_max))
    # a dedicated stream (graph capture needs one other than the legacy default)
    stream = torch.cuda.Stream(device=dev)
    torch.cuda.set_stream(stream)

    # The serving form of the path: the attention kernel derives the window
    # indices from the positions (the same values dsv4sa_window_indices writes).
    def topk_attn(rope_cs=None, rope_pos=None):
        L.dsv4sa_topk_sparse_attn_decode(
            d.logits, d.n_vis_idx, n_max, w.k, d.q, d.sink, d.q_seq, d.comp, d.comp_pt, d.idx_c, d.win, d.win_pt,
            None, d.out, w.softmax_scale, lse=d.lse, ws=d.attn_ws, topk_ws=d.topk_ws, stream=stream, win_pos=d.pos,
            kw=w.kw, win_ring=w.win_ring, flags=L.ATTN_EARLY_WINDOW, rope_cs=rope_cs, rope_pos=rope_pos)

    def attn(rope_cs=None, rope_pos=None):
        L.dsv4sa_sparse_attn_decode(
            d.q, d.sink, d.q_seq, d.comp, d.comp_pt, d.idx_c, d.win, d.win_pt, None, d.out, w.softmax_scale,
            lse=d.lse, ws=d.attn_ws, stream=stream, win_pos=d.pos, kw=w.kw, win_ring=w.win_ring,
            flags=L.ATTN_EARLY_WINDOW, rope_cs=rope_cs, rope_pos=rope_pos)

    # The serving form of the path: indexer, top-k (which also prefetches the
    # selected rows into L2), attention with the window indices derived from
    # the positions.  (The one-call form, dsv4sa_topk_sparse_attn_decode, is
    # timed separately as `one_call_step_us`.)
    kernels = [
        ("indexer_logits", lambda: L.dsv4sa_indexer_logits(d.keys, d.comp_pt, d.q_seq, d.n_vis_idx, d.q_idx,
                                                           d.q_idx_scale, d.wts, n_max, d.logits, stream)),
        ("topk", lambda: L.dsv4sa_topk_prefetch(d.logits, d.n_vis_idx, n_max, w.k, d.idx_c, d.comp, d.comp_pt,
                                                d.q_seq, d.topk_ws, stream)),
        ("sparse_attn_decode", attn),
    ]

    def step(ev=None, marks=(0, 1, 2)):
        """One pass of the path; ev[j] is recorded before the j-th marked kernel and
        ev[-1] after the last one."""
        j = 0
        for i, (_, fn) in enumerate(kernels):
            if ev is not None and i in marks:
                ev[j].record(stream)
                j += 1
            fn()
        if ev is not None:
            ev[j].record(stream)

    attn_plan = L.dsv4sa_attn_plan(L.ATTN_DECODE, w.T, w.H, w.kc, w.kw)
    launches_per_step = 1 + (2 if d.topk_ws is not None else 1) + attn_plan["launches"]
    if args.profile:
        for _ in range(args.warmup + args.steps):
            step()
        torch.cuda.synchronize()
        st, bits = L.dsv4sa_check_errors()
        print(json.dumps({"profile_driver": True, "batch": w.T, "launches": launches_per_step * (args.warmup + args.steps),
                          "status": st, "bits": bits}))
        if st != 0:
            raise SystemExit(1)
        return

    for _ in range(args.warmup):
        flush_l2()
        step()
    torch.cuda.synchronize()
    st, bits = L.dsv4sa_check_errors()
    if st != 0:
        raise RuntimeError(f"device error word after warm-up: {st} ({bits})")

    # The step as one CUDA graph of the three calls (programmatic-dependent
    # launches become graph edges).
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step()
    stream.synchronize()

    # Timed region: 2 K steps.  Even steps are graph replays between one event
    # before and one after (the step time); odd steps launch the three calls
    # directly with events around the indexer (the roofline kernel's launch
    # time).  An event between two kernels ends their programmatic overlap, so
    # the step time is taken on the steps without inner events.
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(2 * args.steps)]
    with ClockSampler(dev.index) as clocks:
        if dist:
            dist.barrier()
        torch.cuda.synchronize()
        for k in range(2 * args.steps):
            flush_l2()
            torch.cuda._sleep(SLEEP_CYCLES)
            if k % 2 == 0:
                evs[k][0].record(stream)
                graph.replay()
                evs[k][1].record(stream)
            else:
                step(evs[k], (0, 1))
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
    st, bits = L.dsv4sa_check_errors()
    if st != 0:
        raise RuntimeError(f"device error word after the timed region: {st} ({bits})")
    step_ms = [evs[k][0].elapsed_time(evs[k][1]) for k in range(0, 2 * args.steps, 2)]
    idx_ms = statistics.mean(evs[k][0].elapsed_time(evs[k][1]) for k in range(1, 2 * args.steps, 2))
    ms = reduce_max(statistics.mean(step_ms), dist, dev)
    value = job_throughput(world, w.T, ms)

    # Per-kernel breakdown, after the timed region: an event around every kernel.
    bevs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(kernels) + 1)] for _ in range(args.steps)]
    for k in range(args.steps):
        flush_l2()
        torch.cuda._sleep(SLEEP_CYCLES)
        step(bevs[k])
    torch.cuda.synchronize()
    part_ms = {name: statistics.mean(e[i].elapsed_time(e[i + 1]) for e in bevs)
               for i, (name, _) in enumerate(kernels)}

    # Warm reference (not the reported value): the same graph replayed with no
    # L2 flush in between, so the step's 88 MB are largely L2-resident.
    wevs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    for k in range(args.steps):
        torch.cuda._sleep(SLEEP_CYCLES)
        wevs[k][0].record(stream)
        graph.replay()
        wevs[k][1].record(stream)
    torch.cuda.synchronize()
    warm_ms = [a.elapsed_time(b) for a, b in wevs]

    # The one-call form of the top-k and the attention (dsv4sa_topk_sparse_attn_decode:
    # the attention's clusters select their own rows), as a graph of two calls.
    one_call_ms = None
    if attn_plan["nsplit"] >= 2 and attn_plan["launches"] == 1 and n_max <= 16384 and w.kc == w.k:
        graph1 = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph1, stream=stream):
            kernels[0][1]()
            topk_attn()
        stream.synchronize()
        oevs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
        for k in range(args.steps):
            flush_l2()
            torch.cuda._sleep(SLEEP_CYCLES)
            oevs[k][0].record(stream)
            graph1.replay()
            oevs[k][1].record(stream)
        torch.cuda.synchronize()
        one_call_ms = statistics.mean(a.elapsed_time(b) for a, b in oevs)

    # ---- end to end through the C ABI with host buffers (pinned), copies inside the timed region:
    # the serving-loop form, one CUDA graph per step (H2D of the step's inputs, the path, D2H
    # of out and lse), replayed and synchronised every step
    sg = L.StepGraph(d)
    h2d, d2h = sg.h2d_bytes, sg.d2h_bytes
    e2e_s = []
    for k in range(args.warmup + args.steps):
        flush_l2()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        sg.replay()
        sg.stream.synchronize()
        if k >= args.warmup:
            e2e_s.append(time.perf_counter() - t0)
    e2e_torch = reduce_max(statistics.mean(e2e_s), dist, dev)
    # the same step built and launched by the library itself (dsv4sa_step_create /
    # dsv4sa_step_launch: one C-ABI call per step, no torch graph in between)
    ns = L.NativeStep(d)
    e2e_n = []
    for k in range(args.warmup + args.steps):
        flush_l2()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        ns.launch()
        ns.stream.synchronize()
        if k >= args.warmup:
            e2e_n.append(time.perf_counter() - t0)
    ns.close()
    e2e_mean = reduce_max(statistics.mean(e2e_n), dist, dev)
    st, bits = L.dsv4sa_check_errors()
    if st != 0:
        raise RuntimeError(f"device error word after the timed region: {st} ({bits})")

    if rank != 0:
        dist.destroy_process_group()
        return
    hbm, bf16_tf, peak_kind = measured_peaks()
    writer = measure_cache_writer(L, torch, dev, stream, flush_l2, hbm)
    inv_rope = measure_inverse_rope(L, torch, d, w, stream, kernels, flush_l2)
    compressor = measure_compressor(L, torch, dev, stream, flush_l2, hbm)
    idx_c = d.idx_c.cpu().numpy()
    idx_w = d.idx_w.cpu().numpy()
    idx_bytes, step_bytes, fp8_flops, bf16_flops = algorithmic_work(w, idx_c, idx_w)
    achieved = idx_bytes / (idx_ms / 1e3) / 1e9
    traffic = profiled_traffic("compressed_sparse_attention_c4_gb300/csrc/indexer.cu",
                               "profiles/indexer_logits_decode64k.md")
    fp8_tf = 2 * bf16_tf     # FP8 dense peak not measured: nominal 2x the measured BF16 figure
    roof_us = max(step_bytes / (hbm * 1e9), fp8_flops / (fp8_tf * 1e12) + bf16_flops / (bf16_tf * 1e12)) * 1e6
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        cpu = run_cpu_baseline()
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "fp8e4m3+bf16", "data": "synthetic",
        "config": {"workload": WORKLOAD, "global_batch": world * w.T, "seq_len": 65536,
                   "parallelism": f"dp{world} (independent sequences per GPU)",
                   "l2": "before every timed step: 512 MB written then 512 MB read (L2 cold and clean)",
                   "timing": "2K steps in the timed region: K replays of a CUDA graph of the three calls give "
                             "ms_per_step, K direct launches with events around the indexer give its launch time"},
        "roofline": {"bound": "hbm", "kernel": "indexer_logits", "achieved": achieved, "peak": hbm,
                     "unit": "GB/s", "frac": achieved / hbm, "traffic": traffic,
                     "peak_source": f"{peak_kind} hbm_gbs", "bytes_per_launch": idx_bytes},
        "step_roofline": {"bytes": step_bytes, "fp8_flops": fp8_flops, "bf16_flops": bf16_flops,
                          "time_us": roof_us, "frac": roof_us / (ms * 1e3),
                          "note": f"max(bytes / {peak_kind} HBM, FLOPs / peak); FP8 peak taken as 2x measured BF16"},
        "step_us_median": statistics.median(step_ms) * 1e3,
        "warm_step_us": {"mean": statistics.mean(warm_ms) * 1e3, "median": statistics.median(warm_ms) * 1e3,
                         "note": "the same graph without the L2 flush between replays (reference only)"},
        "one_call_step_us": None if one_call_ms is None else one_call_ms * 1e3,
        "kernels_ms": part_ms,
        "kernels_ms_note": "event pair around each kernel in a separate pass after the timed region "
                           "(includes about 2 us of event overhead each; no overlap between kernels)",
        "cpu_baseline": cpu,
        "e2e": {"value": job_throughput(world, w.T, e2e_mean * 1e3), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_mean * 1e3,
                "torch_graph_ms_per_step": e2e_torch * 1e3,
                "note": "wall clock per step of dsv4sa_step_launch + stream synchronise: the library's graph of "
                        "the H2D copy kernels of the step's queries and page tables from pinned memory, the "
                        "path, out and lse written into pinned memory; the cache pools stay resident "
                        "(torch_graph_ms_per_step: the same step as a torch CUDA graph of the C-ABI calls)"},
        "gpu_launches": launches_per_step * 2 * args.steps,
        "clocks": clocks.summary(),
        "inverse_rope": inv_rope,
        "compressor": compressor,
        "cache_writer": dict(writer, note="dsv4sa_cache_write, KV rows then indexer keys (two launches), "
                                          "bytes = bf16 rows read + codes, scales and rope written; "
                                          "one CUDA graph of both launches, event-timed after an L2 flush, "
                                          "outside the decode step"),
    }
    print(json.dumps(line))
    if dist:
        dist.destroy_process_group()


def main():
    args = parse_args()
    if args.cpu_child:
        cpu_child(args.cpu_child)
        return
    if args.impl == "reference":
        reference_arm(args)
        return
    gpu_arm(args)


if __name__ == "__main__":
    main()
