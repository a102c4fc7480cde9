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
import atexit
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
    ap.add_argument("--no-configs", action="store_true", help="skip the prefill, 1M-context and ragged workloads")
    ap.add_argument("--batch", type=int, default=32, help="sequences per GPU (profiling only)")
    ap.add_argument("--profile", action="store_true",
                    help="profiling driver for ncu: the path only, no L2 flush buffer, no e2e / CPU legs")
    ap.add_argument("--profile-feeders", action="store_true",
                    help="profiling driver for ncu: the KV-cache writer and compressor cases once each, no step")
    ap.add_argument("--profile-fp4", action="store_true",
                    help="profiling driver for ncu: the FP4 indexer on the decode64k shape, warmup + steps launches")
    ap.add_argument("--profile-config", choices=["prefill", "longctx", "ragged"], default=None,
                    help="profiling driver for ncu: one of the other workloads' path, warmup + steps passes")
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
    """nvidia-smi polled every 20 ms from before the timed region to the end of
    the GPU measurements; `window()` marks the timed region so its samples can
    be told apart from those of the passes after it."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []       # (host time, csv line)
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "20"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            atexit.register(self.stop)   # also when a measurement raises
        except OSError:
            self.proc = None
            return self
        t0 = time.time()     # measurements start once the sampler reports
        while not self.lines and time.time() - t0 < 3.0 and self.proc.poll() is None:
            time.sleep(0.01)
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def window(self, begin: bool):
        if begin:
            self.t0 = time.time()
        else:
            self.t1 = time.time()

    def stop(self):
        if self.proc is not None and self.proc.poll() is None:
            time.sleep(0.05)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def _parse(self, rows):
        sm, mx, reasons = [], [], set()
        for _, line in rows:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(self.NAMES, parts[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return sm, mx, reasons

    def summary(self):
        timed = [r for r in self.lines if self.t0 is not None and self.t1 is not None and self.t0 <= r[0] <= self.t1]
        sm_t, _, reasons_t = self._parse(timed)
        sm, mx, reasons = self._parse(self.lines)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm_t) if sm_t else None, "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm_t),
                "timed_region_s": None if self.t0 is None or self.t1 is None else self.t1 - self.t0,
                "sm_mhz_all": statistics.median(sm), "samples_all": len(sm),
                "note": "nvidia-smi every 20 ms: sm_mhz / samples over the timed region, *_all and reasons over "
                        "it and every GPU measurement after it"}


def measure_fp8_peak(torch, dev, n=8192, reps=10):
    """Dense FP8 (e4m3 x e4m3 -> bf16, per-tensor scales) tensor throughput of
    cuBLASLt through torch._scaled_mm at n^3, best of `reps` event-timed calls."""
    try:
        g = torch.Generator(device=dev).manual_seed(3)
        a = torch.randn((n, n), generator=g, device=dev).to(torch.float8_e4m3fn)
        b = torch.randn((n, n), generator=g, device=dev).to(torch.float8_e4m3fn).t()   # column-major operand
        one = torch.ones((), dtype=torch.float32, device=dev)
        for _ in range(3):
            torch._scaled_mm(a, b, one, one, out_dtype=torch.bfloat16)
        best = float("inf")
        for _ in range(reps):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
            torch._scaled_mm(a, b, one, one, out_dtype=torch.bfloat16)
            e1.record()
            torch.cuda.synchronize()
            best = min(best, e0.elapsed_time(e1))
        del a, b
        return 2 * n ** 3 / (best / 1e3) / 1e12, f"measured: torch._scaled_mm e4m3 {n}^3, best of {reps}"
    except Exception as e:   # noqa: BLE001 -- an unsupported build reports the nominal ratio instead
        return None, f"unmeasured ({type(e).__name__}): nominal 2x the measured BF16 peak"


# ---------------------------------------------------------------- algorithmic work

def algorithmic_work(w, idx_c, idx_w):
    """Bytes each kernel must move and FLOPs it must do for one step.  A key or
    KV row that several queries of one sequence use (prefill) counts once; the
    logits are the top-k's input, not part of the step's bytes."""
    import numpy as np
    seq = np.asarray(w.q_seq, np.int64)
    nvis = np.where(w.c128, 0, w.n_vis).astype(np.int64)    # C128 rows are not scored
    longest = np.zeros(int(seq.max()) + 1, np.int64)
    np.maximum.at(longest, seq, nvis)                      # each sequence's keys read once

    def distinct(idx):
        v = idx >= 0
        return int(np.unique((seq[:, None] << 32 | idx.astype(np.int64))[v]).size)

    valid = int((idx_c >= 0).sum() + (idx_w >= 0).sum())
    idx_bytes = int(longest.sum()) * KEY_ROW_BYTES + w.T * w.Hi * (128 + 8 + 4)
    attn_bytes = ((distinct(idx_c) + distinct(idx_w)) * KV_ROW_BYTES + 2 * w.T * w.H * 512 * 2
                  + w.T * (w.kc + w.kw) * 4)
    topk_bytes = int(nvis.sum()) * 4 + w.T * w.k * 4
    misc = w.T * w.k * 4 + w.T * w.kw * 4
    return {"indexer": {"bytes": idx_bytes, "fp8_flops": 2 * w.Hi * 128 * int(nvis.sum()), "bf16_flops": 0},
            "topk": {"bytes": topk_bytes, "fp8_flops": 0, "bf16_flops": 0},
            "attention": {"bytes": attn_bytes, "fp8_flops": 0, "bf16_flops": 4 * w.H * 512 * valid},
            "step_bytes": idx_bytes + attn_bytes + misc}


def kernel_roofline(work, us, hbm, fp8_tf, bf16_tf, peak_note):
    """The bound a kernel's algorithmic work sets (HBM bytes or tensor FLOPs,
    whichever takes longer at the peaks) and the fraction of it reached in `us`."""
    t_mem = work["bytes"] / (hbm * 1e9)
    t_tc = work["fp8_flops"] / (fp8_tf * 1e12) + work["bf16_flops"] / (bf16_tf * 1e12)
    if t_mem >= t_tc:
        ach = work["bytes"] / (us / 1e6) / 1e9
        return {"bound": "hbm", "achieved": ach, "peak": hbm, "unit": "GB/s", "frac": ach / hbm,
                "bytes_per_launch": work["bytes"], "us": us, "peak_source": peak_note["hbm"]}
    flops = work["fp8_flops"] + work["bf16_flops"]
    peak = flops / t_tc / 1e12          # the FP8/BF16 mix's peak
    ach = flops / (us / 1e6) / 1e12
    return {"bound": "tensor", "achieved": ach, "peak": peak, "unit": "TFLOP/s", "frac": ach / peak,
            "flops_per_launch": flops, "bytes_per_launch": work["bytes"], "us": us,
            "peak_source": peak_note["tensor"]}


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


CONFIGS = {
    "prefill": "prefill64k: one sequence of 65536 tokens, a chunk of 4096 queries at its last positions "
               "(causal: query t sees (pos_t + 1) // 4 C4 entries), H=64, Hi=64, top-512 + 128-token window",
    "longctx": "decode1m: B=4 sequences x 1048576 tokens (C4 N=262144 entries), H=64, Hi=64, top-512 + "
               "128-token window, 1 % heavy-tailed rows",
    "ragged": "ragged: B=128 sequences, log-normal lengths 64..131072 (median 8192), odd sequences C128 "
              "(dense over all N/128 entries, no indexer), 5 % empty, H=8, Hi=64",
}


def config_calls(L, W, dev, stream, name):
    """The workload `name` on the device and the calls of its path in order:
    index assembly, indexer, top-k with prefetch, attention."""
    w = W.make(name)
    d = L.upload(w, dev)
    fused = d.mode != L.ATTN_PREFILL      # decode modes: window indices derived in the attention kernel
    n_max = max(1, int(w.n_max))
    calls = []
    if d.has_c128 or w.kc > w.k:
        calls.append(("compress_indices", lambda: L.dsv4sa_compress_indices(d.n_vis_c128, w.kc, d.idx_c, stream)))
    if not fused:
        calls.append(("window_indices", lambda: L.dsv4sa_window_indices(d.pos, w.kw, w.win_ring, d.idx_w, stream)))
    calls.append(("indexer", lambda: L.dsv4sa_indexer_logits(d.keys, d.comp_pt, d.q_seq, d.n_vis_idx, d.q_idx,
                                                             d.q_idx_scale, d.wts, n_max, d.logits, stream)))
    calls.append(("topk", lambda: L.dsv4sa_topk_prefetch(d.logits, d.n_vis_idx, n_max, w.k, d.idx_c, d.comp,
                                                         d.comp_pt, d.q_seq, d.topk_ws, stream)))
    attn_fn = L.dsv4sa_sparse_attn_prefill if d.mode == L.ATTN_PREFILL else L.dsv4sa_sparse_attn_decode
    if fused:
        calls.append(("attention", lambda: attn_fn(
            d.q, d.sink, d.q_seq, d.comp, d.comp_pt, d.idx_c, d.win, d.win_pt, None, d.out, w.softmax_scale,
            lse=d.lse, ws=d.attn_ws, stream=stream, win_pos=d.pos, kw=w.kw, win_ring=w.win_ring,
            flags=L.ATTN_EARLY_WINDOW)))
    else:
        calls.append(("attention", lambda: attn_fn(
            d.q, d.sink, d.q_seq, d.comp, d.comp_pt, d.idx_c, d.win, d.win_pt, d.idx_w, d.out, w.softmax_scale,
            lse=d.lse, ws=d.attn_ws, stream=stream)))
    return w, d, fused, calls


def measure_config(L, W, torch, dev, stream, flush_l2, name, peaks, peak_note, reps=20):
    """One of the other workloads through the whole path (index assembly,
    indexer, top-k with prefetch, attention), as one CUDA graph replayed after
    an L2 flush and a GPU sleep, event-timed; plus each kernel event-timed on
    its own in direct launches.  Throughput in query-tokens/s and the step's
    and every kernel's roofline fraction."""
    hbm, fp8_tf, bf16_tf = peaks
    w, d, fused, calls = config_calls(L, W, dev, stream, name)

    def run():
        for _, fn in calls:
            fn()
    for _ in range(3):
        run()
    stream.synchronize()
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gr, stream=stream):
        run()
    stream.synchronize()
    step_ev, kern_ev = [], []
    for k in range(2 * (reps + 3)):
        flush_l2()
        torch.cuda._sleep(SLEEP_CYCLES)
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(len(calls) + 1)]
        if k % 2 == 0:
            ev[0].record(stream)
            gr.replay()
            ev[1].record(stream)
        else:
            for i, (_, fn) in enumerate(calls):
                ev[i].record(stream)
                fn()
            ev[-1].record(stream)
        if k >= 6:
            (step_ev if k % 2 == 0 else kern_ev).append(ev)
    torch.cuda.synchronize()
    st, bits = L.dsv4sa_check_errors()
    if st != 0:
        raise RuntimeError(f"device error word after the {name} workload: {st} ({bits})")
    ms = statistics.mean(e[0].elapsed_time(e[1]) for e in step_ev)
    kus = {n: statistics.mean(e[i].elapsed_time(e[i + 1]) for e in kern_ev) * 1e3 for i, (n, _) in enumerate(calls)}
    if fused:
        L.dsv4sa_window_indices(d.pos, w.kw, w.win_ring, d.idx_w, stream)   # for the byte count only
    work = algorithmic_work(w, d.idx_c.cpu().numpy(), d.idx_w.cpu().numpy())
    roof = {n: kernel_roofline(work[n], kus[n], hbm, fp8_tf, bf16_tf, peak_note)
            for n in ("indexer", "topk", "attention")}
    fl8 = sum(work[n]["fp8_flops"] for n in roof)
    fl16 = sum(work[n]["bf16_flops"] for n in roof)
    roof_us = max(work["step_bytes"] / (hbm * 1e9), fl8 / (fp8_tf * 1e12) + fl16 / (bf16_tf * 1e12)) * 1e6
    out = {"workload": CONFIGS[name], "queries": w.T, "value": w.T / (ms / 1e3), "unit": UNIT,
           "ms_per_step": ms, "launches": len(calls) + (1 if d.topk_ws is not None else 0),
           "step_roofline": {"bytes": work["step_bytes"], "fp8_flops": fl8, "bf16_flops": fl16, "time_us": roof_us,
                             "frac": roof_us / (ms * 1e3),
                             "bound": "tensor" if roof_us > work["step_bytes"] / (hbm * 1e9) * 1e6 else "hbm"},
           "kernels_us": kus, "kernels_roofline": roof}
    del d
    torch.cuda.empty_cache()
    return out


def measure_fp4_indexer(L, W, torch, dev, stream, flush_l2, hbm_gbs, reps=20):
    """The FP4 indexer (IDXK_FP4 keys: 64 code bytes + 4 E8M0 bytes per entry;
    FP4 q) on the decode64k shape: B = 32 queries x 16384 entries, Hi = 64, as a
    one-launch CUDA graph after an L2 flush, event-timed."""
    w = W.make_fp4_indexer("fp4d", B=32, L=65536, Hi=64, seed=2202)
    buf, desc = L.pack_key_pool_fp4(w.key_codes, w.key_e8m0, dev)
    pt = torch.from_numpy(w.comp_pt).to(dev)
    q_seq = torch.from_numpy(w.q_seq).to(dev)
    n_vis = torch.from_numpy(w.n_vis).to(dev)
    q = torch.from_numpy(L.pack_fp4_codes(w.q_codes)).to(dev)
    qe = torch.from_numpy(w.q_e8m0).to(dev)
    wt = torch.from_numpy(w.w).to(dev)
    logits = torch.empty((w.T, w.n_max), dtype=torch.float32, device=dev)

    def fn():
        L.dsv4sa_indexer_logits_fp4(desc, pt, q_seq, n_vis, q, qe, wt, w.n_max, logits, stream)
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
    st, bits = L.dsv4sa_check_errors()
    if st != 0:
        raise RuntimeError(f"device error word after the FP4 indexer: {st} ({bits})")
    us = statistics.mean(a.elapsed_time(b) for a, b in ms) * 1e3
    nbytes = int(w.n_vis.sum()) * 68 + w.T * w.Hi * (64 + 4 + 4)
    return {"workload": "B=32 queries x 16384 FP4 keys (68 B each), Hi=64, FP4 q", "us": us, "bytes": nbytes,
            "achieved_gbs": nbytes / us / 1e3, "frac_of_hbm": nbytes / us / 1e3 / hbm_gbs,
            "note": "dsv4sa_indexer_logits_fp4 alone, one-launch CUDA graph after an L2 flush (launch included)"}


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

def _oracle_worker(i, barrier, stop, out_q):
    """One host core: its own decode sequence (same shapes as the bench's, its own
    seed), then one query row through the oracle per step, in lock step with
    the other workers (a step starts and ends at a barrier)."""
    import oracle
    from compressed_sparse_attention_c4_gb300 import workloads as W
    w = W.make("decode", B=1, seed=W.SEEDS["decode"] + 7919 * (i + 1))
    work = w.as_dict()
    barrier.wait()
    rows = 0
    while True:
        barrier.wait()            # step start
        if stop.value:
            break
        oracle.decode_step(work, rows=[0], k=w.k)
        rows += 1
        barrier.wait()            # step end
    out_q.put(rows)


class OraclePool:
    """The fp64 oracle on every host core: one single-threaded worker process
    per core (spawned), each step one query row per worker."""

    def __init__(self, workers=None):
        import multiprocessing as mp
        for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
            os.environ[v] = "1"          # inherited by the spawned workers: one thread each
        ctx = mp.get_context("spawn")
        self.n = workers or os.cpu_count() or 1
        self.barrier = ctx.Barrier(self.n + 1)
        self.stop = ctx.Value("i", 0)
        self.out_q = ctx.Queue()
        self.procs = [ctx.Process(target=_oracle_worker, args=(i, self.barrier, self.stop, self.out_q), daemon=True)
                      for i in range(self.n)]
        for pr in self.procs:
            pr.start()
        self.barrier.wait(timeout=600)    # every worker has built its sequence

    def step(self) -> float:
        """One row per worker; returns the wall time of the step in seconds."""
        t0 = time.perf_counter()
        self.barrier.wait(timeout=600)
        self.barrier.wait(timeout=600)
        return time.perf_counter() - t0

    def close(self):
        self.stop.value = 1
        self.barrier.wait(timeout=600)
        rows = [self.out_q.get(timeout=60) for _ in self.procs]
        for pr in self.procs:
            pr.join(timeout=60)
        return sum(rows)


def run_cpu_baseline(seconds=10.0):
    """cpu_baseline: the oracle on every host core for about `seconds`."""
    try:
        pool = OraclePool()
        pool.step()                         # warm-up step
        steps, dt = 0, 0.0
        while dt < seconds:
            dt += pool.step()
            steps += 1
        pool.close()
    except Exception as e:   # noqa: BLE001 -- reported in the line, never fatal for the GPU numbers
        return {"value": None, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle", "error": repr(e)[-300:]}
    return {"value": steps * pool.n / dt, "unit": UNIT, "cores": pool.n, "kind": "oracle",
            "sample": f"{steps} steps x {pool.n} query rows (one per core; each core its own 65536-token "
                      f"sequence, H=64, Hi=64, the oracle's indexer, top-k and attention), {dt:.1f} s, "
                      f"numpy fp64, one thread per process"}


def reference_arm(args):
    rank, _, _ = rank_env()
    if rank != 0:
        return
    pool = OraclePool()
    for _ in range(args.warmup):
        pool.step()
    dt = sum(pool.step() for _ in range(args.steps))
    pool.close()
    value = args.steps * pool.n / dt
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * dt / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "step": f"{pool.n} query rows (one per host core, each its own "
                                                 f"65536-token sequence) through the fp64 oracle"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": pool.n, "kind": "oracle",
                         "sample": f"{args.steps} steps x {pool.n} query rows, numpy fp64, one thread per process"},
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
    if args.profile_fp4:
        stream = torch.cuda.Stream(device=dev)
        torch.cuda.set_stream(stream)
        w = W.make_fp4_indexer("fp4d", B=args.batch, L=65536, Hi=64, seed=2202)
        buf, desc = L.pack_key_pool_fp4(w.key_codes, w.key_e8m0, dev)
        args4 = (desc, torch.from_numpy(w.comp_pt).to(dev), torch.from_numpy(w.q_seq).to(dev),
                 torch.from_numpy(w.n_vis).to(dev), torch.from_numpy(L.pack_fp4_codes(w.q_codes)).to(dev),
                 torch.from_numpy(w.q_e8m0).to(dev), torch.from_numpy(w.w).to(dev), w.n_max,
                 torch.empty((w.T, w.n_max), dtype=torch.float32, device=dev))
        for _ in range(args.warmup + args.steps):
            L.dsv4sa_indexer_logits_fp4(*args4, stream)
        torch.cuda.synchronize()
        st, bits = L.dsv4sa_check_errors()
        print(json.dumps({"profile_fp4": True, "batch": w.T, "launches": args.warmup + args.steps, "status": st,
                          "bits": bits}))
        if st != 0:
            raise SystemExit(1)
        return
    if args.profile_config:
        stream = torch.cuda.Stream(device=dev)
        torch.cuda.set_stream(stream)
        w, d, _, calls = config_calls(L, W, dev, stream, args.profile_config)
        for _ in range(args.warmup + args.steps):
            for _, fn in calls:
                fn()
        torch.cuda.synchronize()
        st, bits = L.dsv4sa_check_errors()
        print(json.dumps({"profile_config": args.profile_config, "queries": w.T,
                          "launches": [n for n, _ in calls], "passes": args.warmup + args.steps,
                          "status": st, "bits": bits}))
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
        raise RuntimeError(f"device error word after the warm-up: {st} ({bits})")

    # The step as one CUDA graph of the three calls (programmatic-dependent
    # launches become graph edges).
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step()
    stream.synchronize()

    # Timed region: 2 K steps.  Even steps are graph replays between one event
    # before and one after (the step time); odd steps launch the three calls
    # directly with an event between every two (each kernel's launch time).
    # An event between two kernels ends their programmatic overlap, so the step
    # time is taken on the steps without inner events.
    nk = len(kernels)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(nk + 1)] for _ in range(2 * args.steps)]
    clocks = ClockSampler(dev.index).start()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.window(True)
    for k in range(2 * args.steps):
        flush_l2()
        torch.cuda._sleep(SLEEP_CYCLES)
        if k % 2 == 0:
            evs[k][0].record(stream)
            graph.replay()
            evs[k][1].record(stream)
        else:
            step(evs[k])
    torch.cuda.synchronize()
    clocks.window(False)
    if dist:
        dist.barrier()
    st, bits = L.dsv4sa_check_errors()
    if st != 0:
        raise RuntimeError(f"device error word after the timed region: {st} ({bits})")
    step_ms = [evs[k][0].elapsed_time(evs[k][1]) for k in range(0, 2 * args.steps, 2)]
    part_ms = {name: statistics.mean(evs[k][i].elapsed_time(evs[k][i + 1]) for k in range(1, 2 * args.steps, 2))
               for i, (name, _) in enumerate(kernels)}
    ms = reduce_max(statistics.mean(step_ms), dist, dev)
    value = job_throughput(world, w.T, ms)

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
        clocks.stop()
        dist.destroy_process_group()
        return
    hbm, bf16_tf, peak_kind = measured_peaks()
    fp8_tf, fp8_how = measure_fp8_peak(torch, dev)
    if fp8_tf is None:
        fp8_tf = 2 * bf16_tf
    peaks = (hbm, fp8_tf, bf16_tf)
    peak_note = {"hbm": f"{peak_kind} hbm_gbs (MEASURED_PEAKS.json)",
                 "tensor": f"FP8 {fp8_how}; BF16 {peak_kind} bf16_tflops (burst)"}
    idx_c = d.idx_c.cpu().numpy()
    L.dsv4sa_window_indices(d.pos, w.kw, w.win_ring, d.idx_w, stream)   # for the byte count only
    idx_w = d.idx_w.cpu().numpy()
    work = algorithmic_work(w, idx_c, idx_w)
    names = {"indexer_logits": "indexer", "topk": "topk", "sparse_attn_decode": "attention"}
    roofs = {k: kernel_roofline(work[names[k]], part_ms[k] * 1e3, hbm, fp8_tf, bf16_tf, peak_note)
             for k in part_ms}
    dominant = max(part_ms, key=part_ms.get)
    fl8 = sum(work[n]["fp8_flops"] for n in names.values())
    fl16 = sum(work[n]["bf16_flops"] for n in names.values())
    roof_us = max(work["step_bytes"] / (hbm * 1e9), fl8 / (fp8_tf * 1e12) + fl16 / (bf16_tf * 1e12)) * 1e6
    traffic = {"indexer_logits": profiled_traffic("compressed_sparse_attention_c4_gb300/csrc/indexer.cu",
                                                  "profiles/indexer_logits_decode64k.md"),
               "topk": profiled_traffic("compressed_sparse_attention_c4_gb300/csrc/topk.cu",
                                        "profiles/topk_decode64k.md"),
               "sparse_attn_decode": profiled_traffic("compressed_sparse_attention_c4_gb300/csrc/attn_decode.cu",
                                                      "profiles/sparse_attn_decode64k.md")}
    for k in roofs:
        roofs[k]["traffic"] = traffic[k]
    configs = {}
    if not args.no_configs:
        for name in ("prefill", "longctx", "ragged"):
            configs[name] = measure_config(L, W, torch, dev, stream, flush_l2, name, peaks, peak_note)
    fp4_indexer = measure_fp4_indexer(L, W, torch, dev, stream, flush_l2, hbm)
    writer = measure_cache_writer(L, torch, dev, stream, flush_l2, hbm)
    inv_rope = measure_inverse_rope(L, torch, d, w, stream, kernels, flush_l2)
    compressor = measure_compressor(L, torch, dev, stream, flush_l2, hbm)
    clocks.stop()
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
                             "ms_per_step, K direct launches with events between the kernels give each "
                             "kernel's launch time"},
        "roofline": dict(roofs[dominant], kernel=dominant,
                         note="the kernel with the largest event-timed share of the step"),
        "kernels_roofline": roofs,
        "step_roofline": {"bytes": work["step_bytes"], "fp8_flops": fl8, "bf16_flops": fl16,
                          "time_us": roof_us, "frac": roof_us / (ms * 1e3),
                          "note": "max(bytes / HBM peak, FP8 FLOPs / FP8 peak + BF16 FLOPs / BF16 peak)"},
        "peaks": {"hbm_gbs": hbm, "bf16_tflops": bf16_tf, "fp8_tflops": fp8_tf, "fp8_source": fp8_how,
                  "hbm_bf16_source": f"{peak_kind} (MEASURED_PEAKS.json)"},
        "step_us_median": statistics.median(step_ms) * 1e3,
        "warm_step_us": {"mean": statistics.mean(warm_ms) * 1e3, "median": statistics.median(warm_ms) * 1e3,
                         "note": "the same graph without the L2 flush between replays (reference only)"},
        "one_call_step_us": None if one_call_ms is None else one_call_ms * 1e3,
        "kernels_ms": part_ms,
        "kernels_ms_note": "events between the kernels on the odd steps of the timed region (each includes "
                           "about 2 us of event overhead; no overlap between kernels)",
        "configs": configs,
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
        "fp4_indexer": fp4_indexer,
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
    if args.impl == "reference":
        reference_arm(args)
        return
    gpu_arm(args)


if __name__ == "__main__":
    main()
