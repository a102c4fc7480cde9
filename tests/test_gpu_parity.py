"""GPU parity: the CUDA path through the C ABI against the fp64 CPU oracle.

Every input is seeded and synthetic (compressed_sparse_attention_c4_gb300.workloads).
Small cases are compared in full (every logit, every index, every output
element); the full-size workloads (64K-context decode, 1M-context decode,
4096-token chunked prefill) run exactly as bench.py runs them and are compared
on sampled query rows.  Tolerances are in tests/parity.py.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from compressed_sparse_attention_c4_gb300 import workloads as W

from parity import (GpuRun, check_attention, check_row, check_topk_exact, oracle_attention)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="session", autouse=True)
def built():
    from compressed_sparse_attention_c4_gb300 import build, dsv4sa
    import os
    if not os.path.exists(dsv4sa.LIB_PATH):
        build.build()
    torch.cuda.init()


def test_tiny_decode_full():
    run = GpuRun(W.make("tiny"))
    check_row(run, 0)


def test_tiny_decode_sharp_softmax():
    run = GpuRun(W.make("tiny", q_mult=8.0))
    check_row(run, 0)


def test_edge_lengths_and_ragged_tails():
    # n_vis = 1000 (ragged last tile), 513 (one past k), 25, 2049, 0 (empty), 512 (exactly k)
    w = W.make_decode_like("edges", B=6, L=[4000, 2052, 100, 8196, 3, 2048], H=16, Hi=8,
                           kv_std=1.0, key_std=1 / math.sqrt(128), seed=7)
    run = GpuRun(w)
    for t in range(w.T):
        check_row(run, t)


@pytest.mark.parametrize("H", [8, 48, 128])
def test_head_counts(H):
    w = W.make_decode_like(f"heads{H}", B=3, L=[3000, 5000, 700], H=H, Hi=16, kv_std=1.0,
                           key_std=1 / math.sqrt(128), seed=100 + H)
    run = GpuRun(w)
    for t in range(w.T):
        check_row(run, t)


def test_ragged_mixed_batch_full():
    w = W.make("ragged")
    run = GpuRun(w)
    empty = np.nonzero(w.n_vis == 0)[0]
    for t in range(w.T):
        check_row(run, t)
    for t in empty:
        if w.pos[t] < 0:
            assert (run.out[t] == 0).all()
            np.testing.assert_allclose(run.lse[t], w.sink, rtol=1e-5, atol=1e-5)


def test_decode_64k_all_rows():
    """The 64K-context decode batch as the benchmark runs it: every query row."""
    w = W.make("decode")
    run = GpuRun(w, serving=True)
    for t in range(w.T):
        check_row(run, t)


def prefill_rows(w, every=16, per_class=12):
    """Every `every`-th query of the chunk, its first and last four, and for each
    boundary class the first `per_class` queries in it: the query's raw token at
    the first or last slot of a window page, its visible C4 entries ending at
    the first or last slot of a page, and n_vis just below, at or just above a
    multiple of 128 (one 128-entry tile more or less to score and select)."""
    pos, nv = w.pos.astype(np.int64), w.n_vis.astype(np.int64)
    rows = set(range(0, w.T, every)) | set(range(4)) | set(range(w.T - 4, w.T))
    classes = [pos % 64 == 0, pos % 64 == 63, nv % 64 == 1, nv % 64 == 0,
               nv % 128 == 127, nv % 128 == 0, nv % 128 == 1]
    for c in classes:
        rows |= set(np.nonzero(c)[0][:per_class].tolist())
    return sorted(rows)


def test_prefill_sampled():
    """The 4096-query prefill chunk: at least 256 rows, every page and tile boundary class."""
    w = W.make("prefill")
    run = GpuRun(w)
    rows = prefill_rows(w)
    assert len(rows) >= 256
    for t in rows:
        check_row(run, t)


def test_longctx_1m_all_rows():
    """The 1M-context decode batch as the benchmark would run it: every query row
    (two-stage top-k over 16 chunks of 16384 entries)."""
    w = W.make("longctx")
    run = GpuRun(w, serving=True)
    for t in range(w.T):
        check_row(run, t)


def test_deterministic_bits():
    w = W.make("tiny")
    a, b = GpuRun(w), GpuRun(w)
    assert np.array_equal(a.logits, b.logits)
    assert np.array_equal(a.idx_c, b.idx_c)
    assert np.array_equal(a.out.view(np.uint32), b.out.view(np.uint32))


def test_topk_direct_ties_and_chunks():
    """Top-k kernel alone on integer-valued scores (heavy ties), row lengths
    from 0 to 262144 (one- and two-stage), one row left untouched (n_vis < 0)."""
    from compressed_sparse_attention_c4_gb300 import dsv4sa as L
    rng = np.random.default_rng(11)
    lens = [0, 5, 512, 513, 4096, 4097, 16384, 16385, 32768, 70000, 262144, -1]
    n_max = 262144
    T, k = len(lens), 512
    x = rng.integers(-50, 50, size=(T, n_max)).astype(np.float32)
    x[3, :] = 7.0                                   # every score tied
    x[5, ::3] = -0.0                                # signed zeros tie with +0
    logits = torch.from_numpy(x).cuda()
    n_vis = torch.tensor(lens, dtype=torch.int32, device="cuda")
    idx = torch.full((T, k), -7, dtype=torch.int32, device="cuda")
    ws = torch.empty(L.dsv4sa_topk_workspace_size(T, n_max, k), dtype=torch.uint8, device="cuda")
    L.dsv4sa_topk(logits, n_vis, n_max, k, idx, ws)
    got = idx.cpu().numpy()
    for t, n in enumerate(lens):
        if n < 0:
            assert (got[t] == -7).all()
        else:
            assert np.array_equal(got[t], oracle.topk_row(x[t, :n].astype(np.float64), k)), t


@pytest.mark.parametrize("k", [1, 512, 2048])
def test_topk_value_distributions(k):
    """Top-k kernel alone on continuous scores: a wide normal row, a row in a
    narrow band (only the low key bits vary), a row where many scores sit on the
    k-th value's first radix digit (more than the directly ranked few), a row
    with NaN, +-inf and signed zeros; lengths around the one-CTA row limit."""
    from compressed_sparse_attention_c4_gb300 import dsv4sa as L
    rng = np.random.default_rng(29 + k)
    lens = [16383, 16384, 16385, 100000, 3000, 40000]
    n_max = max(lens)
    T = len(lens)
    x = rng.standard_normal((T, n_max)).astype(np.float32)
    x[1] = (1000.0 + 0.01 * rng.random(n_max)).astype(np.float32)          # narrow band
    x[2] = rng.standard_normal(n_max).astype(np.float32) - 4.0
    x[2, rng.choice(16385, 3000, replace=False)] = np.float32(2.0) + rng.integers(0, 64, 3000).astype(np.float32) * np.float32(2.0 ** -22)
    x[3, rng.choice(100000, 50, replace=False)] = np.nan
    x[3, rng.choice(100000, 20, replace=False)] = np.inf
    x[3, rng.choice(100000, 20, replace=False)] = -np.inf
    x[3, rng.choice(100000, 300, replace=False)] = -0.0
    x[3, rng.choice(100000, 300, replace=False)] = 0.0
    x[5] = np.round(x[5] * 4) / 4                                          # coarse ties
    logits = torch.from_numpy(x).cuda()
    n_vis = torch.tensor(lens, dtype=torch.int32, device="cuda")
    idx = torch.full((T, k), -7, dtype=torch.int32, device="cuda")
    ws = torch.empty(max(1, L.dsv4sa_topk_workspace_size(T, n_max, k)), dtype=torch.uint8, device="cuda")
    L.dsv4sa_topk(logits, n_vis, n_max, k, idx, ws)
    got = idx.cpu().numpy()
    for t, n in enumerate(lens):
        assert np.array_equal(got[t], oracle.topk_row(x[t, :n].astype(np.float64), k)), t


def test_index_helpers():
    from compressed_sparse_attention_c4_gb300 import dsv4sa as L
    pos = torch.tensor([-1, 0, 5, 127, 128, 65535], dtype=torch.int32, device="cuda")
    for ring in (0, 128):
        out = torch.empty((6, 128), dtype=torch.int32, device="cuda")
        L.dsv4sa_window_indices(pos, 128, ring, out)
        for t, p in enumerate(pos.tolist()):
            assert np.array_equal(out[t].cpu().numpy(), oracle.window_indices(p, 128, ring))
    n_vis = torch.tensor([0, 3, 1024, 2000], dtype=torch.int32, device="cuda")
    out = torch.empty((4, 1024), dtype=torch.int32, device="cuda")
    L.dsv4sa_compress_indices(n_vis, 1024, out)
    for t, n in enumerate(n_vis.tolist()):
        assert np.array_equal(out[t].cpu().numpy(), oracle.compress_indices(n, 1024))


def test_out_of_range_index_is_flagged_and_skipped():
    from compressed_sparse_attention_c4_gb300 import dsv4sa as L
    w = W.make("tiny")
    run = GpuRun(w)
    d = run.d
    bad = d.idx_c.clone()
    bad[0, 3] = d.comp_pt.shape[1] * 64 + 5          # beyond the page table: invalid + flagged
    L.dsv4sa_sparse_attn_decode(d.q, d.sink, d.q_seq, d.comp, d.comp_pt, bad, d.win, d.win_pt, d.idx_w,
                                d.out, w.softmax_scale, lse=d.lse, ws=d.attn_ws)
    st, bits = L.dsv4sa_check_errors()
    assert st == 5 and bits & 1
    ic = run.idx_c[0].copy()
    ic[3] = -1
    ref = oracle_attention(w, 0, ic, run.idx_w[0])
    got = d.out.float().cpu().numpy()[0]
    assert np.abs(got - ref).max() <= 2e-2 * np.abs(ref).max()
    assert L.dsv4sa_check_errors() == (0, 0)         # the word was cleared


def test_all_invalid_rows_give_zeros_and_sink_lse():
    from compressed_sparse_attention_c4_gb300 import dsv4sa as L
    w = W.make("tiny")
    run = GpuRun(w)
    d = run.d
    none_c = torch.full_like(d.idx_c, -1)
    none_w = torch.full_like(d.idx_w, -1)
    for fn in (L.dsv4sa_sparse_attn_decode, L.dsv4sa_sparse_attn_prefill):
        d.out.fill_(1.0)
        fn(d.q, d.sink, d.q_seq, d.comp, d.comp_pt, none_c, d.win, d.win_pt, none_w, d.out,
           w.softmax_scale, lse=d.lse, ws=d.attn_ws)
        torch.cuda.synchronize()
        assert (d.out == 0).all()
        np.testing.assert_allclose(d.lse.cpu().numpy()[0], w.sink, rtol=1e-6, atol=1e-6)


@pytest.mark.parametrize("B,H,c128", [(64, 64, False), (40, 16, False), (1, 16, False), (64, 16, True)])
def test_split_merge_paths(B, H, c128):
    """Decode splits each query's rows over several CTAs.  By batch size this
    gives clusters of 2, 4 and 8 CTAs merging behind a cluster barrier, and
    (64 queries, one C128 row of 1024 entries: 1152 rows over 2 splits) the
    workspace + merge kernel path."""
    from compressed_sparse_attention_c4_gb300 import dsv4sa as L
    lens = [16000 + 997 * i for i in range(B)]
    c128_rows = None
    if c128:
        lens = [131072, 65536, 9000] + lens[3:]
        c128_rows = [True] + [False] * (B - 1)
    w = W.make_decode_like(f"split{B}", B=B, L=lens, H=H, Hi=16, kv_std=1.0, key_std=1 / math.sqrt(128),
                           c128_rows=c128_rows, seed=300 + B)
    run = GpuRun(w, mode=L.ATTN_DECODE)
    plan = L.dsv4sa_attn_plan(L.ATTN_DECODE, w.T, w.H, w.kc, w.kw)
    assert plan["nsplit"] * plan["rows_per_split"] >= w.kc + w.kw
    assert plan["launches"] == (2 if c128 else 1)
    for t in range(w.T):
        check_attention(run, t)


def test_decode_and_prefill_modes_agree():
    from compressed_sparse_attention_c4_gb300 import dsv4sa as L
    w = W.make_decode_like("modes", B=4, L=[9000, 12000, 3000, 60000], H=64, Hi=64, kv_std=1.0,
                           key_std=1 / math.sqrt(128), seed=21)
    a = GpuRun(w, mode=L.ATTN_DECODE)
    b = GpuRun(w, mode=L.ATTN_PREFILL)
    assert np.array_equal(a.idx_c, b.idx_c)
    for t in range(w.T):
        check_attention(a, t)
        check_attention(b, t)
    assert np.abs(a.out - b.out).max() <= 2e-2 * np.abs(a.out).max()


def test_step_graph_matches_eager():
    """The serving-loop form (one CUDA graph: H2D of the inputs, the path, D2H
    of out and lse) gives the eager path's bits, replay after replay, and picks
    up new host inputs."""
    from compressed_sparse_attention_c4_gb300 import dsv4sa as L
    w = W.make("tiny")
    run = GpuRun(w)
    sg = L.StepGraph(run.d)
    for _ in range(2):
        sg.replay()
        sg.stream.synchronize()
        assert np.array_equal(sg.host_out["out"].float().numpy(), run.out)
        assert np.array_equal(sg.host_out["lse"].numpy(), run.lse)
    sg.host_in["q"].view(torch.int16).fill_(0x3F80)   # every query element 1.0: a different softmax
    sg.replay()
    sg.stream.synchronize()
    got = sg.host_out["out"].float().numpy()
    assert np.isfinite(got).all()
    assert np.abs(got - run.out).max() > 0.05 * np.abs(run.out).max()


@pytest.mark.parametrize("name", ["tiny", "decode"])
def test_native_step_matches_eager(name):
    """The step built by the library (dsv4sa_step_create: the copy kernels and
    the three calls captured in C++, one dsv4sa_step_launch per step) gives the
    eager path's bits, launch after launch, and picks up new host inputs."""
    from compressed_sparse_attention_c4_gb300 import dsv4sa as L
    w = W.make(name)
    run = GpuRun(w)
    ns = L.NativeStep(run.d)
    for _ in range(2):
        ns.host_out["out"].fill_(7.0)
        ns.launch()
        ns.stream.synchronize()
        assert np.array_equal(ns.host_out["out"].float().numpy(), run.out)
        assert np.array_equal(ns.host_out["lse"].numpy(), run.lse)
    ns.host_in["q"].view(torch.int16).fill_(0x3F80)   # every query element 1.0: a different softmax
    ns.launch()
    ns.stream.synchronize()
    got = ns.host_out["out"].float().numpy()
    assert np.isfinite(got).all()
    assert np.abs(got - run.out).max() > 0.05 * np.abs(run.out).max()
    ns.close()
    assert L.dsv4sa_check_errors() == (0, 0)


@pytest.mark.parametrize("name", ["tiny", "ragged", "decode"])
@pytest.mark.parametrize("mode_name", ["ATTN_DECODE", "ATTN_PREFILL"])
@pytest.mark.parametrize("flags", [0, 1])
def test_window_indices_in_kernel_match_explicit(name, mode_name, flags):
    """Attention with the window indices derived in the kernel from the
    positions (empty rows with pos < 0, short histories, the ring of the window
    cache) gives the bits of attention over the explicit dsv4sa_window_indices
    list, with and without the early start of the window rows."""
    from compressed_sparse_attention_c4_gb300 import dsv4sa as L
    mode = getattr(L, mode_name)
    w = W.make(name)
    run = GpuRun(w, mode=mode)
    d = run.d
    fn = L.dsv4sa_sparse_attn_prefill if mode == L.ATTN_PREFILL else L.dsv4sa_sparse_attn_decode
    d.out.fill_(7.0)
    d.lse.fill_(7.0)
    fn(d.q, d.sink, d.q_seq, d.comp, d.comp_pt, d.idx_c, d.win, d.win_pt, None, d.out, w.softmax_scale,
       lse=d.lse, ws=d.attn_ws, win_pos=d.pos, kw=w.kw, win_ring=w.win_ring, flags=flags)
    torch.cuda.synchronize()
    assert L.dsv4sa_check_errors() == (0, 0)
    assert np.array_equal(d.out.float().cpu().numpy(), run.out)
    assert np.array_equal(d.lse.cpu().numpy(), run.lse)


def test_indexer_scales_outside_the_ratio_form():
    """The indexer's epilogue factors out positive q and key scales; a query with a
    negative or zero q-block scale, and keys with a zero block scale, take the
    general form.  Every logit still matches the oracle."""
    from parity import check_logits
    w = W.make_decode_like("scales", B=3, L=[6000, 9000, 20000], H=16, Hi=8, kv_std=1.0,
                           key_std=1 / math.sqrt(128), seed=77)
    w.q_idx_scale[0, 1, 0] *= -1.0          # query 0: one head's first block negative
    w.q_idx_scale[1, 3, :] = 0.0            # query 1: one head's scales zero
    ks = w.key_pool["scale"]
    ks[w.comp_pt[w.q_seq[2]][0], :10, 0] = 0.0    # query 2: ten keys with a zero first-block scale
    ks[w.comp_pt[w.q_seq[2]][1], 5:9, 1] = 0.0
    run = GpuRun(w)
    for t in range(w.T):
        check_logits(run, t)


@pytest.mark.parametrize("Hi", [96, 128])
def test_indexer_wide_heads(Hi):
    """More than 64 indexer heads: two accumulator stages of 2 x HiP TMEM
    columns, taken by two epilogue groups.  Every logit of every row."""
    from parity import check_logits
    w = W.make_decode_like(f"wide{Hi}", B=6, L=[3000, 9000, 600, 20000, 12, 4100], H=16, Hi=Hi, kv_std=1.0,
                           key_std=1 / math.sqrt(128), seed=300 + Hi)
    run = GpuRun(w)
    for t in range(w.T):
        check_logits(run, t)


@pytest.mark.parametrize("Hi", [64, 8])
def test_indexer_many_short_rows(Hi):
    """600 sequences of 0 to 300 entries (0 to 3 tiles each): a CTA's range
    holds many one-tile queries, which the indexer's two MMA issuers (alternate
    tiles) pass without issuing for them; the q blocks alternate between two
    buffers per query and are loaded one query ahead.  Every logit of every
    row is compared with the oracle; Hi = 8 also covers the zero rows of the
    padded q block (Hi < 16)."""
    from parity import check_logits
    rng = np.random.default_rng(4242 + Hi)
    L = rng.integers(0, 1204, size=600)
    L[rng.random(600) < 0.1] = 2            # empty rows among them
    w = W.make_decode_like(f"short{Hi}", B=600, L=L.tolist(), H=16, Hi=Hi, kv_std=1.0,
                           key_std=1 / math.sqrt(128), seed=900 + Hi)
    run = GpuRun(w)
    for t in range(w.T):
        check_logits(run, t)


@pytest.mark.parametrize("B,H,c128,mode_name", [
    (4, 16, False, "ATTN_DECODE"),     # 8 splits: cluster merge
    (24, 64, False, "ATTN_DECODE"),    # 4 splits: cluster merge
    (48, 16, False, "ATTN_DECODE"),    # 2 splits: cluster merge
    (48, 16, True, "ATTN_DECODE"),     # one C128 row of 1024 entries: workspace + merge kernel
    (24, 64, False, "ATTN_PREFILL"),   # one CTA per query: no merge
])
def test_sink_minus_infinity(B, H, c128, mode_name):
    """attn_sink = -inf on every other head (the sink then adds nothing to the
    denominator: plain softmax over the selected rows) on normal rows and on an
    all-invalid row, through every way the splits of a query are merged.  The
    empty row must give exact zeros (lse -inf where the sink is -inf), never NaN."""
    from compressed_sparse_attention_c4_gb300 import dsv4sa as L
    lens = [3000 + 101 * i for i in range(B)]
    c128_rows = None
    if c128:
        lens[0] = 131072
        c128_rows = [True] + [False] * (B - 1)
    empty = [False] * B
    empty[1] = True
    w = W.make_decode_like(f"sinkinf{B}", B=B, L=lens, H=H, Hi=16, kv_std=1.0, key_std=1 / math.sqrt(128),
                           c128_rows=c128_rows, empty_rows=empty, seed=500 + B + H)
    w.sink[::2] = -np.inf
    mode = getattr(L, mode_name)
    run = GpuRun(w, mode=mode)
    if mode == L.ATTN_DECODE:
        plan = L.dsv4sa_attn_plan(mode, w.T, w.H, w.kc, w.kw)
        assert plan["launches"] == (2 if c128 else 1)
    assert np.isfinite(run.out).all()
    assert (run.out[1] == 0).all()
    lse_empty = run.lse[1]
    assert np.all(np.isneginf(lse_empty[::2]))
    np.testing.assert_allclose(lse_empty[1::2], w.sink[1::2], rtol=1e-6, atol=1e-6)
    for t in range(w.T):
        if t != 1:
            check_attention(run, t)


@pytest.mark.parametrize("name", ["decode", "ragged", "longctx"])
def test_topk_prefetch_matches_topk(name):
    """dsv4sa_topk_prefetch (the selection plus L2 prefetches of the selected
    KV rows) writes exactly what dsv4sa_topk writes, including rows left
    untouched (n_vis < 0), short rows and the two-stage path of long rows."""
    from compressed_sparse_attention_c4_gb300 import dsv4sa as L
    w = W.make(name)
    d = L.upload(w, "cuda")
    n_max = max(1, int(w.n_max))
    L.dsv4sa_indexer_logits(d.keys, d.comp_pt, d.q_seq, d.n_vis_idx, d.q_idx, d.q_idx_scale, d.wts, n_max, d.logits)
    a = torch.full_like(d.idx_c, -7)
    b = torch.full_like(d.idx_c, -7)
    L.dsv4sa_topk(d.logits, d.n_vis_idx, n_max, w.k, a, d.topk_ws)
    L.dsv4sa_topk_prefetch(d.logits, d.n_vis_idx, n_max, w.k, b, d.comp, d.comp_pt, d.q_seq, d.topk_ws)
    torch.cuda.synchronize()
    assert L.dsv4sa_check_errors() == (0, 0)
    assert torch.equal(a, b)


@pytest.mark.parametrize("name,B", [("decode", None), ("tiny", None), ("decode", 8), ("decode", 40), ("longctx", None)])
def test_topk_attention_one_call_matches_two(name, B):
    """dsv4sa_topk_sparse_attn_decode gives the bits of dsv4sa_topk followed by
    dsv4sa_sparse_attn_decode: the same indices in idx_c and the same output and
    lse.  decode (4-CTA clusters) and decode with 8 or 40 queries (8- and
    2-CTA clusters), tiny (16 heads, 8 CTAs), longctx (rows past 16384 entries:
    the two run as separate kernels)."""
    from compressed_sparse_attention_c4_gb300 import dsv4sa as L
    w = W.make(name) if B is None else W.make(name, B=B)
    for fused_window in (False, True):
        a = GpuRun(w, mode=L.ATTN_DECODE)
        b_d = L.upload(w, "cuda", L.ATTN_DECODE)
        b_d.idx_c.fill_(-7)
        L.run_path(b_d, fused_window=fused_window, fused_topk=True)
        torch.cuda.synchronize()
        assert L.dsv4sa_check_errors() == (0, 0)
        ref_out = a.out
        if fused_window:
            L.run_path(a.d, fused_window=True)
            torch.cuda.synchronize()
            ref_out = a.d.out.float().cpu().numpy()
        assert np.array_equal(b_d.idx_c.cpu().numpy(), a.idx_c)
        assert np.array_equal(b_d.out.float().cpu().numpy(), ref_out)
        assert np.array_equal(b_d.lse.cpu().numpy(), a.d.lse.cpu().numpy())
    for t in range(min(w.T, 4)):
        check_row(a, t)
