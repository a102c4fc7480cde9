"""The sequence-sharded long-context decode's host steps
(compressed_sparse_attention_c4_gb300.sharded) on CPU.

* merge_candidates against the oracle's top-k rule on candidate sets with
  ties, NaN and signed zeros;
* lse_combine against one softmax over the union of the rows;
* two gloo ranks, each holding half of two long sequences' entries: local top-k
  on each shard (the oracle stands in for the library's kernels on the rank's
  GPU), all-gather of (score, index), global merge -- equal to the top-k over
  the whole row -- then per-rank attention partials over the entries each rank
  holds (window on rank 0) combined with the sink added once, against the
  oracle's attention over the whole selection.
"""
import math
import os
import socket

import numpy as np
import pytest
import torch

import oracle
from compressed_sparse_attention_c4_gb300 import sharded as S
from compressed_sparse_attention_c4_gb300 import workloads as W


def test_shard_ranges_cover_page_aligned():
    for n, world in [(10000, 2), (7500, 3), (64, 4), (262144, 8)]:
        r = S.shard_ranges(n, world)
        assert r[0][0] == 0 and r[-1][1] == n
        for (a, b), (c, d) in zip(r, r[1:]):
            assert b == c and a % 64 == 0
        assert all(b >= a for a, b in r)


def test_merge_candidates_matches_topk_rule():
    rng = np.random.default_rng(5)
    for trial in range(40):
        n, k, R = int(rng.integers(20, 300)), int(rng.integers(1, 40)), int(rng.integers(1, 5))
        s = rng.normal(size=n)
        if trial % 3 == 0:
            s = np.round(s * 2) / 2                          # heavy ties
        if trial % 4 == 1:
            s[rng.integers(0, n, 5)] = np.nan
        if trial % 5 == 2:
            s[rng.integers(0, n, 6)] = 0.0
            s[rng.integers(0, n, 6)] = -0.0
        ref = oracle.topk_row(s, k)
        # split into R contiguous shards, each sends its own top-k (global indices)
        cuts = np.linspace(0, n, R + 1).astype(int)
        sc, ix = [], []
        for a, b in zip(cuts, cuts[1:]):
            loc = oracle.topk_row(s[a:b], k)
            loc = loc[loc >= 0]
            sc.append(np.concatenate([s[a:b][loc], np.zeros(k - loc.size)]))
            ix.append(np.concatenate([loc + a, -np.ones(k - loc.size, np.int64)]))
        got = S.merge_candidates(torch.tensor(np.concatenate(sc))[None], torch.tensor(np.concatenate(ix))[None], k)
        assert np.array_equal(got[0].numpy(), ref), (trial, got[0].numpy(), ref)


def _lse(q, rows, scale):
    if rows.shape[0] == 0:
        return np.full(q.shape[0], -np.inf)
    a = scale * (q @ rows.T)
    m = a.max(axis=1)
    return m + np.log(np.exp(a - m[:, None]).sum(axis=1))


def test_lse_combine_equals_one_softmax():
    rng = np.random.default_rng(9)
    H, D = 4, 512
    q = rng.normal(size=(H, D)) / math.sqrt(D)
    rows = rng.normal(size=(30, D))
    sink = rng.normal(size=H)
    ref = oracle.sink_softmax_attention(q, rows, sink, 1.0)
    parts = [rows[:7], rows[7:7], rows[7:30]]               # one empty part
    o = np.stack([oracle.sink_softmax_attention(q, p, np.full(H, -np.inf), 1.0) for p in parts])
    lse = np.stack([_lse(q, p, 1.0) for p in parts])
    got, glse = S.lse_combine(torch.tensor(o)[:, None], torch.tensor(lse)[:, None], torch.tensor(sink))
    assert np.allclose(got[0].numpy(), ref, rtol=1e-12, atol=1e-12)
    full_lse = np.logaddexp(_lse(q, rows, 1.0), sink)
    assert np.allclose(glse[0].numpy(), full_lse, rtol=1e-12, atol=1e-12)
    # every part empty, sink -inf: zeros and lse -inf
    z, zl = S.lse_combine(torch.zeros(2, 1, H, D), torch.full((2, 1, H), -math.inf), torch.full((H,), -math.inf))
    assert (z == 0).all() and torch.isneginf(zl).all()


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w = W.make_decode_like("shard", B=2, L=[40000, 30000], H=8, Hi=4, kv_std=1.0, key_std=1 / math.sqrt(128),
                           seed=4242)
    k = w.k
    res = []
    for t in range(w.T):
        s = int(w.q_seq[t])
        n = int(w.n_vis[t])
        lo, hi = S.shard_ranges(n, world)[rank]
        scores = oracle.indexer_logits_row(w.q_idx[t], w.q_idx_scale[t], w.w[t], w.key_pool, w.comp_pt[s], n)
        # 1. this rank's exact top-k over the entries it holds
        loc = oracle.topk_row(scores[lo:hi], k)
        loc = loc[loc >= 0].astype(np.int64)
        cs = np.zeros(k)
        ci = -np.ones(k, np.int64)
        cs[:loc.size] = scores[lo:hi][loc]
        ci[:loc.size] = loc + lo
        # 2, 3. all-gather and global merge
        gs, gi = S.gather_candidates(torch.tensor(cs)[None], torch.tensor(ci)[None])
        idx = S.merge_candidates(gs, gi, k)[0].numpy()
        # 4. the partial over the selected entries this rank holds (+ the window on rank 0), no sink
        mine = idx[(idx >= lo) & (idx < hi)]
        idx_w = oracle.window_indices(int(w.pos[t]), w.kw, w.win_ring) if rank == 0 else np.full(w.kw, -1)
        rows = oracle.gather_rows(mine, w.comp_pool, w.comp_pt[s], idx_w, w.win_pool, w.win_pt[s])
        qv = oracle.bf16_decode(w.q[t])
        o_r = oracle.sink_softmax_attention(qv, rows, np.full(w.H, -np.inf), w.softmax_scale)
        lse_r = _lse(qv, rows, w.softmax_scale)
        # 5. combine with the sink once
        o, lse = S.combine_partials(torch.tensor(o_r)[None], torch.tensor(lse_r)[None], torch.tensor(w.sink))
        res.append((idx, o[0].numpy(), lse[0].numpy()))
    q.put((rank, res))
    dist.destroy_process_group()


@pytest.mark.timeout(600)
def test_two_rank_sharded_decode_matches_single():
    world = 2
    port = _free_port()
    ctx = torch.multiprocessing.get_context("spawn")
    qq = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, qq)) for r in range(world)]
    for p in procs:
        p.start()
    got = dict(qq.get(timeout=540) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    w = W.make_decode_like("shard", B=2, L=[40000, 30000], H=8, Hi=4, kv_std=1.0, key_std=1 / math.sqrt(128),
                           seed=4242)
    for t in range(w.T):
        s = int(w.q_seq[t])
        n = int(w.n_vis[t])
        scores = oracle.indexer_logits_row(w.q_idx[t], w.q_idx_scale[t], w.w[t], w.key_pool, w.comp_pt[s], n)
        idx = oracle.topk_row(scores, w.k)
        idx_w = oracle.window_indices(int(w.pos[t]), w.kw, w.win_ring)
        ref = oracle.sparse_attn_row(w.q[t], w.sink, w.softmax_scale, idx, w.comp_pool, w.comp_pt[s], idx_w,
                                     w.win_pool, w.win_pt[s])
        rows = oracle.gather_rows(idx, w.comp_pool, w.comp_pt[s], idx_w, w.win_pool, w.win_pt[s])
        ref_lse = np.logaddexp(_lse(oracle.bf16_decode(w.q[t]), rows, w.softmax_scale), w.sink)
        for rank in range(world):
            gidx, o, lse = got[rank][t]
            assert np.array_equal(gidx, idx)                 # the global top-k of the whole row
            assert np.allclose(o, ref, rtol=1e-10, atol=1e-12)
            assert np.allclose(lse, ref_lse, rtol=1e-12, atol=1e-12)
