"""Sequence-sharded long-context decode across ranks: the host-side steps.

A 1M-token context has N = 262144 C4 entries; its pages can be spread over R
GPUs, each holding a contiguous, page-aligned range of entries (its part of the
KV and indexer-key pools).  One decode step then runs ("DeepSeek-V4 in SGLang"
MQALayer / attention tensor parallelism; the top-512 of 算法2 over a sharded
cache):

1. every rank scores its own entries (dsv4sa_indexer_logits on its pool shard)
   and selects its exact local top-k (dsv4sa_topk): every member of the global
   top-k is in the top-k of the rank that holds it, under the same order;
2. the ranks exchange their candidates, (score, global entry index) pairs, with
   one all-gather;
3. every rank selects the global top-k from the R k candidates
   (``merge_candidates``: score descending, NaN lowest, -0 equal to +0, the
   lower entry index first among equal scores, output in ascending index
   order) -- the same selection as one GPU's top-k over the whole row;
4. each rank attends over the selected entries it holds (plus, on rank 0, the
   raw window), with the sink left out (attn_sink = -inf): a partial output
   o_r normalised over its own rows and its log-sum-exp lse_r;
5. the partials are combined with the sink added once (``lse_combine``):
   M = max(max_r lse_r, sink), o = sum_r e^(lse_r - M) o_r / (sum_r e^(lse_r - M)
   + e^(sink - M)), lse = M + log(that denominator).

This module holds steps 2, 3 and 5 (tensor operations on any device, and the
collectives); steps 1 and 4 are the library's kernels on each rank's shard.
"""
from __future__ import annotations

import math

import torch


def shard_ranges(n_entries: int, world: int, page: int = 64) -> list[tuple[int, int]]:
    """Contiguous, page-aligned entry ranges [lo, hi) of ranks 0..world-1."""
    pages = (n_entries + page - 1) // page
    out = []
    for r in range(world):
        p0, p1 = pages * r // world, pages * (r + 1) // world
        out.append((min(n_entries, p0 * page), min(n_entries, p1 * page)))
    return out


def merge_candidates(scores: torch.Tensor, idx: torch.Tensor, k: int) -> torch.Tensor:
    """Global top-k from candidates: scores [T, M] (float), idx [T, M] (int,
    global entry index, -1 for none).  Returns int32 [T, k]: the k candidates
    with the largest score (NaN lowest, -0 == +0, the lower entry index first
    among equal scores), in ascending entry-index order, -1 padded."""
    s = scores.to(torch.float64) + 0.0        # -0 -> +0
    ix = idx.to(torch.int64)
    valid = ix >= 0
    nan = torch.isnan(s) & valid
    cls = torch.where(valid, torch.where(nan, 1, 2), 0)      # numbers, then NaNs, then nothing
    val = torch.where(valid & ~nan, s, torch.zeros_like(s))
    big = torch.iinfo(torch.int64).max
    # three stable sorts: index ascending, then score descending, then class descending
    o = torch.sort(torch.where(valid, ix, big), dim=1, stable=True).indices
    o = o.gather(1, torch.sort(val.gather(1, o), dim=1, descending=True, stable=True).indices)
    o = o.gather(1, torch.sort(cls.gather(1, o), dim=1, descending=True, stable=True).indices)
    top = o[:, :k]
    sel = torch.where(cls.gather(1, top) > 0, ix.gather(1, top), torch.full_like(top, big))
    sel = torch.sort(sel, dim=1).values
    out = torch.where(sel == big, torch.full_like(sel, -1), sel)
    if out.shape[1] < k:
        out = torch.cat([out, torch.full((out.shape[0], k - out.shape[1]), -1, dtype=out.dtype,
                                         device=out.device)], dim=1)
    return out.to(torch.int32)


def lse_combine(o_parts: torch.Tensor, lse_parts: torch.Tensor, sink: torch.Tensor):
    """o_parts [R, T, H, D] (each normalised over its own rows), lse_parts
    [R, T, H] (-inf for a rank with no rows), sink [H] -> (o [T, H, D],
    lse [T, H]) with the sink counted once.  An all-empty row with sink = -inf
    gives zeros and lse = -inf."""
    o_parts = o_parts.to(torch.float64)
    lse_parts = lse_parts.to(torch.float64)
    sk = sink.to(torch.float64).view(1, -1).expand_as(lse_parts[0])
    M = torch.maximum(lse_parts.max(dim=0).values, sk)
    finite = torch.isfinite(M)
    Ms = torch.where(finite, M, torch.zeros_like(M))
    a = torch.where(torch.isfinite(lse_parts), torch.exp(lse_parts - Ms), torch.zeros_like(lse_parts))
    a_s = torch.where(torch.isfinite(sk), torch.exp(sk - Ms), torch.zeros_like(sk))
    den = a.sum(dim=0) + a_s
    num = (a.unsqueeze(-1) * o_parts).sum(dim=0)
    ok = finite & (den > 0)
    o = torch.where(ok.unsqueeze(-1), num / torch.where(ok, den, torch.ones_like(den)).unsqueeze(-1),
                    torch.zeros_like(num))
    lse = torch.where(ok, Ms + torch.log(torch.where(ok, den, torch.ones_like(den))),
                      torch.full_like(Ms, -math.inf))
    return o, lse


def gather_candidates(scores: torch.Tensor, idx: torch.Tensor, group=None):
    """Step 2: all-gather every rank's [T, k] candidates -> [T, R k], rank-major."""
    import torch.distributed as dist
    world = dist.get_world_size(group)
    s_all = [torch.empty_like(scores) for _ in range(world)]
    i_all = [torch.empty_like(idx) for _ in range(world)]
    dist.all_gather(s_all, scores.contiguous(), group=group)
    dist.all_gather(i_all, idx.contiguous(), group=group)
    return torch.cat(s_all, dim=1), torch.cat(i_all, dim=1)


def combine_partials(o: torch.Tensor, lse: torch.Tensor, sink: torch.Tensor, group=None):
    """Step 5: all-gather the partials (o [T, H, D], lse [T, H]) and combine them."""
    import torch.distributed as dist
    world = dist.get_world_size(group)
    o_all = [torch.empty_like(o) for _ in range(world)]
    l_all = [torch.empty_like(lse) for _ in range(world)]
    dist.all_gather(o_all, o.contiguous(), group=group)
    dist.all_gather(l_all, lse.contiguous(), group=group)
    return lse_combine(torch.stack(o_all), torch.stack(l_all), sink)
