"""Seeded synthetic workloads for the C4 compressed-sparse-attention path.

This module only draws random numbers and lays them out; it holds none of the
method's arithmetic.  Both the CUDA library (through the binding) and the CPU
oracle consume what it returns, so it imports neither.

Values are drawn in fp32 with ``numpy.random.default_rng(seed)`` and stored in
the cache formats: q in BF16; KV nope in FP8 E4M3 with one fp32 scale per 64
elements, KV rope in BF16; indexer q and keys in E4M3 with one fp32 scale per
64 elements.  The format conversions use torch's own casts (``to(bfloat16)``,
``to(float8_e4m3fn)``), which round to nearest even; a block scale is
max(amax, 1e-4) / 448 and the scaled values are clamped to +-448 before the
cast (the act_quant rules of the DeepSeek-V4 kernel walk-through, §3.4).
This is data preparation: parity compares the library and the oracle on the
same stored codes.

Cache pages are scattered over a pool 1.25x the pages in use, in a random
order; the unused pages are filled with NaN patterns so a stray read shows up
as NaN in a result.

Workloads (shapes and distributions, by name):

* ``tiny``     B=1 decode, L=4096 -> N=1024, H=16, Hi=4, q/kv/iq/ik ~ N(0,1)/sqrt(dim)
* ``decode``   B=32 decode, L=65536 -> N=16384, H=64, Hi=64, q ~ N(0,1)/sqrt(512),
               kv ~ N(0,1), iq/ik ~ N(0,1)/sqrt(128)
* ``prefill``  B=1, T=4096 queries at positions 61440..65535 of 65536, causal,
               H=64, Hi=64, distributions of ``tiny``
* ``longctx``  B=4 decode, L=1048576 -> N=262144, H=64, Hi=64, kv and keys ~ N(0,1)
               with the same random 1% of entries scaled x8 in both pools
* ``ragged``   B=128 decode, L ~ lognormal(ln 8192, 1) clipped to [64, 131072],
               H=8, even rows C4 (top-k over N=L/4), odd rows C128 (all N=L/128
               entries), 5% of rows with every index -1

Common: w ~ U(0,1)/2, attn_sink ~ N(0,1), softmax scale 1/sqrt(512), window 128.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

PAGE = 64
NOPE = 448
ROPE = 64
HEAD_DIM = 512
IDX_DIM = 128
WINDOW = 128
TOPK = 512

SEEDS = {"tiny": 1001, "decode": 1002, "prefill": 1003, "longctx": 1004, "ragged": 1005}
NAMES = ("tiny", "decode", "prefill", "longctx", "ragged")


# ---------------------------------------------------------------------------
# format conversions (library casts; data preparation)
# ---------------------------------------------------------------------------

def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def quant_e4m3_blocks(x: np.ndarray, block: int = 64):
    """fp32 [..., D] -> (E4M3 codes uint8 [..., D], fp32 scales [..., D/block])."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    shp = x.shape
    xb = torch.from_numpy(x).reshape(*shp[:-1], shp[-1] // block, block)
    amax = xb.abs().amax(dim=-1).clamp_min(1e-4)
    scale = amax / 448.0
    y = (xb / scale.unsqueeze(-1)).clamp(-448.0, 448.0)
    codes = y.to(torch.float8_e4m3fn).view(torch.uint8).reshape(shp)
    return codes.numpy(), scale.numpy().astype(np.float32)


# ---------------------------------------------------------------------------
# pools
# ---------------------------------------------------------------------------

def _normal(rng, shape, std):
    return (rng.standard_normal(size=shape, dtype=np.float32) * np.float32(std))


def _poison_kv(n_pages):
    return {
        "nope_codes": np.full((n_pages, PAGE, NOPE), 0x7F, np.uint8),
        "nope_scale": np.full((n_pages, PAGE, NOPE // 64), np.nan, np.float32),
        "rope_bits": np.full((n_pages, PAGE, ROPE), 0x7FC0, np.uint16),
    }


def _poison_keys(n_pages):
    return {
        "codes": np.full((n_pages, PAGE, IDX_DIM), 0x7F, np.uint8),
        "scale": np.full((n_pages, PAGE, 2), np.nan, np.float32),
    }


def _fill_kv(pool, phys_pages, rng, std, heavy_mask=None, chunk=1024):
    """Draw KV rows for the given physical pages (iid, so page order is free)."""
    for i in range(0, len(phys_pages), chunk):
        pages = phys_pages[i:i + chunk]
        x = _normal(rng, (len(pages), PAGE, HEAD_DIM), std)
        if heavy_mask is not None:
            x *= np.where(heavy_mask[pages], np.float32(8.0), np.float32(1.0))[..., None]
        codes, scale = quant_e4m3_blocks(x[..., :NOPE])
        pool["nope_codes"][pages] = codes
        pool["nope_scale"][pages] = scale
        pool["rope_bits"][pages] = to_bf16_bits(x[..., NOPE:])


def _fill_keys(pool, phys_pages, rng, std, heavy_mask=None, chunk=4096):
    for i in range(0, len(phys_pages), chunk):
        pages = phys_pages[i:i + chunk]
        x = _normal(rng, (len(pages), PAGE, IDX_DIM), std)
        if heavy_mask is not None:
            x *= np.where(heavy_mask[pages], np.float32(8.0), np.float32(1.0))[..., None]
        codes, scale = quant_e4m3_blocks(x)
        pool["codes"][pages] = codes
        pool["scale"][pages] = scale


def _page_tables(rng, pages_per_seq, total_pages):
    """Scatter each sequence's logical pages over a shuffled pool of total_pages.
    Returns (page_table [B, max_pages] int32, used physical pages)."""
    B = len(pages_per_seq)
    width = max(1, int(max(pages_per_seq)))
    perm = rng.permutation(total_pages).astype(np.int32)
    pt = np.zeros((B, width), dtype=np.int32)
    used = []
    off = 0
    unused = perm[int(sum(pages_per_seq)):]
    filler = int(unused[0]) if len(unused) else int(perm[0])
    for b, n in enumerate(pages_per_seq):
        n = int(n)
        pt[b, :n] = perm[off:off + n]
        pt[b, n:] = filler          # valid page id that is never referenced (poisoned)
        used.append(perm[off:off + n])
        off += n
    return pt, (np.concatenate(used) if used else np.zeros(0, np.int32))


@dataclass
class Workload:
    name: str
    B: int
    T: int
    H: int
    Hi: int
    k: int
    kc: int
    kw: int
    softmax_scale: float
    q: np.ndarray            # uint16 [T, H, 512] bf16 bits
    q_idx: np.ndarray        # uint8  [T, Hi, 128]
    q_idx_scale: np.ndarray  # f32    [T, Hi, 2]
    w: np.ndarray            # f32    [T, Hi]
    sink: np.ndarray         # f32    [H]
    comp_pool: dict
    key_pool: dict
    comp_pt: np.ndarray      # int32 [B, P]
    win_pool: dict
    win_pt: np.ndarray       # int32 [B, Pw]
    win_ring: int            # >0: window indices are ring slots
    q_seq: np.ndarray        # int32 [T]
    pos: np.ndarray          # int32 [T]  0-based raw position of the query token (-1: none)
    n_vis: np.ndarray        # int32 [T]
    c128: np.ndarray         # bool [T]: row takes all entries, no indexer
    n_max: int
    meta: dict = field(default_factory=dict)

    def as_dict(self) -> dict:
        return dict(q=self.q, q_idx=self.q_idx, q_idx_scale=self.q_idx_scale, w=self.w,
                    sink=self.sink, softmax_scale=self.softmax_scale, comp_pool=self.comp_pool,
                    key_pool=self.key_pool, comp_pt=self.comp_pt, win_pool=self.win_pool,
                    win_pt=self.win_pt, win_ring=self.win_ring, kw=self.kw, q_seq=self.q_seq,
                    n_vis=self.n_vis, pos=self.pos, c128=self.c128, kc=self.kc)


def _queries(rng, T, H, Hi, q_std, iq_std, q_mult):
    q = to_bf16_bits(_normal(rng, (T, H, HEAD_DIM), q_std) * np.float32(q_mult))
    qi, qs = quant_e4m3_blocks(_normal(rng, (T, Hi, IDX_DIM), iq_std))
    w = (rng.random((T, Hi), dtype=np.float32) * np.float32(0.5)).astype(np.float32)
    return q, qi, qs, w


def make_decode_like(name, B, L, H, Hi, kv_std, key_std, q_std=1 / math.sqrt(512),
                     iq_std=1 / math.sqrt(128), heavy=0.0, c128_rows=None, empty_rows=None,
                     seed=None, q_mult=1.0, k=TOPK):
    """B sequences with one decode query each (the last token of each sequence)."""
    rng = np.random.default_rng(SEEDS.get(name, 1000) if seed is None else seed)
    L = np.asarray(L, dtype=np.int64).reshape(-1)
    if L.size == 1:
        L = np.full(B, int(L[0]), np.int64)
    T = B
    c128 = np.zeros(T, bool) if c128_rows is None else np.asarray(c128_rows, bool)
    ratio = np.where(c128, 128, 4)
    N = (L // ratio).astype(np.int64)
    pages = (N + PAGE - 1) // PAGE
    total = max(1, int(math.ceil(1.25 * max(1, pages.sum()))))
    comp_pt, used = _page_tables(rng, pages, total)
    heavy_mask = None
    if heavy > 0:
        heavy_mask = rng.random((total, PAGE)) < heavy
    comp_pool = _poison_kv(total)
    key_pool = _poison_keys(total)
    _fill_kv(comp_pool, used, rng, kv_std, heavy_mask)
    _fill_keys(key_pool, used, rng, key_std, heavy_mask)
    # window: ring of 128 raw-token slots (2 pages) per sequence
    wtotal = max(1, int(math.ceil(1.25 * 2 * B)))
    win_pt, wused = _page_tables(rng, np.full(B, 2), wtotal)
    win_pool = _poison_kv(wtotal)
    _fill_kv(win_pool, wused, rng, kv_std)
    q, qi, qs, w = _queries(rng, T, H, Hi, q_std, iq_std, q_mult)
    sink = rng.standard_normal(H).astype(np.float32)
    pos = (L - 1).astype(np.int32)
    n_vis = N.astype(np.int32)
    if empty_rows is not None:
        empty = np.asarray(empty_rows, bool)
        n_vis = np.where(empty, 0, n_vis).astype(np.int32)
        pos = np.where(empty, -1, pos).astype(np.int32)   # no raw token visible either
    kc = k if not c128.any() else max(k, int(N[c128].max(initial=0)))
    return Workload(name=name, B=B, T=T, H=H, Hi=Hi, k=k, kc=kc, kw=WINDOW,
                    softmax_scale=1.0 / math.sqrt(HEAD_DIM), q=q, q_idx=qi, q_idx_scale=qs,
                    w=w, sink=sink, comp_pool=comp_pool, key_pool=key_pool, comp_pt=comp_pt,
                    win_pool=win_pool, win_pt=win_pt, win_ring=2 * PAGE,
                    q_seq=np.arange(T, dtype=np.int32), pos=pos, n_vis=n_vis, c128=c128, n_max=int(max(1, n_vis.max(initial=0))),
                    meta=dict(L=L.tolist() if B <= 256 else None))


def make_prefill(name="prefill", L=65536, T=4096, H=64, Hi=64, seed=None, q_mult=1.0, k=TOPK):
    """One sequence; T query tokens at the last T positions; causal visibility."""
    rng = np.random.default_rng(SEEDS.get(name, 1000) if seed is None else seed)
    std = 1.0 / math.sqrt(HEAD_DIM)
    N = L // 4
    pages = (N + PAGE - 1) // PAGE
    total = int(math.ceil(1.25 * pages))
    comp_pt, used = _page_tables(rng, [pages], total)
    comp_pool = _poison_kv(total)
    key_pool = _poison_keys(total)
    _fill_kv(comp_pool, used, rng, std)
    _fill_keys(key_pool, used, rng, 1.0 / math.sqrt(IDX_DIM))
    pos = np.arange(L - T, L, dtype=np.int64)
    # window pool: raw tokens from the first window position of the chunk on
    first = max(0, int(pos[0]) - (WINDOW - 1))
    p0, p1 = first // PAGE, (L - 1) // PAGE
    wpages = p1 + 1
    wtotal = int(math.ceil(1.25 * (p1 - p0 + 1))) + 1
    perm = rng.permutation(wtotal).astype(np.int32)
    win_pt = np.full((1, wpages), perm[-1], np.int32)        # unreferenced -> poisoned page
    win_pt[0, p0:p1 + 1] = perm[:p1 - p0 + 1]
    win_pool = _poison_kv(wtotal)
    _fill_kv(win_pool, perm[:p1 - p0 + 1], rng, std)
    q, qi, qs, w = _queries(rng, T, H, Hi, std, 1.0 / math.sqrt(IDX_DIM), q_mult)
    sink = rng.standard_normal(H).astype(np.float32)
    n_vis = ((pos + 1) // 4).astype(np.int32)
    return Workload(name=name, B=1, T=T, H=H, Hi=Hi, k=k, kc=k, kw=WINDOW,
                    softmax_scale=1.0 / math.sqrt(HEAD_DIM), q=q, q_idx=qi, q_idx_scale=qs,
                    w=w, sink=sink, comp_pool=comp_pool, key_pool=key_pool, comp_pt=comp_pt,
                    win_pool=win_pool, win_pt=win_pt, win_ring=0,
                    q_seq=np.zeros(T, np.int32), pos=pos.astype(np.int32), n_vis=n_vis,
                    c128=np.zeros(T, bool), n_max=int(N),
                    meta=dict(L=L))


def make(name: str, seed=None, q_mult=1.0, **kw) -> Workload:
    """Build one of the named workloads (see module docstring)."""
    if name == "tiny":
        s = 1.0 / math.sqrt(HEAD_DIM)
        return make_decode_like("tiny", B=1, L=4096, H=16, Hi=4, kv_std=s,
                                key_std=1 / math.sqrt(IDX_DIM), seed=seed, q_mult=q_mult, **kw)
    if name == "decode":
        return make_decode_like("decode", B=kw.pop("B", 32), L=kw.pop("L", 65536), H=64, Hi=64,
                                kv_std=1.0, key_std=1 / math.sqrt(IDX_DIM), seed=seed,
                                q_mult=q_mult, **kw)
    if name == "prefill":
        return make_prefill(seed=seed, q_mult=q_mult, **kw)
    if name == "longctx":
        return make_decode_like("longctx", B=kw.pop("B", 4), L=kw.pop("L", 1 << 20), H=64,
                                Hi=64, kv_std=1.0, key_std=1.0, heavy=0.01, seed=seed,
                                q_mult=q_mult, **kw)
    if name == "ragged":
        rng = np.random.default_rng((SEEDS["ragged"] if seed is None else seed) + 7)
        B = kw.pop("B", 128)
        L = np.clip(np.exp(rng.normal(math.log(8192), 1.0, size=B)), 64, 131072).astype(np.int64)
        c128 = (np.arange(B) % 2) == 1
        empty = rng.random(B) < 0.05
        return make_decode_like("ragged", B=B, L=L, H=8, Hi=64, kv_std=1.0,
                                key_std=1 / math.sqrt(IDX_DIM), c128_rows=c128,
                                empty_rows=empty, seed=seed, q_mult=q_mult, **kw)
    raise ValueError(f"unknown workload {name!r}")


# ---------------------------------------------------------------------------
# FP4 indexer inputs (E2M1 codes with E8M0 block exponents, drawn directly)
# ---------------------------------------------------------------------------

@dataclass
class Fp4IndexerWorkload:
    """Inputs of the FP4 indexer: an IDXK_FP4 pool (logical codes, one per
    byte, [P, 64, 128]; E8M0 bytes [P, 64, 4]), page tables, FP4 queries
    (codes [T, Hi, 128], E8M0 [T, Hi, 4]) and head weights."""
    name: str
    T: int
    Hi: int
    key_codes: np.ndarray
    key_e8m0: np.ndarray
    comp_pt: np.ndarray
    q_codes: np.ndarray
    q_e8m0: np.ndarray
    w: np.ndarray
    q_seq: np.ndarray
    n_vis: np.ndarray
    n_max: int


def make_fp4_indexer(name="fp4", B=3, L=(6000, 9000, 20000), Hi=8, seed=2001, e_lo=122, e_hi=130):
    """B sequences with one decode query each; N = L // 4 visible entries.
    Codes are uniform over the 16 E2M1 patterns, exponents uniform in
    [e_lo, e_hi]; pages not referenced by any table hold E8M0 0xFF (NaN)."""
    rng = np.random.default_rng(seed)
    L = np.asarray(L, dtype=np.int64).reshape(-1)
    if L.size == 1:
        L = np.full(B, int(L[0]), np.int64)
    N = (L // 4).astype(np.int64)
    pages = (N + PAGE - 1) // PAGE
    total = max(1, int(math.ceil(1.25 * max(1, pages.sum()))))
    comp_pt, used = _page_tables(rng, pages, total)
    codes = rng.integers(0, 16, size=(total, PAGE, IDX_DIM), dtype=np.uint8)
    e8 = np.full((total, PAGE, IDX_DIM // 32), 0xFF, np.uint8)
    e8[used] = rng.integers(e_lo, e_hi + 1, size=(len(used), PAGE, IDX_DIM // 32)).astype(np.uint8)
    q_codes = rng.integers(0, 16, size=(B, Hi, IDX_DIM), dtype=np.uint8)
    q_e8 = rng.integers(e_lo, e_hi + 1, size=(B, Hi, IDX_DIM // 32)).astype(np.uint8)
    w = (rng.random((B, Hi)) * 0.5).astype(np.float32)
    return Fp4IndexerWorkload(name=name, T=B, Hi=Hi, key_codes=codes, key_e8m0=e8, comp_pt=comp_pt, q_codes=q_codes,
                              q_e8m0=q_e8, w=w, q_seq=np.arange(B, dtype=np.int32), n_vis=N.astype(np.int32),
                              n_max=int(max(1, N.max(initial=0))))
