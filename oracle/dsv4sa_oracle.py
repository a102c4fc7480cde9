"""fp64 CPU oracle for the C4 compressed-sparse-attention hot path.

TEST INFRASTRUCTURE ONLY.  This module is the plain, slow, obviously correct
definition that the CUDA library is checked against.  Only ``tests/``,
``__graft_entry__.smoke()`` and the ``cpu_baseline`` / ``--impl reference`` legs
of ``bench.py`` may import it.  It shares no code, table or constant with the
CUDA path (``compressed_sparse_attention_c4_gb300``) and imports nothing from it.

Sources (cited by page title and section):

* P1 = "DeepSeek-V4 全面解读：架构设计与 inference/encoding 源码深度解析"
  (wangjunjian.com), §2.5 RMSNorm, §2.6 RoPE 位置编码, §2.8 KV Cache 索引辅助函数, §2.9 Compressor,
  §2.10 Indexer, §2.11 Attention,
  §3.2 数据类型别名, §3.7 sparse_attn_kernel.
* P2 = "DeepSeek-V4 in SGLang 深度理解分析", 概念2 分层压缩, 概念3 C4 Indexer, MQALayer, 算法3 在线压缩,
  概念5 DeepSeekV4TokenToKVPool, 算法2 Paged MQA Logits + TopK.
* P3 = "tilelang量化内核拆解DeepSeek-V4.1-Flash-NVFP4的fp4_gemm与sparse_attn实现",
  section "sparse_attn 实现拆解".

The oracle works on the *logical* cache arrays (page-structured numpy arrays),
not on the library's packed byte layout:

* compressed / window KV pool: ``nope_codes`` uint8 [P, 64, 448] (E4M3 codes),
  ``nope_scale`` float32 [P, 64, 7] (one scale per 64 nope elements),
  ``rope_bits`` uint16 [P, 64, 64] (BF16 bit patterns).  (P2 概念5: nope in FP8
  with a per-block scale, rope in BF16; P1 §2.2: head_dim 512, rope 64.)
* indexer-key pool: ``codes`` uint8 [P, 64, 128], ``scale`` float32 [P, 64, 2].

Entry ``s`` of a sequence lives at slot ``s % 64`` of page ``page_table[seq][s // 64]``.

Every function below states the passage it follows.  All arithmetic is fp64.
Readings of points the pages leave open are listed in the docstrings:

* attention: the result is the sink-softmax over the multiset of valid indices,
  evaluated stably by subtracting max(scores, sink).  With no valid index the
  result is exactly zero (P3: running max starts at -1e30 so an all-(-1) row
  outputs zeros).
* top-k: ties at the threshold go to the lower entry index; output ascending;
  padded with -1; fewer than k visible entries -> all of them (P2 算法2 退化场景).

Parity status: every public function here (the KV-cache writer, the inverse rotary
embedding of the output and the KV compressor included) is pinned by tests in
``tests/test_oracle_pins.py`` against values or routines that do not come from
this module (torch's FP8/BF16 decoders, brute-force loops, scipy softmax,
torch scaled_dot_product_attention, closed forms, invariants).  The FP4 (E2M1 +
E8M0) indexer variant at the end of the module is pinned the same way (hand
codes and ties, the pages' exponent-field rule for the scale, brute-force
loops, equality with the FP8 definition on values both formats hold), and so
is the Hadamard rotation of the compressor's rotate path
(``hadamard_rotate_to_bf16``: the exact rotation rounded once to BF16, pinned
against scipy's Hadamard matrix, torch's BF16 rounding, and fp32 evaluations in
several orders that stay inside ``hadamard_rotate_fp32_bound``).  The
FP4 key writes (plain and rotated) have CUDA counterparts; the FP4 scores
(``indexer_logits_row_fp4``) have none yet.
"""
from __future__ import annotations

import math

import numpy as np

PAGE = 64          # slots per page (P2 概念5 paged pool; 64-token pages)
NOPE = 448         # FP8 part of a KV row (P1 §2.2 head_dim 512 - rope 64)
ROPE = 64          # BF16 part of a KV row (P1 §2.2 rope_head_dim 64)
HEAD_DIM = NOPE + ROPE
SCALE_BLOCK = 64   # elements per FP8 scale
IDX_DIM = 128      # indexer head dim


# ---------------------------------------------------------------------------
# Number formats (P1 §3.2: FP8 = float8_e4m3, BF16 = bfloat16)
# ---------------------------------------------------------------------------

def e4m3_decode(codes) -> np.ndarray:
    """Decode FP8 E4M3 (the 'fn' variant: no infinities) byte codes to fp64.

    From the format definition: 1 sign bit, 4 exponent bits with bias 7,
    3 mantissa bits.  Exponent field 0 is subnormal (2^-6 * m/8).  Exponent 15
    with mantissa 7 is NaN (codes 0x7F and 0xFF); every other code is finite,
    the largest being 448 (0x7E).
    """
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    normal = sign * np.ldexp(1.0 + m / 8.0, (e - 7).astype(np.int64))
    subnormal = sign * np.ldexp(m / 8.0, -6)
    out = np.where(e == 0, subnormal, normal)
    out = np.where((e == 15) & ((c & 7) == 7), np.nan, out)
    return out


def bf16_decode(bits) -> np.ndarray:
    """Decode BF16 bit patterns (uint16) to fp64: they are the top half of an fp32."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


# ---------------------------------------------------------------------------
# Cache rows
# ---------------------------------------------------------------------------

def _locate(page_table_row, entries):
    e = np.asarray(entries, dtype=np.int64)
    pages = np.asarray(page_table_row, dtype=np.int64)[e // PAGE]
    return pages, e % PAGE


def kv_rows(pool: dict, page_table_row, entries) -> np.ndarray:
    """Dequantised KV rows [n, 512] in fp64 for the given entry numbers.

    Row = [e4m3(nope_code[d]) * nope_scale[d // 64] for d < 448] ++ bf16(rope).
    (P2 概念5 NopeFp8RopeBf16Pack; the rope part is the last 64 dims, P1 §2.11
    step 8 applies the inverse RoPE to o[..., -64:].)
    """
    pages, slots = _locate(page_table_row, entries)
    codes = pool["nope_codes"][pages, slots]                 # [n, 448]
    scale = pool["nope_scale"][pages, slots].astype(np.float64)  # [n, 7]
    nope = e4m3_decode(codes) * np.repeat(scale, SCALE_BLOCK, axis=1)
    rope = bf16_decode(pool["rope_bits"][pages, slots])      # [n, 64]
    return np.concatenate([nope, rope], axis=1)


def index_keys(pool: dict, page_table_row, entries) -> np.ndarray:
    """Dequantised indexer keys [n, 128] in fp64: e4m3(code) * scale[d // 64]."""
    pages, slots = _locate(page_table_row, entries)
    codes = pool["codes"][pages, slots]
    scale = pool["scale"][pages, slots].astype(np.float64)
    return e4m3_decode(codes) * np.repeat(scale, SCALE_BLOCK, axis=1)


def index_query(q_codes, q_scale) -> np.ndarray:
    """Dequantised indexer query [Hi, 128] in fp64 (same per-64 block scaling)."""
    return e4m3_decode(q_codes) * np.repeat(np.asarray(q_scale, np.float64), SCALE_BLOCK, axis=-1)


# ---------------------------------------------------------------------------
# Stage 1: indexer logits (P1 §2.10 steps 6-8; P2 算法2)
# ---------------------------------------------------------------------------

def indexer_logits_row(q_codes, q_scale, w, key_pool, page_table_row, n_vis) -> np.ndarray:
    """Index scores I[s] for s < n_vis of one query, fp64 [n_vis].

    I[s] = sum_h w[h] * ReLU( sum_d q[h, d] * k[s, d] )
    P1 §2.10: the score is einsum('bshd,btd->bsht', q, kv) (step 6), ReLU and
    then multiplied by the per-head weights (step 7), summed over heads (step 8).
    ``w`` is taken as the final per-head weight (the softmax_scale * n_heads^-0.5
    factor of step 5 is already folded into it by the caller).
    """
    n = int(n_vis)
    if n <= 0:
        return np.zeros(0, dtype=np.float64)
    q = index_query(q_codes, q_scale)                  # [Hi, 128]
    k = index_keys(key_pool, page_table_row, np.arange(n))  # [n, 128]
    dots = k @ q.T                                      # [n, Hi]
    return np.maximum(dots, 0.0) @ np.asarray(w, np.float64)


def indexer_logits(q_codes, q_scale, w, key_pool, page_table, q_seq, n_vis, rows=None):
    """Index scores for each query row (a list of fp64 arrays of length n_vis[t])."""
    T = len(n_vis)
    rows = range(T) if rows is None else rows
    return {int(t): indexer_logits_row(q_codes[t], q_scale[t], w[t], key_pool,
                                       page_table[q_seq[t]], n_vis[t]) for t in rows}


# ---------------------------------------------------------------------------
# Stage 2: top-k (P1 §2.10 step 9; P2 概念3, 算法2)
# ---------------------------------------------------------------------------

def topk_row(scores, k: int) -> np.ndarray:
    """Top-k entry indices of one query, int32 [k], ascending, -1 padded.

    The k entries with the largest score; among equal scores the lower entry
    index ranks first.  If n_vis <= k every visible entry is taken (P2 算法2:
    below 512 compressed entries no top-k is needed).  The order of the output
    is ascending entry index (attention is order-independent).
    """
    s = np.asarray(scores, dtype=np.float64)
    n = s.shape[0]
    out = np.full(k, -1, dtype=np.int32)
    if n <= k:
        out[:n] = np.arange(n, dtype=np.int32)
        return out
    # exhaustive sort by (score descending, index ascending)
    order = np.lexsort((np.arange(n), -s))   # primary key -s, secondary key index
    sel = np.sort(order[:k].astype(np.int64))
    out[:] = sel.astype(np.int32)
    return out


# ---------------------------------------------------------------------------
# Index assembly (P1 §2.8 get_window_topk_idxs / get_compress_topk_idxs, §2.11 step 4)
# ---------------------------------------------------------------------------

def window_indices(pos: int, window: int = 128, ring: int = 0) -> np.ndarray:
    """Raw-token window of the query at 0-based position ``pos``: positions
    pos-window+1 .. pos (the current token included); positions < 0 -> -1.
    With ``ring`` > 0 the stored index is the slot of a circular buffer of that
    size (position mod ring), as in the decode-time window cache (P1 §2.8).
    """
    p = np.arange(pos - window + 1, pos + 1, dtype=np.int64)
    out = np.where(p < 0, -1, p % ring if ring > 0 else p)
    return out.astype(np.int32)


def compress_indices(n_vis: int, kc: int) -> np.ndarray:
    """All visible compressed entries 0..n_vis-1 then -1 up to kc (no indexer,
    as for the C128 layers; P1 §2.8 get_compress_topk_idxs)."""
    out = np.full(kc, -1, dtype=np.int32)
    n = min(int(n_vis), kc)
    out[:n] = np.arange(n, dtype=np.int32)
    return out


def n_visible(pos: int, ratio: int = 4) -> int:
    """Compressed entries complete at 0-based raw position ``pos``: entry c
    covers raw tokens ratio*c .. ratio*c+ratio-1 (P2 概念2: every 4 tokens become
    one entry), so floor((pos+1)/ratio) entries are visible."""
    return (int(pos) + 1) // ratio


# ---------------------------------------------------------------------------
# Stage 3: sparse attention with attn_sink (P1 §3.7 sparse_attn_kernel; P3 sparse_attn)
# ---------------------------------------------------------------------------

def sink_softmax_attention(q, rows, sink, softmax_scale) -> np.ndarray:
    """o[h] = sum_j e^{a_hj} kv_j / (sum_j e^{a_hj} + e^{sink_h}),  a_hj = scale * q[h].kv_j

    q [H, 512] fp64, rows [n, 512] fp64 (the gathered valid rows; a multiset),
    sink [H].  K and V are the same rows (P2 MQALayer: k=kv, v=kv).  The sink
    adds to the denominator only (P1 §3.7: sum_exp += exp(attn_sink - max)).
    Evaluated stably by subtracting M = max(max_j a_hj, sink_h).  With no rows
    the numerator is empty and the output is exactly 0 (P3: an all -1 row
    yields zeros).
    """
    q = np.asarray(q, np.float64)
    rows = np.asarray(rows, np.float64).reshape(-1, HEAD_DIM)
    sink = np.asarray(sink, np.float64)
    H = q.shape[0]
    out = np.zeros((H, HEAD_DIM), dtype=np.float64)
    if rows.shape[0] == 0:
        return out
    a = softmax_scale * (q @ rows.T)                   # [H, n]
    M = np.maximum(a.max(axis=1), sink)                # [H]
    p = np.exp(a - M[:, None])
    den = p.sum(axis=1) + np.exp(sink - M)
    return (p @ rows) / den[:, None]


def gather_rows(idx_c, comp_pool, comp_pt_row, idx_w, win_pool, win_pt_row) -> np.ndarray:
    """Rows selected by the concatenated index list (compressed ++ window);
    index -1 is an invalid slot and contributes nothing (P1 §2.11 step 4:
    window and compressed indices are concatenated; §3.7: -1 -> not loaded)."""
    parts = []
    ic = np.asarray(idx_c, np.int64)
    ic = ic[ic >= 0]
    if ic.size:
        parts.append(kv_rows(comp_pool, comp_pt_row, ic))
    if idx_w is not None:
        iw = np.asarray(idx_w, np.int64)
        iw = iw[iw >= 0]
        if iw.size:
            parts.append(kv_rows(win_pool, win_pt_row, iw))
    if not parts:
        return np.zeros((0, HEAD_DIM), dtype=np.float64)
    return np.concatenate(parts, axis=0)


def sparse_attn_row(q_bits, sink, softmax_scale, idx_c, comp_pool, comp_pt_row,
                    idx_w=None, win_pool=None, win_pt_row=None) -> np.ndarray:
    """One query token: q given as BF16 bits [H, 512]; returns o [H, 512] fp64."""
    q = bf16_decode(q_bits)
    rows = gather_rows(idx_c, comp_pool, comp_pt_row, idx_w, win_pool, win_pt_row)
    return sink_softmax_attention(q, rows, sink, softmax_scale)


def sparse_attn(q_bits, sink, softmax_scale, idx_c, comp_pool, comp_pt, q_seq,
                idx_w=None, win_pool=None, win_pt=None, rows=None):
    """sparse_attn over query rows ``rows`` (default all): {t: o[t] [H, 512]}."""
    T = q_bits.shape[0]
    rows = range(T) if rows is None else rows
    out = {}
    for t in rows:
        t = int(t)
        s = int(q_seq[t])
        out[t] = sparse_attn_row(
            q_bits[t], sink, softmax_scale, idx_c[t], comp_pool, comp_pt[s],
            None if idx_w is None else idx_w[t], win_pool,
            None if win_pt is None else win_pt[s])
    return out


def decode_step(work: dict, rows=None, k: int = 512):
    """The whole hot path for query rows ``rows``: indexer logits -> top-k ->
    sparse attention over top-k ++ window.  ``work`` holds the logical arrays
    (see module docstring).  Returns (scores, idx_c, out) dicts keyed by row.
    Rows flagged as C128 (``work['c128'][t]``) take all visible entries with no
    indexer (P2 概念2); rows with n_vis <= k take all visible entries.  The
    window list is ``work['idx_w'][t]`` if given, else the window of the query
    position ``work['pos'][t]`` (ring slots when ``work['win_ring']`` > 0).
    """
    T = work["q"].shape[0]
    rows = range(T) if rows is None else rows
    scores, idxc, out = {}, {}, {}
    kc = work.get("kc", k)
    c128 = work.get("c128")
    for t in rows:
        t = int(t)
        s = int(work["q_seq"][t])
        n = int(work["n_vis"][t])
        if c128 is not None and c128[t]:
            ic = compress_indices(n, kc)
        else:
            sc = indexer_logits_row(work["q_idx"][t], work["q_idx_scale"][t], work["w"][t],
                                    work["key_pool"], work["comp_pt"][s], n)
            scores[t] = sc
            ic = np.full(kc, -1, np.int32)
            ic[:k] = topk_row(sc, k)
        idxc[t] = ic
        if "idx_w" in work:
            iw = work["idx_w"][t]
        else:
            iw = window_indices(int(work["pos"][t]), int(work.get("kw", 128)), int(work.get("win_ring", 0)))
        out[t] = sparse_attn_row(work["q"][t], work["sink"], work["softmax_scale"], ic,
                                 work["comp_pool"], work["comp_pt"][s],
                                 iw, work["win_pool"], work["win_pt"][s])
    return scores, idxc, out


SOFTMAX_SCALE_512 = 1.0 / math.sqrt(HEAD_DIM)


# ---------------------------------------------------------------------------
# KV-cache writer (P1 §3.4 act_quant_kernel; P2 概念5 DeepSeekV4TokenToKVPool)
# ---------------------------------------------------------------------------
#
# Quantising a new row into the cache.  The decision "which FP8 code" is taken
# in fp32, the precision the pages' kernel works in (P1 §3.4: FP32 scale,
# absmax per block, amax = max(amax, 1e-4), scale = amax * fp8_max_inv, FP8
# output clamped to [-448, 448]).  Reading of what the pages leave open: the
# value quantised is x / scale (fp32 division), rounded to the nearest E4M3 code
# with ties to the even code; fp8_max_inv is 1/448 rounded to fp32.

FP8_MAX = 448.0
AMAX_FLOOR = 1e-4

_E4M3_FINITE = None   # (values, codes) of every finite code >= 0, ascending


def _e4m3_table():
    global _E4M3_FINITE
    if _E4M3_FINITE is None:
        codes = np.arange(0, 0x7F, dtype=np.uint8)          # 0x00 .. 0x7E: +0 .. 448
        _E4M3_FINITE = (e4m3_decode(codes), codes)
    return _E4M3_FINITE


def e4m3_encode(x) -> np.ndarray:
    """fp32 values in [-448, 448] -> E4M3 codes, round to nearest, ties to the
    even code (the code whose mantissa bit 0 is clear), by search over every
    finite code of the format (P1 §3.2 float8_e4m3).  -0.0 encodes as 0x80."""
    x = np.asarray(x, dtype=np.float32).astype(np.float64)
    vals, codes = _e4m3_table()
    a = np.abs(x)
    if np.any(a > FP8_MAX) or np.any(np.isnan(x)):
        raise ValueError("e4m3_encode expects values in [-448, 448]")
    hi = np.searchsorted(vals, a, side="left")                 # first value >= a
    hi = np.minimum(hi, len(vals) - 1)
    lo = np.maximum(hi - 1, 0)
    d_lo = a - vals[lo]
    d_hi = vals[hi] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & ((codes[hi] & 1) == 0))
    mag = np.where(pick_hi, codes[hi], codes[lo]).astype(np.uint8)
    mag = np.where(a == vals[hi], codes[hi], mag).astype(np.uint8)
    sign = np.signbit(x)
    return np.where(sign, mag | np.uint8(0x80), mag).astype(np.uint8)


def quantize_blocks(x_bf16_bits, block: int = SCALE_BLOCK):
    """One row of BF16 values (bit patterns) -> (E4M3 codes, fp32 scales), one
    scale per `block` consecutive values (P1 §3.4 steps 3-7, in fp32)."""
    x = bf16_decode(x_bf16_bits).astype(np.float32)
    xb = x.reshape(-1, block)
    amax = np.max(np.abs(xb), axis=1).astype(np.float32)
    amax = np.maximum(amax, np.float32(AMAX_FLOOR))
    scale = (amax * np.float32(1.0 / FP8_MAX)).astype(np.float32)
    y = (xb / scale[:, None]).astype(np.float32)
    y = np.clip(y, np.float32(-FP8_MAX), np.float32(FP8_MAX))
    return e4m3_encode(y).reshape(x.shape), scale


def kv_write(pool: dict, page_table_row, entries, kv_bf16_bits) -> None:
    """Write rows into a KV pool in place: entry s goes to slot s % 64 of page
    page_table_row[s // 64]; the 448 nope values become E4M3 codes with one fp32
    scale per 64, the 64 rope values are stored as BF16 unchanged (P2 概念5:
    nope in FP8 with per-block scales, rope in BF16)."""
    pages, slots = _locate(page_table_row, entries)
    for r, (pg, sl) in enumerate(zip(pages, slots)):
        bits = np.asarray(kv_bf16_bits[r], dtype=np.uint16)
        codes, scale = quantize_blocks(bits[:NOPE])
        pool["nope_codes"][pg, sl] = codes
        pool["nope_scale"][pg, sl] = scale
        pool["rope_bits"][pg, sl] = bits[NOPE:]


def key_write(pool: dict, page_table_row, entries, key_bf16_bits) -> None:
    """Write indexer keys in place: 128 values -> E4M3 codes, two fp32 scales."""
    pages, slots = _locate(page_table_row, entries)
    for r, (pg, sl) in enumerate(zip(pages, slots)):
        codes, scale = quantize_blocks(np.asarray(key_bf16_bits[r], dtype=np.uint16))
        pool["codes"][pg, sl] = codes
        pool["scale"][pg, sl] = scale


# ---------------------------------------------------------------- rotary embedding of the output

ROPE_DIM = 64   # the last 64 of the 512 dims carry the rotary part (P1 §2.2 qk_rope_head_dim)


def rope_table(freqs, rows: int) -> np.ndarray:
    """The complex rotation table (P1 §2.6 precompute_freqs_cis, steps 3-4):
    table[p, i] = exp(1j * p * freqs[i]) for positions p < rows, fp64 complex
    [rows, 32].  ``freqs`` are the per-pair angular frequencies: the plain
    1 / base^(2i / 64) of step 1, or any interpolated (YaRN, step 2) variant the
    caller chooses; the rotation below only consumes the table."""
    freqs = np.asarray(freqs, np.float64)
    assert freqs.shape == (ROPE_DIM // 2,)
    ang = np.outer(np.arange(rows, dtype=np.float64), freqs)
    return np.cos(ang) + 1j * np.sin(ang)


def base_freqs(base: float = 10000.0) -> np.ndarray:
    """Step 1 of P1 §2.6 precompute_freqs_cis: 1 / base^(j / 64) for j = 0, 2, .., 62."""
    return 1.0 / (float(base) ** (np.arange(0, ROPE_DIM, 2, dtype=np.float64) / ROPE_DIM))


def _rotate(x, table_rows, conjugate: bool) -> np.ndarray:
    """P1 §2.6 apply_rotary_emb on the last 64 dims of x [..., 512]: the dims are
    taken as 32 complex pairs (x[2i], x[2i + 1]) ("split into complex pairs
    (-1, 2)"), multiplied by the table row, or by its conjugate for the inverse."""
    x = np.array(x, np.float64, copy=True)
    z = x[..., -ROPE_DIM::2] + 1j * x[..., -ROPE_DIM + 1::2]
    r = np.conj(table_rows) if conjugate else table_rows
    z = z * r
    x[..., -ROPE_DIM::2] = z.real
    x[..., -ROPE_DIM + 1::2] = z.imag
    return x


def apply_rope(x, table, pos) -> np.ndarray:
    """Forward rotation of x [T, H, 512] (or [H, 512] with scalar pos) by
    table[pos[t]] (P1 §2.6 apply_rotary_emb, inverse=False)."""
    x = np.asarray(x, np.float64)
    rows = np.asarray(table)[np.asarray(pos)]
    if x.ndim == 3:
        rows = rows[:, None, :]
    return _rotate(x, rows, conjugate=False)


def inverse_rope(o, table, pos) -> np.ndarray:
    """P1 §2.11 step 8 (apply_rotary_emb(o[..., -rd:], freqs_cis, inverse=True));
    P2 MQALayer step 7 (inverse RoPE on the attention output): the last 64 dims
    of o [T, H, 512] (or [H, 512] with scalar pos) rotated by the conjugate of
    table[pos[t]]; the first 448 dims unchanged."""
    o = np.asarray(o, np.float64)
    rows = np.asarray(table)[np.asarray(pos)]
    if o.ndim == 3:
        rows = rows[:, None, :]
    return _rotate(o, rows, conjugate=True)


# ---------------------------------------------------------------- KV compressor (gated pooling)
#
# P1 §2.9 Compressor; P2 概念2 (C4 / C128), 算法3 (online C128), 概念5
# (CompressStatePool).  Readings of what the pages leave open (each stated where used):
#  * the projections wkv / wgate are plain GEMMs of the model: the compressor here
#    starts from their outputs kv, score [tokens, coff * 512] (BF16 bits), coff = 2
#    with overlap (ratio 4), 1 without (ratio 128);
#  * ape [ratio, coff * 512] (fp32) is added to the score of the j-th token of every
#    window before the overlap transform;
#  * overlap transform of window s: slots [0, r) hold the tokens of window s - 1,
#    their first 512 features (the overlapping half; absent for s = 0: kv 0,
#    score -inf); slots [r, 2r) hold the tokens of window s, their last 512
#    features (the normal half, placed directly);
#  * the window's slot scores are softmax-normalised per feature and weight the
#    slot kv; the result is RMS-normalised (P1 §2.5) with weight norm_w and eps,
#    its last 64 dims rotated forward (P1 §2.6) by the table row of position
#    r * s (the window's first raw token); only complete windows are compressed.

COMPRESS_DIM = 512


def rms_norm(x, weight, eps: float) -> np.ndarray:
    """P1 §2.5 RMSNorm: x * rsqrt(mean(x^2) + eps) * weight, over the last axis."""
    x = np.asarray(x, np.float64)
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps) * np.asarray(weight, np.float64)


def _softmax_pool(kv_slots, score_slots) -> np.ndarray:
    """Per feature: softmax over the slots (axis 0) of the scores, weighting the kv.
    Slots with score -inf take no weight."""
    m = np.max(score_slots, axis=0)
    e = np.exp(score_slots - m)
    return (e * kv_slots).sum(axis=0) / e.sum(axis=0)


def compress_windows(kv_bits, score_bits, ape, norm_w, ratio: int, overlap: bool, table,
                     eps: float = 1e-6, first_entry: int = 0) -> np.ndarray:
    """Compressed entries (fp64 [n, 512]) of the complete windows of a token
    sequence (P1 §2.9 forward, prefill steps 1-6).  kv_bits / score_bits: BF16
    bits [tokens, coff * 512]; window s covers tokens [r s, r s + r); with
    ``first_entry`` > 0 the rows start at window ``first_entry`` - 1 (its tokens
    serve only as the previous window of the first compressed one)."""
    d = COMPRESS_DIM
    kv = bf16_decode(kv_bits)
    sc = bf16_decode(score_bits)
    ape = np.asarray(ape, np.float64)
    coff = 2 if overlap else 1
    assert kv.shape[1] == coff * d and sc.shape == kv.shape and ape.shape == (ratio, coff * d)
    start = ratio if (overlap and first_entry > 0) else 0
    n = (kv.shape[0] - start) // ratio
    out = np.zeros((n, d))
    for s in range(n):
        cur = slice(start + ratio * s, start + ratio * s + ratio)
        csc = sc[cur] + ape
        if overlap:
            if start + ratio * s >= ratio:
                prev = slice(start + ratio * s - ratio, start + ratio * s)
                psc = sc[prev] + ape
                kv_slots = np.concatenate([kv[prev, :d], kv[cur, d:]])
                sc_slots = np.concatenate([psc[:, :d], csc[:, d:]])
            else:
                kv_slots = np.concatenate([np.zeros((ratio, d)), kv[cur, d:]])
                sc_slots = np.concatenate([np.full((ratio, d), -np.inf), csc[:, d:]])
        else:
            kv_slots, sc_slots = kv[cur], csc
        c = rms_norm(_softmax_pool(kv_slots, sc_slots), norm_w, eps)
        pos = ratio * (first_entry + s)
        out[s] = apply_rope(c, table, pos)
    return out


def online_c128_init() -> dict:
    """The per-sequence state of online C128 compression (P2 算法3; P2 概念5
    CompressStatePool): running max, sum and weighted kv per feature, and the
    number of tokens of the open window."""
    return {"m": np.full(COMPRESS_DIM, -np.inf), "l": np.zeros(COMPRESS_DIM), "acc": np.zeros(COMPRESS_DIM), "n": 0}


def online_c128_step(state: dict, kv_bits, score_bits, ape, norm_w, table, entry: int, eps: float = 1e-6,
                     ratio: int = 128):
    """Fold one token (kv, score BF16 bits [512]) into the state (P2 算法3: O(1)
    per token, running max / sum).  The token is the state's n-th of window
    ``entry``; ape row n is added to its score.  When the window completes the
    entry (fp64 [512], normalised and rotated as in ``compress_windows``) is
    returned and the state reset; otherwise None."""
    kv = bf16_decode(kv_bits)
    sc = bf16_decode(score_bits) + np.asarray(ape, np.float64)[state["n"]]
    m = np.maximum(state["m"], sc)
    a = np.exp(state["m"] - m)
    b = np.exp(sc - m)
    state["l"] = state["l"] * a + b
    state["acc"] = state["acc"] * a + b * kv
    state["m"] = m
    state["n"] += 1
    if state["n"] < ratio:
        return None
    c = rms_norm(state["acc"] / state["l"], norm_w, eps)
    state.update(online_c128_init())
    return apply_rope(c, table, ratio * entry)


# ---------------------------------------------------------------- FP4 (E2M1) indexer variant
# P1 §3.5 fp4_quant_kernel: blocks of 32 values, fp4_max 6.0, the scale always a
# power of two (§3.3 fast_round_scale: 2 ** ceil(log2(amax * fp4_max_inv))),
# amax floored at 6 * 2^-126; P1 §2.10 step 3 runs the indexer's q through this
# quantisation ("FP4 量化模拟"), and P3 gives the indexer's q and k 32-element
# E8M0 scales.  Logical layout of an FP4 indexer-key pool (the oracle's view):
#   codes uint8 [P, 64, 128] -- one E2M1 code per value in the low 4 bits,
#   e8m0  uint8 [P, 64, 4]   -- the biased exponent of each 32-value block's scale.
# Readings of what the pages leave open: the quotient x / scale is an fp32
# division (exact, the scale being a power of two, unless it underflows), clamped
# to [-6, 6] and rounded to the nearest E2M1 value with ties to the even code
# (mantissa bit clear); fp4_max_inv is 1/6 rounded to fp32.

FP4_BLOCK = 32
FP4_MAX = 6.0
FP4_AMAX_FLOOR = 6.0 * 2.0 ** -126


def e2m1_decode(codes) -> np.ndarray:
    """E2M1 codes -> fp64 (OCP MX FP4: bit 3 sign, bits 2-1 exponent with bias 1,
    bit 0 mantissa; exponent field 0 is subnormal, m * 0.5; no inf or NaN).
    Only the low 4 bits of each code are read."""
    c = np.asarray(codes).astype(np.int64) & 0xF
    e = (c >> 1) & 0x3
    m = (c & 0x1).astype(np.float64)
    mag = np.where(e == 0, 0.5 * m, (1.0 + 0.5 * m) * np.exp2(e.astype(np.float64) - 1.0))
    return np.where(c & 0x8, -mag, mag)


def e8m0_decode(b) -> np.ndarray:
    """E8M0 scale bytes -> fp64 2 ** (b - 127); 0xFF is NaN (OCP MX E8M0)."""
    b = np.asarray(b).astype(np.int64)
    return np.where(b == 0xFF, np.nan, np.exp2(b.astype(np.float64) - 127.0))


def fp4_scale_exponent(amax) -> np.ndarray:
    """The power of two of a block's FP4 scale: ceil(log2(t)) with
    t = fp32(max(amax, 6 * 2^-126) * fp32(1/6)) (P1 §3.5 and §3.3).  t is a
    normal fp32 number, so the fp64 log2 of it lands on the right side of every
    integer and the ceiling is exact."""
    a = np.maximum(np.asarray(amax, np.float32), np.float32(FP4_AMAX_FLOOR))
    t = (a * np.float32(1.0 / FP4_MAX)).astype(np.float32)
    return np.ceil(np.log2(t.astype(np.float64))).astype(np.int64)


_E2M1_MAGS = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])   # codes 0..7


def e2m1_encode(y) -> np.ndarray:
    """fp32 values in [-6, 6] -> E2M1 codes: the nearest magnitude of codes 0..7,
    ties to the even code, sign in bit 3 (-0.0 -> 0x8)."""
    y = np.asarray(y, dtype=np.float32).astype(np.float64)
    a = np.abs(y)
    if np.any(a > FP4_MAX) or np.any(np.isnan(y)):
        raise ValueError("e2m1_encode expects values in [-6, 6]")
    hi = np.minimum(np.searchsorted(_E2M1_MAGS, a, side="left"), 7)
    lo = np.maximum(hi - 1, 0)
    d_lo = a - _E2M1_MAGS[lo]
    d_hi = _E2M1_MAGS[hi] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & ((hi & 1) == 0))
    mag = np.where(pick_hi, hi, lo)
    mag = np.where(a == _E2M1_MAGS[hi], hi, mag)
    return np.where(np.signbit(y), mag | 0x8, mag).astype(np.uint8)


def fp4_quantize(x_bf16_bits):
    """One row of BF16 values (bit patterns, a multiple of 32 of them) -> (E2M1
    codes uint8 [n], E8M0 scale bytes uint8 [n / 32]) (P1 §3.5, in fp32)."""
    x = bf16_decode(x_bf16_bits).astype(np.float32)
    xb = x.reshape(-1, FP4_BLOCK)
    e = fp4_scale_exponent(np.max(np.abs(xb), axis=1))
    scale = np.exp2(e.astype(np.float64)).astype(np.float32)
    y = np.clip((xb / scale[:, None]).astype(np.float32), np.float32(-FP4_MAX), np.float32(FP4_MAX))
    return e2m1_encode(y).reshape(x.shape), (e + 127).astype(np.uint8)


def fp4_dequantize(codes, e8m0) -> np.ndarray:
    """E2M1 codes [..., n] with E8M0 bytes [..., n / 32] -> fp64 values."""
    return e2m1_decode(codes) * np.repeat(e8m0_decode(e8m0), FP4_BLOCK, axis=-1)


def index_keys_fp4(pool: dict, page_table_row, entries) -> np.ndarray:
    """Dequantised FP4 indexer keys [n, 128] in fp64 from an FP4 key pool."""
    pages, slots = _locate(page_table_row, entries)
    return fp4_dequantize(pool["codes"][pages, slots], pool["e8m0"][pages, slots])


def key_write_fp4(pool: dict, page_table_row, entries, key_bf16_bits) -> None:
    """Write indexer keys into an FP4 key pool in place (fp4_quantize per key)."""
    pages, slots = _locate(page_table_row, entries)
    for r, (pg, sl) in enumerate(zip(pages, slots)):
        codes, e8m0 = fp4_quantize(np.asarray(key_bf16_bits[r], dtype=np.uint16))
        pool["codes"][pg, sl] = codes
        pool["e8m0"][pg, sl] = e8m0


def indexer_logits_row_fp4(q_codes, q_e8m0, w, key_pool, page_table_row, n_vis) -> np.ndarray:
    """Index scores of one query with FP4 q [Hi, 128] / E8M0 [Hi, 4] over an FP4
    key pool: the same sum over heads of w * ReLU(q . k) as ``indexer_logits_row``
    (P1 §2.10 steps 6-8), on the FP4-dequantised operands."""
    n = int(n_vis)
    if n <= 0:
        return np.zeros(0, dtype=np.float64)
    q = fp4_dequantize(q_codes, q_e8m0)                      # [Hi, 128]
    k = index_keys_fp4(key_pool, page_table_row, np.arange(n))
    return np.maximum(k @ q.T, 0.0) @ np.asarray(w, np.float64)


# ---------------------------------------------------------------- Hadamard rotation before FP4 (compressor rotate path)
# P1 §2.7 rotate_activation: hadamard_transform(x, scale=d ** -0.5) applied to an
# activation before low-precision quantisation; P1 §2.9 step 7: with rotate=True
# the compressor's output is rotated and FP4-quantised (the indexer's keys);
# P1 §2.10 step 2 rotates the indexer's q the same way.  The transform is the
# Sylvester (Walsh) Hadamard matrix in natural order, H_1 = [1],
# H_2n = [[H_n, H_n], [H_n, -H_n]].  Reading of what the pages leave open: the
# rotated activation keeps the activation's type, BF16, so the definition is the
# exact product H x d^-0.5 rounded once to BF16 (nearest, ties to even), then
# FP4-quantised.  A GPU evaluates the product in fp32; ``hadamard_rotate_fp32_bound``
# states how far any fp32 evaluation can be from the exact value, which is the
# band within which a BF16 rounding decision may legitimately differ.

def hadamard_matrix(d: int) -> np.ndarray:
    """The Sylvester Hadamard matrix of order d (a power of two), fp64."""
    if d < 1 or d & (d - 1):
        raise ValueError("d must be a power of two")
    h = np.ones((1, 1))
    while h.shape[0] < d:
        h = np.block([[h, h], [h, -h]])
    return h


def hadamard_rotate(x) -> np.ndarray:
    """x [..., d] -> H_d x * d^-0.5 in fp64 (the plain definition)."""
    x = np.asarray(x, np.float64)
    d = x.shape[-1]
    return x @ hadamard_matrix(d).T * d ** -0.5


def hadamard_rotate_fp32_bound(x) -> np.ndarray:
    """x [..., d] (d = 2^m) -> a bound, per row, on |fp32 evaluation - H x d^-0.5|.

    Any fp32 evaluation that sums the 2^m signed inputs of an output through a
    tree of depth m (the butterfly network in any stage order) rounds m times,
    each time by at most u = 2^-24 of a partial sum no larger than sum |x|, so it
    is off by at most ((1 + u)^m - 1) sum |x| <= 1.01 m u sum |x|; the scale
    fp32(d^-0.5) and the product each add a relative u.  The bound returned is
    (m + 3) u d^-0.5 sum |x|, which covers both."""
    x = np.asarray(x, np.float64)
    d = x.shape[-1]
    m = int(round(math.log2(d)))
    return (m + 3) * 2.0 ** -24 * d ** -0.5 * np.abs(x).sum(axis=-1, keepdims=True)


def fp64_to_bf16_bits(v) -> np.ndarray:
    """fp64 values -> BF16 bit patterns, rounded once from the exact fp64 value:
    nearest, ties to even (finite values inside the BF16 range)."""
    v = np.asarray(v, np.float64)
    _, e = np.frexp(v)
    step = np.maximum(e - 8, -133)          # BF16: 8 significant bits; subnormal spacing 2^-133
    q = np.ldexp(np.rint(np.ldexp(v, -step)), step)   # exact scalings by powers of two; rint ties to even
    return (q.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)


def hadamard_rotate_to_bf16(x_bf16_bits) -> np.ndarray:
    """BF16 bit patterns [..., d] -> BF16 bit patterns of H x d^-0.5: the exact
    rotation (``hadamard_rotate``) rounded once to BF16."""
    return fp64_to_bf16_bits(hadamard_rotate(bf16_decode(x_bf16_bits)))


def fp32_to_bf16_bits(v) -> np.ndarray:
    """fp32 values -> BF16 bit patterns, round to nearest, ties to even (finite inputs)."""
    u = np.asarray(v, np.float32).view(np.uint32).astype(np.uint64)
    lower = u & 0xFFFF
    upper = u >> 16
    up = (lower > 0x8000) | ((lower == 0x8000) & ((upper & 1) == 1))
    return (upper + up.astype(np.uint64)).astype(np.uint16)


def key_write_fp4_rotated(pool: dict, page_table_row, entries, key_bf16_bits) -> None:
    """The compressor's rotate path into an FP4 key pool (P1 §2.9 step 7): each
    key rotated (``hadamard_rotate_to_bf16``), then written as ``key_write_fp4``."""
    key_write_fp4(pool, page_table_row, entries, hadamard_rotate_to_bf16(np.asarray(key_bf16_bits, np.uint16)))
