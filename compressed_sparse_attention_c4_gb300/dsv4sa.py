"""ctypes binding of libdsv4sa.so (include/dsv4sa.h): same names, torch tensors in.

Argument marshalling only: every function here checks that its tensors live on
a CUDA device with the expected dtype and shape, passes their data pointers and
the current torch stream to the C entry point of the same name, and raises
``DSV4SAError`` on a non-zero status.  There is no fallback: if the shared
library is missing or a tensor is on the CPU, the call fails loudly.

``pack_kv_pool`` / ``pack_key_pool`` lay logical cache arrays out in the
library's paged byte layout (offsets taken from ``dsv4sa_pool_desc_init``),
and ``DeviceWorkload`` + ``run_path`` drive the whole hot path through the C
ABI for tests and the benchmark.
"""
from __future__ import annotations

import ctypes
import math
import os
from dataclasses import dataclass

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdsv4sa.so")

POOL_KV = 0
POOL_IDXK = 1
POOL_IDXK_FP4 = 2
ATTN_DECODE = 0
ATTN_PREFILL = 1
PAGE = 64
HEAD_DIM = 512

STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported size", 3: "workspace missing or too small",
          4: "CUDA runtime error", 5: "index or page id out of range (device)", 6: "device wait timed out"}


class DSV4SAError(RuntimeError):
    def __init__(self, fn, status):
        super().__init__(f"{fn} failed: {status} ({STATUS.get(status, 'unknown')})")
        self.status = status


class PoolDesc(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("page_size", ctypes.c_int32), ("nope_dim", ctypes.c_int32),
                ("rope_dim", ctypes.c_int32), ("scale_group", ctypes.c_int32), ("n_scales", ctypes.c_int32),
                ("num_pages", ctypes.c_int64), ("page_stride", ctypes.c_int64), ("nope_off", ctypes.c_int64),
                ("rope_off", ctypes.c_int64), ("scale_off", ctypes.c_int64), ("nope_row", ctypes.c_int32),
                ("rope_row", ctypes.c_int32), ("scale_row", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("base", ctypes.c_void_p)]


class AttnArgs(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("T", ctypes.c_int32), ("H", ctypes.c_int32),
                ("softmax_scale", ctypes.c_float), ("flags", ctypes.c_int32),
                ("attn_sink", ctypes.c_void_p), ("q_seq", ctypes.c_void_p),
                ("comp", ctypes.POINTER(PoolDesc)), ("comp_pt", ctypes.c_void_p),
                ("comp_pt_stride", ctypes.c_int32), ("kc", ctypes.c_int32), ("idx_c", ctypes.c_void_p),
                ("idx_c_stride", ctypes.c_int32), ("kw", ctypes.c_int32),
                ("win", ctypes.POINTER(PoolDesc)), ("win_pt", ctypes.c_void_p),
                ("win_pt_stride", ctypes.c_int32), ("idx_w_stride", ctypes.c_int32),
                ("idx_w", ctypes.c_void_p), ("out", ctypes.c_void_p), ("lse", ctypes.c_void_p),
                ("ws", ctypes.c_void_p), ("ws_bytes", ctypes.c_size_t),
                ("win_pos", ctypes.c_void_p), ("win_ring", ctypes.c_int32), ("reserved1", ctypes.c_int32),
                ("rope_cs", ctypes.c_void_p), ("rope_pos", ctypes.c_void_p), ("rope_rows", ctypes.c_int32),
                ("reserved2", ctypes.c_int32)]


class StepDesc(ctypes.Structure):
    _fields_ = [("host_in", ctypes.c_void_p), ("dev_in", ctypes.c_void_p), ("in_bytes", ctypes.c_size_t),
                ("in_split", ctypes.c_size_t), ("kpool", ctypes.POINTER(PoolDesc)), ("page_table", ctypes.c_void_p),
                ("pt_stride", ctypes.c_int32), ("T", ctypes.c_int32), ("q_seq", ctypes.c_void_p),
                ("n_vis", ctypes.c_void_p), ("q_fp8", ctypes.c_void_p), ("q_scale", ctypes.c_void_p),
                ("w", ctypes.c_void_p), ("Hi", ctypes.c_int32), ("n_max", ctypes.c_int32), ("logits", ctypes.c_void_p),
                ("logits_stride", ctypes.c_int64), ("k", ctypes.c_int32), ("idx_stride", ctypes.c_int32),
                ("idx", ctypes.c_void_p), ("topk_ws", ctypes.c_void_p), ("topk_ws_bytes", ctypes.c_size_t),
                ("attn", ctypes.POINTER(AttnArgs))]


_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64
_SZ = ctypes.c_size_t
_SIGS = {
    "dsv4sa_version": ([], ctypes.c_int),
    "dsv4sa_status_string": ([ctypes.c_int], ctypes.c_char_p),
    "dsv4sa_pool_bytes": ([_I32, _I64], _SZ),
    "dsv4sa_pool_desc_init": ([ctypes.POINTER(PoolDesc), _I32, _P, _I64], ctypes.c_int),
    "dsv4sa_indexer_logits": ([ctypes.POINTER(PoolDesc), _P, _I32, _P, _P, _P, _P, _P, _I32, _I32, _I32, _P,
                               _I64, _P], ctypes.c_int),
    "dsv4sa_indexer_logits_fp4": ([ctypes.POINTER(PoolDesc), _P, _I32, _P, _P, _P, _P, _P, _I32, _I32, _I32,
                                   _P, _I64, _P], ctypes.c_int),
    "dsv4sa_topk_workspace_size": ([_I32, _I32, _I32], _SZ),
    "dsv4sa_attn_plan": ([_I32, _I32, _I32, _I32, _I32, ctypes.POINTER(_I32), ctypes.POINTER(_I32),
                          ctypes.POINTER(_I32)], ctypes.c_int),
    "dsv4sa_topk": ([_P, _I64, _P, _I32, _I32, _I32, _P, _I32, _P, _SZ, _P], ctypes.c_int),
    "dsv4sa_topk_noalloc": ([_P, _I64, _P, _I32, _I32, _I32, _P, _I32, _P], ctypes.c_int),
    "dsv4sa_topk_prefetch": ([_P, _I64, _P, _I32, _I32, _I32, _P, _I32, _P, _SZ, ctypes.POINTER(PoolDesc), _P, _I32,
                              _P, _P], ctypes.c_int),
    "dsv4sa_window_indices": ([_P, _I32, _I32, _I32, _P, _I32, _P], ctypes.c_int),
    "dsv4sa_cache_write": ([ctypes.POINTER(PoolDesc), _P, _I32, _P, _P, _P, _I32, _P], ctypes.c_int),
    "dsv4sa_cache_write_rotated": ([ctypes.POINTER(PoolDesc), _P, _I32, _P, _P, _P, _I32, _P], ctypes.c_int),
    "dsv4sa_compress_indices": ([_P, _I32, _I32, _P, _I32, _P], ctypes.c_int),
    "dsv4sa_selftest_wait_timeout": ([_P, _P], ctypes.c_int),
    "dsv4sa_copy_async": ([_P, _P, _SZ, _P], ctypes.c_int),
    "dsv4sa_copy_async_background": ([_P, _P, _SZ, _P], ctypes.c_int),
    "dsv4sa_compress_windows": ([_P, _P, _I64, _I64, _P, _P, _P, _I32, _I32, _I32, _P, _P, ctypes.c_float, _P, _I32,
                                 _P, _P], ctypes.c_int),
    "dsv4sa_compress_online_c128": ([_P, _P, _I64, _I32, _P, _P, _P, _I32, _P, _P, _P, ctypes.c_float, _P, _I32,
                                     _P, _P, _P], ctypes.c_int),
    "dsv4sa_attn_workspace_size": ([_I32, _I32, _I32, _I32, _I32], _SZ),
    "dsv4sa_sparse_attn_decode": ([ctypes.POINTER(AttnArgs), _P], ctypes.c_int),
    "dsv4sa_topk_sparse_attn_decode": ([ctypes.POINTER(AttnArgs), _P, _I64, _P, _I32, _I32, _P, _SZ, _P], ctypes.c_int),
    "dsv4sa_sparse_attn_prefill": ([ctypes.POINTER(AttnArgs), _P], ctypes.c_int),
    "dsv4sa_check_errors": ([_P, ctypes.POINTER(ctypes.c_uint32)], ctypes.c_int),
    "dsv4sa_step_create": ([ctypes.POINTER(_P), ctypes.POINTER(StepDesc), _P], ctypes.c_int),
    "dsv4sa_step_launch": ([_P, _P], ctypes.c_int),
    "dsv4sa_step_destroy": ([_P], ctypes.c_int),
}

_LIB = None


def lib() -> ctypes.CDLL:
    """The loaded shared library (loaded on first use; raises if it is not built)."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is not built: run `python -m compressed_sparse_attention_c4_gb300.build`")
        L = ctypes.CDLL(LIB_PATH)
        for name, (args, res) in _SIGS.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = res
        _LIB = L
    return _LIB


def exported_symbols():
    return list(_SIGS)


def _check(fn, status):
    if status != 0:
        raise DSV4SAError(fn, status)


def _dev(t: torch.Tensor, name: str, dtype=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (the library has no CPU path)")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _dev_or_pinned(t: torch.Tensor, name: str, dtype=None):
    """A CUDA tensor, or a pinned host tensor: with unified addressing its
    pointer is valid on the device and the kernel's stores cross the host link."""
    if isinstance(t, torch.Tensor) and not t.is_cuda and t.is_pinned():
        if dtype is not None and t.dtype != dtype:
            raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
        return ctypes.c_void_p(t.data_ptr())
    return _dev(t, name, dtype)


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


# ---------------------------------------------------------------- pools

def dsv4sa_pool_bytes(kind: int, num_pages: int) -> int:
    return int(lib().dsv4sa_pool_bytes(kind, num_pages))


def dsv4sa_pool_desc_init(kind: int, base: int | torch.Tensor, num_pages: int) -> PoolDesc:
    d = PoolDesc()
    ptr = base.data_ptr() if isinstance(base, torch.Tensor) else int(base)
    _check("dsv4sa_pool_desc_init", lib().dsv4sa_pool_desc_init(ctypes.byref(d), kind, ctypes.c_void_p(ptr), num_pages))
    return d


def _layout(kind: int, num_pages: int) -> PoolDesc:
    return dsv4sa_pool_desc_init(kind, 1 << 20, num_pages)   # any aligned base: offsets only


def _alloc_pool(kind: int, num_pages: int, device) -> torch.Tensor:
    nbytes = dsv4sa_pool_bytes(kind, num_pages)
    buf = torch.empty(nbytes + 1024, dtype=torch.uint8, device=device)
    off = (-buf.data_ptr()) % 1024
    return buf[off:off + nbytes]


def pack_kv_pool(nope_codes: np.ndarray, nope_scale: np.ndarray, rope_bits: np.ndarray, device="cuda"):
    """Logical KV pool arrays -> (device byte tensor, PoolDesc) in the library layout."""
    P = nope_codes.shape[0]
    L = _layout(POOL_KV, P)
    host = np.zeros((P, L.page_stride), dtype=np.uint8)
    host[:, L.nope_off:L.nope_off + PAGE * L.nope_row] = nope_codes.reshape(P, -1)
    host[:, L.rope_off:L.rope_off + PAGE * L.rope_row] = np.ascontiguousarray(rope_bits).view(np.uint8).reshape(P, -1)
    sc = np.zeros((P, PAGE, L.scale_row // 4), dtype=np.float32)
    sc[:, :, :nope_scale.shape[-1]] = nope_scale
    host[:, L.scale_off:L.scale_off + PAGE * L.scale_row] = sc.view(np.uint8).reshape(P, -1)
    dev = _alloc_pool(POOL_KV, P, device)
    dev.copy_(torch.from_numpy(host.reshape(-1)))
    return dev, dsv4sa_pool_desc_init(POOL_KV, dev, P)


def pack_key_pool(codes: np.ndarray, scale: np.ndarray, device="cuda"):
    """Logical indexer-key pool arrays -> (device byte tensor, PoolDesc)."""
    P = codes.shape[0]
    L = _layout(POOL_IDXK, P)
    host = np.zeros((P, L.page_stride), dtype=np.uint8)
    host[:, L.nope_off:L.nope_off + PAGE * L.nope_row] = codes.reshape(P, -1)
    host[:, L.scale_off:L.scale_off + PAGE * L.scale_row] = \
        np.ascontiguousarray(scale, dtype=np.float32).view(np.uint8).reshape(P, -1)
    dev = _alloc_pool(POOL_IDXK, P, device)
    dev.copy_(torch.from_numpy(host.reshape(-1)))
    return dev, dsv4sa_pool_desc_init(POOL_IDXK, dev, P)


def pack_key_pool_fp4(codes: np.ndarray, e8m0: np.ndarray, device="cuda"):
    """Logical FP4 indexer-key pool arrays (E2M1 codes uint8 [P, 64, 128], one
    per byte; E8M0 bytes [P, 64, 4]) -> (device byte tensor, PoolDesc): codes two
    per byte, value 2j in the low nibble of byte j."""
    P = codes.shape[0]
    L = _layout(POOL_IDXK_FP4, P)
    c = np.asarray(codes, np.uint8) & 0xF
    packed = (c[..., 0::2] | (c[..., 1::2] << 4)).astype(np.uint8)
    host = np.zeros((P, L.page_stride), dtype=np.uint8)
    host[:, L.nope_off:L.nope_off + PAGE * L.nope_row] = packed.reshape(P, -1)
    host[:, L.scale_off:L.scale_off + PAGE * L.scale_row] = np.asarray(e8m0, np.uint8).reshape(P, -1)
    dev = _alloc_pool(POOL_IDXK_FP4, P, device)
    dev.copy_(torch.from_numpy(host.reshape(-1)))
    return dev, dsv4sa_pool_desc_init(POOL_IDXK_FP4, dev, P)


# ---------------------------------------------------------------- stage 1: indexer

def dsv4sa_indexer_logits(kpool: PoolDesc, page_table, q_seq, n_vis, q_fp8, q_scale, w, n_max: int, logits,
                          stream=None):
    T, Hi = q_fp8.shape[0], q_fp8.shape[1]
    st = lib().dsv4sa_indexer_logits(
        ctypes.byref(kpool), _dev(page_table, "page_table", torch.int32), page_table.shape[-1],
        _dev(q_seq, "q_seq", torch.int32), _dev(n_vis, "n_vis", torch.int32), _dev(q_fp8, "q_fp8", torch.uint8),
        _dev(q_scale, "q_scale", torch.float32), _dev(w, "w", torch.float32), T, Hi, n_max,
        _dev(logits, "logits", torch.float32), logits.shape[-1], _stream(stream))
    _check("dsv4sa_indexer_logits", st)


def pack_fp4_codes(codes: np.ndarray) -> np.ndarray:
    """E2M1 codes one per byte [..., 2 m] -> packed bytes [..., m], value 2j in
    the low nibble of byte j (the layout of FP4 q and FP4 pool codes)."""
    c = np.asarray(codes, np.uint8) & 0xF
    return (c[..., 0::2] | (c[..., 1::2] << 4)).astype(np.uint8)


def dsv4sa_indexer_logits_fp4(kpool: PoolDesc, page_table, q_seq, n_vis, q_fp4, q_e8m0, w, n_max: int, logits,
                              stream=None):
    """q_fp4: device uint8 [T, Hi, 64] packed E2M1 codes; q_e8m0: uint8 [T, Hi, 4]."""
    T, Hi = q_fp4.shape[0], q_fp4.shape[1]
    st = lib().dsv4sa_indexer_logits_fp4(
        ctypes.byref(kpool), _dev(page_table, "page_table", torch.int32), page_table.shape[-1],
        _dev(q_seq, "q_seq", torch.int32), _dev(n_vis, "n_vis", torch.int32), _dev(q_fp4, "q_fp4", torch.uint8),
        _dev(q_e8m0, "q_e8m0", torch.uint8), _dev(w, "w", torch.float32), T, Hi, n_max,
        _dev(logits, "logits", torch.float32), logits.shape[-1], _stream(stream))
    _check("dsv4sa_indexer_logits_fp4", st)


# ---------------------------------------------------------------- stage 2: top-k

def dsv4sa_topk_workspace_size(T: int, n_max: int, k: int) -> int:
    return int(lib().dsv4sa_topk_workspace_size(T, n_max, k))


def dsv4sa_topk(logits, n_vis, n_max: int, k: int, idx, ws=None, stream=None):
    T = n_vis.shape[0]
    wsp = _dev(ws, "ws", torch.uint8) if ws is not None else None
    st = lib().dsv4sa_topk(_dev(logits, "logits", torch.float32), logits.shape[-1], _dev(n_vis, "n_vis", torch.int32),
                           T, n_max, k, _dev(idx, "idx", torch.int32), idx.shape[-1], wsp,
                           0 if ws is None else ws.numel(), _stream(stream))
    _check("dsv4sa_topk", st)


def dsv4sa_topk_prefetch(logits, n_vis, n_max: int, k: int, idx, kv_pool: PoolDesc, kv_pt, q_seq, ws=None,
                         stream=None):
    """dsv4sa_topk, with each selected entry's row of the compressed KV pool
    prefetched into L2 for the attention that gathers it next."""
    T = n_vis.shape[0]
    wsp = _dev(ws, "ws", torch.uint8) if ws is not None else None
    st = lib().dsv4sa_topk_prefetch(_dev(logits, "logits", torch.float32), logits.shape[-1],
                                    _dev(n_vis, "n_vis", torch.int32), T, n_max, k, _dev(idx, "idx", torch.int32),
                                    idx.shape[-1], wsp, 0 if ws is None else ws.numel(), ctypes.byref(kv_pool),
                                    _dev(kv_pt, "kv_pt", torch.int32), kv_pt.shape[-1],
                                    _dev(q_seq, "q_seq", torch.int32), _stream(stream))
    _check("dsv4sa_topk_prefetch", st)


def dsv4sa_topk_noalloc(logits, n_vis, n_max: int, k: int, idx, stream=None):
    """dsv4sa_topk without a workspace: for callers that cannot allocate device
    memory when they call; uses the library's fixed 8 MiB device scratch (see
    include/dsv4sa.h for the size limit and the sharing rules)."""
    T = n_vis.shape[0]
    st = lib().dsv4sa_topk_noalloc(_dev(logits, "logits", torch.float32), logits.shape[-1],
                                   _dev(n_vis, "n_vis", torch.int32), T, n_max, k, _dev(idx, "idx", torch.int32),
                                   idx.shape[-1], _stream(stream))
    _check("dsv4sa_topk_noalloc", st)


# ---------------------------------------------------------------- index assembly

def dsv4sa_window_indices(pos, window: int, ring: int, idx_w, stream=None):
    st = lib().dsv4sa_window_indices(_dev(pos, "pos", torch.int32), pos.shape[0], window, ring,
                                     _dev(idx_w, "idx_w", torch.int32), idx_w.shape[-1], _stream(stream))
    _check("dsv4sa_window_indices", st)


def dsv4sa_cache_write(pool: PoolDesc, page_table, row_seq, row_entry, rows, stream=None):
    """Quantise BF16 rows [n, 512] (KV pool) or [n, 128] (indexer-key pool) into the pool."""
    want = HEAD_DIM if pool.kind == POOL_KV else 128
    if rows.dim() != 2 or rows.shape[1] != want:
        raise ValueError(f"rows must be [n, {want}]")
    n = rows.shape[0]
    _check("dsv4sa_cache_write", lib().dsv4sa_cache_write(
        ctypes.byref(pool), _dev(page_table, "page_table", torch.int32), page_table.shape[-1],
        _dev(row_seq, "row_seq", torch.int32), _dev(row_entry, "row_entry", torch.int32),
        _dev(rows, "rows", torch.bfloat16), n, _stream(stream)))


def dsv4sa_cache_write_rotated(pool: PoolDesc, page_table, row_seq, row_entry, rows, stream=None):
    """Rotate BF16 keys [n, 128] by the order-128 Hadamard transform, then quantise
    them into an FP4 indexer-key pool."""
    if rows.dim() != 2 or rows.shape[1] != 128:
        raise ValueError("rows must be [n, 128]")
    _check("dsv4sa_cache_write_rotated", lib().dsv4sa_cache_write_rotated(
        ctypes.byref(pool), _dev(page_table, "page_table", torch.int32), page_table.shape[-1],
        _dev(row_seq, "row_seq", torch.int32), _dev(row_entry, "row_entry", torch.int32),
        _dev(rows, "rows", torch.bfloat16), rows.shape[0], _stream(stream)))


def dsv4sa_compress_windows(kv, score, first_tok, prev_tok, position, ratio: int, overlap: bool, ape, norm_w,
                            rope_cs, out, eps: float = 1e-6, stream=None):
    """Pool windows of projected tokens into compressed entries (see dsv4sa.h).
    kv, score: bf16 [n_tok, coff * 512] (rows may be strided); first_tok,
    prev_tok (overlap only), position: int32 [n]; ape fp32 [ratio, coff * 512];
    norm_w fp32 [512]; rope_cs fp32 [rows, 32, 2]; out bf16 [n, 512]."""
    n = first_tok.shape[0]
    if kv.stride(1) != 1 or score.stride(0) != kv.stride(0) or score.shape != kv.shape:
        raise ValueError("kv and score must be row-major with the same row stride")
    _check("dsv4sa_compress_windows", lib().dsv4sa_compress_windows(
        _dev(kv, "kv", torch.bfloat16), _dev(score, "score", torch.bfloat16), kv.stride(0), kv.shape[0],
        _dev(first_tok, "first_tok", torch.int32), _dev(prev_tok, "prev_tok", torch.int32) if overlap else None,
        _dev(position, "position", torch.int32), n, int(ratio), 1 if overlap else 0,
        _dev(ape, "ape", torch.float32), _dev(norm_w, "norm_w", torch.float32), float(eps),
        _dev(rope_cs, "rope_cs", torch.float32), rope_cs.shape[0], _dev(out, "out", torch.bfloat16), _stream(stream)))


def dsv4sa_compress_online_c128(kv, score, state_idx, state, state_count, position, ape, norm_w, rope_cs, out,
                                done, eps: float = 1e-6, stream=None):
    """Fold one new token per sequence into its online C128 state (see dsv4sa.h).
    kv, score: bf16 [T, 512]; state fp32 [slots, 3, 512]; state_count int32
    [slots]; out bf16 [T, 512]; done int32 [T]."""
    T = kv.shape[0]
    if kv.stride(1) != 1 or score.stride(0) != kv.stride(0) or score.shape != kv.shape:
        raise ValueError("kv and score must be row-major with the same row stride")
    _check("dsv4sa_compress_online_c128", lib().dsv4sa_compress_online_c128(
        _dev(kv, "kv", torch.bfloat16), _dev(score, "score", torch.bfloat16), kv.stride(0), T,
        _dev(state_idx, "state_idx", torch.int32), _dev(state, "state", torch.float32),
        _dev(state_count, "state_count", torch.int32), state.shape[0], _dev(position, "position", torch.int32),
        _dev(ape, "ape", torch.float32), _dev(norm_w, "norm_w", torch.float32), float(eps),
        _dev(rope_cs, "rope_cs", torch.float32), rope_cs.shape[0], _dev(out, "out", torch.bfloat16),
        _dev(done, "done", torch.int32), _stream(stream)))


def dsv4sa_selftest_wait_timeout(result, stream=None):
    """Launch the failure-path self-test (a bounded wait that runs out; see dsv4sa.h)."""
    _check("dsv4sa_selftest_wait_timeout", lib().dsv4sa_selftest_wait_timeout(_dev(result, "result", torch.int32),
                                                                              _stream(stream)))


def dsv4sa_copy_async(dst, src, stream=None):
    """Copy src into dst (same byte size, a multiple of 16) with the library's copy
    kernel; either may be a CUDA tensor or a pinned host tensor."""
    if dst.numel() * dst.element_size() != src.numel() * src.element_size():
        raise ValueError("dst and src differ in size")
    _check("dsv4sa_copy_async", lib().dsv4sa_copy_async(_dev_or_pinned(dst, "dst"), _dev_or_pinned(src, "src"),
                                                        dst.numel() * dst.element_size(), _stream(stream)))


def dsv4sa_copy_async_background(dst, src, stream=None):
    """dsv4sa_copy_async by one warp per SM: for a copy on a side stream that runs
    beside the indexer (see dsv4sa.h)."""
    if dst.numel() * dst.element_size() != src.numel() * src.element_size():
        raise ValueError("dst and src differ in size")
    _check("dsv4sa_copy_async_background",
           lib().dsv4sa_copy_async_background(_dev_or_pinned(dst, "dst"), _dev_or_pinned(src, "src"),
                                              dst.numel() * dst.element_size(), _stream(stream)))


def online_c128_state(slots: int, device="cuda"):
    """Fresh online C128 states: (state fp32 [slots, 3, 512] = (-inf, 0, 0), count int32 [slots] = 0)."""
    state = torch.zeros((slots, 3, 512), dtype=torch.float32, device=device)
    state[:, 0] = float("-inf")
    return state, torch.zeros(slots, dtype=torch.int32, device=device)


def dsv4sa_compress_indices(n_vis, kc: int, idx, stream=None):
    st = lib().dsv4sa_compress_indices(_dev(n_vis, "n_vis", torch.int32), n_vis.shape[0], kc,
                                       _dev(idx, "idx", torch.int32), idx.shape[-1], _stream(stream))
    _check("dsv4sa_compress_indices", st)


# ---------------------------------------------------------------- stage 3: attention

def dsv4sa_attn_workspace_size(mode: int, T: int, H: int, kc: int, kw: int) -> int:
    return int(lib().dsv4sa_attn_workspace_size(mode, T, H, kc, kw))


def dsv4sa_attn_plan(mode: int, T: int, H: int, kc: int, kw: int) -> dict:
    """Splits, rows per split and kernel launches of an attention call on the current device."""
    ns, rps, nl = _I32(), _I32(), _I32()
    _check("dsv4sa_attn_plan", lib().dsv4sa_attn_plan(mode, T, H, kc, kw, ctypes.byref(ns), ctypes.byref(rps),
                                                      ctypes.byref(nl)))
    return {"nsplit": ns.value, "rows_per_split": rps.value, "launches": nl.value}


ATTN_EARLY_WINDOW = 1


def _attn_args(q, sink, q_seq, comp, comp_pt, idx_c, win, win_pt, idx_w, out, softmax_scale, lse, ws,
               win_pos=None, kw=None, win_ring=0, flags=0, rope_cs=None, rope_pos=None):
    a = AttnArgs()
    a.q = _dev(q, "q", torch.bfloat16)
    a.T, a.H = q.shape[0], q.shape[1]
    if q.shape[2] != HEAD_DIM:
        raise ValueError("q must be [T, H, 512]")
    a.softmax_scale = float(softmax_scale)
    a.flags = int(flags)
    a.attn_sink = _dev(sink, "attn_sink", torch.float32)
    a.q_seq = _dev(q_seq, "q_seq", torch.int32)
    if idx_c is not None:
        a.comp = ctypes.pointer(comp)
        a.comp_pt = _dev(comp_pt, "comp_pt", torch.int32)
        a.comp_pt_stride = comp_pt.shape[-1]
        a.idx_c = _dev(idx_c, "idx_c", torch.int32)
        a.kc = idx_c.shape[-1]
        a.idx_c_stride = idx_c.shape[-1]
    if idx_w is not None:
        a.win = ctypes.pointer(win)
        a.win_pt = _dev(win_pt, "win_pt", torch.int32)
        a.win_pt_stride = win_pt.shape[-1]
        a.idx_w = _dev(idx_w, "idx_w", torch.int32)
        a.kw = idx_w.shape[-1]
        a.idx_w_stride = idx_w.shape[-1]
    elif win_pos is not None and kw:
        # window indices computed in the kernel from the positions
        a.win = ctypes.pointer(win)
        a.win_pt = _dev(win_pt, "win_pt", torch.int32)
        a.win_pt_stride = win_pt.shape[-1]
        a.win_pos = _dev(win_pos, "win_pos", torch.int32)
        a.kw = int(kw)
        a.win_ring = int(win_ring)
    a.out = _dev_or_pinned(out, "out", torch.bfloat16)
    a.lse = _dev_or_pinned(lse, "lse", torch.float32) if lse is not None else None
    if ws is not None:
        a.ws = _dev(ws, "ws", torch.uint8)
        a.ws_bytes = ws.numel()
    if rope_cs is not None:
        # (cos, sin) table [rows, 32, 2] fp32: the inverse rotary embedding of the output
        if rope_cs.dim() != 3 or rope_cs.shape[1:] != (32, 2):
            raise ValueError("rope_cs must be [rows, 32, 2]")
        a.rope_cs = _dev(rope_cs, "rope_cs", torch.float32)
        a.rope_pos = _dev(rope_pos, "rope_pos", torch.int32)
        a.rope_rows = rope_cs.shape[0]
    return a


def dsv4sa_sparse_attn_decode(q, sink, q_seq, comp, comp_pt, idx_c, win, win_pt, idx_w, out, softmax_scale,
                              lse=None, ws=None, stream=None, win_pos=None, kw=None, win_ring=0, flags=0,
                              rope_cs=None, rope_pos=None):
    """idx_w=None with win_pos, kw (and win_ring) given: the window indices are
    computed in the kernel from the positions.  flags: ATTN_EARLY_WINDOW (see
    dsv4sa.h).  rope_cs [rows, 32, 2] with rope_pos [T]: the output's last 64
    dims are rotated back by the table row of each query."""
    a = _attn_args(q, sink, q_seq, comp, comp_pt, idx_c, win, win_pt, idx_w, out, softmax_scale, lse, ws,
                   win_pos, kw, win_ring, flags, rope_cs, rope_pos)
    _check("dsv4sa_sparse_attn_decode", lib().dsv4sa_sparse_attn_decode(ctypes.byref(a), _stream(stream)))


def dsv4sa_topk_sparse_attn_decode(logits, n_vis, n_max: int, k: int, q, sink, q_seq, comp, comp_pt, idx_c, win,
                                   win_pt, idx_w, out, softmax_scale, lse=None, ws=None, topk_ws=None, stream=None,
                                   win_pos=None, kw=None, win_ring=0, flags=0, rope_cs=None, rope_pos=None):
    """dsv4sa_topk into idx_c, then dsv4sa_sparse_attn_decode over it, as one call
    (one kernel when the decode runs as clusters over rows of <= 16384 entries)."""
    a = _attn_args(q, sink, q_seq, comp, comp_pt, idx_c, win, win_pt, idx_w, out, softmax_scale, lse, ws,
                   win_pos, kw, win_ring, flags, rope_cs, rope_pos)
    twp = _dev(topk_ws, "topk_ws", torch.uint8) if topk_ws is not None else None
    _check("dsv4sa_topk_sparse_attn_decode", lib().dsv4sa_topk_sparse_attn_decode(
        ctypes.byref(a), _dev(logits, "logits", torch.float32), logits.shape[-1], _dev(n_vis, "n_vis", torch.int32),
        n_max, k, twp, 0 if topk_ws is None else topk_ws.numel(), _stream(stream)))


def dsv4sa_sparse_attn_prefill(q, sink, q_seq, comp, comp_pt, idx_c, win, win_pt, idx_w, out, softmax_scale,
                               lse=None, ws=None, stream=None, win_pos=None, kw=None, win_ring=0, flags=0,
                               rope_cs=None, rope_pos=None):
    a = _attn_args(q, sink, q_seq, comp, comp_pt, idx_c, win, win_pt, idx_w, out, softmax_scale, lse, ws,
                   win_pos, kw, win_ring, flags, rope_cs, rope_pos)
    _check("dsv4sa_sparse_attn_prefill", lib().dsv4sa_sparse_attn_prefill(ctypes.byref(a), _stream(stream)))


def dsv4sa_check_errors(stream=None) -> tuple[int, int]:
    bits = ctypes.c_uint32(0)
    st = lib().dsv4sa_check_errors(_stream(stream), ctypes.byref(bits))
    return int(st), int(bits.value)


# ---------------------------------------------------------------- whole path (tests / bench)

@dataclass
class DeviceWorkload:
    """A workload resident on the GPU: pools, page tables, queries, outputs, workspaces."""
    w: object
    mode: int
    comp_buf: torch.Tensor
    comp: PoolDesc
    key_buf: torch.Tensor
    keys: PoolDesc
    win_buf: torch.Tensor
    win: PoolDesc
    comp_pt: torch.Tensor
    win_pt: torch.Tensor
    q: torch.Tensor
    q_idx: torch.Tensor
    q_idx_scale: torch.Tensor
    wts: torch.Tensor
    sink: torch.Tensor
    q_seq: torch.Tensor
    pos: torch.Tensor
    n_vis_idx: torch.Tensor      # indexer / top-k rows (-1: not routed through top-k)
    n_vis_c128: torch.Tensor     # rows taking every visible entry (0 otherwise)
    has_c128: bool
    logits: torch.Tensor
    idx_c: torch.Tensor
    idx_w: torch.Tensor
    out: torch.Tensor
    lse: torch.Tensor
    topk_ws: torch.Tensor | None
    attn_ws: torch.Tensor | None
    in_arena: torch.Tensor       # the STEP_INPUTS tensors are views of this buffer
    in_layout: list
    out_arena: torch.Tensor      # out and lse are views of this buffer
    out_layout: list


# indexer / top-k inputs first, then those only the attention reads (the graph
# step copies the second group while the indexer runs)
STEP_INPUTS = ("q_idx", "q_idx_scale", "wts", "q_seq", "n_vis_idx", "comp_pt", "q", "sink", "pos", "win_pt")
ATTN_ONLY_INPUTS = ("q", "sink", "pos", "win_pt")
STEP_OUTPUTS = ("out", "lse")


def _arena_layout(specs):
    """Byte offsets of tensors packed into one buffer, each 256-byte aligned; the
    buffer size is a multiple of 256 bytes (whole 16-byte units for the copy
    kernel)."""
    off, layout = 0, []
    for name, shape, dtype in specs:
        off = (off + 255) // 256 * 256
        nbytes = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        layout.append((name, off, nbytes, tuple(shape), dtype))
        off += nbytes
    return layout, max((off + 255) // 256 * 256, 256)


def _arena_views(buf, layout):
    return {name: buf[o:o + nb].view(dtype).view(shape) for name, o, nb, shape, dtype in layout}


def upload(w, device="cuda", mode=None) -> DeviceWorkload:
    """Copy a workloads.Workload to the GPU in the library's formats."""
    dev = torch.device(device)
    if mode is None:
        mode = ATTN_PREFILL if w.T > 4 * w.B else ATTN_DECODE
    comp_buf, comp = pack_kv_pool(w.comp_pool["nope_codes"], w.comp_pool["nope_scale"], w.comp_pool["rope_bits"], dev)
    key_buf, keys = pack_key_pool(w.key_pool["codes"], w.key_pool["scale"], dev)
    win_buf, win = pack_kv_pool(w.win_pool["nope_codes"], w.win_pool["nope_scale"], w.win_pool["rope_bits"], dev)

    def t(x, dt):
        return torch.from_numpy(np.ascontiguousarray(x)).to(dt).to(dev)

    c128 = np.asarray(w.c128, bool)
    n_max = max(1, int(w.n_max))
    logits_stride = (n_max + 3) // 4 * 4
    topk_ws_bytes = dsv4sa_topk_workspace_size(w.T, n_max, w.k)
    attn_ws_bytes = dsv4sa_attn_workspace_size(mode, w.T, w.H, w.kc, w.kw)
    # the per-step inputs and outputs each live in one buffer, so a step moves
    # them with one host-to-device and one device-to-host copy
    host = {
        "q": torch.from_numpy(np.ascontiguousarray(w.q).view(np.int16)).view(torch.bfloat16),
        "q_idx": torch.from_numpy(np.ascontiguousarray(w.q_idx, np.uint8)),
        "q_idx_scale": torch.from_numpy(np.ascontiguousarray(w.q_idx_scale, np.float32)),
        "wts": torch.from_numpy(np.ascontiguousarray(w.w, np.float32)),
        "sink": torch.from_numpy(np.ascontiguousarray(w.sink, np.float32)),
        "q_seq": torch.from_numpy(np.ascontiguousarray(w.q_seq, np.int32)),
        "pos": torch.from_numpy(np.ascontiguousarray(w.pos, np.int32)),
        "n_vis_idx": torch.from_numpy(np.where(c128, -1, w.n_vis).astype(np.int32)),
        "comp_pt": torch.from_numpy(np.ascontiguousarray(w.comp_pt, np.int32)),
        "win_pt": torch.from_numpy(np.ascontiguousarray(w.win_pt, np.int32)),
    }
    in_layout, in_bytes = _arena_layout([(n, host[n].shape, host[n].dtype) for n in STEP_INPUTS])
    in_arena = torch.empty(in_bytes, dtype=torch.uint8, device=dev)
    ins = _arena_views(in_arena, in_layout)
    for n in STEP_INPUTS:
        ins[n].copy_(host[n])
    out_layout, out_bytes = _arena_layout([("out", (w.T, w.H, HEAD_DIM), torch.bfloat16),
                                           ("lse", (w.T, w.H), torch.float32)])
    out_arena = torch.empty(out_bytes, dtype=torch.uint8, device=dev)
    outs = _arena_views(out_arena, out_layout)
    return DeviceWorkload(
        w=w, mode=mode, comp_buf=comp_buf, comp=comp, key_buf=key_buf, keys=keys, win_buf=win_buf, win=win,
        in_arena=in_arena, in_layout=in_layout, out_arena=out_arena, out_layout=out_layout,
        n_vis_c128=t(np.where(c128, w.n_vis, 0), torch.int32), has_c128=bool(c128.any()),
        logits=torch.empty((w.T, logits_stride), dtype=torch.float32, device=dev),
        idx_c=torch.empty((w.T, w.kc), dtype=torch.int32, device=dev),
        idx_w=torch.empty((w.T, w.kw), dtype=torch.int32, device=dev),
        topk_ws=torch.empty(topk_ws_bytes, dtype=torch.uint8, device=dev) if topk_ws_bytes else None,
        attn_ws=torch.empty(attn_ws_bytes, dtype=torch.uint8, device=dev) if attn_ws_bytes else None,
        **ins, **outs)


def run_path(d: DeviceWorkload, stream=None, fused_window=False, before_attention=None, out=None, lse=None,
             after_indexer=None, fused_topk=False):
    """One pass of the hot path on the GPU, every step in the library's kernels:
    index assembly -> indexer logits -> top-k -> sparse attention.  With
    fused_window the attention kernel computes the window indices from the
    positions itself (one launch fewer; d.idx_w is then not written)."""
    w = d.w
    n_max = max(1, int(w.n_max))
    if d.has_c128 or w.kc > w.k:
        dsv4sa_compress_indices(d.n_vis_c128, w.kc, d.idx_c, stream)
    if not fused_window:
        dsv4sa_window_indices(d.pos, w.kw, w.win_ring, d.idx_w, stream)
    dsv4sa_indexer_logits(d.keys, d.comp_pt, d.q_seq, d.n_vis_idx, d.q_idx, d.q_idx_scale, d.wts, n_max, d.logits,
                          stream)
    if after_indexer is not None:
        after_indexer()
    if fused_topk and d.mode != ATTN_PREFILL and w.kc == w.k:
        # the top-k and the decode attention as one call (fused_window: window indices from positions)
        if before_attention is not None:
            before_attention()
        dsv4sa_topk_sparse_attn_decode(
            d.logits, d.n_vis_idx, n_max, w.k, d.q, d.sink, d.q_seq, d.comp, d.comp_pt, d.idx_c, d.win, d.win_pt,
            None if fused_window else d.idx_w, d.out if out is None else out, w.softmax_scale,
            lse=d.lse if lse is None else lse, ws=d.attn_ws, topk_ws=d.topk_ws, stream=stream,
            win_pos=d.pos if fused_window else None, kw=w.kw if fused_window else None,
            win_ring=w.win_ring if fused_window else 0, flags=ATTN_EARLY_WINDOW if fused_window else 0)
        return
    # the top-k also prefetches the selected compressed rows into L2 for the attention
    dsv4sa_topk_prefetch(d.logits, d.n_vis_idx, n_max, w.k, d.idx_c, d.comp, d.comp_pt, d.q_seq, d.topk_ws, stream)
    if before_attention is not None:
        before_attention()
    fn = dsv4sa_sparse_attn_prefill if d.mode == ATTN_PREFILL else dsv4sa_sparse_attn_decode
    if fused_window:
        # the kernels before it on the stream (indexer, top-k) write only logits and idx_c
        fn(d.q, d.sink, d.q_seq, d.comp, d.comp_pt, d.idx_c, d.win, d.win_pt, None,
           d.out if out is None else out, w.softmax_scale, lse=d.lse if lse is None else lse, ws=d.attn_ws,
           stream=stream, win_pos=d.pos, kw=w.kw, win_ring=w.win_ring, flags=ATTN_EARLY_WINDOW)
    else:
        fn(d.q, d.sink, d.q_seq, d.comp, d.comp_pt, d.idx_c, d.win, d.win_pt, d.idx_w, d.out, w.softmax_scale,
           lse=d.lse, ws=d.attn_ws, stream=stream)


class StepGraph:
    """One step of a serving loop as a single CUDA graph launch.

    The graph holds: two host-to-device copies of the step's packed inputs
    (`d.in_arena`) from a pinned host buffer of the same layout, made by the
    library's copy kernels (a copy-engine transfer node costs about 20 us of
    latency in the graph) -- the indexer's part first, the attention-only part
    (mostly q) on a side stream beside the indexer (dsv4sa_copy_async_background,
    one warp per SM) -- and the whole path (run_path, window indices
    derived in the attention kernel), whose attention kernel writes out and lse
    straight into a pinned host buffer over the host link.  `host_in[name]` / `host_out[name]` are views of
    those host buffers: the caller fills host_in, calls replay(), and
    synchronises `stream` before reading host_out.  The cache pools stay
    resident on the device; programmatic-dependent launches keep their overlap
    inside the graph."""

    def __init__(self, d: DeviceWorkload):
        self.d = d
        # byte offset where the attention-only inputs start in the packed layout
        self.split = min(o for n, o, _, _, _ in d.in_layout if n in ATTN_ONLY_INPUTS)
        self.side = torch.cuda.Stream(device=d.in_arena.device)
        self.host_in_arena = torch.empty_like(d.in_arena, device="cpu").pin_memory()
        self.host_out_arena = torch.empty_like(d.out_arena, device="cpu").pin_memory()
        self.host_in = _arena_views(self.host_in_arena, d.in_layout)
        self.host_out = _arena_views(self.host_out_arena, d.out_layout)
        self.host_in_arena.copy_(d.in_arena)
        self.stream = torch.cuda.Stream(device=d.in_arena.device)
        self.h2d_bytes = self.host_in_arena.numel()
        self.d2h_bytes = self.host_out_arena.numel()
        # one eager pass first: per-device set-up (kernel attributes, driver
        # entry points) happens outside the capture
        self.stream.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(self.stream):
            self._body()
        self.stream.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph, stream=self.stream):
            self._body()
        self.stream.synchronize()

    def _body(self):
        # the indexer's inputs first; the attention-only inputs (mostly q) then
        # travel on a side stream, by one warp per SM beside the indexer (it
        # leaves a warp's worth of registers free on every SM), joined before
        # the attention
        dsv4sa_copy_async(self.d.in_arena[:self.split], self.host_in_arena[:self.split], self.stream)
        joined = torch.cuda.Event()
        ev = torch.cuda.Event()
        ev.record(self.stream)
        self.side.wait_event(ev)
        with torch.cuda.stream(self.side):
            dsv4sa_copy_async_background(self.d.in_arena[self.split:], self.host_in_arena[self.split:], self.side)
        joined.record(self.side)
        # the attention writes out and lse straight into the pinned host buffer
        run_path(self.d, self.stream, fused_window=True,
                 before_attention=lambda: self.stream.wait_event(joined),
                 out=self.host_out["out"], lse=self.host_out["lse"])

    def replay(self):
        """Launch the step on `stream` (the graph is launched on the current stream)."""
        with torch.cuda.stream(self.stream):
            self.graph.replay()


class NativeStep:
    """The same serving step as StepGraph, built and owned by the library
    (dsv4sa_step_create: a CUDA graph of the copy kernels and the three calls,
    captured in C++), launched by one C-ABI call with no torch graph in
    between.  host_in / host_out are views of pinned host buffers with the
    packed layouts of `d`; the caller fills host_in, calls launch() and
    synchronises `stream` before reading host_out."""

    def __init__(self, d: DeviceWorkload):
        w = d.w
        self.d = d
        self.split = min(o for n, o, _, _, _ in d.in_layout if n in ATTN_ONLY_INPUTS)
        self.host_in_arena = torch.empty_like(d.in_arena, device="cpu").pin_memory()
        self.host_out_arena = torch.empty_like(d.out_arena, device="cpu").pin_memory()
        self.host_in = _arena_views(self.host_in_arena, d.in_layout)
        self.host_out = _arena_views(self.host_out_arena, d.out_layout)
        self.host_in_arena.copy_(d.in_arena)
        self.stream = torch.cuda.Stream(device=d.in_arena.device)
        self.h2d_bytes = self.host_in_arena.numel()
        self.d2h_bytes = self.host_out_arena.numel()
        self.attn = _attn_args(d.q, d.sink, d.q_seq, d.comp, d.comp_pt, d.idx_c, d.win, d.win_pt, None,
                               self.host_out["out"], w.softmax_scale, self.host_out["lse"], d.attn_ws,
                               win_pos=d.pos, kw=w.kw, win_ring=w.win_ring, flags=ATTN_EARLY_WINDOW)
        n_max = max(1, int(w.n_max))
        sd = StepDesc()
        sd.host_in = self.host_in_arena.data_ptr()
        sd.dev_in = d.in_arena.data_ptr()
        sd.in_bytes = d.in_arena.numel()
        sd.in_split = self.split
        sd.kpool = ctypes.pointer(d.keys)
        sd.page_table = _dev(d.comp_pt, "page_table", torch.int32)
        sd.pt_stride = d.comp_pt.shape[-1]
        sd.T = w.T
        sd.q_seq = _dev(d.q_seq, "q_seq", torch.int32)
        sd.n_vis = _dev(d.n_vis_idx, "n_vis", torch.int32)
        sd.q_fp8 = _dev(d.q_idx, "q_fp8", torch.uint8)
        sd.q_scale = _dev(d.q_idx_scale, "q_scale", torch.float32)
        sd.w = _dev(d.wts, "w", torch.float32)
        sd.Hi = d.q_idx.shape[1]
        sd.n_max = n_max
        sd.logits = _dev(d.logits, "logits", torch.float32)
        sd.logits_stride = d.logits.shape[-1]
        sd.k = w.k
        sd.idx_stride = d.idx_c.shape[-1]
        sd.idx = _dev(d.idx_c, "idx", torch.int32)
        sd.topk_ws = d.topk_ws.data_ptr() if d.topk_ws is not None else None
        sd.topk_ws_bytes = d.topk_ws.numel() if d.topk_ws is not None else 0
        sd.attn = ctypes.pointer(self.attn)
        self.desc = sd
        self.handle = ctypes.c_void_p()
        _check("dsv4sa_step_create", lib().dsv4sa_step_create(ctypes.byref(self.handle), ctypes.byref(sd),
                                                              ctypes.c_void_p(self.stream.cuda_stream)))

    def launch(self):
        _check("dsv4sa_step_launch", lib().dsv4sa_step_launch(self.handle, ctypes.c_void_p(self.stream.cuda_stream)))

    def close(self):
        if self.handle:
            self.stream.synchronize()
            lib().dsv4sa_step_destroy(self.handle)
            self.handle = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
