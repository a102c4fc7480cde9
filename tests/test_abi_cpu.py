"""C-ABI checks that need no GPU: the library loads, exports every entry point
include/dsv4sa.h declares, and rejects bad arguments on the host before any
CUDA call (no compute call is made here)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dsv4sa.h")


@pytest.fixture(scope="module")
def L():
    from compressed_sparse_attention_c4_gb300 import build, dsv4sa
    if not os.path.exists(dsv4sa.LIB_PATH):
        build.build()
    return dsv4sa


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"DSV4SA_API\s+[\w\s\*]+?\b(dsv4sa_\w+)\s*\(", text)))


def test_header_declares_expected_entry_points():
    names = declared_functions()
    for must in ("dsv4sa_indexer_logits", "dsv4sa_topk", "dsv4sa_sparse_attn_decode",
                 "dsv4sa_sparse_attn_prefill", "dsv4sa_pool_desc_init"):
        assert must in names


def test_library_exports_every_declared_symbol(L):
    lib = L.lib()
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert set(declared_functions()) <= set(L.exported_symbols()) | {"dsv4sa_status_string", "dsv4sa_version"}


def test_binding_signatures_match_the_header(L):
    """The binding's ctypes signature table names exactly the header's entry
    points, so every call the header declares is typed on the Python side."""
    assert set(L._SIGS) == set(declared_functions())


def test_version_and_status_strings(L):
    lib = L.lib()
    assert lib.dsv4sa_version() >= 100
    for s in range(7):
        assert lib.dsv4sa_status_string(s).decode() == L.STATUS[s]


def test_pool_layout(L):
    assert L.dsv4sa_pool_bytes(L.POOL_KV, 3) == 3 * 38912
    assert L.dsv4sa_pool_bytes(L.POOL_IDXK, 5) == 5 * 8704
    assert L.dsv4sa_pool_bytes(7, 5) == 0
    d = L.dsv4sa_pool_desc_init(L.POOL_KV, 1 << 20, 10)
    assert (d.page_stride, d.nope_off, d.rope_off, d.scale_off) == (38912, 0, 28672, 36864)
    assert (d.nope_row, d.rope_row, d.scale_row, d.n_scales) == (448, 128, 32, 7)
    k = L.dsv4sa_pool_desc_init(L.POOL_IDXK, 1 << 20, 10)
    assert (k.page_stride, k.scale_off, k.nope_row, k.scale_row) == (8704, 8192, 128, 8)
    f = L.dsv4sa_pool_desc_init(L.POOL_IDXK_FP4, 1 << 20, 10)
    assert L.dsv4sa_pool_bytes(L.POOL_IDXK_FP4, 5) == 5 * 4352
    assert (f.page_stride, f.scale_off, f.nope_row, f.scale_row, f.scale_group, f.n_scales) == (4352, 4096, 64, 4, 32, 4)
    # every block offset and row is 16-byte aligned (vector / TMA loads)
    for v in (d.rope_off, d.scale_off, d.nope_row, d.rope_row, d.scale_row, k.scale_off, k.nope_row):
        assert v % 8 == 0
    with pytest.raises(L.DSV4SAError):
        L.dsv4sa_pool_desc_init(L.POOL_KV, (1 << 20) + 16, 10)     # not 1024-aligned
    with pytest.raises(L.DSV4SAError):
        L.dsv4sa_pool_desc_init(L.POOL_KV, 1 << 20, 0)


def test_workspace_sizes(L):
    assert L.dsv4sa_topk_workspace_size(32, 4096, 512) == 0          # one chunk per row
    assert L.dsv4sa_topk_workspace_size(32, 16384, 512) == 0
    assert L.dsv4sa_topk_workspace_size(32, 16385, 512) == 32 * 2 * 512 * 8
    assert L.dsv4sa_topk_workspace_size(4, 262144, 512) == 4 * 16 * 512 * 8
    assert L.dsv4sa_topk_workspace_size(4, 1 << 20, 512) == 4 * 64 * 512 * 8
    assert L.dsv4sa_topk_workspace_size(4, (1 << 20) + 1, 512) == 0  # beyond 64 chunks: unsupported
    assert L.dsv4sa_attn_workspace_size(L.ATTN_PREFILL, 4096, 64, 512, 128) == 0
    assert L.dsv4sa_attn_workspace_size(L.ATTN_DECODE, 32, 64, 512, 128) == 32 * 8 * 64 * 514 * 4   # up to 8 splits
    assert L.dsv4sa_attn_workspace_size(L.ATTN_DECODE, 2, 64, 2048, 128) == 2 * 17 * 64 * 514 * 4
    assert L.dsv4sa_attn_workspace_size(L.ATTN_DECODE, 1, 16, 0, 128) == 0   # one chunk: no split


def test_host_validation_rejects_before_launch(L):
    lib = L.lib()
    d = L.dsv4sa_pool_desc_init(L.POOL_IDXK, 1 << 20, 4)
    fake = ctypes.c_void_p(1 << 21)
    # indexer: unsupported head counts, missing pointers, n_max beyond the page table / logits row
    st = lib.dsv4sa_indexer_logits(ctypes.byref(d), fake, 4, fake, fake, fake, fake, fake, 2, 0, 256, fake, 256, None)
    assert st == 2
    st = lib.dsv4sa_indexer_logits(ctypes.byref(d), fake, 4, fake, fake, fake, fake, fake, 2, 129, 256, fake, 256, None)
    assert st == 2
    st = lib.dsv4sa_indexer_logits(ctypes.byref(d), None, 4, fake, fake, fake, fake, fake, 2, 64, 256, fake, 256, None)
    assert st == 1
    st = lib.dsv4sa_indexer_logits(ctypes.byref(d), fake, 4, fake, fake, fake, fake, fake, 2, 64, 257, fake, 512, None)
    assert st == 1
    st = lib.dsv4sa_indexer_logits(ctypes.byref(d), fake, 4, fake, fake, fake, fake, fake, 2, 64, 256, fake, 100, None)
    assert st == 1
    kv = L.dsv4sa_pool_desc_init(L.POOL_KV, 1 << 20, 4)           # wrong pool kind
    st = lib.dsv4sa_indexer_logits(ctypes.byref(kv), fake, 4, fake, fake, fake, fake, fake, 2, 64, 256, fake, 256, None)
    assert st == 1
    # top-k: k out of range, idx row too short, missing workspace for a chunked row
    assert lib.dsv4sa_topk(fake, 4096, fake, 2, 4096, 0, fake, 512, None, 0, None) == 2
    assert lib.dsv4sa_topk(fake, 4096, fake, 2, 4096, 4096, fake, 4096, None, 0, None) == 2
    assert lib.dsv4sa_topk(fake, 4096, fake, 2, 4096, 512, fake, 100, None, 0, None) == 1
    assert lib.dsv4sa_topk(fake, 20000, fake, 2, 20000, 512, fake, 512, None, 0, None) == 3
    assert lib.dsv4sa_topk(fake, 300000, fake, 2, 300000, 2048, fake, 2048, None, 0, None) == 2   # 19 x 2048 > 32768
    # cache writer: negative n, bad pool descriptor, missing pointers
    kvd = L.dsv4sa_pool_desc_init(L.POOL_KV, 1 << 20, 4)
    assert lib.dsv4sa_cache_write(ctypes.byref(kvd), fake, 4, fake, fake, fake, -1, None) == 1
    bad = L.dsv4sa_pool_desc_init(L.POOL_KV, 1 << 20, 4)
    bad.page_stride += 16
    assert lib.dsv4sa_cache_write(ctypes.byref(bad), fake, 4, fake, fake, fake, 3, None) == 1
    assert lib.dsv4sa_cache_write(ctypes.byref(kvd), None, 4, fake, fake, fake, 3, None) == 1
    assert lib.dsv4sa_cache_write(ctypes.byref(kvd), fake, 4, fake, fake, ctypes.c_void_p((1 << 21) + 2), 3, None) == 1
    assert lib.dsv4sa_cache_write(ctypes.byref(kvd), fake, 4, fake, fake, fake, 0, None) == 0   # nothing to do
    # rotated FP4 key writer: FP4 pools only, then the same checks
    f4 = L.dsv4sa_pool_desc_init(L.POOL_IDXK_FP4, 1 << 20, 4)
    idxk = L.dsv4sa_pool_desc_init(L.POOL_IDXK, 1 << 20, 4)
    assert lib.dsv4sa_cache_write_rotated(ctypes.byref(kvd), fake, 4, fake, fake, fake, 3, None) == 1
    assert lib.dsv4sa_cache_write_rotated(ctypes.byref(idxk), fake, 4, fake, fake, fake, 3, None) == 1
    assert lib.dsv4sa_cache_write_rotated(ctypes.byref(f4), fake, 4, fake, fake, fake, -1, None) == 1
    assert lib.dsv4sa_cache_write_rotated(ctypes.byref(f4), fake, 0, fake, fake, fake, 3, None) == 1
    assert lib.dsv4sa_cache_write_rotated(ctypes.byref(f4), fake, 4, None, fake, fake, 3, None) == 1
    assert lib.dsv4sa_cache_write_rotated(ctypes.byref(f4), fake, 4, fake, fake, ctypes.c_void_p((1 << 21) + 2), 3,
                                          None) == 1
    assert lib.dsv4sa_cache_write_rotated(ctypes.byref(f4), fake, 4, fake, fake, fake, 0, None) == 0
    # index helpers
    assert lib.dsv4sa_window_indices(fake, 2, 128, 0, fake, 64, None) == 1
    assert lib.dsv4sa_compress_indices(None, 2, 16, fake, 16, None) == 1
    # attention plan: argument checks come before any device query
    assert lib.dsv4sa_attn_plan(0, 1, 0, 512, 128, None, None, None) == 1
    assert lib.dsv4sa_attn_plan(7, 1, 64, 512, 128, None, None, None) == 1
    # attention
    assert lib.dsv4sa_sparse_attn_decode(None, None) == 1
    a = L.AttnArgs()
    a.T, a.H = 1, 0
    assert lib.dsv4sa_sparse_attn_decode(ctypes.byref(a), None) == 2
    a.H = 129
    assert lib.dsv4sa_sparse_attn_prefill(ctypes.byref(a), None) == 2
    a.H, a.q = 16, None
    assert lib.dsv4sa_sparse_attn_decode(ctypes.byref(a), None) == 1
    a.q = ctypes.c_void_p((1 << 21) + 8)                           # misaligned q
    a.attn_sink = a.q_seq = a.out = fake
    assert lib.dsv4sa_sparse_attn_decode(ctypes.byref(a), None) == 1
    a.q = fake
    a.kc, a.idx_c_stride = 512, 512
    assert lib.dsv4sa_sparse_attn_decode(ctypes.byref(a), None) == 1   # kc > 0 without a pool
    a.comp = ctypes.pointer(kv)
    a.comp_pt, a.comp_pt_stride, a.idx_c = fake, 4, fake
    assert lib.dsv4sa_sparse_attn_decode(ctypes.byref(a), None) == 3   # two chunks need a workspace
    # the inverse rotary embedding: a table needs positions, rows and 16-byte alignment
    a.rope_cs, a.rope_rows = fake, 8
    assert lib.dsv4sa_sparse_attn_decode(ctypes.byref(a), None) == 1   # no rope_pos
    a.rope_pos = fake
    a.rope_rows = 0
    assert lib.dsv4sa_sparse_attn_decode(ctypes.byref(a), None) == 1   # empty table
    a.rope_rows, a.rope_cs = 8, ctypes.c_void_p((1 << 21) + 8)
    assert lib.dsv4sa_sparse_attn_decode(ctypes.byref(a), None) == 1   # misaligned table
    a.rope_cs = fake
    assert lib.dsv4sa_sparse_attn_decode(ctypes.byref(a), None) == 3   # valid table: on to the workspace check


def test_python_binding_refuses_cpu_tensors(L):
    import torch
    d = L.dsv4sa_pool_desc_init(L.POOL_IDXK, 1 << 20, 4)
    x = torch.zeros(4, dtype=torch.int32)
    with pytest.raises(ValueError, match="CUDA"):
        L.dsv4sa_indexer_logits(d, x.view(1, 4), x[:1], x[:1], torch.zeros(1, 4, 128, dtype=torch.uint8),
                                torch.zeros(1, 4, 2), torch.zeros(1, 4), 64, torch.zeros(1, 64))


def test_compressor_validation_without_a_gpu(L):
    """Host-side checks of the compressor entry points (no launch reaches a GPU)."""
    lib = L.lib()
    fake = ctypes.c_void_p(1 << 21)
    odd = ctypes.c_void_p((1 << 21) + 4)
    f = ctypes.c_float(1e-6)
    # windows: ratio 4 needs overlap-sized rows; overlap only with ratio 4
    args = lambda stride, n, ratio, overlap, kv=fake, rows=8: (kv, fake, stride, 64, fake, fake, fake, n, ratio, overlap,
                                                                 fake, fake, f, fake, rows, fake, None)
    assert lib.dsv4sa_compress_windows(*args(1024, 0, 4, 1)) == 0            # nothing to do
    assert lib.dsv4sa_compress_windows(*args(512, 3, 4, 1)) == 1             # rows too short for the overlap
    assert lib.dsv4sa_compress_windows(*args(1028, 3, 4, 1)) == 1            # stride not a multiple of 8
    assert lib.dsv4sa_compress_windows(*args(1024, 3, 8, 1)) == 2            # overlap needs ratio 4
    assert lib.dsv4sa_compress_windows(*args(512, 3, 2048, 0)) == 2          # window too long
    assert lib.dsv4sa_compress_windows(*args(1024, 3, 4, 1, kv=odd)) == 1    # misaligned rows
    assert lib.dsv4sa_compress_windows(*args(1024, 3, 4, 1, rows=0)) == 1    # empty rotation table
    assert lib.dsv4sa_compress_windows(*args(1024, -1, 4, 1)) == 1
    on = lambda T, slots, stride=512, st=fake: (fake, fake, stride, T, fake, st, fake, slots, fake, fake, fake, f,
                                                fake, 8, fake, fake, None)
    assert lib.dsv4sa_compress_online_c128(*on(0, 4)) == 0
    assert lib.dsv4sa_compress_online_c128(*on(2, 0)) == 1                   # no state slots
    assert lib.dsv4sa_compress_online_c128(*on(2, 4, stride=500)) == 1
    assert lib.dsv4sa_compress_online_c128(*on(2, 4, st=odd)) == 1           # misaligned state


def test_step_validation_without_a_gpu(L):
    lib = L.lib()
    h = ctypes.c_void_p()
    assert lib.dsv4sa_step_create(ctypes.byref(h), None, None) == 1
    d = L.StepDesc()                                  # no buffers: rejected before any CUDA call
    assert lib.dsv4sa_step_create(ctypes.byref(h), ctypes.byref(d), None) == 1
    assert lib.dsv4sa_step_launch(None, None) == 1 and lib.dsv4sa_step_destroy(None) == 1


def test_copy_validation_without_a_gpu(L):
    lib = L.lib()
    fake = ctypes.c_void_p(1 << 21)
    assert lib.dsv4sa_copy_async(fake, fake, 0, None) == 0                           # nothing to copy
    assert lib.dsv4sa_copy_async(fake, fake, 24, None) == 1                          # not a multiple of 16
    assert lib.dsv4sa_copy_async(ctypes.c_void_p((1 << 21) + 8), fake, 32, None) == 1   # misaligned
    assert lib.dsv4sa_copy_async(None, fake, 32, None) == 1
    for fn in (lib.dsv4sa_copy_async_background,):
        assert fn(fake, fake, 0, None) == 0
        assert fn(fake, fake, 24, None) == 1
        assert fn(ctypes.c_void_p((1 << 21) + 8), fake, 32, None) == 1
        assert fn(fake, None, 32, None) == 1


def test_header_is_plain_c(tmp_path):
    """include/dsv4sa.h is a C header: a C11 translation unit that uses every
    public type compiles with -pedantic and no warnings."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    cuda_inc = "/usr/local/cuda/include"
    if gcc is None or not os.path.exists(os.path.join(cuda_inc, "cuda_runtime_api.h")):
        pytest.skip("gcc or the CUDA headers are not available")
    src = tmp_path / "uses_header.c"
    src.write_text(
        '#include "dsv4sa.h"\n'
        "int main(void) {\n"
        "  dsv4sa_pool_desc p; dsv4sa_attn_args a; dsv4sa_step_desc s; dsv4sa_step* st = 0;\n"
        "  dsv4sa_status e = DSV4SA_OK; dsv4sa_pool_kind k = DSV4SA_POOL_IDXK_FP4;\n"
        "  int (*attn)(const dsv4sa_attn_args*, cudaStream_t) = dsv4sa_sparse_attn_decode;\n"
        "  int (*create)(dsv4sa_step**, const dsv4sa_step_desc*, cudaStream_t) = dsv4sa_step_create;\n"
        "  size_t (*pool_bytes)(int32_t, int64_t) = dsv4sa_pool_bytes;\n"
        "  (void)p; (void)a; (void)s; (void)st; (void)e; (void)k; (void)attn; (void)create; (void)pool_bytes;\n"
        "  return 0;\n"
        "}\n")
    include = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")
    r = subprocess.run([gcc, "-std=c11", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", include, "-I", cuda_inc,
                        "-c", str(src), "-o", str(tmp_path / "uses_header.o")], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
