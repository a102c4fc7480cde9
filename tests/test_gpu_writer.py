"""GPU parity of the KV-cache writer (dsv4sa_cache_write) against the fp64/fp32
oracle (oracle.kv_write / oracle.key_write): every code byte, scale bit and
rope bit of every slot, written or not, must match.  The quantised code is an
integer decided in fp32 on both sides, so the comparison is exact."""
import numpy as np
import pytest
import torch

import oracle
from compressed_sparse_attention_c4_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    import os
    from compressed_sparse_attention_c4_gb300 import build, dsv4sa
    if not os.path.exists(dsv4sa.LIB_PATH):
        build.build()
    return dsv4sa


def unpack_kv(L, buf, P):
    d = L.dsv4sa_pool_desc_init(L.POOL_KV, 1 << 20, P)
    host = buf.cpu().numpy().reshape(P, d.page_stride)
    codes = host[:, d.nope_off:d.nope_off + 64 * d.nope_row].reshape(P, 64, 448)
    rope = np.ascontiguousarray(host[:, d.rope_off:d.rope_off + 64 * d.rope_row]).view(np.uint16).reshape(P, 64, 64)
    sc = np.ascontiguousarray(host[:, d.scale_off:d.scale_off + 64 * d.scale_row]).view(np.float32)
    return {"nope_codes": codes.copy(), "nope_scale": sc.reshape(P, 64, 8)[:, :, :7].copy(), "rope_bits": rope.copy()}


def unpack_keys(L, buf, P):
    d = L.dsv4sa_pool_desc_init(L.POOL_IDXK, 1 << 20, P)
    host = buf.cpu().numpy().reshape(P, d.page_stride)
    codes = host[:, d.nope_off:d.nope_off + 64 * d.nope_row].reshape(P, 64, 128)
    sc = np.ascontiguousarray(host[:, d.scale_off:d.scale_off + 64 * d.scale_row]).view(np.float32)
    return {"codes": codes.copy(), "scale": sc.reshape(P, 64, 2).copy()}


def unpack_keys_fp4(L, buf, P):
    d = L.dsv4sa_pool_desc_init(L.POOL_IDXK_FP4, 1 << 20, P)
    host = buf.cpu().numpy().reshape(P, d.page_stride)
    packed = host[:, d.nope_off:d.nope_off + 64 * d.nope_row].reshape(P, 64, 64)
    codes = np.empty((P, 64, 128), np.uint8)
    codes[..., 0::2] = packed & 0xF
    codes[..., 1::2] = packed >> 4
    e8m0 = host[:, d.scale_off:d.scale_off + 64 * d.scale_row].reshape(P, 64, 4)
    return {"codes": codes, "e8m0": e8m0.copy()}


def bf16(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16)


def rows_mix(rng, n, dim):
    """Rows with very different block magnitudes, zero blocks, blocks under the
    amax floor, negative zeros and values on E4M3 rounding ties."""
    x = rng.standard_normal((n, dim)).astype(np.float32) * rng.uniform(1e-3, 30, (n, 1)).astype(np.float32)
    special = [lambda r: r.__setitem__(slice(None), 0.0),
               lambda r: r.__setitem__(slice(0, 64), 3e-5),
               lambda r: r.__setitem__(slice(None, None, 7), -0.0),
               lambda r: r.__setitem__(slice(0, 64), np.arange(64, dtype=np.float32) / 8 - 4),  # many ties
               lambda r: r.__setitem__(slice(64, 128), 1e4)]
    for i, f in enumerate(special[:n]):
        f(x[i])
    if n == 1:
        x[0, :64] = np.arange(64, dtype=np.float32) / 8 - 4
    return x


def assert_pools_equal(a, b):
    for k in a:
        x, y = np.ascontiguousarray(a[k]), np.ascontiguousarray(b[k])
        bad = np.argwhere(x.view(np.uint8) != y.view(np.uint8))
        assert bad.size == 0, f"{k}: {len(bad)} bytes differ, first at {bad[:4].tolist()}: " \
                              f"{[(x[tuple(i)], y[tuple(i)]) for i in bad[:4]]}"


@pytest.mark.parametrize("n", [1, 37, 640])
def test_kv_write_matches_oracle(L, n):
    rng = np.random.default_rng(500 + n)
    P, B = 24, 3
    pool = {"nope_codes": rng.integers(0, 0x70, (P, 64, 448)).astype(np.uint8),
            "nope_scale": rng.uniform(0.01, 1, (P, 64, 7)).astype(np.float32),
            "rope_bits": rng.integers(0, 0x7F00, (P, 64, 64)).astype(np.uint16)}
    pt = rng.permutation(P)[:B * 8].reshape(B, 8).astype(np.int32)   # 8 pages per sequence, no page shared
    # distinct slots: distinct (sequence, entry) pairs on disjoint pages
    pairs = rng.permutation(B * 512)[:n]
    seq, ent = (pairs // 512).astype(np.int32), (pairs % 512).astype(np.int32)
    x = rows_mix(rng, n, 512)
    xb = bf16(x)
    buf, desc = L.pack_kv_pool(pool["nope_codes"], pool["nope_scale"], pool["rope_bits"], "cuda")
    L.dsv4sa_cache_write(desc, torch.from_numpy(pt).cuda(), torch.from_numpy(seq).cuda(), torch.from_numpy(ent).cuda(),
                         xb.cuda())
    torch.cuda.synchronize()
    assert L.dsv4sa_check_errors() == (0, 0)
    ref = {k: v.copy() for k, v in pool.items()}
    bits = xb.view(torch.int16).numpy().view(np.uint16)
    for r in range(n):
        oracle.kv_write(ref, pt[seq[r]], [ent[r]], bits[r:r + 1])
    assert_pools_equal(unpack_kv(L, buf, P), ref)


def test_key_write_matches_oracle(L):
    rng = np.random.default_rng(600)
    P, n = 10, 300
    pool = {"codes": rng.integers(0, 0x70, (P, 64, 128)).astype(np.uint8),
            "scale": rng.uniform(0.01, 1, (P, 64, 2)).astype(np.float32)}
    pt = rng.permutation(P).astype(np.int32).reshape(1, P)
    ent = rng.permutation(P * 64)[:n].astype(np.int32)
    seq = np.zeros(n, np.int32)
    x = rows_mix(rng, n, 128)
    xb = bf16(x)
    buf, desc = L.pack_key_pool(pool["codes"], pool["scale"], "cuda")
    L.dsv4sa_cache_write(desc, torch.from_numpy(pt).cuda(), torch.from_numpy(seq).cuda(), torch.from_numpy(ent).cuda(),
                         xb.cuda())
    torch.cuda.synchronize()
    assert L.dsv4sa_check_errors() == (0, 0)
    ref = {k: v.copy() for k, v in pool.items()}
    oracle.key_write(ref, pt[0], ent, xb.view(torch.int16).numpy().view(np.uint16))
    assert_pools_equal(unpack_keys(L, buf, P), ref)


def test_fp4_key_write_matches_oracle(L):
    """FP4 indexer keys (E2M1 codes two per byte, E8M0 per 32 values) byte for
    byte against the oracle's fp4 writer, slots not written included; rows with
    zero blocks, blocks on E2M1 rounding ties, tiny and large blocks, negative
    zeros; one row past the page table is flagged and skipped."""
    rng = np.random.default_rng(602)
    P, n = 10, 301
    pool = {"codes": rng.integers(0, 16, (P, 64, 128)).astype(np.uint8),
            "e8m0": rng.integers(1, 255, (P, 64, 4)).astype(np.uint8)}
    pt = rng.permutation(P).astype(np.int32).reshape(1, P)
    ent = rng.permutation(P * 64)[:n].astype(np.int32)
    ent[-1] = P * 64 + 5                                          # past the page table
    seq = np.zeros(n, np.int32)
    x = rows_mix(rng, n, 128)
    ties = np.array([6.0, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -2.5, -0.75, 0.2500001, 4.5] + [0.0] * 20, np.float32)
    x[10, :32] = ties                                             # amax 6: scale 1, every E2M1 tie
    x[10, 32:64] = ties * 2.0 ** -20                              # the same ties, scale 2^-20
    x[11, :] = rng.standard_normal(128).astype(np.float32) * 1e-30
    x[12, :] = rng.standard_normal(128).astype(np.float32) * 1e30
    xb = bf16(x)
    buf, desc = L.pack_key_pool_fp4(pool["codes"], pool["e8m0"], "cuda")
    L.dsv4sa_cache_write(desc, torch.from_numpy(pt).cuda(), torch.from_numpy(seq).cuda(), torch.from_numpy(ent).cuda(),
                         xb.cuda())
    torch.cuda.synchronize()
    st, bits = L.dsv4sa_check_errors()
    assert st == 5 and bits != 0                                  # the out-of-range row
    assert L.dsv4sa_check_errors() == (0, 0)
    ref = {k: v.copy() for k, v in pool.items()}
    oracle.key_write_fp4(ref, pt[0], ent[:-1], xb[:-1].view(torch.int16).numpy().view(np.uint16))
    assert_pools_equal(unpack_keys_fp4(L, buf, P), ref)


def check_rotated_fp4_row(codes, e8m0, key_bits):
    """One key written by the rotated FP4 writer against the plain definition:
    the exact rotation H x d^-0.5 (fp64), rounded once to BF16, FP4-quantised.
    A GPU evaluates the rotation in fp32, so each rotated value may land
    anywhere in [exact - b, exact + b] (b = oracle.hadamard_rotate_fp32_bound)
    before its BF16 rounding.  Where that band holds one BF16 value (almost
    every element) the code and the block's scale byte must be the oracle's
    exactly; where it straddles a rounding boundary, the code must be one that
    some value of the band quantises to."""
    x = oracle.bf16_decode(key_bits)
    exact = oracle.hadamard_rotate(x)
    band = oracle.hadamard_rotate_fp32_bound(x)
    lo = oracle.bf16_decode(oracle.fp64_to_bf16_bits(exact - band))
    hi = oracle.bf16_decode(oracle.fp64_to_bf16_bits(exact + band))
    ambiguous = 0
    for b in range(len(x) // 32):
        sl = slice(32 * b, 32 * b + 32)
        blo, bhi = lo[sl], hi[sl]
        straddle = (blo <= 0) & (bhi >= 0)
        amax_lo = np.where(straddle, 0.0, np.minimum(np.abs(blo), np.abs(bhi))).max()
        amax_hi = np.maximum(np.abs(blo), np.abs(bhi)).max()
        e_lo, e_hi = int(oracle.fp4_scale_exponent(amax_lo)), int(oracle.fp4_scale_exponent(amax_hi))
        e = int(e8m0[b]) - 127
        assert e_lo <= e <= e_hi, (b, e, e_lo, e_hi)
        scale = np.float32(2.0 ** e)
        ylo = np.clip((blo.astype(np.float32) / scale).astype(np.float32), -6, 6)
        yhi = np.clip((bhi.astype(np.float32) / scale).astype(np.float32), -6, 6)
        clo, chi = oracle.e2m1_encode(ylo), oracle.e2m1_encode(yhi)
        got = codes[sl]
        exact_elems = clo == chi
        assert np.array_equal(got[exact_elems], clo[exact_elems]), b
        vg, vlo, vhi = oracle.e2m1_decode(got), oracle.e2m1_decode(clo), oracle.e2m1_decode(chi)
        assert np.all((vg >= vlo) & (vg <= vhi)), b
        zero = vg == 0
        sign_ok = ((got & 8) == (clo & 8)) | ((got & 8) == (chi & 8))
        assert np.all(~zero | sign_ok), b
        ambiguous += int((~exact_elems).sum()) + (e_lo != e_hi)
    return ambiguous


def test_fp4_rotated_key_write_matches_oracle(L):
    """The compressor's rotate path: keys rotated by the order-128 Hadamard
    transform and FP4-quantised by dsv4sa_cache_write_rotated, checked against
    the plain definition (exact rotation, one BF16 rounding, FP4 quantisation)
    with the fp32 evaluation band; one row past the page table is flagged and
    skipped, and slots not written keep their bytes."""
    rng = np.random.default_rng(603)
    P, n = 10, 301
    pool = {"codes": rng.integers(0, 16, (P, 64, 128)).astype(np.uint8),
            "e8m0": rng.integers(1, 255, (P, 64, 4)).astype(np.uint8)}
    pt = rng.permutation(P).astype(np.int32).reshape(1, P)
    ent = rng.permutation(P * 64)[:n].astype(np.int32)
    ent[-1] = P * 64 + 5                                          # past the page table
    seq = np.zeros(n, np.int32)
    x = rows_mix(rng, n, 128)
    x[10, :] = 0.0
    x[10, 0] = 1.0                                                # rotates to +-128^-0.5 everywhere
    x[11, :] = rng.standard_normal(128).astype(np.float32) * 1e-30
    x[12, :] = rng.standard_normal(128).astype(np.float32) * 1e30
    xb = bf16(x)
    buf, desc = L.pack_key_pool_fp4(pool["codes"], pool["e8m0"], "cuda")
    L.dsv4sa_cache_write_rotated(desc, torch.from_numpy(pt).cuda(), torch.from_numpy(seq).cuda(),
                                 torch.from_numpy(ent).cuda(), xb.cuda())
    torch.cuda.synchronize()
    st, bits = L.dsv4sa_check_errors()
    assert st == 5 and bits != 0                                  # the out-of-range row
    assert L.dsv4sa_check_errors() == (0, 0)
    got = unpack_keys_fp4(L, buf, P)
    keys = xb.view(torch.int16).numpy().view(np.uint16)
    written = np.zeros((P, 64), bool)
    ambiguous = 0
    for r in range(n - 1):
        pg, sl = pt[0, ent[r] // 64], ent[r] % 64
        written[pg, sl] = True
        ambiguous += check_rotated_fp4_row(got["codes"][pg, sl], got["e8m0"][pg, sl], keys[r])
    assert ambiguous <= 0.01 * (n - 1) * 128                      # the band is narrow: nearly every code is exact
    assert np.array_equal(got["codes"][~written], pool["codes"][~written])
    assert np.array_equal(got["e8m0"][~written], pool["e8m0"][~written])


def test_write_then_read_through_the_path(L):
    """Rows written by the writer are read back by the attention exactly as the
    oracle's cache (the tiny workload, its first compressed entries replaced)."""
    from parity import GpuRun, check_attention
    w = W.make("tiny")
    rng = np.random.default_rng(601)
    n = 96
    x = (rng.standard_normal((n, 512)) * 0.7).astype(np.float32)
    xb = bf16(x)
    bits = xb.view(torch.int16).numpy().view(np.uint16)
    ent = np.arange(n, dtype=np.int32)
    for r in range(n):
        oracle.kv_write(w.comp_pool, w.comp_pt[0], [ent[r]], bits[r:r + 1])
    run = GpuRun(w)                                    # cache uploaded with the oracle's writes
    d = run.d
    xw = torch.from_numpy(rng.standard_normal((n, 512)).astype(np.float32)).to(torch.bfloat16)
    # overwrite on the GPU with the writer, the oracle cache with the oracle writer: same bytes
    L.dsv4sa_cache_write(d.comp, d.comp_pt, torch.zeros(n, dtype=torch.int32, device="cuda"),
                         torch.from_numpy(ent).cuda(), xw.cuda())
    oracle.kv_write(w.comp_pool, w.comp_pt[0], ent, xw.view(torch.int16).numpy().view(np.uint16))
    torch.cuda.synchronize()
    L.run_path(d)
    torch.cuda.synchronize()
    run.out = d.out.float().cpu().numpy()
    run.lse = d.lse.cpu().numpy()
    run.idx_c = d.idx_c.cpu().numpy()
    check_attention(run, 0)


def test_out_of_range_rows_are_flagged_and_skipped(L):
    rng = np.random.default_rng(602)
    P = 4
    pool = {"codes": rng.integers(0, 0x70, (P, 64, 128)).astype(np.uint8),
            "scale": rng.uniform(0.01, 1, (P, 64, 2)).astype(np.float32)}
    pt = np.array([[0, 1, 7, 2]], np.int32)            # page id 7 is out of range
    ent = np.array([3, 130, 64 * 4 + 1, -1], np.int32)  # entry 130 -> page 7; 257 beyond the row; -1
    buf, desc = L.pack_key_pool(pool["codes"], pool["scale"], "cuda")
    xb = bf16(rng.standard_normal((4, 128)))
    L.dsv4sa_cache_write(desc, torch.from_numpy(pt).cuda(), torch.zeros(4, dtype=torch.int32, device="cuda"),
                         torch.from_numpy(ent).cuda(), xb.cuda())
    st, bits = L.dsv4sa_check_errors()
    assert st == 5 and bits & 1
    ref = {k: v.copy() for k, v in pool.items()}
    oracle.key_write(ref, pt[0], ent[:1], xb.view(torch.int16).numpy().view(np.uint16)[:1])
    assert_pools_equal(unpack_keys(L, buf, P), ref)


@pytest.mark.parametrize("kind,n", [("kv", 20000), ("keys", 40000)])
def test_large_batches_walk_the_grid(L, kind, n):
    """More rows than the resident grid holds, so every warp takes several rows;
    rows arrive in random slot order over several sequences."""
    rng = np.random.default_rng(700 + n)
    B = 5
    per_seq = (n + B - 1) // B
    pages_per_seq = (per_seq + 63) // 64 + 1
    P = B * pages_per_seq
    pt = rng.permutation(P).astype(np.int32).reshape(B, pages_per_seq)
    order = rng.permutation(B * pages_per_seq * 64)[:n]
    seq, ent = (order // (pages_per_seq * 64)).astype(np.int32), (order % (pages_per_seq * 64)).astype(np.int32)
    dim = 512 if kind == "kv" else 128
    x = (rng.standard_normal((n, dim)) * rng.uniform(1e-3, 50, (n, 1))).astype(np.float32)
    xb = bf16(x)
    bits = xb.view(torch.int16).numpy().view(np.uint16)
    if kind == "kv":
        pool = {"nope_codes": np.zeros((P, 64, 448), np.uint8), "nope_scale": np.zeros((P, 64, 7), np.float32),
                "rope_bits": np.zeros((P, 64, 64), np.uint16)}
        buf, desc = L.pack_kv_pool(pool["nope_codes"], pool["nope_scale"], pool["rope_bits"], "cuda")
    else:
        pool = {"codes": np.zeros((P, 64, 128), np.uint8), "scale": np.zeros((P, 64, 2), np.float32)}
        buf, desc = L.pack_key_pool(pool["codes"], pool["scale"], "cuda")
    L.dsv4sa_cache_write(desc, torch.from_numpy(pt).cuda(), torch.from_numpy(seq).cuda(), torch.from_numpy(ent).cuda(),
                         xb.cuda())
    torch.cuda.synchronize()
    assert L.dsv4sa_check_errors() == (0, 0)
    ref = {k: v.copy() for k, v in pool.items()}
    write = oracle.kv_write if kind == "kv" else oracle.key_write
    for b in range(B):
        m = seq == b
        write(ref, pt[b], ent[m], bits[m])
    got = unpack_kv(L, buf, P) if kind == "kv" else unpack_keys(L, buf, P)
    assert_pools_equal(got, ref)
