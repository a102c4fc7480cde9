"""GPU parity of the KV compressor (dsv4sa_compress_windows,
dsv4sa_compress_online_c128) against the fp64 oracle (oracle.compress_windows,
oracle.online_c128_step).

Tolerance: the kernels pool, normalise and rotate in fp32 and round once to
BF16, the oracle in fp64; an element may land on the other side of a BF16
rounding boundary, so |gpu - oracle| <= 2^-8 |oracle| + 1e-6 max|row| (one BF16
unit in the last place plus fp32 noise)."""
import math

import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu
REL = 2.0 ** -8


@pytest.fixture(scope="module")
def L():
    import os
    from compressed_sparse_attention_c4_gb300 import build, dsv4sa
    if not os.path.exists(dsv4sa.LIB_PATH):
        build.build()
    return dsv4sa


def bf16(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16)


def bits(t):
    return t.view(torch.int16).numpy().view(np.uint16)


def table(rows):
    t = oracle.rope_table(oracle.base_freqs(160000.0), rows)
    cs = np.stack([t.real, t.imag], axis=-1).astype(np.float32)
    return torch.from_numpy(cs), cs[..., 0].astype(np.float64) + 1j * cs[..., 1].astype(np.float64)


def check(got, ref):
    got = np.asarray(got, np.float64)
    assert got.shape == ref.shape and np.isfinite(got).all()
    err = np.abs(got - ref)
    lim = REL * np.abs(ref) + 1e-6 * np.abs(ref).max(axis=-1, keepdims=True)
    bad = np.argwhere(err > lim)
    assert bad.size == 0, f"{len(bad)} values off, first {bad[:3].tolist()}: {err[tuple(bad[0])]} vs {lim[tuple(bad[0])]}"


def inputs(rng, n_tok, width, score_scale=2.0, ratio=4):
    kv = bf16(rng.standard_normal((n_tok, width)))
    sc = bf16(rng.standard_normal((n_tok, width)) * score_scale)
    ape = (rng.standard_normal((ratio, width)) * 0.3).astype(np.float32)
    w = rng.uniform(0.5, 1.5, 512).astype(np.float32)
    return kv, sc, ape, w


@pytest.mark.parametrize("n_tok", [4, 7, 1003])
def test_c4_prefill_windows(L, n_tok):
    rng = np.random.default_rng(900 + n_tok)
    kv, sc, ape, w = inputs(rng, n_tok, 1024)
    n = n_tok // 4
    cs, tab = table(4 * n + 1)
    first = torch.arange(n, dtype=torch.int32) * 4
    prev = torch.where(first > 0, first - 4, torch.full_like(first, -1))
    pos = first.clone()
    out = torch.zeros((n, 512), dtype=torch.bfloat16, device="cuda")
    L.dsv4sa_compress_windows(kv.cuda(), sc.cuda(), first.cuda(), prev.cuda(), pos.cuda(), 4, True,
                              torch.from_numpy(ape).cuda(), torch.from_numpy(w).cuda(), cs.cuda(), out)
    torch.cuda.synchronize()
    assert L.dsv4sa_check_errors() == (0, 0)
    ref = oracle.compress_windows(bits(kv), bits(sc), ape, w, 4, True, tab)
    check(out.float().cpu().numpy(), ref)


def test_c4_decode_windows_from_a_state_buffer(L):
    """Decode: each sequence keeps its last 8 tokens (the previous window and the
    one just completed); the entry number sets the rotation."""
    rng = np.random.default_rng(910)
    B = 33
    kv, sc, ape, w = inputs(rng, 8 * B, 1024)
    entries = rng.integers(1, 5000, B)
    entries[0] = 0                                  # a first window: no previous one
    cs, tab = table(4 * int(entries.max()) + 1)
    first = torch.arange(B, dtype=torch.int32) * 8 + 4
    prev = first - 4
    prev[0] = -1
    pos = torch.from_numpy((4 * entries).astype(np.int32))
    out = torch.zeros((B, 512), dtype=torch.bfloat16, device="cuda")
    L.dsv4sa_compress_windows(kv.cuda(), sc.cuda(), first.cuda(), prev.cuda(), pos.cuda(), 4, True,
                              torch.from_numpy(ape).cuda(), torch.from_numpy(w).cuda(), cs.cuda(), out)
    torch.cuda.synchronize()
    assert L.dsv4sa_check_errors() == (0, 0)
    got = out.float().cpu().numpy()
    kb, sb = bits(kv), bits(sc)
    for b in range(B):
        rows = slice(8 * b + (4 if b == 0 else 0), 8 * b + 8)
        ref = oracle.compress_windows(kb[rows], sb[rows], ape, w, 4, True, tab, first_entry=int(entries[b]))
        check(got[b:b + 1], ref)


def test_c128_offline_windows_and_cache_write(L):
    """Ratio 128 without overlap, then the entries quantised into a KV pool: the
    pool bytes equal the oracle writer's on the same BF16 entries."""
    rng = np.random.default_rng(920)
    n_tok = 128 * 3 + 50
    kv, sc, ape, w = inputs(rng, n_tok, 512, ratio=128)
    n = 3
    cs, tab = table(128 * n)
    first = torch.arange(n, dtype=torch.int32) * 128
    out = torch.zeros((n, 512), dtype=torch.bfloat16, device="cuda")
    L.dsv4sa_compress_windows(kv.cuda(), sc.cuda(), first.cuda(), None, first.cuda(), 128, False,
                              torch.from_numpy(ape).cuda(), torch.from_numpy(w).cuda(), cs.cuda(), out)
    torch.cuda.synchronize()
    assert L.dsv4sa_check_errors() == (0, 0)
    check(out.float().cpu().numpy(), oracle.compress_windows(bits(kv), bits(sc), ape, w, 128, False, tab))
    # into the pool
    P = 2
    pool = {"nope_codes": np.zeros((P, 64, 448), np.uint8), "nope_scale": np.ones((P, 64, 7), np.float32),
            "rope_bits": np.zeros((P, 64, 64), np.uint16)}
    buf, desc = L.pack_kv_pool(pool["nope_codes"], pool["nope_scale"], pool["rope_bits"], "cuda")
    pt = torch.tensor([[1, 0]], dtype=torch.int32).cuda()
    ent = torch.tensor([0, 1, 65], dtype=torch.int32).cuda()
    L.dsv4sa_cache_write(desc, pt, torch.zeros(3, dtype=torch.int32).cuda(), ent, out)
    torch.cuda.synchronize()
    assert L.dsv4sa_check_errors() == (0, 0)
    oracle.kv_write(pool, np.array([1, 0]), np.array([0, 1, 65]), bits(out.cpu()))
    host = buf.cpu().numpy().reshape(P, desc.page_stride)
    codes = host[:, desc.nope_off:desc.nope_off + 64 * desc.nope_row].reshape(P, 64, 448)
    assert np.array_equal(codes, pool["nope_codes"])


def test_online_c128_matches_offline(L):
    """Five sequences, one token per call, states starting at different counts;
    every completed window equals the offline oracle's entry for it."""
    rng = np.random.default_rng(930)
    B, steps = 5, 300
    kv, sc, ape, w = inputs(rng, B * steps, 512, ratio=128)
    kvb, scb = bits(kv).reshape(B, steps, 512), bits(sc).reshape(B, steps, 512)
    cs, tab = table(128 * 4)
    state, count = L.online_c128_state(B)
    # sequence b has already folded (b * 29) tokens of window 0 when this test's tokens start: replay them
    pre = [b * 29 for b in range(B)]
    dev_ape, dev_w, dev_cs = torch.from_numpy(ape).cuda(), torch.from_numpy(w).cuda(), cs.cuda()
    kvd = kv.view(B, steps, 512).cuda()
    scd = sc.view(B, steps, 512).cuda()
    finished = {b: [] for b in range(B)}
    for i in range(steps):
        idx = torch.arange(B, dtype=torch.int32).cuda()
        tok = torch.arange(B) * 0 + i
        entry = torch.tensor([(pre[b] + i) // 128 if i >= 0 else 0 for b in range(B)], dtype=torch.int32)
        out = torch.zeros((B, 512), dtype=torch.bfloat16, device="cuda")
        done = torch.zeros(B, dtype=torch.int32, device="cuda")
        rows_kv = kvd[torch.arange(B), tok]
        rows_sc = scd[torch.arange(B), tok]
        if i == 0:
            # pre-fold b * 29 tokens of sequence b from its own token list (tokens 0 .. pre[b] - 1 reused)
            for k in range(max(pre)):
                act = [b for b in range(B) if k < pre[b]]
                if not act:
                    continue
                a = torch.tensor(act, dtype=torch.int32).cuda()
                o2 = torch.zeros((len(act), 512), dtype=torch.bfloat16, device="cuda")
                d2 = torch.zeros(len(act), dtype=torch.int32, device="cuda")
                L.dsv4sa_compress_online_c128(kvd[a.long(), k].contiguous(), scd[a.long(), k].contiguous(), a,
                                              state, count, torch.zeros(len(act), dtype=torch.int32).cuda(),
                                              dev_ape, dev_w, dev_cs, o2, d2)
        L.dsv4sa_compress_online_c128(rows_kv.contiguous(), rows_sc.contiguous(), idx, state, count,
                                      (entry * 128).cuda(), dev_ape, dev_w, dev_cs, out, done)
        dn = done.cpu().numpy()
        for b in np.nonzero(dn)[0]:
            finished[int(b)].append(out[b].float().cpu().numpy())
    torch.cuda.synchronize()
    assert L.dsv4sa_check_errors() == (0, 0)
    for b in range(B):
        seq_kv = np.concatenate([kvb[b, :pre[b]], kvb[b]])
        seq_sc = np.concatenate([scb[b, :pre[b]], scb[b]])
        ref = oracle.compress_windows(seq_kv, seq_sc, ape, w, 128, False, tab)
        assert len(finished[b]) == ref.shape[0]
        check(np.array(finished[b]), ref)
    # the counts are where the sequences stand in their open windows
    assert count.cpu().numpy().tolist() == [(pre[b] + steps) % 128 for b in range(B)]


def test_out_of_range_windows_and_states_are_flagged(L):
    rng = np.random.default_rng(940)
    kv, sc, ape, w = inputs(rng, 16, 1024)
    cs, _ = table(64)
    first = torch.tensor([0, 12, 14], dtype=torch.int32)      # the last window runs past 16 tokens
    prev = torch.tensor([-1, 8, 10], dtype=torch.int32)
    out = torch.full((3, 512), 7.0, dtype=torch.bfloat16, device="cuda")
    L.dsv4sa_compress_windows(kv.cuda(), sc.cuda(), first.cuda(), prev.cuda(), first.cuda(), 4, True,
                              torch.from_numpy(ape).cuda(), torch.from_numpy(w).cuda(), cs.cuda(), out)
    st, b = L.dsv4sa_check_errors()
    assert st == 5 and b & 1
    assert (out[2] == 0).all() and torch.isfinite(out[:2].float()).all() and (out[:2] != 7.0).any()
    state, count = L.online_c128_state(2)
    kv2, sc2, ape2, w2 = inputs(rng, 2, 512, ratio=128)
    done = torch.full((2,), 9, dtype=torch.int32, device="cuda")
    L.dsv4sa_compress_online_c128(kv2.cuda(), sc2.cuda(), torch.tensor([1, 5], dtype=torch.int32).cuda(), state,
                                  count, torch.zeros(2, dtype=torch.int32).cuda(), torch.from_numpy(ape2).cuda(),
                                  torch.from_numpy(w2).cuda(), cs.cuda(), torch.zeros((2, 512), dtype=torch.bfloat16,
                                                                                      device="cuda"), done)
    st, b = L.dsv4sa_check_errors()
    assert st == 5 and b & 1
    assert done.cpu().tolist() == [0, 0] and count.cpu().tolist() == [0, 1]
