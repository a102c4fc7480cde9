"""Pins of the CPU oracle against things other than itself (CPU only).

Each test checks the oracle against a value or routine that does not come from
the oracle: hand-derived cases (tests/golden/hand_cases.json), torch's own
FP8/BF16 decoders, brute-force loops, scipy's softmax, torch's
scaled_dot_product_attention, closed forms and invariants.  A plausible slip in
the oracle (a dropped scale, ReLU in the wrong place, a wrong index, the sink
in the numerator, a reversed tie rule) fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))
GOLD = json.load(open(os.path.join(HERE, "golden", "hand_cases.json")))


def torch_e4m3(codes):
    return torch.from_numpy(np.asarray(codes, np.uint8).copy()).view(torch.float8_e4m3fn).double().numpy()


def torch_bf16(bits):
    return torch.from_numpy(np.asarray(bits, np.uint16).view(np.int16).copy()).view(torch.bfloat16).double().numpy()


# ---------------------------------------------------------------- formats

def test_e4m3_all_codes_match_torch():
    codes = np.arange(256, dtype=np.uint8)
    mine = oracle.e4m3_decode(codes)
    ref = torch_e4m3(codes)
    assert np.array_equal(np.isnan(mine), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(mine[ok], ref[ok])
    assert np.array_equal(np.signbit(mine[ok]), np.signbit(ref[ok]))


def test_e4m3_hand_values():
    g = GOLD["e4m3"]
    v = oracle.e4m3_decode(g["codes"])
    assert v.tolist() == g["values"]
    assert np.signbit(v[g["codes"].index(128)])
    assert np.isnan(oracle.e4m3_decode(g["nan_codes"])).all()


def test_bf16_matches_torch():
    rng = np.random.default_rng(0)
    bits = rng.integers(0, 65536, size=5000).astype(np.uint16)
    bits = bits[(bits & 0x7F80) != 0x7F80]          # drop inf/nan patterns
    assert np.array_equal(oracle.bf16_decode(bits), torch_bf16(bits))


# ---------------------------------------------------------------- helpers

def small_key_pool(rng, n_pages):
    codes = rng.integers(0, 256, size=(n_pages, 64, 128)).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x30               # no NaN codes
    scale = rng.uniform(0.01, 0.2, size=(n_pages, 64, 2)).astype(np.float32)
    return {"codes": codes, "scale": scale}


def small_kv_pool(rng, n_pages):
    codes = rng.integers(0, 256, size=(n_pages, 64, 448)).astype(np.uint8)
    codes[(codes & 0x7F) >= 0x70] = 0x28               # finite, moderate magnitudes
    scale = rng.uniform(0.005, 0.05, size=(n_pages, 64, 7)).astype(np.float32)
    rope = torch.from_numpy(rng.standard_normal((n_pages, 64, 64)).astype(np.float32)) \
        .to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    return {"nope_codes": codes, "nope_scale": scale, "rope_bits": rope}


def brute_kv_row(pool, page, slot):
    """Row via torch's decoders and an explicit per-element loop over scale blocks."""
    codes = torch_e4m3(pool["nope_codes"][page, slot])
    out = np.empty(512)
    for d in range(448):
        out[d] = codes[d] * float(pool["nope_scale"][page, slot, d // 64])
    out[448:] = torch_bf16(pool["rope_bits"][page, slot])
    return out


# ---------------------------------------------------------------- indexer

def test_indexer_hand_cases():
    for c in GOLD["indexer"]["cases"]:
        H = c["heads"]
        qc = np.array(c.get("q_codes_per_head", [c.get("q_code")] * H), np.uint8)
        q_codes = np.repeat(qc[:, None], 128, axis=1)
        q_scale = np.tile(np.array(c["q_scales"], np.float32), (H, 1))
        pool = {"codes": np.full((1, 64, 128), c["key_code"], np.uint8),
                "scale": np.tile(np.array(c["key_scales"], np.float32), (1, 64, 1))}
        got = oracle.indexer_logits_row(q_codes, q_scale, np.array(c["w"], np.float32), pool,
                                        np.array([0]), 1)
        assert got.tolist() == [c["expect"]]


def test_indexer_brute_force_loops():
    rng = np.random.default_rng(1)
    Hi, n_pages, n_vis = 3, 4, 150
    pool = small_key_pool(rng, n_pages)
    pt = rng.permutation(n_pages)[:3]
    qc = rng.integers(0, 256, size=(Hi, 128)).astype(np.uint8)
    qc[(qc & 0x7F) == 0x7F] = 0x31
    qs = rng.uniform(0.5, 2.0, size=(Hi, 2)).astype(np.float32)
    w = rng.uniform(-1, 1, size=Hi).astype(np.float32)
    got = oracle.indexer_logits_row(qc, qs, w, pool, pt, n_vis)
    qv = torch_e4m3(qc)
    ref = []
    for s in range(n_vis):
        page, slot = pt[s // 64], s % 64
        kv = torch_e4m3(pool["codes"][page, slot])
        tot = 0.0
        for h in range(Hi):
            dot = 0.0
            for d in range(128):
                dot += (qv[h, d] * float(qs[h, d // 64])) * (kv[d] * float(pool["scale"][page, slot, d // 64]))
            tot += float(w[h]) * max(dot, 0.0)
        ref.append(tot)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


def test_indexer_invariants():
    rng = np.random.default_rng(2)
    Hi, n_pages, n = 5, 6, 300
    pool = small_key_pool(rng, n_pages)
    pt = np.arange(5)
    qc = rng.integers(0, 0x70, size=(Hi, 128)).astype(np.uint8) | (rng.integers(0, 2, (Hi, 128)) * 0x80).astype(np.uint8)
    qs = rng.uniform(0.5, 2.0, size=(Hi, 2)).astype(np.float32)
    w = rng.uniform(0, 1, size=Hi).astype(np.float32)
    base = oracle.indexer_logits_row(qc, qs, w, pool, pt, n)
    # physical page order is irrelevant
    perm = rng.permutation(n_pages)                 # new physical page i holds old page perm[i]
    pool2 = {k: v[perm] for k, v in pool.items()}
    pt2 = np.array([int(np.where(perm == p)[0][0]) for p in pt])
    np.testing.assert_array_equal(oracle.indexer_logits_row(qc, qs, w, pool2, pt2, n), base)
    # positive homogeneity in w
    np.testing.assert_allclose(oracle.indexer_logits_row(qc, qs, 3.0 * w.astype(np.float64), pool, pt, n), 3.0 * base, rtol=1e-12)
    # I(q) - I(-q) = sum_h w_h (q_h . k): ReLU(x) - ReLU(-x) = x, checked with an einsum
    neg = qc ^ np.uint8(0x80)
    diff = base - oracle.indexer_logits_row(neg, qs, w, pool, pt, n)
    qv = torch_e4m3(qc) * np.repeat(qs.astype(np.float64), 64, axis=1)
    keys = np.stack([torch_e4m3(pool["codes"][pt[s // 64], s % 64]) *
                     np.repeat(pool["scale"][pt[s // 64], s % 64].astype(np.float64), 64) for s in range(n)])
    lin = np.einsum("hd,sd,h->s", qv, keys, w.astype(np.float64))
    np.testing.assert_allclose(diff, lin, rtol=1e-10, atol=1e-10)


def test_indexer_empty():
    rng = np.random.default_rng(3)
    pool = small_key_pool(rng, 1)
    assert oracle.indexer_logits_row(np.zeros((2, 128), np.uint8), np.ones((2, 2), np.float32),
                                     np.ones(2, np.float32), pool, np.array([0]), 0).shape == (0,)


# ---------------------------------------------------------------- top-k

def test_topk_hand_cases():
    for c in GOLD["topk"]["cases"]:
        assert oracle.topk_row(np.array(c["scores"], float), c["k"]).tolist() == c["expect"]


def check_topk_invariants(scores, k, sel):
    n = len(scores)
    m = min(k, n)
    assert sel.dtype == np.int32 and sel.shape == (k,)
    chosen = sel[:m]
    assert (sel[m:] == -1).all()
    assert (np.diff(chosen) > 0).all()
    rest = np.setdiff1d(np.arange(n), chosen)
    if rest.size and chosen.size:
        thr = scores[chosen].min()
        assert scores[rest].max() <= thr
        eq_rest = rest[scores[rest] == thr]
        eq_sel = chosen[scores[chosen] == thr]
        if eq_rest.size:
            assert eq_sel.max() < eq_rest.min()      # ties go to the lower index


@pytest.mark.parametrize("n,k,levels", [(40, 10, 5), (1000, 512, 0), (600, 512, 3), (512, 512, 0),
                                        (300, 512, 0), (2048, 7, 2)])
def test_topk_invariants(n, k, levels):
    rng = np.random.default_rng(n + k)
    scores = rng.integers(0, levels, n).astype(float) if levels else rng.standard_normal(n)
    check_topk_invariants(scores, k, oracle.topk_row(scores, k))


def test_topk_matches_torch_topk_on_distinct():
    rng = np.random.default_rng(4)
    for n in (513, 4096, 20000):
        s = rng.standard_normal(n)
        ref = np.sort(torch.topk(torch.from_numpy(s), 512).indices.numpy())
        assert np.array_equal(oracle.topk_row(s, 512), ref.astype(np.int32))


# ---------------------------------------------------------------- index assembly

def test_window_and_compress_indices():
    for c in GOLD["window"]["cases"]:
        assert oracle.window_indices(c["pos"], c["window"], c["ring"]).tolist() == c["expect"]
    w = oracle.window_indices(5, 128)
    assert (w[:122] == -1).all() and w[122:].tolist() == list(range(6))
    assert oracle.compress_indices(3, 6).tolist() == [0, 1, 2, -1, -1, -1]
    assert oracle.compress_indices(9, 4).tolist() == [0, 1, 2, 3]
    for pos, n in GOLD["n_visible"]["cases"]:
        assert oracle.n_visible(pos) == n


# ---------------------------------------------------------------- attention

def dense_sink_softmax(q, rows, sink, scale):
    """Textbook route: append the sink as one more logit with a zero value row
    and apply scipy's softmax over the extended vector."""
    H = q.shape[0]
    out = np.zeros((H, 512))
    for h in range(H):
        logits = np.concatenate([scale * rows @ q[h], [sink[h]]])
        vals = np.concatenate([rows, np.zeros((1, 512))])
        out[h] = scipy.special.softmax(logits) @ vals
    return out


def sparse(v: dict, dim=512):
    x = np.zeros(dim)
    for k, val in v.items():
        x[int(k)] = val
    return x


def test_attention_hand_cases():
    for c in GOLD["attention"]["cases"]:
        q = sparse(c["q"])[None]
        rows = np.array([sparse(r) for r in c["rows"]]).reshape(-1, 512)
        got = oracle.sink_softmax_attention(q, rows, np.array([c["sink"]]), c["scale"])[0]
        np.testing.assert_allclose(got, sparse(c["expect"]), rtol=1e-14, atol=1e-15)


def test_attention_brute_force_softmax():
    rng = np.random.default_rng(5)
    for n in (1, 5, 33):
        q = rng.standard_normal((3, 512))
        rows = rng.standard_normal((n, 512))
        sink = rng.standard_normal(3) * 3
        got = oracle.sink_softmax_attention(q, rows, sink, 0.2)
        np.testing.assert_allclose(got, dense_sink_softmax(q, rows, sink, 0.2), rtol=1e-12, atol=1e-13)


def test_attention_large_scores_stable():
    rng = np.random.default_rng(6)
    q = rng.standard_normal((2, 512)) * 40
    rows = rng.standard_normal((9, 512))
    sink = np.array([800.0, -5.0])
    got = oracle.sink_softmax_attention(q, rows, sink, 1.0)
    assert np.isfinite(got).all()
    np.testing.assert_allclose(got, dense_sink_softmax(q, rows, sink, 1.0), rtol=1e-10, atol=1e-12)


def test_attention_no_sink_is_sdpa():
    rng = np.random.default_rng(7)
    q = rng.standard_normal((4, 512))
    rows = rng.standard_normal((17, 512))
    got = oracle.sink_softmax_attention(q, rows, np.full(4, -np.inf), 1 / math.sqrt(512))
    tq = torch.from_numpy(q)[None, :, None, :]            # [1, H, 1, D]
    tk = torch.from_numpy(rows)[None, None].expand(1, 4, 17, 512)
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tk, scale=1 / math.sqrt(512))
    np.testing.assert_allclose(got, ref[0, :, 0].numpy(), rtol=1e-12, atol=1e-13)


def test_attention_closed_forms():
    rng = np.random.default_rng(8)
    q = rng.standard_normal((2, 512))
    r = rng.standard_normal((1, 512))
    sink = np.array([0.3, -1.2])
    a = 0.1 * (q @ r[0])
    one = oracle.sink_softmax_attention(q, r, sink, 0.1)
    np.testing.assert_allclose(one, (np.exp(a) / (np.exp(a) + np.exp(sink)))[:, None] * r, rtol=1e-13)
    two = oracle.sink_softmax_attention(q, np.concatenate([r, r]), sink, 0.1)   # duplicate index
    np.testing.assert_allclose(two, (2 * np.exp(a) / (2 * np.exp(a) + np.exp(sink)))[:, None] * r, rtol=1e-13)
    assert (oracle.sink_softmax_attention(q, np.zeros((0, 512)), sink, 0.1) == 0).all()


def test_sparse_attn_gather_and_order():
    rng = np.random.default_rng(9)
    comp = small_kv_pool(rng, 4)
    win = small_kv_pool(rng, 2)
    cpt = np.array([2, 0, 3])
    wpt = np.array([1, 0])
    H = 3
    q = torch.from_numpy(rng.standard_normal((H, 512)).astype(np.float32)).to(torch.bfloat16) \
        .view(torch.int16).numpy().view(np.uint16)
    sink = rng.standard_normal(H).astype(np.float32)
    idx_c = np.array([5, -1, 130, 64, 5, -1], np.int32)
    idx_w = np.array([-1, 3, 127, 64], np.int32)
    got = oracle.sparse_attn_row(q, sink, 0.05, idx_c, comp, cpt, idx_w, win, wpt)
    # brute force: rows built element by element, textbook softmax
    rows = [brute_kv_row(comp, cpt[e // 64], e % 64) for e in idx_c if e >= 0] + \
           [brute_kv_row(win, wpt[e // 64], e % 64) for e in idx_w if e >= 0]
    ref = dense_sink_softmax(torch_bf16(q), np.array(rows), sink.astype(np.float64), 0.05)
    np.testing.assert_allclose(got, ref, rtol=1e-11, atol=1e-13)
    # order of the index list and the split between the two lists do not matter
    got2 = oracle.sparse_attn_row(q, sink, 0.05, idx_c[::-1].copy(), comp, cpt, idx_w[::-1].copy(), win, wpt)
    np.testing.assert_allclose(got2, got, rtol=1e-12, atol=1e-14)
    # all -1 -> exactly zero
    z = oracle.sparse_attn_row(q, sink, 0.05, np.full(6, -1, np.int32), comp, cpt,
                               np.full(4, -1, np.int32), win, wpt)
    assert (z == 0).all()


def test_topk_all_entries_is_full_attention():
    """k >= N: the indexer + top-k path attends to every compressed entry, which
    is dense sink-softmax attention over all of them plus the window."""
    rng = np.random.default_rng(10)
    comp, win = small_kv_pool(rng, 2), small_kv_pool(rng, 2)
    keys = small_key_pool(rng, 2)
    N, H, Hi = 100, 2, 3
    q = torch.from_numpy(rng.standard_normal((1, H, 512)).astype(np.float32)).to(torch.bfloat16) \
        .view(torch.int16).numpy().view(np.uint16)
    work = dict(q=q, q_idx=rng.integers(0, 0x70, (1, Hi, 128)).astype(np.uint8),
                q_idx_scale=np.ones((1, Hi, 2), np.float32), w=np.ones((1, Hi), np.float32),
                sink=np.array([0.5, -0.5], np.float32), softmax_scale=0.05, comp_pool=comp,
                key_pool=keys, comp_pt=np.array([[1, 0]]), win_pool=win, win_pt=np.array([[0, 1]]),
                q_seq=np.array([0]), n_vis=np.array([N]), idx_w=np.array([[3, 4, -1]], np.int32))
    _, idxc, out = oracle.decode_step(work, k=128)
    assert idxc[0][:N].tolist() == list(range(N)) and (idxc[0][N:] == -1).all()
    rows = [brute_kv_row(comp, [1, 0][e // 64], e % 64) for e in range(N)] + \
           [brute_kv_row(win, 0, 3), brute_kv_row(win, 0, 4)]
    ref = dense_sink_softmax(torch_bf16(q[0]), np.array(rows), np.array([0.5, -0.5]), 0.05)
    np.testing.assert_allclose(out[0], ref, rtol=1e-11, atol=1e-13)


# ---------------------------------------------------------------- KV-cache writer

def torch_e4m3_cast(x):
    """torch's fp32 -> float8_e4m3fn conversion (round to nearest even) as codes."""
    return torch.from_numpy(np.asarray(x, np.float32).copy()).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_e4m3_encode_matches_torch_cast():
    vals = oracle.e4m3_decode(np.arange(0, 0x7F, dtype=np.uint8))            # +0 .. 448
    mids = (vals[:-1] + vals[1:]) / 2                                        # exact ties
    f32 = lambda a: np.asarray(a, np.float64).astype(np.float32)
    up = np.nextafter(f32(mids), np.float32(np.inf))
    dn = np.nextafter(f32(mids), np.float32(-np.inf))
    rng = np.random.default_rng(40)
    rand = np.concatenate([rng.uniform(-448, 448, 20000), rng.uniform(-0.02, 0.02, 5000),
                           rng.standard_normal(5000) * 3]).astype(np.float32)
    x = np.concatenate([f32(vals), -f32(vals), f32(mids), -f32(mids), up, dn, -up, -dn, rand,
                        np.array([0.0, -0.0], np.float32)])
    x = x[np.abs(x) <= 448]
    assert np.array_equal(oracle.e4m3_encode(x), torch_e4m3_cast(x))


def test_e4m3_encode_decode_roundtrip():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)
    assert np.array_equal(oracle.e4m3_encode(oracle.e4m3_decode(codes).astype(np.float32)), codes)


def bf16_bits(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_quantize_hand_block():
    g = GOLD["quantize"]
    x = np.zeros(64, np.float32)
    x[:len(g["values"])] = g["values"]
    codes, scale = oracle.quantize_blocks(bf16_bits(x))
    assert codes[:len(g["codes"])].tolist() == g["codes"]
    assert (codes[len(g["codes"]):] == g["zero_rest_code"]).all()
    assert scale.view(np.uint32).tolist() == [g["scale_bits"]]


def test_quantize_invariants():
    rng = np.random.default_rng(41)
    x = (rng.standard_normal((20, 448)) * rng.uniform(1e-3, 50, (20, 1))).astype(np.float32)
    x[3, 64:128] = 0.0                                  # an all-zero block
    x[4, :64] = 1e-6                                    # below the amax floor
    for r in range(20):
        bits = bf16_bits(x[r])
        xr = torch_bf16(bits).reshape(7, 64)
        codes, scale = oracle.quantize_blocks(bits)
        codes = codes.reshape(7, 64)
        assert scale.shape == (7,) and (scale > 0).all()
        for b in range(7):
            amax = np.abs(xr[b]).max()
            if amax >= 1e-4:
                # the largest magnitude maps to the format's maximum
                assert (torch_e4m3(codes[b]) == np.sign(xr[b][np.argmax(np.abs(xr[b]))]) * 448).any()
            else:
                assert np.isclose(scale[b], 1e-4 / 448, rtol=1e-6)
            # dequantised values are within half an E4M3 step (relative 2^-4, or the subnormal step)
            deq = torch_e4m3(codes[b]) * float(scale[b])
            step = np.maximum(np.abs(xr[b]) * 2.0 ** -4, 2.0 ** -9 * float(scale[b]))
            assert (np.abs(deq - xr[b]) <= step * 1.0001).all()
        if r == 3:
            assert (codes[1] == 0).all()                # an all-zero block gives zero codes
    # blocks are independent: changing one block leaves the others' codes and scales alone
    y = x[0].copy()
    y[64:128] *= 7.0
    c0, s0 = oracle.quantize_blocks(bf16_bits(x[0]))
    c1, s1 = oracle.quantize_blocks(bf16_bits(y))
    keep = np.ones(448, bool)
    keep[64:128] = False
    assert np.array_equal(c0[keep], c1[keep]) and np.array_equal(np.delete(s0, 1), np.delete(s1, 1))


def test_kv_and_key_write_roundtrip():
    rng = np.random.default_rng(42)
    pool = small_kv_pool(rng, 3)
    before = {k: v.copy() for k, v in pool.items()}
    pt = np.array([2, 0, 1])
    entries = np.array([5, 64, 130, 191])
    rows = (rng.standard_normal((4, 512)) * 2).astype(np.float32)
    bits = bf16_bits(rows)
    oracle.kv_write(pool, pt, entries, bits)
    got = oracle.kv_rows(pool, pt, entries)
    ref = torch_bf16(bits)
    np.testing.assert_array_equal(got[:, 448:], ref[:, 448:])              # rope stored as is
    assert (np.abs(got[:, :448] - ref[:, :448]) <= np.abs(ref[:, :448]) * 2.0 ** -4 + 1e-3).all()
    touched = np.zeros((3, 64), bool)
    touched[pt[entries // 64], entries % 64] = True
    for k in pool:
        assert np.array_equal(pool[k][~touched], before[k][~touched])   # nothing else written
    keys = small_key_pool(rng, 2)
    kb = bf16_bits((rng.standard_normal((3, 128)) * 0.3).astype(np.float32))
    oracle.key_write(keys, np.array([1, 0]), np.array([0, 63, 64]), kb)
    kref = torch_bf16(kb)
    kgot = oracle.index_keys(keys, np.array([1, 0]), np.array([0, 63, 64]))
    assert (np.abs(kgot - kref) <= np.abs(kref) * 2.0 ** -4 + 1e-4).all()


# ---------------------------------------------------------------- inverse rotary embedding of the output

def _table_with(angle_of_pair: dict, rows: int = 4) -> np.ndarray:
    """A rotation table equal to 1 everywhere except the given (row, pair) angles."""
    t = np.ones((rows, 32), np.complex128)
    for (r, i), a in angle_of_pair.items():
        t[r, i] = np.exp(1j * a)
    return t


def test_inverse_rope_hand_cases():
    g = GOLD["inverse_rope"]
    angles = {"pi/2": np.pi / 2, "pi": np.pi, "-pi/2": -np.pi / 2}
    for case in g["cases"]:
        for i in (0, 17, 31):
            o = np.zeros((2, 512))
            o[1, 448 + 2 * i:450 + 2 * i] = g["pair"]
            out = oracle.inverse_rope(o, _table_with({(2, i): angles[case["angle"]]}), 2)
            np.testing.assert_allclose(out[1, 448 + 2 * i:450 + 2 * i], case["expect"], atol=1e-12)
            rest = np.delete(out, [448 + 2 * i, 449 + 2 * i], axis=1)
            assert not rest.any()


def test_inverse_rope_is_the_transposed_rotation_matrix():
    """Each pair (x, y) -> (c x + s y, -s x + c y), c = cos(p f_i), s = sin(p f_i),
    computed here from the angles directly (not from the complex table)."""
    rng = np.random.default_rng(70)
    freqs = oracle.base_freqs(10000.0)
    table = oracle.rope_table(freqs, 300)
    o = rng.standard_normal((5, 3, 512))
    pos = np.array([0, 1, 57, 200, 299])
    out = oracle.inverse_rope(o, table, pos)
    np.testing.assert_array_equal(out[..., :448], o[..., :448])
    for t in range(5):
        for i in range(32):
            c, s = np.cos(pos[t] * freqs[i]), np.sin(pos[t] * freqs[i])
            x, y = o[t, :, 448 + 2 * i], o[t, :, 449 + 2 * i]
            np.testing.assert_allclose(out[t, :, 448 + 2 * i], c * x + s * y, atol=1e-12)
            np.testing.assert_allclose(out[t, :, 449 + 2 * i], -s * x + c * y, atol=1e-12)


def test_rope_invariants():
    rng = np.random.default_rng(71)
    freqs = oracle.base_freqs(10000.0)
    # the frequencies: 1 at pair 0, a geometric sequence of ratio base^(-1/32), 10000^(-1/2) = 0.01 at pair 16
    assert freqs[0] == 1.0 and abs(freqs[16] - 0.01) < 1e-15
    np.testing.assert_allclose(freqs[1:] / freqs[:-1], 10000.0 ** (-1 / 32), rtol=1e-12)
    table = oracle.rope_table(freqs, 64)
    np.testing.assert_allclose(np.abs(table), 1.0, atol=1e-12)
    np.testing.assert_array_equal(table[0], np.ones(32))                      # position 0: identity
    np.testing.assert_allclose(table[9], table[1] ** 9, atol=1e-12)          # rows are powers of row 1
    o = rng.standard_normal((4, 2, 512))
    pos = np.array([3, 0, 63, 10])
    out = oracle.inverse_rope(o, table, pos)
    np.testing.assert_allclose(out[1], o[1], atol=0)                          # position 0 changes nothing
    norm = lambda a: a[..., 448::2] ** 2 + a[..., 449::2] ** 2
    np.testing.assert_allclose(norm(out), norm(o), rtol=1e-12)               # each pair keeps its length
    np.testing.assert_allclose(oracle.apply_rope(out, table, pos), o, atol=1e-12)   # forward undoes inverse
    # linear in o
    o2 = rng.standard_normal(o.shape)
    np.testing.assert_allclose(oracle.inverse_rope(2 * o - o2, table, pos),
                               2 * out - oracle.inverse_rope(o2, table, pos), atol=1e-12)


# ---------------------------------------------------------------- KV compressor

def _bf16(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16)


def _bits(x):
    return _bf16(x).view(torch.int16).numpy().view(np.uint16)


def _vals(bits):
    return torch.from_numpy(np.asarray(bits).view(np.int16)).view(torch.bfloat16).double().numpy()


def test_rms_norm_pins():
    rng = np.random.default_rng(80)
    x = rng.standard_normal((5, 512)) * 3
    y = oracle.rms_norm(x, np.ones(512), 0.0)
    np.testing.assert_allclose(np.mean(y * y, axis=1), 1.0, rtol=1e-12)          # unit mean square
    np.testing.assert_allclose(oracle.rms_norm(7.5 * x, np.ones(512), 0.0), y, rtol=1e-12)   # scale-free
    w = rng.uniform(0.5, 2, 512)
    np.testing.assert_allclose(oracle.rms_norm(x, w, 0.0), y * w, rtol=1e-12)
    # eps: a constant row c gives c / sqrt(c^2 + eps)
    np.testing.assert_allclose(oracle.rms_norm(np.full(512, 0.01), np.ones(512), 1e-4), 0.01 / math.sqrt(1e-4 + 1e-4))


def test_compressor_matches_brute_force_c4_overlap():
    """Window by window, feature by feature, with the slots listed explicitly and
    scipy's softmax (tiny sizes)."""
    from scipy.special import softmax
    rng = np.random.default_rng(81)
    T, d = 12, 512
    kv, sc = _bits(rng.standard_normal((T, 2 * d))), _bits(rng.standard_normal((T, 2 * d)) * 2)
    ape = rng.standard_normal((4, 2 * d)) * 0.3
    w = rng.uniform(0.5, 1.5, d)
    table = oracle.rope_table(oracle.base_freqs(160000.0), 16)
    got = oracle.compress_windows(kv, sc, ape, w, 4, True, table, eps=1e-6)
    K, S = _vals(kv), _vals(sc)
    assert got.shape == (3, d)
    for s in range(3):
        pooled = np.zeros(d)
        for f in range(d):
            slots_kv, slots_sc = [], []
            if s > 0:
                for j in range(4):
                    tok = 4 * (s - 1) + j
                    slots_kv.append(K[tok, f])
                    slots_sc.append(S[tok, f] + ape[j, f])
            for j in range(4):
                tok = 4 * s + j
                slots_kv.append(K[tok, d + f])
                slots_sc.append(S[tok, d + f] + ape[j, d + f])
            pooled[f] = np.dot(softmax(np.array(slots_sc)), np.array(slots_kv))
        normed = pooled / math.sqrt(np.mean(pooled ** 2) + 1e-6) * w
        ang = 4 * s * oracle.base_freqs(160000.0)
        z = (normed[448::2] + 1j * normed[449::2]) * np.exp(1j * ang)
        ref = normed.copy()
        ref[448::2], ref[449::2] = z.real, z.imag
        np.testing.assert_allclose(got[s], ref, rtol=1e-10, atol=1e-12)


def test_compressor_special_cases():
    rng = np.random.default_rng(82)
    d = 512
    kv_vals = rng.standard_normal((8, 2 * d))
    kv = _bits(kv_vals)
    K = _vals(kv)
    ape = np.zeros((4, 2 * d))
    ones = np.ones(d)
    table = oracle.rope_table(np.zeros(32), 8)          # zero frequencies: no rotation at all
    # equal scores: window 0 averages its own 4 tokens' last half (the previous-window slots are empty),
    # window 1 averages 8 slots: window 0's first halves and window 1's last halves
    sc = _bits(np.zeros((8, 2 * d)))
    got = oracle.compress_windows(kv, sc, ape, ones, 4, True, table, eps=0.0)
    p0 = K[0:4, d:].mean(axis=0)
    p1 = np.concatenate([K[0:4, :d], K[4:8, d:]]).mean(axis=0)
    np.testing.assert_allclose(got[0], p0 / np.sqrt(np.mean(p0 ** 2)), rtol=1e-10)
    np.testing.assert_allclose(got[1], p1 / np.sqrt(np.mean(p1 ** 2)), rtol=1e-10)
    # one dominant slot per feature: the pooled value is that slot's kv
    s = np.full((8, 2 * d), -30.0)
    s[2, :d] = 30.0          # token 2 of window 0, overlapping half: slot 2 of window 1
    s[1, d:] = 30.0          # token 1 of window 0, normal half: slot 5 of window 0
    got = oracle.compress_windows(kv, _bits(s), ape, ones, 4, True, table, eps=0.0)
    np.testing.assert_allclose(got[0], K[1, d:] / np.sqrt(np.mean(K[1, d:] ** 2)), rtol=1e-9)
    w1 = K[4:8, d:]          # window 1: the dominant slot is window 0's token 2, first half
    np.testing.assert_allclose(got[1], K[2, :d] / np.sqrt(np.mean(K[2, :d] ** 2)), rtol=1e-9)
    assert w1.shape == (4, d)


def test_online_c128_equals_offline():
    """Running max / sum over the tokens (P2 算法3) gives the window softmax exactly
    (up to rounding), window after window, and resets between windows."""
    rng = np.random.default_rng(83)
    d = 512
    kv, sc = _bits(rng.standard_normal((384, d))), _bits(rng.standard_normal((384, d)) * 3)
    ape = rng.standard_normal((128, d)) * 0.2
    w = rng.uniform(0.5, 1.5, d)
    table = oracle.rope_table(oracle.base_freqs(160000.0), 400)
    off = oracle.compress_windows(kv, sc, ape, w, 128, False, table)
    st = oracle.online_c128_init()
    on = []
    for i in range(384):
        r = oracle.online_c128_step(st, kv[i], sc[i], ape, w, table, i // 128)
        assert (r is None) == ((i + 1) % 128 != 0)
        if r is not None:
            on.append(r)
    np.testing.assert_allclose(np.array(on), off, rtol=1e-10, atol=1e-12)


# ---------------------------------------------------------------- FP4 (E2M1) indexer variant

def bf16_bits_of(values):
    """BF16 bit patterns of values that BF16 holds exactly."""
    v = np.asarray(values, np.float32)
    bits = (v.view(np.uint32) >> 16).astype(np.uint16)
    assert np.array_equal(torch_bf16(bits), v.astype(np.float64)), "value not exact in BF16"
    return bits


def test_e2m1_hand_values():
    g = GOLD["e2m1"]
    got = oracle.e2m1_decode(g["codes"])
    assert np.array_equal(got, np.array(g["values"]))
    assert np.array_equal(np.signbit(got), np.signbit(np.array(g["values"])))   # -0 for code 8
    assert np.array_equal(oracle.e2m1_decode(np.array(g["codes"]) | 0xF0), got)   # high bits ignored


def test_e2m1_encode_ties_and_roundtrip():
    g = GOLD["e2m1"]
    assert oracle.e2m1_encode(g["ties"]["values"]).tolist() == g["ties"]["codes"]
    for c in range(16):
        assert int(oracle.e2m1_encode(oracle.e2m1_decode(c))) == c
    # brute force over all 16 codes on fp32 values across [-6, 6], just off every midpoint too
    mags = np.array(GOLD["e2m1"]["values"][:8])
    mids = (mags[1:] + mags[:-1]) / 2
    xs = np.concatenate([np.linspace(-6, 6, 2001), mids, -mids,
                         np.nextafter(mids.astype(np.float32), np.float32(0)),
                         np.nextafter(mids.astype(np.float32), np.float32(7))]).astype(np.float32)
    table = np.array(GOLD["e2m1"]["values"])
    for x in xs:
        d = np.abs(table - float(x))
        best = [c for c in range(16) if d[c] == d.min() and (np.signbit(table[c]) == np.signbit(x) or table[c] != 0)]
        best = [c for c in best if (c & 1) == 0] or best          # ties to the even code
        if x == 0:
            best = [8 if np.signbit(x) else 0]
        assert int(oracle.e2m1_encode(x)) == best[0], (float(x), best)
    with pytest.raises(ValueError):
        oracle.e2m1_encode(6.5)


def test_e8m0_decode():
    assert oracle.e8m0_decode(127) == 1.0 and oracle.e8m0_decode(128) == 2.0 and oracle.e8m0_decode(124) == 0.125
    assert oracle.e8m0_decode(1) == 2.0 ** -126 and np.isnan(oracle.e8m0_decode(255))


def test_fp4_scale_exponent_hand_and_bitfield_rule():
    g = GOLD["fp4_scale"]
    assert oracle.fp4_scale_exponent(g["amax"]).tolist() == g["exponent"]
    # against the exponent / mantissa field rule of P1 §3.3 fast_log2_ceil, on fp32 values
    rng = np.random.default_rng(41)
    amax = np.concatenate([np.exp2(rng.uniform(-130, 120, 4000)), 6.0 * np.exp2(np.arange(-126, 120))]).astype(np.float32)
    t = (np.maximum(amax, np.float32(6.0 * 2.0 ** -126)) * np.float32(1.0 / 6.0)).astype(np.float32)
    bits = t.view(np.uint32)
    field = ((bits >> 23) & 0xFF).astype(np.int64) - 127 + ((bits & 0x7FFFFF) != 0)
    assert np.array_equal(oracle.fp4_scale_exponent(amax), field)


def test_fp4_quantize_hand_blocks():
    for blk in GOLD["fp4_scale"]["blocks"]:
        codes, e8m0 = oracle.fp4_quantize(bf16_bits_of(blk["values"]))
        assert codes.tolist() == blk["codes"] and e8m0.tolist() == [blk["e8m0"]]


def test_fp4_quantize_invariants():
    rng = np.random.default_rng(42)
    x = (rng.standard_normal((64, 128)) * np.exp2(rng.integers(-20, 20, (64, 1)))).astype(np.float32)
    x[3, :32] = 0.0                       # a zero block: the floor scale, zero codes
    x[5, 32:64] = 1e-39                   # under the floor
    for row in x:
        bits = (row.view(np.uint32) >> 16).astype(np.uint16)      # truncation to BF16 is data generation
        xv = torch_bf16(bits).reshape(-1, 32)
        codes, e8m0 = oracle.fp4_quantize(bits)
        scale = np.exp2(e8m0.astype(np.float64) - 127)
        deq = oracle.e2m1_decode(codes).reshape(-1, 32) * scale[:, None]
        for b in range(4):
            amax = np.abs(xv[b]).max()
            if amax > 6.0 * 2.0 ** -126:
                m = np.abs(deq[b]).max() / scale[b]
                assert 3.0 <= m <= 6.0                               # the block max lands in the top binade
            else:
                assert e8m0[b] == 1
            # error: at most half the grid step at the value's magnitude (0.5 below 2, 1 up to 4, 2 above)
            y = np.abs(xv[b]) / scale[b]
            half_step = np.where(y < 2, 0.25, np.where(y < 4, 0.5, 1.0))
            assert np.all(np.abs(xv[b] / scale[b] - deq[b] / scale[b]) <= half_step + 1e-12)


def test_indexer_fp4_equals_fp8_on_the_same_values():
    """An FP4 pool whose two 32-value blocks of each 64-dim half share their
    exponent holds values an FP8 pool (E4M3 codes, fp32 scale 2^e per 64) holds
    exactly: both oracles must give the same scores bit for bit."""
    rng = np.random.default_rng(43)
    P, n, Hi = 6, 300, 8
    pt = rng.permutation(P).astype(np.int32)
    e64 = rng.integers(120, 132, (P, 64, 2))
    fp4 = {"codes": rng.integers(0, 16, (P, 64, 128)).astype(np.uint8), "e8m0": np.repeat(e64, 2, axis=2).astype(np.uint8)}
    fp8 = {"codes": oracle.e4m3_encode(oracle.e2m1_decode(fp4["codes"])),
           "scale": np.exp2(e64.astype(np.float64) - 127).astype(np.float32)}
    qe = rng.integers(124, 130, (Hi, 2))
    q4, q4e = rng.integers(0, 16, (Hi, 128)).astype(np.uint8), np.repeat(qe, 2, axis=1).astype(np.uint8)
    q8, q8s = oracle.e4m3_encode(oracle.e2m1_decode(q4)), np.exp2(qe.astype(np.float64) - 127).astype(np.float32)
    w = rng.uniform(-0.5, 1.0, Hi)
    a = oracle.indexer_logits_row_fp4(q4, q4e, w, fp4, pt, n)
    b = oracle.indexer_logits_row(q8, q8s, w, fp8, pt, n)
    assert np.array_equal(a, b)


def test_indexer_fp4_brute_force_loops():
    rng = np.random.default_rng(44)
    P, n, Hi = 2, 70, 3
    pt = np.array([1, 0], np.int32)
    pool = {"codes": rng.integers(0, 16, (P, 64, 128)).astype(np.uint8), "e8m0": rng.integers(118, 136, (P, 64, 4)).astype(np.uint8)}
    q, qe = rng.integers(0, 16, (Hi, 128)).astype(np.uint8), rng.integers(120, 134, (Hi, 4)).astype(np.uint8)
    w = [0.7, -0.2, 1.3]
    table = GOLD["e2m1"]["values"]
    ref = []
    for s in range(n):
        pg, sl = pt[s // 64], s % 64
        tot = 0.0
        for h in range(Hi):
            dot = 0.0
            for d in range(128):
                kv = table[pool["codes"][pg, sl, d]] * 2.0 ** (int(pool["e8m0"][pg, sl, d // 32]) - 127)
                qv = table[q[h, d]] * 2.0 ** (int(qe[h, d // 32]) - 127)
                dot += qv * kv
            tot += w[h] * max(dot, 0.0)
        ref.append(tot)
    got = oracle.indexer_logits_row_fp4(q, qe, w, pool, pt, n)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-300)


def test_key_write_fp4_roundtrip():
    rng = np.random.default_rng(45)
    P = 3
    pool = {"codes": np.zeros((P, 64, 128), np.uint8), "e8m0": np.zeros((P, 64, 4), np.uint8)}
    pt = np.array([2, 0, 1], np.int32)
    entries = np.array([0, 65, 130, 191])
    keys = (rng.standard_normal((4, 128)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    oracle.key_write_fp4(pool, pt, entries, keys)
    got = oracle.index_keys_fp4(pool, pt, entries)
    for r in range(4):
        codes, e8m0 = oracle.fp4_quantize(keys[r])
        assert np.array_equal(got[r], oracle.fp4_dequantize(codes, e8m0))
        x = torch_bf16(keys[r])
        assert np.all(np.abs(got[r] - x) <= np.repeat(np.exp2(e8m0.astype(np.float64) - 127), 32) * 1.0 + 1e-30)


# ---------------------------------------------------------------- Hadamard rotation (compressor rotate path)

def test_hadamard_matrix_is_scipys():
    import scipy.linalg
    for d in (1, 2, 4, 8, 16, 32, 64, 128, 256):
        assert np.array_equal(oracle.hadamard_matrix(d), scipy.linalg.hadamard(d))
    with pytest.raises(ValueError):
        oracle.hadamard_matrix(96)


def test_hadamard_rotate_is_orthonormal_and_an_involution():
    rng = np.random.default_rng(50)
    x = rng.standard_normal((20, 128))
    y = oracle.hadamard_rotate(x)
    np.testing.assert_allclose(np.linalg.norm(y, axis=1), np.linalg.norm(x, axis=1), rtol=1e-12)
    np.testing.assert_allclose(oracle.hadamard_rotate(y), x, atol=1e-12)
    e = np.zeros(128)
    e[37] = 1.0                                            # a unit vector: column 37 of H / sqrt(128)
    np.testing.assert_allclose(oracle.hadamard_rotate(e) * math.sqrt(128), oracle.hadamard_matrix(128)[:, 37],
                               rtol=1e-15, atol=0)


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(51)
    v = np.concatenate([rng.standard_normal(5000) * np.exp2(rng.integers(-30, 30, 5000)),
                        # exact ties between two BF16 values, both parities of the lower one
                        (np.arange(1, 2000, dtype=np.uint32) << 15).view(np.float32).astype(np.float64)]).astype(np.float32)
    want = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle.fp32_to_bf16_bits(v), want)


def _fp32_butterflies(v, strides):
    """fp32 Hadamard butterflies over the last axis in the given stride order
    (a, b) -> (a + b, a - b), then the fp32 scale d^-0.5 (an evaluation a GPU may use)."""
    v = np.asarray(v, np.float32).copy()
    d = v.shape[-1]
    for h in strides:
        w = v.reshape(v.shape[:-1] + (d // (2 * h), 2, h))
        a, b = w[..., 0, :], w[..., 1, :]
        v = np.stack([(a + b).astype(np.float32), (a - b).astype(np.float32)], axis=-2).reshape(v.shape)
    return (v * np.float32(d ** -0.5)).astype(np.float32)


def _fp32_pairwise(v, h):
    """fp32 products H[i, j] x[j] summed by a balanced pairwise tree (depth log2 d), then scaled."""
    v = np.asarray(v, np.float32)
    prod = (v[..., None, :] * h.astype(np.float32)).astype(np.float32)     # [..., d, d]
    while prod.shape[-1] > 1:
        prod = (prod[..., 0::2] + prod[..., 1::2]).astype(np.float32)
    return (prod[..., 0] * np.float32(v.shape[-1] ** -0.5)).astype(np.float32)


def test_fp64_to_bf16_rounding_matches_torch():
    """The one rounding of the exact rotation: on values that fp32 holds exactly,
    it must be torch's fp32 -> BF16 cast (nearest, ties to even)."""
    rng = np.random.default_rng(54)
    v = np.concatenate([rng.standard_normal(5000) * np.exp2(rng.integers(-60, 60, 5000)),
                        (np.arange(1, 2000, dtype=np.uint32) << 15).view(np.float32).astype(np.float64),
                        -(np.arange(1, 500, dtype=np.uint32) << 15).view(np.float32).astype(np.float64),
                        [0.0, -0.0, 2.0 ** -130, 3 * 2.0 ** -134]]).astype(np.float32)
    want = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle.fp64_to_bf16_bits(v.astype(np.float64)), want)
    # an fp64 value just above a BF16 tie rounds up even when fp32 would have rounded it onto the tie
    tie = np.float64(1.0 + 2.0 ** -8)
    assert oracle.fp64_to_bf16_bits(tie) == 0x3F80                     # tie: to the even neighbour 1.0
    assert oracle.fp64_to_bf16_bits(tie + 2.0 ** -40) == 0x3F81        # above the tie: up


def test_fp32_evaluations_stay_inside_the_bound():
    """Three fp32 evaluations of the rotation (butterflies with increasing and
    with decreasing strides, a pairwise-summed product with scipy's matrix) all
    lie within hadamard_rotate_fp32_bound of the exact fp64 rotation, and the
    bound is far below a BF16 half-ulp of a typical output (so the GPU
    comparison that uses it stays exact almost everywhere)."""
    import scipy.linalg
    rng = np.random.default_rng(52)
    x = (rng.standard_normal((200, 128)) * np.exp2(rng.integers(-8, 8, (200, 1)))).astype(np.float32)
    x = oracle.bf16_decode((x.view(np.uint32) >> 16).astype(np.uint16))
    exact = oracle.hadamard_rotate(x)
    bound = oracle.hadamard_rotate_fp32_bound(x)
    h = scipy.linalg.hadamard(128)
    for got in (_fp32_butterflies(x, [1, 2, 4, 8, 16, 32, 64]), _fp32_butterflies(x, [64, 32, 16, 8, 4, 2, 1]),
                _fp32_pairwise(x, h)):
        assert np.all(np.abs(got.astype(np.float64) - exact) <= bound)
    rel = bound / np.maximum(np.abs(exact), 1e-300)
    assert np.median(rel) < 1e-4                   # BF16 half-ulp is 2^-9 relative
    # a constant row: every butterfly exact, the whole mass on element 0
    ones = np.full((1, 128), 0x3F80, np.uint16)                        # BF16 1.0
    r = oracle.bf16_decode(oracle.hadamard_rotate_to_bf16(ones))[0]
    want = torch.tensor(128.0 * 128 ** -0.5, dtype=torch.float64).to(torch.bfloat16).double().item()
    assert r[0] == want and np.all(r[1:] == 0.0)


def test_hadamard_rotate_to_bf16_is_the_rounded_definition():
    """The oracle's rotated BF16 key is the exact rotation rounded once: every
    element within half a BF16 ulp of the fp64 value, and equal to torch's BF16
    cast of it wherever fp32 holds the exact value."""
    rng = np.random.default_rng(55)
    bits = (rng.standard_normal((64, 128)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    got = oracle.bf16_decode(oracle.hadamard_rotate_to_bf16(bits))
    exact = oracle.hadamard_rotate(oracle.bf16_decode(bits))
    _, e = np.frexp(exact)
    assert np.all(np.abs(got - exact) <= np.ldexp(1.0, e - 9))
    f32_exact = exact.astype(np.float32).astype(np.float64) == exact
    via_torch = torch.from_numpy(exact.astype(np.float32)).to(torch.bfloat16).double().numpy()
    assert np.array_equal(got[f32_exact], via_torch[f32_exact])


def test_rotated_fp4_keys_reconstruct_the_keys():
    """Writing rotated keys and rotating the dequantised result back recovers
    the keys within the FP4 error: the rotation is orthonormal, so the error
    norm is the quantisation error of the rotated key plus its BF16 rounding."""
    rng = np.random.default_rng(53)
    P = 2
    pool = {"codes": np.zeros((P, 64, 128), np.uint8), "e8m0": np.zeros((P, 64, 4), np.uint8)}
    pt = np.array([1, 0], np.int32)
    entries = np.array([0, 3, 64, 127])
    keys = (rng.standard_normal((4, 128)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    oracle.key_write_fp4_rotated(pool, pt, entries, keys)
    deq = oracle.index_keys_fp4(pool, pt, entries)
    back = oracle.hadamard_rotate(deq)                       # H / sqrt(d) is its own inverse
    x = oracle.bf16_decode(keys)
    rot = oracle.hadamard_rotate(x)
    # the FP4 grid step is at most 2 * 2^e per value; half of it per value in norm
    scale = np.repeat(oracle.e8m0_decode(pool["e8m0"][pt[entries // 64], entries % 64]), 32, axis=1)
    err_bound = np.linalg.norm(scale, axis=1) + np.linalg.norm(rot, axis=1) * 2.0 ** -8
    assert np.all(np.linalg.norm(back - x, axis=1) <= err_bound)
    assert np.all(np.linalg.norm(back - x, axis=1) < 0.5 * np.linalg.norm(x, axis=1))
