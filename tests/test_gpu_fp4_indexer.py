"""GPU parity of the FP4 indexer (dsv4sa_indexer_logits_fp4) against the fp64
oracle's ``indexer_logits_row_fp4``.

Each 32-value block's E2M1 x E2M1 dot product is exact in fp32 (products are
multiples of 1/4 up to 36, sums of 32 stay below 2^11), and each E8M0 scale is
a power of two, so the only roundings are the three additions of the four
scaled block sums and the 2 x Hi operations of the ReLU-weighted head sum:
|gpu - oracle| <= 2e-5 * sum_h |w_h| sum_d |q_hd k_sd| (the bound the FP8
indexer is held to) is far outside what fp32 can accumulate here.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from compressed_sparse_attention_c4_gb300 import workloads as W

pytestmark = pytest.mark.gpu

LOGIT_REL = 2e-5


def upload(w):
    from compressed_sparse_attention_c4_gb300 import dsv4sa as L
    buf, desc = L.pack_key_pool_fp4(w.key_codes, w.key_e8m0, "cuda")
    d = dict(buf=buf, desc=desc,
             pt=torch.from_numpy(w.comp_pt).cuda(), q_seq=torch.from_numpy(w.q_seq).cuda(),
             n_vis=torch.from_numpy(w.n_vis).cuda(),
             q=torch.from_numpy(L.pack_fp4_codes(w.q_codes)).cuda(),
             qe=torch.from_numpy(np.ascontiguousarray(w.q_e8m0)).cuda(),
             w=torch.from_numpy(w.w).cuda())
    d["logits"] = torch.full((w.T, w.n_max + 5), 7.25, dtype=torch.float32, device="cuda")
    return d


def run(w):
    from compressed_sparse_attention_c4_gb300 import dsv4sa as L
    d = upload(w)
    L.dsv4sa_indexer_logits_fp4(d["desc"], d["pt"], d["q_seq"], d["n_vis"], d["q"], d["qe"], d["w"], w.n_max,
                                d["logits"])
    torch.cuda.synchronize()
    assert L.dsv4sa_check_errors() == (0, 0)
    return d["logits"].cpu().numpy()


def check(w, got, rows=None):
    pool = {"codes": w.key_codes, "e8m0": w.key_e8m0}
    for t in (range(w.T) if rows is None else rows):
        n = int(w.n_vis[t])
        s = int(w.q_seq[t])
        ref = oracle.indexer_logits_row_fp4(w.q_codes[t], w.q_e8m0[t], w.w[t], pool, w.comp_pt[s], n)
        if n:
            qd = np.abs(oracle.fp4_dequantize(w.q_codes[t], w.q_e8m0[t]))
            kd = np.abs(oracle.index_keys_fp4(pool, w.comp_pt[s], np.arange(n)))
            bound = LOGIT_REL * ((kd @ qd.T) @ np.abs(w.w[t].astype(np.float64))) + 1e-30
            err = np.abs(got[t, :n].astype(np.float64) - ref)
            bad = np.nonzero(err > bound)[0]
            assert bad.size == 0, f"row {t}: {bad.size} logits off, worst {err[bad].max()}"
        assert (got[t, n:] == 7.25).all(), f"row {t}: entries past n_vis were written"


@pytest.mark.parametrize("Hi", [1, 8, 16, 40, 64])
def test_fp4_indexer_heads_and_ragged_tails(Hi):
    # N = 1500 (ragged tile), 2250, 5000, 16 (one partial page), 0 (empty), 64 (one full page), 65, 128
    w = W.make_fp4_indexer(f"fp4h{Hi}", B=8, L=[6000, 9000, 20000, 64, 3, 256, 260, 512], Hi=Hi, seed=2000 + Hi)
    check(w, run(w))


def test_fp4_indexer_exponent_extremes():
    """Block exponents far apart inside one key (2^-20 .. 2^20 scales): each
    block's sum is scaled separately, so no block is lost to another's range."""
    w = W.make_fp4_indexer("fp4x", B=4, L=[8000, 4100, 12000, 500], Hi=16, seed=2101, e_lo=107, e_hi=147)
    check(w, run(w))


def test_fp4_indexer_decode64k_sampled():
    """The 64K-context decode shape (B = 32, N = 16384, Hi = 64), every logit of eight rows."""
    w = W.make_fp4_indexer("fp4d", B=32, L=65536, Hi=64, seed=2202)
    got = run(w)
    check(w, got, rows=[0, 5, 11, 16, 21, 26, 30, 31])


def test_fp4_indexer_rejects_wide_heads_and_wrong_pool():
    from compressed_sparse_attention_c4_gb300 import dsv4sa as L
    w = W.make_fp4_indexer("fp4r", B=2, L=[4000, 4000], Hi=8, seed=2303)
    d = upload(w)
    q_wide = torch.zeros((w.T, 65, 64), dtype=torch.uint8, device="cuda")
    e_wide = torch.zeros((w.T, 65, 4), dtype=torch.uint8, device="cuda")
    w_wide = torch.zeros((w.T, 65), dtype=torch.float32, device="cuda")
    with pytest.raises(RuntimeError, match="UNSUPPORTED|unsupported"):
        L.dsv4sa_indexer_logits_fp4(d["desc"], d["pt"], d["q_seq"], d["n_vis"], q_wide, e_wide, w_wide, w.n_max,
                                    d["logits"])
    kbuf = L._alloc_pool(L.POOL_IDXK, 4, "cuda")
    kdesc = L.dsv4sa_pool_desc_init(L.POOL_IDXK, kbuf, 4)
    with pytest.raises(RuntimeError, match="INVALID|invalid"):
        L.dsv4sa_indexer_logits_fp4(kdesc, d["pt"], d["q_seq"], d["n_vis"], d["q"], d["qe"], d["w"], w.n_max,
                                    d["logits"])
