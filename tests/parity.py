"""Comparison helpers shared by the GPU parity tests.

Tolerances (see the test module docstrings for the derivations):
* indexer logits: |gpu - oracle| <= 2e-5 * sum_h |w_h| sum_d |qhat_hd khat_sd|  (fp32 accumulation of
  at most 64 exact FP8 products per scale block, then a 64-term head sum);
* top-k on the library's own logits: bit-exact against the oracle's selection rule;
* top-k end to end: the selected set may differ from the oracle's only by entries whose fp64 score
  lies within 1e-3 relative of the oracle's k-th score;
* attention (BF16 output): max |err| <= 2e-2 and mean |err| <= 2e-3 against the fp64 oracle.
"""
import numpy as np
import torch

import oracle

ATTN_MAX_ABS = 2e-2
ATTN_MEAN_ABS = 2e-3
ATTN_REL = 2e-2     # scale-free check as well: max err <= 2e-2 * max |o| of the row
TIE_REL = 1e-3
LOGIT_REL = 2e-5


class GpuRun:
    """Run the whole path once through the C ABI and bring the results back.
    serving=True runs it as the benchmark does: the window indices derived in
    the attention kernel (early window start); the explicit list is then
    written afterwards by its own kernel, for the checks."""

    def __init__(self, w, mode=None, serving=False):
        from compressed_sparse_attention_c4_gb300 import dsv4sa as L
        self.L = L
        self.w = w
        self.d = L.upload(w, "cuda", mode)
        L.run_path(self.d, fused_window=serving)
        if serving:
            L.dsv4sa_window_indices(self.d.pos, w.kw, w.win_ring, self.d.idx_w)
        torch.cuda.synchronize()
        st, bits = L.dsv4sa_check_errors()
        assert st == 0 and bits == 0, (st, bits)
        self.logits = self.d.logits.cpu().numpy()
        self.idx_c = self.d.idx_c.cpu().numpy()
        self.idx_w = self.d.idx_w.cpu().numpy()
        self.out = self.d.out.float().cpu().numpy()
        self.lse = self.d.lse.cpu().numpy()


_KD = {"w": None, "s": -1, "kd": None}   # the last sequence's |dequantised keys|: its rows share them


def logit_bound(w, t, n):
    qd = np.abs(oracle.index_query(w.q_idx[t], w.q_idx_scale[t]))
    s = int(w.q_seq[t])
    if _KD["w"] is not w or _KD["s"] != s or _KD["kd"].shape[0] < n:
        n_seq = max(n, int(w.n_vis[w.q_seq == s].max()))
        _KD.update(w=w, s=s, kd=np.abs(oracle.index_keys(w.key_pool, w.comp_pt[s], np.arange(n_seq))))
    kd = _KD["kd"][:n]
    return LOGIT_REL * ((kd @ qd.T) @ np.abs(w.w[t].astype(np.float64))) + 1e-30


def check_logits(run, t):
    w = run.w
    n = int(w.n_vis[t])
    ref = oracle.indexer_logits_row(w.q_idx[t], w.q_idx_scale[t], w.w[t], w.key_pool, w.comp_pt[w.q_seq[t]], n)
    got = run.logits[t, :n].astype(np.float64)
    if n:
        err = np.abs(got - ref)
        bound = logit_bound(w, t, n)
        bad = np.nonzero(err > bound)[0]
        assert bad.size == 0, f"row {t}: {bad.size} logits off, worst {err[bad].max()} vs {bound[bad].min()}"
    return ref


def check_topk_exact(run, t):
    """Selection on the library's own fp32 logits must equal the oracle's rule exactly."""
    w = run.w
    n = int(w.n_vis[t])
    ref = oracle.topk_row(run.logits[t, :n].astype(np.float64), w.k)
    got = run.idx_c[t, :w.k]
    assert np.array_equal(got, ref), f"row {t}: top-k differs on identical scores"


def check_topk_vs_oracle(run, t, scores):
    w = run.w
    k = w.k
    ref = oracle.topk_row(scores, k)
    got = run.idx_c[t, :k]
    m = min(k, len(scores))
    assert (got[m:] == -1).all() and (np.diff(got[:m]) > 0).all()
    diff = np.setxor1d(ref[:m], got[:m])
    if diff.size:
        thr = scores[ref[:m]].min()
        far = diff[np.abs(scores[diff] - thr) > TIE_REL * abs(thr)]
        assert far.size == 0, f"row {t}: top-k differs beyond the tie band: {far[:8]}"
    return diff.size


def oracle_attention(w, t, idx_c_row, idx_w_row):
    s = int(w.q_seq[t])
    return oracle.sparse_attn_row(w.q[t], w.sink, w.softmax_scale, idx_c_row, w.comp_pool, w.comp_pt[s],
                                  idx_w_row, w.win_pool, w.win_pt[s])


def lse_reference(w, t, idx_c_row, idx_w_row):
    """log(sum_j e^{a_hj} + e^{sink_h}) from the oracle's gathered rows (the
    kernels' extra lse output; the pages' sparse_attn returns only o)."""
    s = int(w.q_seq[t])
    rows = oracle.gather_rows(idx_c_row, w.comp_pool, w.comp_pt[s], idx_w_row, w.win_pool, w.win_pt[s])
    q = oracle.bf16_decode(w.q[t])
    sink = np.asarray(w.sink, np.float64)
    a = w.softmax_scale * (q @ rows.T) if rows.shape[0] else np.zeros((q.shape[0], 0))
    M = np.maximum(a.max(axis=1, initial=-np.inf), sink)
    return M + np.log(np.exp(a - M[:, None]).sum(axis=1) + np.exp(sink - M))


LSE_ABS = 2e-2   # scores come from BF16 operands; a dropped or doubled split moves lse by ~0.1 or more


def check_attention(run, t, idx_c_row=None):
    w = run.w
    ic = run.idx_c[t] if idx_c_row is None else idx_c_row
    if run.lse is not None:
        lref = lse_reference(w, t, ic, run.idx_w[t])
        lerr = np.abs(run.lse[t] - lref).max()
        assert lerr <= LSE_ABS, f"row {t}: lse err {lerr}"
    ref = oracle_attention(w, t, ic, run.idx_w[t])
    got = run.out[t]
    err = np.abs(got - ref)
    assert np.isfinite(got).all(), f"row {t}: non-finite output"
    assert err.max() <= ATTN_MAX_ABS, f"row {t}: max abs err {err.max()}"
    assert err.mean() <= ATTN_MEAN_ABS, f"row {t}: mean abs err {err.mean()}"
    scale = np.abs(ref).max()
    if scale > 0:
        assert err.max() <= ATTN_REL * scale, f"row {t}: max err {err.max()} vs |o| {scale}"
    else:
        assert err.max() == 0.0, f"row {t}: an empty row must give exact zeros"
    return err.max(), err.mean(), float((err.max(axis=1) / (np.abs(ref).max(axis=1) + 1e-30)).max())


def check_row(run, t):
    """Everything for one query row: logits, exact top-k, top-k vs fp64, attention."""
    w = run.w
    assert np.array_equal(run.idx_w[t], oracle.window_indices(int(w.pos[t]), w.kw, w.win_ring))
    if w.c128[t]:
        assert np.array_equal(run.idx_c[t], oracle.compress_indices(int(w.n_vis[t]), w.kc))
    else:
        scores = check_logits(run, t)
        check_topk_exact(run, t)
        check_topk_vs_oracle(run, t, scores)
        assert (run.idx_c[t, w.k:] == -1).all()
    return check_attention(run, t)
