"""GPU parity of the inverse rotary embedding fused into the attention output
(dsv4sa_attn_args.rope_cs / rope_pos) against oracle.inverse_rope applied to
the fp64 oracle attention.  Covered: the one-CTA-per-query finalisation
(prefill mode), the cluster merge of decode splits, the workspace merge kernel,
and an out-of-range position (flagged; that query left unrotated)."""
import math

import numpy as np
import pytest
import torch

import oracle
from compressed_sparse_attention_c4_gb300 import workloads as W
from parity import ATTN_MAX_ABS, ATTN_MEAN_ABS, ATTN_REL, GpuRun, oracle_attention

pytestmark = pytest.mark.gpu


def fp32_table(rows, base=10000.0):
    """The oracle's rotation table rounded to fp32 pairs [rows, 32, 2] (what a
    caller precomputes once), and the same values back as fp64 complex."""
    t = oracle.rope_table(oracle.base_freqs(base), rows)
    cs = np.stack([t.real, t.imag], axis=-1).astype(np.float32)
    return cs, cs[..., 0].astype(np.float64) + 1j * cs[..., 1].astype(np.float64)


def rerun(run, mode, rope_cs=None, rope_pos=None):
    L, d, w = run.L, run.d, run.w
    fn = L.dsv4sa_sparse_attn_decode if mode == L.ATTN_DECODE else L.dsv4sa_sparse_attn_prefill
    d.out.fill_(0)
    fn(d.q, d.sink, d.q_seq, d.comp, d.comp_pt, d.idx_c, d.win, d.win_pt, d.idx_w, d.out, w.softmax_scale,
       lse=d.lse, ws=d.attn_ws, rope_cs=rope_cs, rope_pos=rope_pos)
    torch.cuda.synchronize()
    return d.out.float().cpu().numpy()


def check_rotated(run, got, table, pos, rows):
    w = run.w
    for t in rows:
        ref = oracle.inverse_rope(oracle_attention(w, t, run.idx_c[t], run.idx_w[t]), table, int(pos[t]))
        err = np.abs(got[t] - ref)
        assert np.isfinite(got[t]).all()
        assert err.max() <= ATTN_MAX_ABS, f"row {t}: max abs err {err.max()}"
        assert err.mean() <= ATTN_MEAN_ABS, f"row {t}: mean abs err {err.mean()}"
        assert err.max() <= ATTN_REL * max(np.abs(ref).max(), 1e-30), f"row {t}: relative err"


@pytest.mark.parametrize("case", ["prefill_finalise", "decode_cluster", "decode_workspace"])
def test_inverse_rope_matches_oracle(case):
    from compressed_sparse_attention_c4_gb300 import dsv4sa as L
    if case == "prefill_finalise":
        w = W.make_decode_like("rope8", B=8, L=[5000 + 3001 * i for i in range(8)], H=64, Hi=16, kv_std=1.0,
                               key_std=1 / math.sqrt(128), seed=409)
        mode = L.ATTN_PREFILL
    elif case == "decode_cluster":
        B = 40
        w = W.make_decode_like("rope40", B=B, L=[16000 + 997 * i for i in range(B)], H=64, Hi=16, kv_std=1.0,
                               key_std=1 / math.sqrt(128), seed=410)
        mode = L.ATTN_DECODE
    else:
        B = 64
        lens = [131072, 65536, 9000] + [16000 + 997 * i for i in range(3, B)]
        w = W.make_decode_like("rope64", B=B, L=lens, H=16, Hi=16, kv_std=1.0, key_std=1 / math.sqrt(128),
                               c128_rows=[True] + [False] * (B - 1), seed=411)
        mode = L.ATTN_DECODE
    run = GpuRun(w, mode=mode)
    plan = L.dsv4sa_attn_plan(mode, w.T, w.H, w.kc, w.kw)
    want = {"prefill_finalise": (1, 1), "decode_cluster": (None, 1), "decode_workspace": (None, 2)}[case]
    assert plan["launches"] == want[1] and (want[0] is None or plan["nsplit"] == want[0]), plan
    if case == "decode_cluster":
        assert plan["nsplit"] > 1
    rows = int(np.max(w.pos)) + 1
    cs, table = fp32_table(rows)
    pos = np.asarray(w.pos, np.int64)
    plain = rerun(run, mode)
    got = rerun(run, mode, torch.from_numpy(cs).cuda(), torch.from_numpy(pos.astype(np.int32)).cuda())
    assert L.dsv4sa_check_errors() == (0, 0)
    # the rotation touches only the last 64 dims, and rotates the same values
    np.testing.assert_array_equal(got[..., :448], plain[..., :448])
    check_rotated(run, got, table, pos, range(min(w.T, 24)))


def test_out_of_range_position_is_flagged_and_left_unrotated():
    from compressed_sparse_attention_c4_gb300 import dsv4sa as L
    w = W.make_decode_like("rope6", B=6, L=[3000, 9000, 40000, 12000, 700, 20000], H=64, Hi=16, kv_std=1.0,
                           key_std=1 / math.sqrt(128), seed=412)
    run = GpuRun(w, mode=L.ATTN_PREFILL)
    rows = int(np.max(w.pos)) + 1
    cs, table = fp32_table(rows)
    pos = np.asarray(w.pos, np.int32).copy()
    bad = [0, w.T - 1]
    pos[bad[0]] = rows          # one past the table
    pos[bad[1]] = -3
    plain = rerun(run, L.ATTN_PREFILL)
    got = rerun(run, L.ATTN_PREFILL, torch.from_numpy(cs).cuda(), torch.from_numpy(pos).cuda())
    st, bits = L.dsv4sa_check_errors()
    assert st == 5 and bits & 1
    for t in bad:
        np.testing.assert_array_equal(got[t], plain[t])
    good = [t for t in range(w.T) if t not in bad]
    check_rotated(run, got, table, pos, good[:8])
