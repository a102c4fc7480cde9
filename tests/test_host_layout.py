"""Host logic of the serving step (no GPU): the packed per-step input buffer.

StepGraph copies the packed inputs in two parts -- bytes [0, split) before the
indexer, [split, end) beside it for the attention -- so the layout must put
every input the indexer and the top-k read before `split`, keep every view
16-byte aligned for the copy kernels, and give views that alias the buffer
exactly (no gaps read as data, no overlaps).
"""
import numpy as np
import torch

from compressed_sparse_attention_c4_gb300 import dsv4sa as L
from compressed_sparse_attention_c4_gb300 import workloads as W


def specs_of(w):
    """The (name, shape, dtype) list upload() packs, from a workload's arrays."""
    shapes = {
        "q_idx": (w.q_idx.shape, torch.uint8), "q_idx_scale": (w.q_idx_scale.shape, torch.float32),
        "wts": (w.w.shape, torch.float32), "q_seq": (w.q_seq.shape, torch.int32),
        "n_vis_idx": (w.n_vis.shape, torch.int32), "comp_pt": (w.comp_pt.shape, torch.int32),
        "q": (w.q.shape, torch.bfloat16), "sink": (w.sink.shape, torch.float32),
        "pos": (w.pos.shape, torch.int32), "win_pt": (w.win_pt.shape, torch.int32),
    }
    return [(n, shapes[n][0], shapes[n][1]) for n in L.STEP_INPUTS]


def test_step_inputs_layout_and_split():
    for name in ("tiny", "decode", "ragged"):
        w = W.make(name)
        layout, total = L._arena_layout(specs_of(w))
        assert total % 256 == 0 and total >= 256
        ends = 0
        spans = []
        for n, off, nbytes, shape, dtype in layout:
            assert off % 256 == 0, (name, n, off)
            assert off >= ends, (name, n)            # packed in order, no overlap
            ends = off + nbytes
            spans.append((n, off, ends))
        assert ends <= total
        split = min(off for n, off, _, _, _ in layout if n in L.ATTN_ONLY_INPUTS)
        assert split % 16 == 0
        for n, off, end in spans:
            if n in L.ATTN_ONLY_INPUTS:
                assert off >= split
            else:
                assert end <= split, (name, n)       # read by the indexer or the top-k: copied first


def test_views_alias_the_buffer():
    w = W.make("tiny")
    layout, total = L._arena_layout(specs_of(w))
    buf = torch.zeros(total, dtype=torch.uint8)
    views = L._arena_views(buf, layout)
    rng = np.random.default_rng(3)
    written = {}
    for n, off, nbytes, shape, dtype in layout:
        v = views[n]
        assert tuple(v.shape) == tuple(shape) and v.dtype == dtype
        raw = torch.from_numpy(rng.integers(0, 256, nbytes, dtype=np.uint8))
        v.view(torch.uint8).view(-1).copy_(raw)
        written[n] = (off, raw)
    for n, (off, raw) in written.items():
        assert torch.equal(buf[off:off + raw.numel()], raw), n
    covered = np.zeros(total, bool)
    for n, off, nbytes, _, _ in layout:
        assert not covered[off:off + nbytes].any()
        covered[off:off + nbytes] = True
