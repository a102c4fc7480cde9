"""The scratch-free top-k entry point (dsv4sa_topk_noalloc).

Some callers cannot allocate device memory when they call the library: a
serving engine that reserves all device memory in its own pool at start-up,
a runtime whose hot path must never take cudaMalloc's implicit
synchronisation, an embedded caller with no allocator.  dsv4sa_topk_noalloc
serves them with a fixed device scratch inside the library.  This test checks
that it returns exactly what dsv4sa_topk (with a caller workspace) returns, on
two calls in a row, and that a request beyond the scratch is refused.

The file is named so that pytest collects it last.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    import os
    from compressed_sparse_attention_c4_gb300 import build, dsv4sa
    if not os.path.exists(dsv4sa.LIB_PATH):
        build.build()
    return dsv4sa


def test_noalloc_topk_matches_workspace_entry_point(L):
    rng = np.random.default_rng(2024)
    lens = [0, 100, 512, 4096, 4097, 16384, 70000, 9000, -1]
    n_max, k, T = 70000, 512, len(lens)
    x = rng.integers(-300, 300, size=(T, n_max)).astype(np.float32)   # many ties
    x[2, :] = 1.5
    logits = torch.from_numpy(x).cuda()
    n_vis = torch.tensor(lens, dtype=torch.int32, device="cuda")
    ref = torch.full((T, k), -7, dtype=torch.int32, device="cuda")
    ws = torch.empty(L.dsv4sa_topk_workspace_size(T, n_max, k), dtype=torch.uint8, device="cuda")
    L.dsv4sa_topk(logits, n_vis, n_max, k, ref, ws)
    for _ in range(2):                               # two calls in a row share the scratch
        got = torch.full((T, k), -7, dtype=torch.int32, device="cuda")
        L.dsv4sa_topk_noalloc(logits, n_vis, n_max, k, got)
        torch.cuda.synchronize()
        assert torch.equal(got, ref)


def test_noalloc_topk_rejects_requests_beyond_the_scratch(L):
    T, n_max, k = 64, 1 << 20, 512                   # 64 x 64 chunks x 512 x 8 B = 16 MiB > 8 MiB
    logits = torch.zeros((T, n_max), dtype=torch.float32, device="cuda")
    n_vis = torch.full((T,), n_max, dtype=torch.int32, device="cuda")
    idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
    with pytest.raises(L.DSV4SAError) as e:
        L.dsv4sa_topk_noalloc(logits, n_vis, n_max, k, idx)
    assert e.value.status == 2
