"""World-size-2 check of bench.py's multi-rank host logic on CPU (gloo).

The path shards by sequence: each rank decodes its own batch with no
collective on the data path; the only collective is the max over ranks of
the step time.  Two gloo ranks check that the shards differ, that the max
reduction gives the slowest rank's time on every rank, and the whole-job
throughput formula."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, q):
    import numpy as np
    import torch
    import torch.distributed as dist
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    from compressed_sparse_attention_c4_gb300 import workloads as W
    r, wsz, local = bench.rank_env()
    ms = bench.reduce_max(10.0 + 5.0 * r, dist, "cpu")
    w = W.make_decode_like("shard", B=2, L=512, H=16, Hi=4, kv_std=1.0, key_std=1.0, seed=bench.shard_seed(r))
    digest = float(np.asarray(w.q[0, 0, :8], dtype=np.float64).sum())
    got = [None] * world
    dist.all_gather_object(got, digest)
    q.put((r, wsz, local, ms, bench.job_throughput(wsz, 32, ms), got))
    dist.destroy_process_group()


@pytest.mark.timeout(300)
def test_two_rank_host_logic():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=240) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r, (rank, wsz, local, ms, thr, digests) in enumerate(res):
        assert (rank, wsz, local) == (r, world, r)
        assert ms == 15.0                                   # the slowest rank's time, on every rank
        assert abs(thr - 2 * 32 / 0.015) < 1e-6
        assert digests[0] != digests[1]                     # independent shards
