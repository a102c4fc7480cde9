"""Failure detection on the GPU without a fault: the library's bounded wait (the
code every kernel's mbarrier waits use) runs out on a barrier nothing arrives
on, reports DSV4SA_ERR_DEVICE_TIMEOUT through the device error word, and the
context stays usable for the path that follows."""
import time

import numpy as np
import pytest
import torch

from compressed_sparse_attention_c4_gb300 import workloads as W
from parity import GpuRun, check_row

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_the_context_survives():
    from compressed_sparse_attention_c4_gb300 import dsv4sa as L
    assert L.dsv4sa_check_errors() == (0, 0)
    res = torch.full((1,), 7, dtype=torch.int32, device="cuda")
    t0 = time.perf_counter()
    L.dsv4sa_selftest_wait_timeout(res)
    st, bits = L.dsv4sa_check_errors()
    elapsed = time.perf_counter() - t0
    assert st == 6 and bits & 2, (st, bits)      # DSV4SA_ERR_DEVICE_TIMEOUT
    assert res.item() == 0                        # the wait gave up
    assert 1.5 <= elapsed <= 30.0                 # after the 2 s wait limit, not never
    assert L.dsv4sa_check_errors() == (0, 0)      # read and cleared
    run = GpuRun(W.make("tiny"))                  # the context still runs the path
    check_row(run, 0)
    assert np.isfinite(run.out).all()


@pytest.mark.parametrize("background", [False, True])
def test_copy_kernel_between_host_and_device(background):
    """dsv4sa_copy_async and dsv4sa_copy_async_background (the step graph's
    input copies): pinned host -> device, device -> pinned host and device ->
    device, sizes with a ragged tail of 16-byte units and sizes above one
    grid-stride sweep."""
    from compressed_sparse_attention_c4_gb300 import dsv4sa as L
    copy = L.dsv4sa_copy_async_background if background else L.dsv4sa_copy_async
    g = torch.Generator().manual_seed(5)
    for n in (16, 4096 + 48, 320000, 2417920, 9 * 2 ** 20 + 16):
        src = torch.randint(0, 256, (n,), dtype=torch.uint8, generator=g).pin_memory()
        dev = torch.zeros(n, dtype=torch.uint8, device="cuda")
        copy(dev, src)
        back = torch.zeros(n, dtype=torch.uint8).pin_memory()
        dev2 = torch.empty_like(dev)
        copy(dev2, dev)
        copy(back, dev2)
        torch.cuda.synchronize()
        assert torch.equal(dev.cpu(), src) and torch.equal(back, src)
