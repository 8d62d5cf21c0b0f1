"""Failure reporting on the GPU without a fault.

The only waits in the library's kernels are the bulk-copy kernel's barrier waits, each bounded
by %globaltimer; on expiry a block sets bit 0 of the device error word and returns. The library's
self-test entry runs that same bounded wait on a barrier nothing completes, with a short limit:
the wait must give up after at least the limit, report through the word, and leave the context
usable for the next copy.
"""
import time

import numpy as np
import pytest

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ss():
    import fsdp_sharded_mixed_ss_gb300 as m
    return m


def test_bounded_wait_runs_out_and_reports(ss):
    import torch
    assert ss.ss_device_error(clear=True) == 0
    limit_ns = 50_000_000
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    ss.ss_selftest_wait_timeout(limit_ns)
    torch.cuda.synchronize()
    waited = time.perf_counter() - t0
    assert waited >= limit_ns * 1e-9                     # it waited out the limit ...
    assert waited < 10.0                                 # ... and then gave up
    assert ss.ss_device_error(clear=False) == 1          # bit 0: a bounded wait ran out
    assert ss.ss_device_error(clear=True) == 1
    assert ss.ss_device_error() == 0

    # the context is intact: a bulk-copy unshard right after runs, waits succeed, no error bit
    N, P = 8, 3 << 20
    _, bounds = ss.ss_flatten_layout([P], N)
    shards = [torch.arange(int(bounds[k]), int(bounds[k + 1]), device="cuda", dtype=torch.int32).to(torch.float32)
              for k in range(N)]
    flat = torch.empty(P, device="cuda")
    ss.ss_unshard(shards, bounds, flat)
    torch.cuda.synchronize()
    assert np.array_equal(flat.cpu().numpy(), np.arange(P, dtype=np.float32))
    assert ss.ss_device_error() == 0


def test_timeout_bit_survives_until_cleared(ss):
    """Two timed-out waits on different streams set the same bit once; clearing resets it."""
    import torch
    assert ss.ss_device_error(clear=True) == 0
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    for st in streams:
        ss.ss_selftest_wait_timeout(5_000_000, stream=st)
    torch.cuda.synchronize()
    assert ss.ss_device_error(clear=True) == 1
    assert ss.ss_device_error() == 0
