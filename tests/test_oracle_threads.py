"""The oracle's results do not depend on how many host threads compute them.

The oracle splits its element-wise loops (reduce, AdamW, casts) over OpenMP threads with a static
schedule, each element computed alone, and sums the squares for the clip norm in one fixed order; so
one thread and every thread must give the same bits. (The timed CPU baseline runs on all cores; this
pins that its results are the one-thread definition's.)
"""
import numpy as np
import pytest

import oracle
import synth


def _inputs(n, N, seed):
    grads = [synth.host_range(synth.normal(1e-3, synth.BF16, synth.GRAD, r, seed), 0, n) for r in range(N)]
    master = synth.host_range(synth.normal(0.02, synth.FP32, synth.MASTER, seed=seed), 0, n).view(np.float32).copy()
    m = synth.host_range(synth.normal(1e-4, synth.FP32, synth.MOM1, seed=seed), 0, n).view(np.float32).copy()
    v = synth.host_range(synth.normal(1e-8, synth.FP32, synth.MOM2, seed=seed, absolute=True), 0,
                         n).view(np.float32).copy()
    return grads, master, m, v


def _run(n, N, seed):
    grads, master, m, v = _inputs(n, N, seed)
    g = oracle.grad_reduce(grads, oracle.BF16, post_scale=0.5)
    p16 = oracle.adamw(1e-3, 0.9, 0.999, 1e-8, 0.01, 7, g, master, m, v, p16_dtype=oracle.BF16, grad_scale=0.75)
    bounds = np.array([0, n // 3, n // 3 + 5, n], dtype=np.int64)
    flat = oracle.unshard([p16[:n // 3], p16[n // 3:n // 3 + 5], p16[n // 3 + 5:]], bounds)
    return g, master, m, v, p16, flat, oracle.sumsq(g)


@pytest.mark.parametrize("n,N", [(1_000_003, 8), (262_147, 3)])
def test_one_thread_and_all_threads_agree_bit_for_bit(n, N):
    threads = oracle.max_threads()
    try:
        oracle.set_threads(1)
        one = _run(n, N, 4)
        oracle.set_threads(max(threads, 4))
        many = _run(n, N, 4)
    finally:
        oracle.set_threads(threads)
    for a, b in zip(one[:6], many[:6]):
        assert np.array_equal(np.asarray(a).view(np.uint8), np.asarray(b).view(np.uint8))
    assert one[6] == many[6]
