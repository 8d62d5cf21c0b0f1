"""GPU parity of the whole shard step on the five workloads, through the C ABI.

Every input is generated on the device by the seeded generator and regenerated
on the host for the oracle. Bars (the stated tolerance): layout and copies
bit-exact; fp32 master, m and v within max(1e-6 * |ref|, 1e-9); 16-bit params
within 1 ulp. Small shards are compared element by element; large ones at
sampled elements (both ends of every shard, 16-element runs, random points),
plus properties over the whole buffer (unshard == concatenation, reshard
round trip bit-exact).
"""
import numpy as np
import pytest

import oracle
from synth import workloads

from parity import compare_workload, gpu_run

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _free_memory():
    yield
    import torch
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def _layout_exact(w, out):
    o, b = oracle.flatten_layout(w.numels, w.n_ranks)
    assert np.array_equal(out["offsets"], o) and np.array_equal(out["bounds"], b)


def test_tiny_mlp_all_elements():
    w = workloads.tiny_mlp()
    out = gpu_run(w)
    _layout_exact(w, out)
    stats = compare_workload(w, out, per_shard_samples=1 << 30)     # every element of every shard
    assert sum(s["n"] for (k, name), s in stats.items() if name == "master") == w.P


def test_gpt2_small_rank0_15_steps_and_unshard():
    w = workloads.gpt2_small()
    out = gpu_run(w)
    _layout_exact(w, out)
    compare_workload(w, out, per_shard_samples=200_000)


def test_llama3_8b_shard():
    w = workloads.llama3_8b_shard()
    out = gpu_run(w)
    _layout_exact(w, out)
    compare_workload(w, out, per_shard_samples=200_000)


def test_llama70b_layer_all_shards_fp16_roundtrip():
    w = workloads.llama70b_layer()
    out = gpu_run(w)
    _layout_exact(w, out)
    compare_workload(w, out, per_shard_samples=4096)


@pytest.mark.parametrize("N", workloads.SWEEP_RANKS)
@pytest.mark.parametrize("n", workloads.SWEEP_SIZES)
def test_size_sweep(n, N):
    w = workloads.sweep(n, N)
    out = gpu_run(w)
    compare_workload(w, out, per_shard_samples=1 << 20 if n < (1 << 21) else 100_000)
