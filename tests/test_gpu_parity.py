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


def test_llama70b_layer_shards_with_offset_views():
    """The config-4 extra: rank gradient views one element off the state's 16-byte phase
    (the shifted-load kernel) on two full-size shards of the 70B layer, fp16."""
    import torch

    import fsdp_sharded_mixed_ss_gb300 as ss
    import synth
    from parity import assert_p16_within_ulp, assert_state_close, gather_np, oracle_shard, sample_indices

    w = workloads.llama70b_layer()
    _, bounds = ss.ss_flatten_layout(w.numels, w.n_ranks)
    for k in (0, 37):
        lo, hi = int(bounds[k]), int(bounds[k + 1])
        n = hi - lo
        G = []
        for r in range(w.n_ranks):
            base = torch.empty(n + 1, dtype=torch.float16, device="cuda")
            synth.device_fill(w.grad(r, 1), base[1:].view(torch.int16), start=lo)
            G.append(base[1:])
        master = torch.empty(n, dtype=torch.float32, device="cuda")
        synth.device_fill(w.master, master.view(torch.int32), start=lo)
        m = torch.zeros(n, device="cuda")
        v = torch.zeros(n, device="cuda")
        p16 = torch.empty(n, dtype=torch.float16, device="cuda")
        ss.ss_adam_step(w.hp(1), n, master, m, v, rank_grads=G, param16=p16)
        idx = sample_indices(lo, hi, 50_000, k)
        ref = oracle_shard(w, idx, range(1, 2))
        loc = idx - lo
        for name, t in (("master", master), ("m", m), ("v", v)):
            assert_state_close(gather_np(t, loc), ref[name], f"shard {k} {name}")
        assert_p16_within_ulp(gather_np(p16.view(torch.int16), loc).view(np.uint16), ref["p16"], synth.FP16, "p16")
        del G
        torch.cuda.empty_cache()


def test_llama3_shard_reduce_bit_exact_sampled():
    """ss_grad_reduce on the Llama-3-8B rank-0 shard (1,003,782,656 elements, 8 ranks) at full
    size: bit-exact against the oracle at sampled elements, with 1% outliers in the gradients."""
    import torch

    import fsdp_sharded_mixed_ss_gb300 as ss
    import synth
    from parity import gather_np, sample_indices

    w = workloads.llama3_8b_shard()
    _, bounds = ss.ss_flatten_layout(w.numels, w.n_ranks)
    n = int(bounds[1])
    G = []
    for r in range(w.n_ranks):
        t = torch.empty(n, dtype=torch.bfloat16, device="cuda")
        synth.device_fill(w.grad(r, 1), t.view(torch.int16))
        G.append(t)
    out = torch.empty(n, dtype=torch.float32, device="cuda")
    ss.ss_grad_reduce(G, n, out)
    idx = sample_indices(0, n, 200_000, 3)
    ref = oracle.grad_reduce([synth.host_gather(w.grad(r, 1), idx) for r in range(w.n_ranks)], oracle.BF16)
    assert np.array_equal(gather_np(out, idx).view(np.uint32), ref.view(np.uint32))
