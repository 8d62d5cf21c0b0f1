"""The sum-of-squares entry point that allocates nothing (collected last on purpose).

Some callers cannot allocate device memory -- plugin code inside a framework
that has already reserved the GPU's memory for its own pool, or a loop where
cudaMalloc's implicit synchronisation is not acceptable -- so they cannot hand
ss_grad_sumsq a workspace. ss_grad_sumsq_noalloc keeps that scratch in a fixed
array inside the library. These tests call it through the C ABI twice in a row
and check it two ways: against ss_grad_sumsq with a caller workspace, which runs
the same kernels in the same order, so the sums must be bit-identical; and
against the oracle's double-precision sum of squares of the oracle's own
rank-ordered gradient sum (regenerated on the host from the same seeded
streams), within the 5e-7 relative bound the header states, with the reduced
gradient written to g_out bit-exact at sampled elements.
"""
import numpy as np
import pytest

import oracle
import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ss():
    import fsdp_sharded_mixed_ss_gb300 as m
    return m


def _spec(r, step):
    return synth.normal(1e-3, synth.BF16, synth.GRAD, r, step)


def _grads(n, N, step):
    import torch
    out = []
    for r in range(N):
        t = torch.empty(n, dtype=torch.bfloat16, device="cuda")
        synth.device_fill(_spec(r, step), t.view(torch.int16))
        out.append(t)
    return out


@pytest.mark.parametrize("n,N", [(1_000_003, 8), (37, 2), (20_000_000, 4)])
def test_noalloc_matches_workspace_version_and_oracle_twice(ss, n, N):
    import torch
    ws = torch.empty(ss.ss_grad_sumsq_workspace(n) // 8, dtype=torch.float64, device="cuda")
    for step in (1, 2):                      # two calls in a row, different inputs
        G = _grads(n, N, step)
        a = torch.zeros(1, dtype=torch.float64, device="cuda")
        b = torch.zeros(1, dtype=torch.float64, device="cuda")
        ga = torch.empty(n, dtype=torch.float32, device="cuda")
        gb = torch.empty(n, dtype=torch.float32, device="cuda")
        fa = torch.zeros(1, dtype=torch.int32, device="cuda")
        fb = torch.zeros(1, dtype=torch.int32, device="cuda")
        ss.ss_grad_sumsq_noalloc(n, a, rank_grads=G, post_scale=0.5, g_out=ga, nonfinite_flag=fa)
        ss.ss_grad_sumsq(n, b, ws, rank_grads=G, post_scale=0.5, g_out=gb, nonfinite_flag=fb)
        torch.cuda.synchronize()
        x, y = a.item(), b.item()
        assert x == y                        # same kernels, same order: the same bits
        assert torch.equal(ga, gb)
        assert fa.item() == fb.item() == 0
        # the oracle: rank-ordered fp32 sum of the host-regenerated gradients, then a double sum of squares
        g = oracle.grad_reduce([synth.host_range(_spec(r, step), 0, n) for r in range(N)], oracle.BF16,
                               post_scale=0.5)
        ref = oracle.sumsq(g)
        assert ref > 0 and abs(x - ref) <= 5e-7 * ref
        idx = np.unique(np.concatenate([np.arange(min(n, 64)), np.arange(max(n - 64, 0), n),
                                        np.random.default_rng(step).integers(0, n, size=min(n, 100_000))]))
        got = ga.index_select(0, torch.from_numpy(idx).cuda()).cpu().numpy()
        assert np.array_equal(got.view(np.uint32), g[idx].view(np.uint32))


def test_noalloc_from_fp32_and_size_limit(ss):
    import torch
    n = 123_457
    spec = synth.normal(1e-2, synth.FP32, synth.GRAD, 0, 3)
    g = torch.empty(n, dtype=torch.float32, device="cuda")
    synth.device_fill(spec, g.view(torch.int32))
    out = torch.zeros(2, dtype=torch.float64, device="cuda")
    ws = torch.empty(ss.ss_grad_sumsq_workspace(n) // 8, dtype=torch.float64, device="cuda")
    ss.ss_grad_sumsq_noalloc(n, out[0:1], g32=g)
    ss.ss_grad_sumsq(n, out[1:2], ws, g32=g)
    o = out.cpu().numpy()
    assert o[0] == o[1]
    ref = oracle.sumsq(synth.host_range(spec, 0, n).view(np.float32))
    assert abs(o[0] - ref) <= 5e-7 * ref
    with pytest.raises(ss.SSError) as e:
        ss.ss_grad_sumsq_noalloc(ss.SS_NOALLOC_SUMSQ_MAX_N + 1, out[0:1], g32=g)
    assert e.value.status == 5
