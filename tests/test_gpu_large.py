"""Shards beyond 2^31 elements: every index in the kernels is 64-bit.

n = 2^31 + 7 elements, N = 2 bf16 ranks (about 39 GB on the device): one fused step, checked on
sampled elements (both ends, runs around 2^31 and random points) against the oracle; then the
16-bit parameters unsharded with a 2^31 + 7-element shard and a small one, checked the same way;
and the same step with both ranks' gradient views one element off the state's 16-byte phase (the
warp-cooperative shifted-load kernel, whose run and group indices then pass 2^31 too); and one
rank's gradient accumulated into an fp32 output of 2^31 + 7 elements, aligned and one element off.
"""
import numpy as np
import pytest

import oracle
import synth

from parity import assert_p16_within_ulp, assert_state_close, sample_indices

pytestmark = pytest.mark.gpu

N_LARGE = (1 << 31) + 7


@pytest.fixture(scope="module")
def ss():
    import fsdp_sharded_mixed_ss_gb300 as m
    return m


def test_step_and_unshard_beyond_2_31(ss):
    import torch
    n, N = N_LARGE, 2
    hp = dict(lr=3e-4, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.1, step=1000)
    gspec = [synth.normal(1e-3, synth.BF16, synth.GRAD, r, 3) for r in range(N)]
    sspec = [synth.normal(0.02, synth.FP32, synth.MASTER), synth.normal(1e-4, synth.FP32, synth.MOM1),
             synth.normal(1e-8, synth.FP32, synth.MOM2, absolute=True)]
    G = []
    for sp in gspec:
        t = torch.empty(n, dtype=torch.bfloat16, device="cuda")
        synth.device_fill(sp, t.view(torch.int16))
        G.append(t)
    st = []
    for sp in sspec:
        t = torch.empty(n, dtype=torch.float32, device="cuda")
        synth.device_fill(sp, t.view(torch.int32))
        st.append(t)
    p16 = torch.empty(n, dtype=torch.bfloat16, device="cuda")
    ss.ss_adam_step(hp, n, *st, rank_grads=G, param16=p16)

    idx = np.unique(np.concatenate([sample_indices(0, n, 200_000, 5),
                                    np.arange((1 << 31) - 40, (1 << 31) + 7)]))
    g = oracle.grad_reduce([synth.host_gather(sp, idx) for sp in gspec], synth.BF16)
    om, omm, ov = (synth.host_gather(sp, idx).view(np.float32).copy() for sp in sspec)
    rp = oracle.adamw(hp["lr"], hp["beta1"], hp["beta2"], hp["eps"], hp["weight_decay"], hp["step"], g, om, omm, ov,
                      p16_dtype=synth.BF16)
    it = torch.from_numpy(idx.astype(np.int64)).cuda()
    assert_state_close(st[0][it].cpu().numpy(), om, "master")
    assert_state_close(st[1][it].cpu().numpy(), omm, "m")
    assert_state_close(st[2][it].cpu().numpy(), ov, "v")
    got16 = p16.view(torch.int16)[it].cpu().numpy().view(np.uint16)
    assert_p16_within_ulp(got16, rp, synth.BF16, "p16")
    del G, st
    torch.cuda.empty_cache()

    # unshard: the large shard first, then 1,000 elements; the flat buffer holds both
    small = torch.arange(1000, device="cuda", dtype=torch.float32).to(torch.bfloat16)
    bounds = np.array([0, n, n + 1000], dtype=np.int64)
    flat = torch.empty(n + 1000, dtype=torch.bfloat16, device="cuda")
    ss.ss_unshard([p16, small], bounds, flat)
    fi = torch.from_numpy(np.concatenate([idx, n + np.arange(1000)]).astype(np.int64)).cuda()
    want = torch.cat([p16[it], small])
    assert torch.equal(flat[fi].view(torch.int16), want.view(torch.int16))


def test_shifted_step_beyond_2_31_elements(ss):
    import torch
    n, N = (1 << 31) + 7, 2
    hp = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01, step=1)
    specs = [synth.normal(1e-3, synth.BF16, synth.GRAD, r, 1) for r in range(N)]
    G = []
    for s in specs:
        base = torch.empty(n + 8, dtype=torch.bfloat16, device="cuda")
        v = base[1:n + 1]
        synth.device_fill(s, v.view(torch.int16))
        G.append(v)
    mspec = synth.normal(0.02, synth.FP32, synth.MASTER)
    master = torch.empty(n, dtype=torch.float32, device="cuda")
    synth.device_fill(mspec, master.view(torch.int32))
    m = torch.zeros(n, dtype=torch.float32, device="cuda")
    v = torch.zeros(n, dtype=torch.float32, device="cuda")
    p16 = torch.empty(n, dtype=torch.bfloat16, device="cuda")
    ss.ss_adam_step(hp, n, master, m, v, rank_grads=G, param16=p16)
    torch.cuda.synchronize()
    idx = np.unique(np.concatenate([sample_indices(0, n, 200_000, 6),
                                    np.arange((1 << 31) - 40, (1 << 31) + 7)]))
    g = oracle.grad_reduce([synth.host_gather(s, idx) for s in specs], oracle.BF16)
    om = synth.host_gather(mspec, idx).view(np.float32).copy()
    omm, ov = np.zeros(idx.size, np.float32), np.zeros(idx.size, np.float32)
    rp = oracle.adamw(hp["lr"], hp["beta1"], hp["beta2"], hp["eps"], hp["weight_decay"], 1, g, om, omm, ov,
                      p16_dtype=oracle.BF16)
    it = torch.from_numpy(idx.astype(np.int64)).cuda()
    for name, t, r in (("master", master, om), ("m", m, omm), ("v", v, ov)):
        assert_state_close(t[it].cpu().numpy(), r, name)
    assert_p16_within_ulp(p16.view(torch.int16)[it].cpu().numpy().view(np.uint16), rp, oracle.BF16, "p16")
    del G, master, m, v, p16
    torch.cuda.empty_cache()


@pytest.mark.parametrize("off", [0, 1])
def test_one_rank_reduce_beyond_2_31_elements(ss, off):
    """One rank's gradient accumulated into the fp32 output, n = 2^31 + 7: aligned (the 4-element
    lane map) or the view one element off the output's phase (several runs a warp at a time, the
    sums stored through shared memory); bit-exact against the oracle on sampled elements."""
    import torch
    n = N_LARGE
    spec = synth.normal(1e-3, synth.BF16, synth.GRAD, 0, 7)
    base = torch.empty(n + 8, dtype=torch.bfloat16, device="cuda")
    g = base[off:off + n]
    synth.device_fill(spec, g.view(torch.int16))
    ospec = synth.normal(1e-2, synth.FP32, synth.MOM1)
    out = torch.empty(n, dtype=torch.float32, device="cuda")
    synth.device_fill(ospec, out.view(torch.int32))
    ss.ss_grad_reduce([g], n, out, post_scale=0.5, accumulate=True)
    torch.cuda.synchronize()
    idx = np.unique(np.concatenate([sample_indices(0, n, 200_000, 8),
                                    np.arange((1 << 31) - 40, (1 << 31) + 7)]))
    acc = synth.host_gather(ospec, idx).view(np.float32).copy()
    oracle.grad_reduce([synth.host_gather(spec, idx)], oracle.BF16, post_scale=0.5, accumulate_into=acc)
    it = torch.from_numpy(idx.astype(np.int64)).cuda()
    assert np.array_equal(out[it].cpu().numpy().view(np.uint32), acc.view(np.uint32))
    del base, out
    torch.cuda.empty_cache()
